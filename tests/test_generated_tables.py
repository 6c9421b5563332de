"""The kernels' generated constant tables are what their generators write:
a hand edit of a generated header, or a generator changed without
regenerating, fails here (no GPU needed)."""
import importlib.util
import pathlib

CSRC = pathlib.Path(__file__).resolve().parent.parent / "elliptic_curve_scalar_gb300" / "csrc"


def _load(name):
    spec = importlib.util.spec_from_file_location(name, CSRC / (name + ".py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_divstep_table_is_regenerated():
    gen = _load("gen_divsteps")
    tab = gen.table()
    assert len(tab) == 1152
    assert (CSRC / "divstep_table.cuh").read_text() == gen.render(tab)


def test_divstep_table_entries_match_four_exact_divsteps():
    gen = _load("gen_divsteps")
    gen.check(gen.table(), trials=20000, seed=11)


def test_divstep_table_clamped_delta_classes():
    """delta <= -4: no swap within four steps, so f is unchanged and
    delta' = delta + 4.  delta >= 4: g = 0 mod 16 takes four halvings
    (delta' = delta + 4); an odd g swaps at once (delta' = 4 - delta)."""
    gen = _load("gen_divsteps")
    tab = gen.table()
    idx = lambda ds, fh, gl: ((ds + 4) * 8 + fh) * 16 + gl
    for fh in range(8):
        for gl in range(16):
            u, v, q, r, s, t = tab[idx(-4, fh, gl)]
            assert (u, v, s, t) == (16, 0, 1, 4)
        u, v, q, r, s, t = tab[idx(4, fh, 0)]
        assert (u, v, q, r, s, t) == (16, 0, 0, 1, 1, 4)
        for gl in range(1, 16, 2):
            s, t = tab[idx(4, fh, gl)][4:]
            assert (s, t) == (-1, 4)


def test_rns_constants_are_regenerated():
    gen = _load("gen_rns")
    assert (CSRC / "rns_consts.cuh").read_text() == gen.render()
