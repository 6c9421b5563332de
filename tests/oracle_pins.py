"""Pins for the CPU oracle: facts fixed by mathematics, not by the oracle itself.

Each ``pin_*`` function raises AssertionError when the active oracle build gets
a fact wrong.  ``tests/test_oracle.py`` runs them against the real oracle;
``tests/test_oracle_mutations.py`` runs them against builds with one planted
mistake each and requires that some pin fails, which shows the pins would
catch that class of bug.

The facts:
* field products and inverses against Python integers (exact, any size);
* Montgomery encoding x -> x * 2^256 mod p against Python integers;
* group sanity: G = (1, 2) on y^2 = x^3 + 3, [r]G = infinity, [r-1]G = -G;
* the curve-membership test rejects what y^2 = x^3 + 3 over F_p excludes: a
  point with x or y moved by one, (1, 3), and coordinates that are not
  canonical residues (x + p or y + p in place of x or y);
* brute force: tiny MSMs against repeated addition with the affine law;
* all-ones scalars give the plain point sum;
* closed form: for P_i = [r_i]G the MSM is [sum k_i r_i mod r]G, with the
  scalar computed in Python integers and the point by the affine law;
* linearity: MSM(k + k') = MSM(k) + MSM(k');
* n = 1 special cases k in {0, 1, 2, r - 1, r, 2^256 - 1};
* exceptional inputs (equal and opposite points) against the affine law;
* agreement with the independent pure-Python oracle on random inputs.
"""
import random

import numpy as np

import oracle
from oracle import pyref
from elliptic_curve_scalar_gb300 import synth

P, R = pyref.P, pyref.R


def _pt(w):
    return oracle.words_to_point(w)


def _words(pts):
    return np.stack([oracle.point_to_words(p) for p in pts])


def _rand_points(rng, n):
    rs = [rng.randrange(1, R) for _ in range(n)]
    return rs, [pyref.mul(r, pyref.G) for r in rs]


def pin_field():
    rng = random.Random(11)
    edges = [0, 1, 2, P - 1, P - 2, P // 2, (1 << 255), (1 << 256) - 1, P, P + 1]
    vals = edges + [rng.randrange(0, 1 << 256) for _ in range(300)]
    for i, a in enumerate(vals):
        b = vals[(i * 7 + 3) % len(vals)]
        got = oracle.limbs_to_int(oracle.fp_mul(oracle.int_to_limbs(a), oracle.int_to_limbs(b)))
        assert got == (a % P) * (b % P) % P, ("fp_mul", a, b)
    # products whose Barrett quotient estimate is furthest off: both operands near p
    for d1 in range(1, 40):
        for d2 in range(1, 40, 7):
            a, b = P - d1, P - d2 * 977
            got = oracle.limbs_to_int(oracle.fp_mul(oracle.int_to_limbs(a), oracle.int_to_limbs(b)))
            assert got == a * b % P, ("fp_mul near p", d1, d2)
    # about one product in a thousand needs Barrett's final correction: cover many
    for _ in range(20000):
        a, b = rng.randrange(0, P), rng.randrange(0, P)
        got = oracle.limbs_to_int(oracle.fp_mul(oracle.int_to_limbs(a), oracle.int_to_limbs(b)))
        assert got == a * b % P, ("fp_mul", a, b)
    for a in [1, 2, P - 1] + [rng.randrange(1, P) for _ in range(20)]:
        inv = oracle.limbs_to_int(oracle.fp_inv(oracle.int_to_limbs(a)))
        assert inv * a % P == 1, ("fp_inv", a)


def pin_montgomery():
    rng = random.Random(12)
    xs = [0, 1, P - 1] + [rng.randrange(0, P) for _ in range(50)]
    enc = oracle.mont_encode(oracle.ints_to_limbs(xs))
    dec = oracle.mont_decode(enc)
    for x, e, d in zip(xs, enc, dec):
        assert oracle.limbs_to_int(e) == x * (1 << 256) % P, ("encode", x)
        assert oracle.limbs_to_int(d) == x, ("decode", x)


def pin_group():
    g = oracle.point_to_words(pyref.G)
    assert pyref.on_curve(pyref.G)
    assert oracle.is_on_curve(g)
    assert _pt(oracle.scalar_mul(g, oracle.int_to_limbs(R))) is None, "[r]G != inf"
    assert _pt(oracle.scalar_mul(g, oracle.int_to_limbs(R - 1))) == pyref.neg(pyref.G), "[r-1]G != -G"
    assert _pt(oracle.scalar_mul(g, oracle.int_to_limbs(2))) == pyref.add(pyref.G, pyref.G), "[2]G"
    big = (1 << 256) - 1
    assert _pt(oracle.scalar_mul(g, oracle.int_to_limbs(big))) == pyref.mul(big % R, pyref.G), "[2^256-1]G"


def pin_on_curve_rejects():
    """Points off y^2 = x^3 + 3, or with a coordinate outside [0, p), are not
    on the curve; both oracles must say so (the points they accept are
    covered by pin_group and the pins that check their outputs)."""
    rng = random.Random(18)
    _, pts = _rand_points(rng, 3)
    bad = [(1, 3), (2, 3), (0, 1)]
    for x, y in pts:
        bad += [(x, (y + 1) % P), ((x + 1) % P, y), (x + P, y), (x, y + P)]
        # (x + 1, y) is on the curve only if 3x^2 + 3x + 1 = 0 mod p: never for these seeds
        assert (y * y - (x + 1) ** 3 - 3) % P != 0
    for x, y in bad:
        assert not pyref.on_curve((x, y)), ("pyref.on_curve accepts", x, y)
        w = np.concatenate([oracle.int_to_limbs(x), oracle.int_to_limbs(y)])
        assert not oracle.is_on_curve(w), ("is_on_curve accepts", x, y)
    for p in pts:
        assert pyref.on_curve(p) and oracle.is_on_curve(oracle.point_to_words(p))


def pin_generator_multiples():
    rng = random.Random(13)
    ks = [0, 1, 2, 255, 256, 0xFF << 248, (1 << 256) - 1, R - 1, R, R + 5]
    ks += [rng.randrange(0, 1 << 256) for _ in range(6)]
    got = oracle.generator_multiples(oracle.ints_to_limbs(ks), threads=2)
    for k, w in zip(ks, got):
        assert _pt(w) == pyref.mul(k % R, pyref.G), ("[k]G", k)
        assert oracle.is_on_curve(w)


def pin_brute_force():
    rng = random.Random(14)
    for n in (1, 2, 3, 5, 8):
        _, pts = _rand_points(rng, n)
        ks = [rng.randrange(0, 16) for _ in range(n)]
        expect = None
        for p, k in zip(pts, ks):
            expect = pyref.add(expect, pyref.mul_repeated(k, p))
        got = oracle.msm(_words(pts), oracle.ints_to_limbs(ks), threads=3)
        assert _pt(got) == expect, ("brute force", n)


def pin_all_ones():
    rng = random.Random(15)
    _, pts = _rand_points(rng, 9)
    expect = None
    for p in pts:
        expect = pyref.add(expect, p)
    got = oracle.msm(_words(pts), oracle.ints_to_limbs([1] * 9), threads=4)
    assert _pt(got) == expect, "all-ones sum"


def pin_closed_form():
    r_vals, k = synth.uniform_workload(48, 1234)
    pts = oracle.generator_multiples(r_vals, threads=4)
    got = oracle.msm(pts, k, threads=4)
    s = sum(a * b for a, b in zip(synth.limbs_to_ints(r_vals), synth.limbs_to_ints(k))) % R
    assert _pt(got) == pyref.mul(s, pyref.G), "closed form"
    assert oracle.is_on_curve(got)


def pin_linearity():
    r_vals, k1 = synth.uniform_workload(20, 77)
    _, k2 = synth.uniform_workload(20, 78)
    pts = oracle.generator_multiples(r_vals, threads=2)
    ks = [(a + b) % R for a, b in zip(synth.limbs_to_ints(k1), synth.limbs_to_ints(k2))]
    lhs = _pt(oracle.msm(pts, oracle.ints_to_limbs(ks), threads=2))
    rhs = pyref.add(_pt(oracle.msm(pts, k1, threads=2)), _pt(oracle.msm(pts, k2, threads=2)))
    assert lhs == rhs, "linearity"


def pin_single_term():
    p = pyref.mul(987654321, pyref.G)
    w = oracle.point_to_words(p)[None]
    cases = {0: None, 1: p, 2: pyref.add(p, p), R - 1: pyref.neg(p), R: None,
             (1 << 256) - 1: pyref.mul(((1 << 256) - 1) % R, p)}
    for k, expect in cases.items():
        got = oracle.msm(w, oracle.int_to_limbs(k)[None], threads=1)
        assert _pt(got) == expect, ("n=1", k)
    zero = oracle.msm(np.repeat(w, 5, axis=0), np.zeros((5, 4), dtype=np.uint64), threads=2)
    assert _pt(zero) is None, "all-zero scalars"


def pin_exceptional():
    rng = random.Random(16)
    _, (a, b) = _rand_points(rng, 2)
    cases = [
        ([a, a], [1, 1], pyref.add(a, a)),                 # doubling inside the sum
        ([a, pyref.neg(a)], [1, 1], None),                 # P + (-P)
        ([a, pyref.neg(a), b], [3, 3, 1], b),
        ([None, a], [5, 1], a),                            # infinity input
        ([a, a, a, a], [1, 1, 1, 1], pyref.mul(4, a)),
    ]
    for pts, ks, expect in cases:
        got = oracle.msm(_words(pts), oracle.ints_to_limbs(ks), threads=1)
        assert _pt(got) == expect, ("exceptional", ks)
    got = _pt(oracle.add(oracle.point_to_words(a), oracle.point_to_words(a)))
    assert got == pyref.add(a, a), "add(P, P)"


def pin_jacobian_normalisation():
    rng = random.Random(17)
    _, (a,) = _rand_points(rng, 1)
    z = rng.randrange(2, P)
    X, Y, Z = a[0] * z * z % P, a[1] * z * z * z % P, z
    jm = oracle.mont_encode(oracle.ints_to_limbs([X, Y, Z])).reshape(12)
    assert _pt(oracle.jacobian_mont_to_affine(jm)) == a
    jm_inf = oracle.mont_encode(oracle.ints_to_limbs([5, 7, 0])).reshape(12)
    assert _pt(oracle.jacobian_mont_to_affine(jm_inf)) is None


def pin_two_oracles():
    r_vals, k = synth.uniform_workload(16, 4242)
    pts = oracle.generator_multiples(r_vals, threads=2)
    got = oracle.msm(pts, k, threads=2)
    expect = pyref.msm([_pt(w) for w in pts], synth.limbs_to_ints(k))
    assert _pt(got) == expect, "C oracle vs Python oracle"


ALL_PINS = [
    pin_field,
    pin_montgomery,
    pin_group,
    pin_on_curve_rejects,
    pin_generator_multiples,
    pin_brute_force,
    pin_all_ones,
    pin_closed_form,
    pin_linearity,
    pin_single_term,
    pin_exceptional,
    pin_jacobian_normalisation,
    pin_two_oracles,
]


def failing_pins():
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError as e:  # a pin rejected the build
            failed.append((pin.__name__, str(e)))
    return failed
