"""bench.py host logic that needs no GPU: the staleness check of the stored
DRAM counters, the closed-form check of the timed output, the per-phase work
counts and the clock summary."""
import json
import os
import random
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402
import oracle  # noqa: E402
from oracle import pyref  # noqa: E402
from elliptic_curve_scalar_gb300 import synth  # noqa: E402

CSRC = os.path.join(ROOT, "elliptic_curve_scalar_gb300", "csrc")


def _local_includes(name, seen):
    if name in seen or "/" in name:  # the public header (include/) holds no device code
        return
    seen.add(name)
    with open(os.path.join(CSRC, name)) as f:
        for inc in re.findall(r'^\s*#include\s+"([^"]+)"', f.read(), re.M):
            _local_includes(inc, seen)


def test_digest_covers_every_kernel_source():
    seen = set()
    _local_includes("msm_g1.cu", seen)
    _local_includes("msm_accum.cu", seen)
    assert seen == set(bench.KERNEL_SOURCES)


def test_digest_follows_every_source():
    base = {name: b"x" for name in bench.KERNEL_SOURCES}
    d0 = bench.kernel_sources_digest(lambda name: base[name])
    assert d0 == bench.kernel_sources_digest(lambda name: base[name])
    for name in bench.KERNEL_SOURCES:
        changed = dict(base, **{name: b"y"})
        assert bench.kernel_sources_digest(lambda nm: changed[nm]) != d0


def test_digest_ignores_comments_but_not_code():
    src = b'int f(int x) { // doubles x\n  return 2 * x; /* block\n comment */ }\nconst char* s = "a // b";\n'
    base = {name: src for name in bench.KERNEL_SOURCES}
    d0 = bench.kernel_sources_digest(lambda name: base[name])
    recommented = src.replace(b"doubles x", b"twice x").replace(b"block", b"a longer block")
    respaced = src.replace(b"return 2 * x;", b"return   2 *  x;")
    for other in (recommented, respaced):
        assert bench.kernel_sources_digest(lambda nm: dict(base, **{"fq.cuh": other})[nm]) == d0
    for other in (src.replace(b"2 * x", b"3 * x"), src.replace(b'"a // b"', b'"a / b"')):
        assert bench.kernel_sources_digest(lambda nm: dict(base, **{"fq.cuh": other})[nm]) != d0
    assert bench.code_only(b'x = 1; // y\n"//z" /* w */ q') == b'x = 1; "//z" q'


def test_traffic_only_for_the_build_it_was_taken_on(tmp_path):
    prof = tmp_path / "traffic.json"
    prof.write_text(json.dumps({"bytes_per_msm": {"n2p16": {"accum_tree": 123}},
                                "sources_sha256": bench.kernel_sources_digest()}))
    assert bench.phase_traffic("n2p16", "accum_tree", str(prof)) == (123, None)
    assert bench.phase_traffic("n2p16", "combine", str(prof)) == (None, None)
    assert bench.phase_traffic("n2p20", "accum_tree", str(prof)) == (None, None)
    prof.write_text(json.dumps({"bytes_per_msm": {"n2p16": {"accum_tree": 123}}, "sources_sha256": "0" * 64}))
    assert bench.phase_traffic("n2p16", "accum_tree", str(prof)) == (None, 123)
    assert bench.phase_traffic("n2p16", "accum_tree", str(tmp_path / "missing.json")) == (None, None)


def test_dot_mod_r_is_exact():
    r, k = synth.uniform_workload(3000, 99)
    expect = sum(a * b for a, b in zip(synth.limbs_to_ints(k), synth.limbs_to_ints(r))) % pyref.R
    assert bench.dot_mod_r(k, r) == expect
    assert bench.dot_mod_r(k, r, chunk=7) == expect  # chunk boundaries change nothing
    top = np.full((5, 4), np.uint64(0xFFFFFFFFFFFFFFFF))
    assert bench.dot_mod_r(top, top) == 5 * ((1 << 256) - 1) ** 2 % pyref.R


def test_generator_multiple_matches_the_python_oracle():
    rng = random.Random(5)
    for s in [0, 1, 2, 3, pyref.R - 1, pyref.R] + [rng.randrange(pyref.R) for _ in range(4)]:
        assert bench.generator_multiple(s) == pyref.mul(s % pyref.R, pyref.G)


def _jac_words(pt, z):
    if pt is None:
        xyz = [1, 1, 0]
    else:
        xyz = [pt[0] * z * z % pyref.P, pt[1] * z * z * z % pyref.P, z]
    mont = [v * (1 << 256) % pyref.P for v in xyz]
    return np.array([(v >> (32 * i)) & 0xFFFFFFFF for v in mont for i in range(8)], dtype=np.uint32)


def test_jacobian_words_to_affine():
    p = pyref.mul(123456789, pyref.G)
    assert bench.jacobian_words_to_affine(_jac_words(p, 1)) == p
    assert bench.jacobian_words_to_affine(_jac_words(p, 987654321987)) == p
    assert bench.jacobian_words_to_affine(_jac_words(None, 0)) is None


def test_closed_form_check_accepts_the_msm_and_rejects_another_point():
    n, K = 24, 2
    r, k = synth.uniform_workload(K * n, 31)
    pts = oracle.generator_multiples(r, threads=2)
    outs = []
    for m in range(K):
        q = oracle.words_to_point(oracle.msm(pts[m * n:(m + 1) * n], k[m * n:(m + 1) * n], threads=2))
        outs.append(_jac_words(q, 5 + m))
    good = np.concatenate(outs)
    assert bench.closed_form_ok(good, r, k, K, n)
    bad = good.copy()
    bad[24:] = _jac_words(pyref.add(oracle.words_to_point(oracle.msm(pts[n:], k[n:], threads=2)), pyref.G), 3)
    assert not bench.closed_form_ok(bad, r, k, K, n)


def _work_by_loops(counts, adds, c, glv, K, T, L):
    """phase_work's bucket-reduction and combination counts, restated as the
    kernels' loops, one bucket and one chunk at a time."""
    nbits = 128 if glv else 255
    W = -(-nbits // c)
    B = 1 << (c - 1)
    madd = jadd = jdbl = 0
    jac = {}
    for g in range(K * W * B):
        h = (int(counts[g]) + 1) // 2
        stride, items = 1, h
        while items > T:
            stride *= 2
            items = -(-h // stride)
        jac[g] = T >= 2 and items >= 2
        if jac[g]:
            madd += items - 1
    G = B // L
    for w in range(K * W):
        for j in range(G):
            run_inf = sum_inf = True
            for b in reversed(range(j * L, (j + 1) * L)):
                g = w * B + b
                if counts[g]:
                    if not run_inf:
                        if jac[g]:
                            jadd += 1
                        else:
                            madd += 1
                    run_inf = False
                if not run_inf:
                    if not sum_inf:
                        jadd += 1
                    sum_inf = False
        lg = G.bit_length() - 1
        jadd += (G - 1) + lg * (G // 2 - 1) + lg
        jdbl += sum(t - 1 + L.bit_length() - 1 for t in range(1, lg + 1))
    return {"madd": madd, "add": jadd, "dbl": jdbl}


def test_phase_work_counts_the_kernels_loops():
    rng = np.random.default_rng(3)
    for c, glv, K, T, L in ((4, 1, 1, 8, 4), (5, 0, 2, 1, 4), (6, 1, 1, 16, 8), (3, 1, 3, 2, 4)):
        nbits = 128 if glv else 255
        W = -(-nbits // c)
        nb = K * W * (1 << (c - 1))
        counts = rng.integers(0, 40, size=nb) * (rng.random(nb) < 0.7)
        stats = {"adds": 10 ** 6, "finish_t": T, "chunk_len": L}
        got = bench.phase_work(counts.astype(np.uint32), stats, c, glv, K)
        assert got["point_ops"]["bucket_reduce"] == _work_by_loops(counts, 0, c, glv, K, T, L)
        assert got["adds_l0"] == int((counts // 2).sum())
        assert got["point_ops"]["combine"] == {"dbl": K * (nbits - nbits // W), "add": K * (W - 1)}


def _row(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return "0, %s, %s, 612.40, 0x0000000000000000, %s, %s, %s, %s\n" % (sm, mx, hw, hwt, swt, cap)


def test_clock_summary_of_a_clean_run():
    c = bench.summarize_clocks([_row(2070, 2070), _row(2055, 2070), _row(2070, 2070)])
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}


def test_clock_summary_reports_every_active_reason():
    lines = [_row(1980, 2070, cap="Active"), _row(1500, 2070, hwt="Active"), _row(2070, 2070),
             "garbled line\n", _row("[N/A]", 2070)]
    c = bench.summarize_clocks(lines)
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert c["samples"] == 4 and c["sm_mhz"] == 1980.0 and c["sm_max_mhz"] == 2070.0


def test_clock_summary_without_samples():
    assert bench.summarize_clocks([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_clock_sampler_without_nvidia_smi_reports_no_samples(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", "")
    s = bench.ClockSampler(tmpdir=str(tmp_path))
    c = s.stop()
    assert c["samples"] == 0 and c["reasons"] == []
    assert not list(tmp_path.iterdir())  # the sample file is removed
