"""MSM parity: the CUDA path against the CPU oracle, bit-exact after both are
normalised to canonical affine coordinates (the MSM has exactly one correct
affine result, so bucket, sort and tie order cannot change it).

Small and medium sizes are compared with oracle.msm directly; the full-size
workloads (n = 2^20, 2^22) are compared with the closed form
[sum_i k_i r_i mod r]G, which holds for any n because P_i = [r_i]G.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import pyref
from elliptic_curve_scalar_gb300 import msm as gm
from elliptic_curve_scalar_gb300 import synth
from tests.gpu_helpers import gpu_points, gpu_scalars, normalise, points_from_r, ints_to_u32

pytestmark = pytest.mark.gpu

_ctx = {}


def ctx(max_n, max_c):
    key = (max_n, max_c)
    if key not in _ctx:
        _ctx[key] = gm.MsmG1(max_n, max_c)
    return _ctx[key]


def run_gpu(points_affine, k, c, max_n=None, max_c=None, batch_s=0, tpb=128, glv=1, place=0, grid=0):
    n = k.shape[0]
    cx = ctx(max_n or max(n, 1), max_c or max(c, 1))
    cx.set_param(gm.PARAM_BATCH_S, batch_s)
    cx.set_param(gm.PARAM_TPB, tpb)
    cx.set_param(gm.PARAM_GLV, glv)
    cx.set_param(gm.PARAM_ACC_PLACEMENT, place)
    cx.set_param(gm.PARAM_GRID, grid)
    try:
        out = cx.run(gpu_points(points_affine), gpu_scalars(k), c)
        res = normalise(out)
        assert cx.stats()["error"] == 0
    finally:
        cx.set_param(gm.PARAM_ACC_PLACEMENT, 0)
        cx.set_param(gm.PARAM_GRID, 0)
    return res


def expect_oracle(points_affine, k):
    return oracle.msm(points_affine, k)


@pytest.mark.parametrize("glv", [1, 0])
def test_config1_n1024_c8(glv):
    """n = 2^10, c = 8, uniform points [r_i]G and scalars (seed 1001)."""
    r, k = synth.uniform_workload(1 << 10, 1001)
    pts = points_from_r(r)
    got = run_gpu(pts, k, 8, glv=glv)
    assert np.array_equal(got, expect_oracle(pts, k))
    assert np.array_equal(got, oracle.closed_form(r, k))
    assert oracle.is_on_curve(got)


@pytest.mark.parametrize("glv", [1, 0])
@pytest.mark.parametrize("n,c", [(1, 4), (2, 3), (3, 8), (7, 5), (31, 6), (33, 7), (100, 9),
                                 (257, 10), (1000, 11), (4097, 12)])
def test_small_sizes(n, c, glv):
    r, k = synth.uniform_workload(n, 2000 + n)
    pts = points_from_r(r)
    assert np.array_equal(run_gpu(pts, k, c, glv=glv), expect_oracle(pts, k))


@pytest.mark.parametrize("glv", [1, 0])
@pytest.mark.parametrize("c", list(range(1, 21)))
def test_every_window_size(c, glv):
    r, k = synth.uniform_workload(1500, 3000 + c)
    pts = points_from_r(r)
    assert np.array_equal(run_gpu(pts, k, c, max_n=1500, max_c=20, glv=glv), expect_oracle(pts, k))


@pytest.fixture(scope="module")
def mid_case():
    r, k = synth.uniform_workload(20000, 4242)
    pts = points_from_r(r)
    return pts, k, expect_oracle(pts, k)


@pytest.mark.parametrize("batch_s", [0, 1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("tpb", [64, 128, 256])
def test_knobs(mid_case, batch_s, tpb):
    """Every batch size S and block size gives the same result (the pages
    verified each S separately because failures were S-specific: PR #23736,
    section "Real-hardware results")."""
    pts, k, expect = mid_case
    assert np.array_equal(run_gpu(pts, k, 13, max_n=20000, max_c=13, batch_s=batch_s, tpb=tpb), expect)


PLACEMENTS = {"local": 0, "shared": 1, "registers": 2}


@pytest.mark.parametrize("place", ["shared", "registers"])
@pytest.mark.parametrize("batch_s", [0, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("tpb", [64, 128, 256])
def test_prefix_placements(mid_case, place, batch_s, tpb):
    """Prefix products in shared memory or in registers (the pages' choice of
    where pref_scratch lives: PR #23738 "stream-walker S-sweep", section "What
    would actually win") give the result of the default placement for every
    batch size and block size; sizes a placement does not hold are clamped."""
    pts, k, expect = mid_case
    got = run_gpu(pts, k, 13, max_n=20000, max_c=13, batch_s=batch_s, tpb=tpb, place=PLACEMENTS[place])
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("place", ["local", "shared", "registers"])
@pytest.mark.parametrize("glv", [1, 0])
def test_prefix_placements_on_exceptional_pairs(place, glv):
    """Equal, opposite and infinite operands inside a batch whose prefix
    products live in each placement."""
    r, k = synth.adversarial_workload(30000, 1007)
    pts = points_from_r(r)
    got = run_gpu(pts, k, 12, max_n=30000, max_c=16, glv=glv, batch_s=8, place=PLACEMENTS[place])
    assert np.array_equal(got, expect_oracle(pts, k))


@pytest.mark.parametrize("grid", [1, 3, 17, 152, 100000])
@pytest.mark.parametrize("batch_s", [0, 1, 8])
def test_grid_cap(mid_case, grid, batch_s):
    """A cap on the accumulation grid (the pages' walkerMaxWg) splits the
    work into consecutive launches; the result does not change."""
    pts, k, expect = mid_case
    got = run_gpu(pts, k, 13, max_n=20000, max_c=13, batch_s=batch_s, grid=grid)
    assert np.array_equal(got, expect)


def test_new_parameters_reject_bad_values():
    cx = ctx(20000, 13)
    for key, bad in ((gm.PARAM_GRID, -1), (gm.PARAM_ACC_PLACEMENT, 3), (gm.PARAM_ACC_PLACEMENT, -1)):
        with pytest.raises(gm.MsmError):
            cx.set_param(key, bad)
    cx.set_param(gm.PARAM_GRID, 5)
    assert cx.get_param(gm.PARAM_GRID) == 5
    cx.set_param(gm.PARAM_ACC_PLACEMENT, gm.ACC_SHARED)
    assert cx.get_param(gm.PARAM_ACC_PLACEMENT) == gm.ACC_SHARED
    cx.set_param(gm.PARAM_GRID, 0)
    cx.set_param(gm.PARAM_ACC_PLACEMENT, gm.ACC_LOCAL)


@pytest.mark.parametrize("groups", [1, 2, 3, 4])
@pytest.mark.parametrize("timing", [0, 1])
def test_window_groups_and_schedules(mid_case, groups, timing):
    """The pipelined schedule (window groups on the context's streams) and the
    serial one (phase timing on) give the same result for every group count."""
    pts, k, expect = mid_case
    cx = ctx(20000, 13)
    cx.set_param(gm.PARAM_GROUPS, groups)
    cx.set_param(gm.PARAM_TIMING, timing)
    try:
        got = normalise(cx.run(gpu_points(pts), gpu_scalars(k), 13))
        if timing:
            assert len(cx.phase_ms()) == 7
    finally:
        cx.set_param(gm.PARAM_GROUPS, 0)
        cx.set_param(gm.PARAM_TIMING, 0)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("finish_t", [1, 2, 3, 4, 8, 16, 64])
def test_small_bucket_finish(mid_case, finish_t):
    """Every small-bucket threshold T (buckets with <= T items summed in
    Jacobian coordinates outside the affine tree) gives the same result."""
    pts, k, expect = mid_case
    cx = ctx(20000, 13)
    cx.set_param(gm.PARAM_FINISH, finish_t)
    try:
        got = normalise(cx.run(gpu_points(pts), gpu_scalars(k), 13))
    finally:
        cx.set_param(gm.PARAM_FINISH, 0)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("c,finish_t", [(8, 4), (8, 32), (16, 2), (16, 8)])
def test_small_bucket_finish_chunk_lengths(mid_case, c, finish_t):
    """The fused finish and chunk sums with chunks of two buckets (c = 8, four
    threads per bucket's chain) and of eight (c = 16, one thread each)."""
    pts, k, expect = mid_case
    cx = ctx(20000, c)
    cx.set_param(gm.PARAM_FINISH, finish_t)
    try:
        got = normalise(cx.run(gpu_points(pts), gpu_scalars(k), c))
    finally:
        cx.set_param(gm.PARAM_FINISH, 0)
    assert np.array_equal(got, expect)


def _host_inputs(pts, k, pin=True):
    p = torch.from_numpy(oracle.points_to_gpu_layout(pts).view(np.int32))
    s_ = torch.from_numpy(synth.scalars_to_u32(k).view(np.int32))
    return (p.pin_memory(), s_.pin_memory()) if pin else (p.contiguous(), s_.contiguous())


@pytest.mark.parametrize("glv", [1, 0])
@pytest.mark.parametrize("timing", [0, 1])
def test_host_buffer_entry(mid_case, glv, timing):
    """msm_g1_run_host (inputs and result in host memory, the points uploaded
    on a context stream beside the sort) gives the oracle's result in both
    schedules."""
    pts, k, expect = mid_case
    cx = ctx(20000, 13)
    cx.set_param(gm.PARAM_GLV, glv)
    cx.set_param(gm.PARAM_TIMING, timing)
    try:
        hp, hs = _host_inputs(pts, k)
        out = cx.run_host(hp, hs, 13)
        got = normalise(out)
    finally:
        cx.set_param(gm.PARAM_GLV, 1)
        cx.set_param(gm.PARAM_TIMING, 0)
    assert np.array_equal(got, expect)


def test_host_buffer_entry_back_to_back():
    """Consecutive host-buffer calls on one stream with no synchronisation in
    between reuse the context's device copies: each must still see its own
    inputs (pinned and pageable host buffers)."""
    cases = []
    for i, n in enumerate((3000, 1500, 2999)):
        r, k = synth.uniform_workload(n, 7100 + i)
        pts = points_from_r(r)
        cases.append((pts, k, oracle.closed_form(r, k), i != 1))
    cx = ctx(3000, 11)
    outs = []
    for pts, k, _, pin in cases:
        hp, hs = _host_inputs(pts, k, pin)
        outs.append(cx.run_host(hp, hs, 11, out=torch.empty(24, dtype=torch.int32).pin_memory()))
    torch.cuda.synchronize()
    for (pts, k, expect, _), out in zip(cases, outs):
        assert np.array_equal(normalise(out), expect)


def test_host_buffer_entry_edges():
    cx = ctx(100, 8)
    empty_p = torch.zeros((0, 16), dtype=torch.int32)
    empty_s = torch.zeros((0, 8), dtype=torch.int32)
    out = cx.run_host(empty_p, empty_s, 8)
    assert oracle.words_to_point(normalise(out)) is None
    r, k = synth.uniform_workload(101, 3)
    hp, hs = _host_inputs(points_from_r(r), k)
    with pytest.raises(gm.MsmError) as e:
        cx.run_host(hp, hs, 8)
    assert e.value.code == gm.ERR_CAPACITY
    out = cx.run_host(hp[:100], hs[:100], 8)
    assert np.array_equal(normalise(out), oracle.closed_form(r[:100], k[:100]))


@pytest.mark.parametrize("inversion", [1, 0])
def test_inversion_choice(mid_case, inversion):
    """Both batch inversions (safegcd divsteps, Fermat) give the oracle's result."""
    pts, k, expect = mid_case
    cx = ctx(20000, 13)
    cx.set_param(gm.PARAM_INVERSION, inversion)
    try:
        got = normalise(cx.run(gpu_points(pts), gpu_scalars(k), 13))
    finally:
        cx.set_param(gm.PARAM_INVERSION, 0)
    assert np.array_equal(got, expect)


def _batch_case(sizes, seed):
    rs, ks = [], []
    for i, n in enumerate(sizes):
        r, k = synth.uniform_workload(n, seed + i) if n else (np.zeros((0, 4), np.uint64), np.zeros((0, 4), np.uint64))
        rs.append(r)
        ks.append(k)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    r_all = np.concatenate(rs)
    return rs, ks, offsets, points_from_r(r_all), np.concatenate(ks)


@pytest.mark.parametrize("glv", [1, 0])
def test_batch_matches_each_msm(glv):
    """msm_g1_run_batch: ragged and empty MSMs fused into one pass give each
    MSM's own result (closed form) and the single-MSM entry's result."""
    sizes = [700, 1, 0, 2500, 33, 1024, 0, 5]
    rs, ks, offsets, pts, k = _batch_case(sizes, 8100)
    cx = ctx(5000, 12)
    cx.set_param(gm.PARAM_GLV, glv)
    try:
        out = cx.run_batch(gpu_points(pts), gpu_scalars(k), offsets, 9)
        torch.cuda.synchronize()
        for m, (r, km) in enumerate(zip(rs, ks)):
            got = oracle.jacobian_mont_to_affine(gm.to_host(out[m]))
            assert np.array_equal(got, oracle.closed_form(r, km)), m
        single = normalise(cx.run(gpu_points(pts[offsets[3]:offsets[4]]), gpu_scalars(k[offsets[3]:offsets[4]]), 9))
        assert np.array_equal(single, oracle.jacobian_mont_to_affine(gm.to_host(out[3])))
    finally:
        cx.set_param(gm.PARAM_GLV, 1)


def test_batch_split_into_passes():
    """A batch larger than the context's buffers runs as several passes:
    200 MSMs at c = 13 need 2000 windows of 4096 buckets, more than a context
    made for 4096 terms holds."""
    sizes = [(37 * i) % 300 + 1 for i in range(200)]
    rs, ks, offsets, pts, k = _batch_case(sizes, 8300)
    cx = ctx(4096, 13)
    out = cx.run_batch(gpu_points(pts), gpu_scalars(k), offsets, 13)
    torch.cuda.synchronize()
    for m in range(0, 200, 7):
        got = oracle.jacobian_mont_to_affine(gm.to_host(out[m]))
        assert np.array_equal(got, oracle.closed_form(rs[m], ks[m])), m
    got = oracle.jacobian_mont_to_affine(gm.to_host(out[199]))
    assert np.array_equal(got, oracle.closed_form(rs[199], ks[199]))


def test_batch_context_fuses_one_pass():
    """A context made for 16 fused MSMs (msm_g1_create_batch) runs 16 MSMs of
    2^12 terms at c = 13 as one pass: one sort, one accumulation, one
    reduction, 16 combination warps."""
    sizes = [1 << 12] * 16
    rs, ks, offsets, pts, k = _batch_case(sizes, 8500)
    with gm.MsmG1(1 << 16, 13, max_batch=16) as cx:
        out = cx.run_batch(gpu_points(pts), gpu_scalars(k), offsets, 13)
        torch.cuda.synchronize()
        for m in range(16):
            got = oracle.jacobian_mont_to_affine(gm.to_host(out[m]))
            assert np.array_equal(got, oracle.closed_form(rs[m], ks[m])), m
    with gm.MsmG1(1 << 16, 13) as cx1:  # sized for one MSM: several passes, same points
        out1 = cx1.run_batch(gpu_points(pts), gpu_scalars(k), offsets, 13)
        torch.cuda.synchronize()
        for m in (0, 7, 15):
            assert np.array_equal(oracle.jacobian_mont_to_affine(gm.to_host(out1[m])),
                                  oracle.jacobian_mont_to_affine(gm.to_host(out[m])))


def test_batch_argument_errors():
    cx = ctx(100, 8)
    r, k = synth.uniform_workload(120, 3)
    pts, ks = gpu_points(points_from_r(r)), gpu_scalars(k)
    with pytest.raises(gm.MsmError) as e:
        cx.run_batch(pts, ks, [0, 120], 8)  # one MSM beyond max_n
    assert e.value.code == gm.ERR_CAPACITY
    out = cx.run_batch(pts, ks, [0, 60, 120], 8)  # two that fit
    torch.cuda.synchronize()
    assert np.array_equal(oracle.jacobian_mont_to_affine(gm.to_host(out[1])), oracle.closed_form(r[60:], k[60:]))
    lib = gm.lib()
    bad = (ctypes.c_size_t * 3)(0, 80, 60)  # decreasing offsets
    assert lib.msm_g1_run_batch(cx._ctx, ctypes.c_void_p(pts.data_ptr()), ctypes.c_void_p(ks.data_ptr()), bad, 2, 8,
                                ctypes.c_void_p(out.data_ptr()), None) == gm.ERR_INVALID_ARG


def test_empty_input():
    cx = ctx(16, 8)
    pts = torch.zeros((0, 16), dtype=torch.int32, device="cuda")
    ks = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    out = cx.run(pts, ks, 8)
    assert oracle.words_to_point(normalise(out)) is None


LAMBDA = 0xb3c4d79d41a917585bfc41088d8daaa78b17ea66b99c90dd  # the endomorphism's eigenvalue (pinned in test_glv)


@pytest.mark.parametrize("glv", [1, 0])
@pytest.mark.parametrize("kval", [0, 1, 2, 3, pyref.R - 1, pyref.R, pyref.R + 1, (1 << 256) - 1, 1 << 255,
                                  LAMBDA, pyref.R - LAMBDA, LAMBDA * LAMBDA % pyref.R, (1 << 127) - 1, 1 << 127])
def test_single_term(kval, glv):
    """One term, including scalars whose GLV halves are zero, one or negative."""
    pts = points_from_r(oracle.ints_to_limbs([987654321]))
    k = oracle.ints_to_limbs([kval])
    assert np.array_equal(run_gpu(pts, k, 8, max_n=16, max_c=8, glv=glv), expect_oracle(pts, k))


@pytest.mark.parametrize("c", [4, 8])
def test_glv_images_collide_with_inputs(c):
    """Inputs P, phi(P) = [lambda]P and -phi(P), all with one scalar k: in the
    GLV path every bucket then holds copies of P, phi(P), -phi(P) and
    phi(phi(P)), so the accumulation meets doublings (equal points), P == -Q
    cancellations and, where a window's two digits coincide, the sum
    P + phi(P) + phi^2(P) = [1 + lambda + lambda^2]P = infinity."""
    assert LAMBDA == gm.glv_constants()[1]
    t = 424242
    r = [t] * 300 + [t * LAMBDA % pyref.R] * 300 + [(pyref.R - t) * LAMBDA % pyref.R] * 150
    kk = synth.limbs_to_ints(synth.uniform_workload(1, 62)[1])[0]
    k = oracle.ints_to_limbs([kk] * len(r))
    pts = points_from_r(oracle.ints_to_limbs(r))
    # max_n = 2 x 750 so that c = 4 (2n x 32 entries) fits the context
    assert np.array_equal(run_gpu(pts, k, c, max_n=1500, max_c=8), expect_oracle(pts, k))


def test_all_zero_scalars():
    r, _ = synth.uniform_workload(300, 5)
    pts = points_from_r(r)
    k = np.zeros((300, 4), dtype=np.uint64)
    assert oracle.words_to_point(run_gpu(pts, k, 8)) is None


@pytest.mark.parametrize("n", [2, 3, 64, 1000])
def test_same_point_same_digit(n):
    """Every entry lands in one bucket with the same point: level 0 pairs are
    all doublings, later levels add equal partial sums (doublings again)."""
    pts = points_from_r(oracle.ints_to_limbs([31337] * n))
    k = np.zeros((n, 4), dtype=np.uint64)
    k[:, 0] = 1
    got = run_gpu(pts, k, 8, max_n=1000, max_c=8)
    assert oracle.words_to_point(got) == pyref.mul(31337 * n % pyref.R, pyref.G)


@pytest.mark.parametrize("n,c,finish_t", [(20000, 13, 0), (20000, 10, 1), (70000, 13, 8)])
def test_equal_scalars_fill_one_bucket_per_window(n, c, finish_t):
    """All scalars equal: every window puts all n (or 2n) terms into one
    bucket, far deeper than the tree levels launched one by one, so the
    deep-level launch sums it (MSM = k sum_i P_i)."""
    r, _ = synth.uniform_workload(n, 2024 + c)
    pts = points_from_r(r)
    kv = 0x1234567890ABCDEF1234567890ABCDEF1234567890ABCDEF1234567890ABCDE % pyref.R
    k = oracle.ints_to_limbs([kv] * n)
    cx = ctx(n, 16)
    cx.set_param(gm.PARAM_FINISH, finish_t)
    cx.set_param(gm.PARAM_STATS, 1)
    try:
        got = run_gpu(pts, k, c, max_n=n, max_c=16)
        levels = cx.stats()["levels"]
    finally:
        cx.set_param(gm.PARAM_FINISH, 0)
        cx.set_param(gm.PARAM_STATS, 0)
    assert np.array_equal(got, oracle.closed_form(r, k))
    if finish_t == 1:
        assert levels >= 14  # the deep levels did the work (log2 n of them)


def test_opposite_points_cancel():
    r = [11 + i for i in range(200)] + [pyref.R - 11 - i for i in range(200)]
    k = oracle.ints_to_limbs([5 + (i % 200) for i in range(400)])
    pts = points_from_r(oracle.ints_to_limbs(r))
    assert oracle.words_to_point(run_gpu(pts, k, 6)) is None


def test_infinity_inputs():
    r, k = synth.uniform_workload(500, 77)
    pts = points_from_r(r)
    pts[::7] = 0  # (0, 0) = infinity
    assert np.array_equal(run_gpu(pts, k, 9), expect_oracle(pts, k))


@pytest.mark.parametrize("scal", ["ones", "uniform"])
def test_progression_points(scal):
    """The pages' failing workload: points in arithmetic progression make
    partial sums collide in x (PR #23736, section "Change (correct, landed)")."""
    r, k = synth.progression_workload(3000, 9, scalars=scal)
    pts = points_from_r(r)
    assert np.array_equal(run_gpu(pts, k, 7), expect_oracle(pts, k))


@pytest.mark.parametrize("glv", [1, 0])
@pytest.mark.parametrize("finish_t", [1, 8])
def test_adversarial_small(finish_t, glv):
    r, k = synth.adversarial_workload(30000, 1005)
    pts = points_from_r(r)
    cx = ctx(30000, 16)
    cx.set_param(gm.PARAM_FINISH, finish_t)
    try:
        got = run_gpu(pts, k, 12, max_n=30000, max_c=16, glv=glv)
    finally:
        cx.set_param(gm.PARAM_FINISH, 0)
    assert np.array_equal(got, expect_oracle(pts, k))


def test_deterministic_result():
    r, k = synth.uniform_workload(5000, 8)
    pts = points_from_r(r)
    a = run_gpu(pts, k, 11)
    b = run_gpu(pts, k, 11)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("glv", [0, 1])
def test_sort_structure(glv):
    """The sorted bucket list: every entry sits in the bucket of its digit,
    with the right negate flag; odd buckets carry one padding entry.  With
    GLV, entries i < n carry the digits of |k1_i| (negated when k1_i < 0) and
    entries n + i those of |k2_i| on phi(P_i)."""
    n, c = 3000, 9
    r, k = synth.uniform_workload(n, 99)
    pts = points_from_r(r)
    cx = ctx(n, c)
    cx.set_param(gm.PARAM_BATCH_S, 8)
    cx.set_param(gm.PARAM_GLV, glv)
    torch.cuda.synchronize()
    cx.run(gpu_points(pts), gpu_scalars(k), c)
    B = 1 << (c - 1)
    if glv:
        halves = gm.to_host(gm.test_glv_split(gpu_scalars(k))).reshape(n, 10)
        words = np.zeros((2 * n, 8), dtype=np.uint32)
        words[:n, :4], words[n:, :4] = halves[:, 0:4], halves[:, 4:8]
        digits = gm.to_host(gm.test_digits(gm.to_device(words), c, gm.GLV_BITS)).view(np.int32)
        flip = np.concatenate([halves[:, 8], halves[:, 9]]).astype(bool)
    else:
        digits = gm.to_host(gm.test_digits(gpu_scalars(k), c)).view(np.int32)
        flip = np.zeros(n, dtype=bool)
    W = digits.shape[1]
    counts, _ = cx.debug_read(0, W * B)
    offsets, _ = cx.debug_read(1, W * B + 1)
    total = int(offsets[-1])
    entries, nbytes = cx.debug_read(2, total)
    assert nbytes == 4 * total
    expect_count = np.zeros(W * B, dtype=np.int64)
    for w in range(W):
        d = digits[:, w]
        nz = d != 0
        np.add.at(expect_count, w * B + np.abs(d[nz]) - 1, 1)
    assert np.array_equal(counts.astype(np.int64), expect_count)
    for g in range(W * B):
        m = int(counts[g])
        o = int(offsets[g])
        assert o % 2 == 0 and int(offsets[g + 1]) - o == m + (m & 1)
        seg = entries[o:o + m]
        w, b = divmod(g, B)
        idx = seg & 0x7FFFFFFF
        neg = (seg >> 31) == 1
        dig = digits[idx, w]
        assert np.all(np.abs(dig) == b + 1) and np.all(((dig < 0) ^ flip[idx]) == neg)
        assert len(set(idx.tolist())) == m
        if m & 1:
            assert entries[o + m] == 0xFFFFFFFF
    cx.set_param(gm.PARAM_GLV, 1)


def test_capacity_and_argument_errors():
    cx = ctx(100, 8)
    r, k = synth.uniform_workload(101, 1)
    pts, ks = gpu_points(points_from_r(r)), gpu_scalars(k)
    with pytest.raises(gm.MsmError) as e:
        cx.run(pts, ks, 8)
    assert e.value.code == gm.ERR_CAPACITY
    with pytest.raises(gm.MsmError) as e:
        cx.run(pts[:100], ks[:100], 9)
    assert e.value.code == gm.ERR_CAPACITY
    with pytest.raises(gm.MsmError) as e:
        cx.run(pts[:100], ks[:100], 21)
    assert e.value.code == gm.ERR_INVALID_ARG
    flat = ks.reshape(-1)[1:8 * 50 + 1].reshape(50, 8)  # 4-byte offset: misaligned
    with pytest.raises(gm.MsmError) as e:
        cx.run(pts[:50], flat, 8)
    assert e.value.code == gm.ERR_INVALID_ARG


def test_mul_generator():
    ks = [0, 1, 2, pyref.R - 1, pyref.R, (1 << 256) - 1] + synth.limbs_to_ints(synth.uniform_workload(3000, 6)[0])
    kl = oracle.ints_to_limbs(ks)
    cx = ctx(16, 8)
    out = cx.mul_generator(gm.to_device(synth.scalars_to_u32(kl)))
    torch.cuda.synchronize()
    got = gm.to_host(out)
    expect = oracle.points_to_gpu_layout(oracle.generator_multiples(kl))
    assert np.array_equal(got, expect)


# ------------------------------------------------------------ full sizes

@pytest.fixture(scope="module")
def big_points():
    """2^22 uniform points [r_i]G from the oracle (prefixes serve 2^16, 2^20)."""
    r, _ = synth.uniform_workload(1 << 22, 1004)
    return r, points_from_r(r)


@pytest.mark.parametrize("glv", [1, 0])
def test_config2_n65536_c13(big_points, glv):
    r_all, pts_all = big_points
    n = 1 << 16
    _, k = synth.uniform_workload(n, 1002)
    r, pts = r_all[:n], pts_all[:n]
    got = run_gpu(pts, k, 13, max_n=n, max_c=13, glv=glv)
    assert np.array_equal(got, expect_oracle(pts, k))
    assert np.array_equal(got, oracle.closed_form(r, k))


@pytest.mark.parametrize("batch_s", [0, 4, 8, 16, 32, 64])
def test_config3_n2p20_c16(big_points, batch_s):
    r_all, pts_all = big_points
    n = 1 << 20
    _, k = synth.uniform_workload(n, 1003)
    got = run_gpu(pts_all[:n], k, 16, max_n=n, max_c=16, batch_s=batch_s)
    assert np.array_equal(got, oracle.closed_form(r_all[:n], k))


@pytest.mark.parametrize("place", ["local", "shared", "registers"])
@pytest.mark.parametrize("tpb", [64, 128, 256])
@pytest.mark.parametrize("batch_s", [4, 8, 16, 32, 64])
def test_config3_sweep(big_points, place, tpb, batch_s):
    """Every cell of the n = 2^20 sweep over S, threads per block and the
    prefix-product placement is bit-exact (the closed form)."""
    r_all, pts_all = big_points
    n = 1 << 20
    k = _config3_scalars()
    got = run_gpu(pts_all[:n], k, 16, max_n=n, max_c=16, batch_s=batch_s, tpb=tpb, place=PLACEMENTS[place])
    assert np.array_equal(got, _config3_expect(r_all[:n], k))


_c3 = {}


def _config3_scalars():
    if "k" not in _c3:
        _c3["k"] = synth.uniform_workload(1 << 20, 1003)[1]
    return _c3["k"]


def _config3_expect(r, k):
    if "e" not in _c3:
        _c3["e"] = oracle.closed_form(r, k)
    return _c3["e"]


@pytest.mark.parametrize("c,glv", [(16, 1), (17, 1), (18, 1), (16, 0)])
def test_config4_n2p22(big_points, c, glv):
    r, pts = big_points
    _, k = synth.uniform_workload(1 << 22, 1005)
    got = run_gpu(pts, k, c, max_n=1 << 22, max_c=18, glv=glv)
    assert np.array_equal(got, oracle.closed_form(r, k))


def test_n2p23_beyond_the_configs(big_points):
    """n = 2^23 (twice the largest configuration): the 2^22 points twice over,
    with independent scalars; the closed form pins the result at any n."""
    r, pts = big_points
    _, k1 = synth.uniform_workload(1 << 22, 1007)
    _, k2 = synth.uniform_workload(1 << 22, 1008)
    r2 = np.concatenate([r, r])
    k = np.concatenate([k1, k2])
    got = run_gpu(np.concatenate([pts, pts]), k, 16, max_n=1 << 23, max_c=16)
    assert np.array_equal(got, oracle.closed_form(r2, k))


@pytest.mark.parametrize("glv", [1, 0])
def test_config5_adversarial_n2p20(glv):
    n = 1 << 20
    r, k = synth.adversarial_workload(n, 1006)
    pts = points_from_r(r)
    got = run_gpu(pts, k, 16, max_n=n, max_c=16, glv=glv)
    assert np.array_equal(got, oracle.closed_form(r, k))


def test_graph_replay_follows_buffer_contents_and_arguments():
    """Small MSMs replay a captured CUDA graph while the pointers, n and c stay
    the same: new scalar values in the same buffer, a new output buffer, a
    parameter change (which drops the graph), the graph switched off, and a run
    captured inside the caller's own CUDA graph all give the oracle's result."""
    n, c = 1000, 8
    cx = gm.MsmG1(n, c)
    r, k = synth.uniform_workload(n, 4242)
    pts = gpu_points(points_from_r(r))
    scal = gpu_scalars(k)
    out = torch.empty(24, dtype=torch.int32, device="cuda")
    for step in range(3):
        cx.run(pts, scal, c, out=out)
        assert np.array_equal(normalise(out), oracle.closed_form(r, k)), step
        if step == 0:  # the same buffer, new values: the replay reads them
            k = synth.uniform_workload(n, 4243)[1]
            scal.copy_(gpu_scalars(k))
    out2 = torch.empty(24, dtype=torch.int32, device="cuda")
    cx.run(pts, scal, c, out=out2)
    assert np.array_equal(normalise(out2), oracle.closed_form(r, k))
    cx.set_param(gm.PARAM_GROUPS, 1)
    cx.run(pts, scal, c, out=out2)
    assert np.array_equal(normalise(out2), oracle.closed_form(r, k))
    cx.set_param(gm.PARAM_GRAPH, 0)
    cx.run(pts, scal, c, out=out)
    assert np.array_equal(normalise(out), oracle.closed_form(r, k))
    cx.set_param(gm.PARAM_GRAPH, 1)
    cx.set_param(gm.PARAM_GROUPS, 0)
    # inside the caller's capture the run becomes part of the caller's graph
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cx.run(pts, scal, c, out=out, stream=s)
    out.zero_()
    torch.cuda.synchronize()
    g.replay()
    assert np.array_equal(normalise(out), oracle.closed_form(r, k))


def test_graph_replay_of_host_buffer_runs():
    """msm_g1_run_host with page-locked buffers replays its captured copies and
    launches: new scalar values in the same host buffer, a new result buffer,
    and pageable buffers (which take the direct path) all give the oracle's
    result."""
    n, c = 900, 9
    cx = gm.MsmG1(n, c)
    r, k = synth.uniform_workload(n, 5151)
    pts = gpu_points(points_from_r(r)).cpu().pin_memory()
    scal = gpu_scalars(k).cpu().pin_memory()
    out = torch.empty(24, dtype=torch.int32).pin_memory()
    for step in range(3):
        cx.run_host(pts, scal, c, out=out)
        torch.cuda.synchronize()
        assert np.array_equal(oracle.jacobian_mont_to_affine(out.numpy().view(np.uint32)), oracle.closed_form(r, k)), step
        if step == 0:
            k = synth.uniform_workload(n, 5152)[1]
            scal.copy_(gpu_scalars(k).cpu())
    out2 = torch.empty(24, dtype=torch.int32).pin_memory()
    cx.run_host(pts, scal, c, out=out2)
    torch.cuda.synchronize()
    assert np.array_equal(oracle.jacobian_mont_to_affine(out2.numpy().view(np.uint32)), oracle.closed_form(r, k))
    out3 = torch.empty(24, dtype=torch.int32)
    cx.run_host(pts.clone(), scal.clone(), c, out=out3)
    torch.cuda.synchronize()
    assert np.array_equal(oracle.jacobian_mont_to_affine(out3.numpy().view(np.uint32)), oracle.closed_form(r, k))
