"""msm_g1_run_noalloc, the MSM entry point for callers that cannot allocate
device memory (their heap belongs to another allocator, they run under a
fixed memory budget, or cudaMalloc's implicit synchronisation is too costly).
It must give exactly the result of the context-based msm_g1_run, call after
call, although every call reuses the same fixed scratch array.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from elliptic_curve_scalar_gb300 import msm as gm
from elliptic_curve_scalar_gb300 import synth
from tests.gpu_helpers import gpu_points, gpu_scalars, normalise, points_from_r

pytestmark = pytest.mark.gpu


def _noalloc(points, scalars, c):
    """Call the entry point through the C ABI directly."""
    out = torch.zeros(24, dtype=torch.int32, device="cuda")
    rc = gm.lib().msm_g1_run_noalloc(ctypes.c_void_p(points.data_ptr()), ctypes.c_void_p(scalars.data_ptr()),
                                     scalars.shape[0], c, ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out


def test_noalloc_matches_msm_g1_run_on_consecutive_calls():
    cases = [(4096, 10, 9101), (2999, 9, 9102), (4096, 10, 9103)]
    for n, c, seed in cases:  # three calls in a row reuse the same scratch array
        r, k = synth.uniform_workload(n, seed)
        pts, ks = gpu_points(points_from_r(r)), gpu_scalars(k)
        rc, out = _noalloc(pts, ks, c)
        assert rc == gm.OK
        got = normalise(out)
        with gm.MsmG1(n, c) as ctx:
            expect = normalise(ctx.run(pts, ks, c))
        assert np.array_equal(got, expect), (n, c, seed)
        assert np.array_equal(got, oracle.closed_form(r, k))


def test_noalloc_rejects_sizes_beyond_its_limit():
    r, k = synth.uniform_workload(4097, 9104)
    pts, ks = gpu_points(points_from_r(r)), gpu_scalars(k)
    rc, _ = _noalloc(pts, ks, 10)
    assert rc == gm.ERR_CAPACITY
    rc, _ = _noalloc(pts[:4096], ks[:4096], 11)
    assert rc == gm.ERR_CAPACITY
    rc, out = _noalloc(pts[:1], ks[:1], 0)  # auto window within the limit
    assert rc == gm.OK
    assert np.array_equal(normalise(out), oracle.closed_form(r[:1], k[:1]))
    # a window below 8 bits takes more entries per point: 4096 points no longer fit at c = 7
    rc, _ = _noalloc(pts[:4096], ks[:4096], 7)
    assert rc == gm.ERR_CAPACITY
    rc, out = _noalloc(pts[:3767], ks[:3767], 7)
    assert rc == gm.OK
    assert np.array_equal(normalise(out), oracle.closed_form(r[:3767], k[:3767]))
    rc, out = _noalloc(pts[:500], ks[:500], 4)  # a small window with few points fits
    assert rc == gm.OK
    assert np.array_equal(normalise(out), oracle.closed_form(r[:500], k[:500]))
