"""The residue-number-system arithmetic of the window combination and the
bucket reduction's shifts (rns.cuh; the two-warp projective chains of
g1_proj.cuh) against Python integers and the oracle's affine law."""
import ctypes
import random

import numpy as np
import pytest
import torch

from oracle import pyref
from elliptic_curve_scalar_gb300 import msm as gm
from tests.gpu_helpers import (P, R, mont, unmont, ints_to_u32, u32_to_ints, point_to_jac_words,
                               jac_words_to_point)

pytestmark = pytest.mark.gpu

OPS = {"mul": 0, "sqr_chain": 1, "dbl_n": 2, "add": 3, "horner": 4, "is_zero": 5}
EDGE = [0, 1, 2, P - 1, P - 2, (1 << 255) % P, (1 << 128) - 1, (1 << 224), P >> 1, (1 << 254) % P]


def rns(op, a, b=None, n=None, arg=0, width=24):
    n = a.shape[0] if n is None else n
    out = torch.zeros((n, width), dtype=torch.int32, device=a.device)
    rc = gm.lib().msm_g1_test_rns(OPS[op], ctypes.c_void_p(a.data_ptr()),
                                  ctypes.c_void_p(b.data_ptr() if b is not None else 0),
                                  ctypes.c_void_p(out.data_ptr()), n, arg,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gm.OK
    return gm.to_host(out)


def _field(n, seed):
    rng = random.Random(seed)
    return EDGE + [rng.randrange(P) for _ in range(n - len(EDGE))]


def test_rns_product_matches_the_positional_product():
    n = 1031
    a, b = _field(n, 11), list(reversed(_field(n, 12)))
    da = gm.to_device(ints_to_u32([mont(x) for x in a]))
    db = gm.to_device(ints_to_u32([mont(x) for x in b]))
    got = u32_to_ints(rns("mul", da, db, width=8))
    assert all(v < P for v in got), "not fully reduced"
    for x, y, g in zip(a, b, got):
        assert unmont(g) == x * y % P, (x, y)
    assert got == u32_to_ints(gm.to_host(gm.test_fq("mul", da, db)))


@pytest.mark.parametrize("k", [1, 2, 13, 117, 300])
def test_rns_squaring_chain_keeps_its_bounds(k):
    """Lazily reduced values fed back into the product k times in a row."""
    a = _field(64, 13 + k)
    da = gm.to_device(ints_to_u32([mont(x) for x in a]))
    got = [unmont(v) for v in u32_to_ints(rns("sqr_chain", da, arg=k, width=8))]
    for x, g in zip(a, got):
        assert g == pow(x, 1 << k, P), (x, k)


def _points(rng, n):
    return [pyref.mul(rng.randrange(1, R), pyref.G) for _ in range(n)]


def _jac(pts, rng):
    return np.stack([point_to_jac_words(p, rng.randrange(2, P)) for p in pts])


@pytest.mark.parametrize("k", [0, 1, 2, 5, 13, 65, 117])
def test_rns_doubling_chain(k):
    rng = random.Random(21 + k)
    pts = _points(rng, 30) + [None, pyref.G]
    da = gm.to_device(_jac(pts, rng))
    got = rns("dbl_n", da, arg=k)
    for p, w in zip(pts, got):
        assert jac_words_to_point(w) == (None if p is None else pyref.mul(1 << k, p)), k


def test_rns_addition_is_complete():
    """The complete projective addition: distinct points, P + P, P + (-P),
    and the identity on either side or both."""
    rng = random.Random(31)
    a = _points(rng, 40) + [None, None]
    b = _points(rng, 36) + [a[0], pyref.neg(a[1]), None, a[3], a[4], None]
    a[36] = a[2]  # a doubling where the operands' Jacobian coordinates differ
    b[36] = a[2]
    ja, jb = _jac(a, rng), _jac(b, rng)
    got = rns("add", gm.to_device(ja), gm.to_device(jb))
    for i, (p, q) in enumerate(zip(a, b)):
        assert jac_words_to_point(got[i]) == pyref.add(p, q), i


def test_rns_horner_with_special_windows():
    """Horner's rule over 10 window sums of 13-bit weight, with infinite
    windows, a window that makes the running value double (equal x) and one
    that cancels it (opposite points)."""
    rng = random.Random(41)
    cases = []
    for t in range(8):
        ws = _points(rng, 10)
        if t == 1:
            ws[3] = None
            ws[9] = None  # the top window infinite: the chain starts lower
        if t == 2:  # running value after the top window and one shift: 2^13 T_9
            ws[8] = pyref.mul(1 << 13, ws[9])
        if t == 3:
            ws[8] = pyref.neg(pyref.mul(1 << 13, ws[9]))
        if t == 4:
            ws = [None] * 10
        cases.append(ws)
    words = np.concatenate([_jac([w for w in ws], rng) for ws in cases])
    got = rns("horner", gm.to_device(words), n=len(cases), arg=10)
    for ws, w in zip(cases, got):
        expect = None
        for t in reversed(ws):
            expect = pyref.add(pyref.mul(1 << 13, expect) if expect is not None else None, t)
        assert jac_words_to_point(w) == expect


def test_rns_zero_test_is_exact():
    rng = random.Random(51)
    bound = 20
    vals = [k * P for k in range(bound)] + [k * P + 1 for k in range(bound)] + [k * P - 1 for k in range(1, bound)]
    vals += [rng.randrange(bound * P) for _ in range(60)] + [1, 2, P >> 1]
    vals = [v for v in vals if v < (1 << 256)]
    da = gm.to_device(ints_to_u32(vals))
    got = rns("is_zero", da, arg=bound, width=1)[:, 0]
    for v, g in zip(vals, got):
        assert g == (1 if v % P == 0 else 0), v
