"""Device primitives (field, curve, batched affine addition, digit recoding)
against the oracle's arithmetic (Python integers and the affine law of
oracle.pyref), element by element and bit-exact."""
import random

import numpy as np
import pytest
import torch

from oracle import pyref
from elliptic_curve_scalar_gb300 import msm as gm
from tests.gpu_helpers import (P, R, mont, unmont, ints_to_u32, u32_to_ints, point_to_aff_words,
                               aff_words_to_point, point_to_jac_words, jac_words_to_point)

pytestmark = pytest.mark.gpu

EDGE = [0, 1, 2, P - 1, P - 2, (1 << 255) % P, (1 << 128) - 1, (1 << 224), P >> 1, (1 << 254) % P]


def _field_inputs(n, seed):
    rng = random.Random(seed)
    vals = EDGE + [rng.randrange(P) for _ in range(n - len(EDGE))]
    return vals


@pytest.mark.parametrize("op", ["mul", "sqr", "add", "sub", "neg", "inv", "inv_fermat", "inv_table", "inv_block"])
def test_fq_ops(op):
    n = 4099  # several blocks and a ragged tail
    a = _field_inputs(n, 1)
    if op == "inv_block":  # the block's shared inversion takes nonzero values only
        a = [x or 1 for x in a]
    b = list(reversed(_field_inputs(n, 2)))
    da = gm.to_device(ints_to_u32([mont(x) for x in a]))
    db = gm.to_device(ints_to_u32([mont(x) for x in b]))
    out = gm.test_fq(op, da, db if op in ("mul", "add", "sub") else None)
    got = [unmont(v) for v in u32_to_ints(gm.to_host(out))]
    raw = u32_to_ints(gm.to_host(out))
    assert all(v < P for v in raw), "result not fully reduced"
    for x, y, g in zip(a, b, got):
        if op == "mul":
            e = x * y % P
        elif op == "sqr":
            e = x * x % P
        elif op == "add":
            e = (x + y) % P
        elif op == "sub":
            e = (x - y) % P
        elif op == "neg":
            e = (-x) % P
        else:  # both inversions: 0 -> 0
            e = pow(x, P - 2, P)
        assert g == e, (op, x, y)


def _rand_points(rng, n):
    return [pyref.mul(rng.randrange(1, R), pyref.G) for _ in range(n)]


def test_jacobian_ops():
    rng = random.Random(5)
    pts = _rand_points(rng, 40)
    a = pts[:20] + [None, pts[0], pts[1], pts[2]]
    b = pts[20:] + [pts[3], None, pts[1], pyref.neg(pts[2])]
    zs = [rng.randrange(2, P) for _ in a]
    ja = np.stack([point_to_jac_words(p, z) for p, z in zip(a, zs)])
    jb = np.stack([point_to_jac_words(p, z + 7) for p, z in zip(b, zs)])
    ab = np.stack([point_to_aff_words(p) for p in b])
    da, db, dab = gm.to_device(ja), gm.to_device(jb), gm.to_device(ab)
    dbl = gm.to_host(gm.test_g1("jac_dbl", da))
    add = gm.to_host(gm.test_g1("jac_add", da, db))
    mix = gm.to_host(gm.test_g1("jac_mixed", da, dab))
    aff = gm.to_host(gm.test_g1("to_affine", da))
    dblc = gm.to_host(gm.test_g1("jac_dbl_coop", da))
    addc = gm.to_host(gm.test_g1("jac_add_coop", da, db))
    # the same sums with the operands of the special cases swapped and with P + P
    addc2 = gm.to_host(gm.test_g1("jac_add_coop", db, da))
    addc3 = gm.to_host(gm.test_g1("jac_add_coop", da, da))
    mixc = gm.to_host(gm.test_g1("jac_mixed_coop", da, dab))
    # groups of 8 lanes: four elements per warp, whose special cases differ
    dbl8 = gm.to_host(gm.test_g1("jac_dbl_coop8", da))
    add8 = gm.to_host(gm.test_g1("jac_add_coop8", da, db))
    add8s = gm.to_host(gm.test_g1("jac_add_coop8", db, da))
    mix8 = gm.to_host(gm.test_g1("jac_mixed_coop8", da, dab))
    dbl5 = gm.to_host(gm.test_g1("jac_dbl5_coop", da))
    # affine + affine (the finish's first step): a's affine words against b's
    aa = gm.to_device(np.stack([point_to_aff_words(p) for p in a]))
    affadd = gm.to_host(gm.test_g1("aff_add", aa, dab))
    affdbl = gm.to_host(gm.test_g1("aff_add", aa, aa))
    for i, (p, q) in enumerate(zip(a, b)):
        assert jac_words_to_point(dbl[i]) == pyref.add(p, p), ("dbl", i)
        assert jac_words_to_point(add[i]) == pyref.add(p, q), ("add", i)
        assert jac_words_to_point(dblc[i]) == pyref.add(p, p), ("dbl_coop", i)
        assert jac_words_to_point(addc[i]) == pyref.add(p, q), ("add_coop", i)
        assert jac_words_to_point(addc2[i]) == pyref.add(q, p), ("add_coop swapped", i)
        assert jac_words_to_point(addc3[i]) == pyref.add(p, p), ("add_coop P+P", i)
        assert jac_words_to_point(mix[i]) == pyref.add(p, q), ("mixed", i)
        assert jac_words_to_point(mixc[i]) == pyref.add(p, q), ("mixed_coop", i)
        assert jac_words_to_point(dbl8[i]) == pyref.add(p, p), ("dbl_coop8", i)
        assert jac_words_to_point(add8[i]) == pyref.add(p, q), ("add_coop8", i)
        assert jac_words_to_point(add8s[i]) == pyref.add(q, p), ("add_coop8 swapped", i)
        assert jac_words_to_point(mix8[i]) == pyref.add(p, q), ("mixed_coop8", i)
        assert jac_words_to_point(dbl5[i]) == pyref.mul(32, p), ("dbl5_coop", i)
        assert jac_words_to_point(affadd[i]) == pyref.add(p, q), ("aff_add", i)
        assert jac_words_to_point(affdbl[i]) == pyref.add(p, p), ("aff_add P+P", i)
        assert aff_words_to_point(aff[i]) == p, ("to_affine", i)


@pytest.mark.parametrize("block", [0, 1])
@pytest.mark.parametrize("inline_back", [0, 1])
@pytest.mark.parametrize("batch_s", [1, 2, 4, 8, 16, 32, 64])
def test_batch_affine_add(batch_s, inline_back, block):
    """Batched affine pair additions, including pairs that would poison a
    shared inversion: equal points (tangent), opposite points, infinity;
    per-thread inversions and one inversion shared by the block's threads
    (whose tail threads have no pairs)."""
    rng = random.Random(100 + batch_s)
    pts = _rand_points(rng, 60)
    a, b = [], []
    for i in range(37):
        kind = i % 6
        p, q = pts[i], pts[i + 20]
        if kind == 1:
            q = p                 # doubling
        elif kind == 2:
            q = pyref.neg(p)      # P + (-P) = infinity
        elif kind == 3:
            p = None              # infinity + Q
        elif kind == 4:
            q = None              # P + infinity
        a.append(p)
        b.append(q)
    da = gm.to_device(np.stack([point_to_aff_words(p) for p in a]))
    db = gm.to_device(np.stack([point_to_aff_words(p) for p in b]))
    out = gm.to_host(gm.test_batch_add(da, db, batch_s, inline_back, block))
    for i, (p, q) in enumerate(zip(a, b)):
        assert aff_words_to_point(out[i]) == pyref.add(p, q), (batch_s, i)


def window_layout(c, nbits):
    """Widths of the W = ceil(nbits / c) windows, balanced: the low
    nbits - W floor(nbits / W) windows are one bit wider than the rest."""
    W = -(-nbits // c)
    q = nbits // W
    wide = nbits - q * W
    return [q + 1 if w < wide else q for w in range(W)]


def test_window_layout_reduces_to_c_and_c_minus_1_for_full_scalars():
    """For 255 bits the balanced layout is c-bit windows with the top
    W c - 255 one bit narrower."""
    for c in range(1, 21):
        W = -(-255 // c)
        narrow = W * c - 255
        if narrow <= W:
            assert window_layout(c, 255) == [c - 1 if w >= W - narrow else c for w in range(W)]


@pytest.mark.parametrize("nbits", [255, 128])
@pytest.mark.parametrize("c", [1, 2, 5, 8, 13, 16, 17, 18, 20])
def test_signed_digits(c, nbits):
    rng = random.Random(c)
    if nbits == 255:
        ks = [0, 1, R - 1, R, R + 1, (1 << 256) - 1, (1 << 254), 2 ** (c - 1), 2 ** c - 1]
        ks += [rng.randrange(0, 1 << 256) for _ in range(300)]
    else:  # GLV halves, < 2^127
        ks = [0, 1, (1 << 127) - 1, 1 << 126, 2 ** (c - 1), 2 ** c - 1, ((1 << 127) - 1) // 3]
        ks += [rng.randrange(0, 1 << 127) for _ in range(300)]
    d = gm.test_digits(gm.to_device(ints_to_u32(ks)), c, nbits)
    digits = gm.to_host(d).view(np.int32)
    widths = window_layout(c, nbits)
    W = -(-nbits // c)
    if nbits == 255:
        assert W == gm.window_count(c)
    assert digits.shape == (len(ks), W) and len(widths) == W and sum(widths) == nbits and max(widths) <= c
    offsets = [sum(widths[:w]) for w in range(W)]
    for k, row in zip(ks, digits):
        assert all(-(1 << (cw - 1)) < int(v) <= (1 << (cw - 1)) for v, cw in zip(row, widths))
        assert sum(int(v) << off for v, off in zip(row, offsets)) == k % R


def test_glv_split_on_device():
    """The device split k -> (k1, k2): k = k1 + lambda k2 (mod r) and
    |k1|, |k2| < 2^127, for reduced and unreduced scalars."""
    _, lam = gm.glv_constants()
    rng = random.Random(11)
    ks = [0, 1, 2, R - 1, R, R + 1, lam, R - lam, (1 << 256) - 1, 1 << 127, (R - 1) // 2]
    ks += [rng.randrange(0, 1 << 256) for _ in range(5000)]
    out = gm.to_host(gm.test_glv_split(gm.to_device(ints_to_u32(ks)))).reshape(-1, 10)
    for k, row in zip(ks, out):
        a = sum(int(v) << (32 * j) for j, v in enumerate(row[0:4]))
        b = sum(int(v) << (32 * j) for j, v in enumerate(row[4:8]))
        assert int(row[8]) in (0, 1) and int(row[9]) in (0, 1)
        k1 = -a if row[8] else a
        k2 = -b if row[9] else b
        assert a < 1 << 127 and b < 1 << 127
        assert (k1 + lam * k2 - k) % R == 0, k
