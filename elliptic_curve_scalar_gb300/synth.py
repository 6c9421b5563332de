"""Seeded synthetic workloads for BN254 G1 multi-scalar multiplication.

This module draws integers only.  It holds no field or curve arithmetic: a
workload is the list of discrete logarithms r_i (the points are P_i = [r_i]G,
computed by whoever consumes the workload) and the list of scalars k_i.
Because P_i = [r_i]G, every MSM over such a workload has the closed form
[sum_i k_i r_i mod r]G, which pins results at any size.

The random source is splitmix64 used as a counter-based generator (Steele,
Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014):
value(seed, stream, i) = mix64(key(seed, stream) + (i + 1) * 0x9E3779B97F4A7C15).
It is written out here with numpy uint64 wrap-around arithmetic so that the
same seed gives the same workload on every host and numpy version.

Workloads (the shape of the pages' measurements: "logn=16, independent random
points" in PR #23736, section "Real-hardware results"; the adversarial mix is
this library's own stress case):

* ``uniform``: r_i and k_i uniform in [0, r).
* ``adversarial``: scalars 12.5 % zero, 12.5 % one, 25 % uniform below 2^64,
  50 % uniform in [0, r), at shuffled positions; points: 5 % exact duplicates
  and 5 % negations of a uniformly chosen earlier point.
* ``progression``: r_i = a + i*d mod r, the arithmetic progression of points
  whose partial sums collide in x (the failure the pages record in PR #23736,
  section "Change (correct, landed)").
"""
import numpy as np

# BN254 scalar-field order r (the prime order of G1).
R_INT = 0x30644E72E131A029B85045B68181585D2833E84879B9709143E1F593F0000001
R_LIMBS = np.array([(R_INT >> (64 * i)) & 0xFFFFFFFFFFFFFFFF for i in range(4)], dtype=np.uint64)

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream identifiers
S_R, S_K, S_KCAT, S_KSMALL, S_PCAT, S_PSRC, S_PERM = range(1, 8)


def _mix64(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed, stream):
    with np.errstate(over="ignore"):
        k = _mix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64) * _GOLDEN + np.uint64(stream))
    return k[0]


def u64_stream(seed, stream, count, offset=0):
    """count uint64 values of stream ``stream`` starting at counter ``offset``."""
    i = np.arange(offset, offset + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(_key(seed, stream) + (i + np.uint64(1)) * _GOLDEN)


def _less_than_r(x):
    """x: uint64[n, 4] -> bool[n], lexicographic compare against r."""
    lt = np.zeros(x.shape[0], dtype=bool)
    eq = np.ones(x.shape[0], dtype=bool)
    for limb in range(3, -1, -1):
        lt |= eq & (x[:, limb] < R_LIMBS[limb])
        eq &= x[:, limb] == R_LIMBS[limb]
    return lt


def uniform_below_r(seed, stream, n):
    """uint64[n, 4]: uniform integers in [0, r) by rejection from 254-bit draws."""
    out = np.zeros((n, 4), dtype=np.uint64)
    todo = np.arange(n)
    round_ = 0
    while todo.size:
        # counter space: round * 2^40 + 4 * index + limb keeps every draw distinct
        base = np.uint64(round_) << np.uint64(40)
        ctr = base + np.repeat(todo.astype(np.uint64) * np.uint64(4), 4) + np.tile(np.arange(4, dtype=np.uint64), todo.size)
        with np.errstate(over="ignore"):
            draw = _mix64(_key(seed, stream) + (ctr + np.uint64(1)) * _GOLDEN).reshape(-1, 4)
        draw[:, 3] &= np.uint64((1 << 62) - 1)  # 254-bit candidates
        ok = _less_than_r(draw)
        out[todo[ok]] = draw[ok]
        todo = todo[~ok]
        round_ += 1
    return out


def _neg_mod_r(x):
    """(r - x) mod r on uint64[n, 4] with x < r."""
    out = np.zeros_like(x)
    borrow = np.zeros(x.shape[0], dtype=np.uint64)
    for limb in range(4):
        a = R_LIMBS[limb]
        b = x[:, limb]
        with np.errstate(over="ignore"):
            d = a - b - borrow
        borrow = ((b > a) | ((b == a) & (borrow == 1))).astype(np.uint64)
        out[:, limb] = d
    zero = np.all(x == 0, axis=1)
    out[zero] = 0
    return out


def uniform_workload(n, seed):
    """(r_values, scalars), both uint64[n, 4] uniform in [0, r)."""
    return uniform_below_r(seed, S_R, n), uniform_below_r(seed, S_K, n)


def adversarial_workload(n, seed):
    """(r_values, scalars) with the zero/one/small/uniform scalar mix and
    duplicated / negated points described in the module docstring."""
    r_values = uniform_below_r(seed, S_R, n)
    k = uniform_below_r(seed, S_K, n)
    cat = u64_stream(seed, S_KCAT, n) % np.uint64(8)
    small = u64_stream(seed, S_KSMALL, n)
    k[cat == 0] = 0
    one = cat == 1
    k[one] = 0
    k[one, 0] = 1
    sm = (cat == 2) | (cat == 3)
    k[sm] = 0
    k[sm, 0] = small[sm]

    pcat = u64_stream(seed, S_PCAT, n) % np.uint64(20)
    src_draw = u64_stream(seed, S_PSRC, n)
    idx = np.arange(n, dtype=np.uint64)
    derived = (pcat <= 1) & (idx > 0)
    src = np.where(derived, src_draw % np.maximum(idx, np.uint64(1)), idx).astype(np.int64)
    flip = (derived & (pcat == 1)).astype(np.int64)
    # follow chains (a copy of a copy) back to an underived point, composing signs
    for _ in range(64):
        nxt = src[src]
        if np.array_equal(nxt, src):
            break
        flip = flip ^ np.where(src != np.arange(n), flip[src], 0)
        src = nxt
    base = r_values[src]
    negd = _neg_mod_r(base)
    r_out = np.where((flip == 1)[:, None], negd, base)
    return np.ascontiguousarray(r_out), np.ascontiguousarray(k)


def progression_workload(n, seed, scalars="uniform"):
    """r_i = a + i*d mod r (small a, d drawn from the seed); scalars uniform or all one."""
    a = int(u64_stream(seed, S_R, 1)[0]) % 1000 + 1
    d = int(u64_stream(seed, S_R, 1, offset=1)[0]) % 1000 + 1
    r_vals = np.zeros((n, 4), dtype=np.uint64)
    for i in range(n):
        v = (a + i * d) % R_INT
        for limb in range(4):
            r_vals[i, limb] = (v >> (64 * limb)) & 0xFFFFFFFFFFFFFFFF
    if scalars == "ones":
        k = np.zeros((n, 4), dtype=np.uint64)
        k[:, 0] = 1
    else:
        k = uniform_below_r(seed, S_K, n)
    return r_vals, k


WORKLOADS = {
    "uniform": uniform_workload,
    "adversarial": adversarial_workload,
    "progression": progression_workload,
}


def workload(kind, n, seed):
    return WORKLOADS[kind](n, seed)


def limbs_to_ints(a):
    a = np.asarray(a, dtype=np.uint64)
    return [int(row[0]) | int(row[1]) << 64 | int(row[2]) << 128 | int(row[3]) << 192 for row in a]


def scalars_to_u32(k):
    """uint64[n, 4] -> uint32[n, 8] (the library's scalar layout, same bytes)."""
    return np.ascontiguousarray(np.asarray(k, dtype=np.uint64)).view(np.uint32).reshape(-1, 8)
