"""The seeded workload generators: determinism, ranges and the adversarial structure."""
import numpy as np

from elliptic_curve_scalar_gb300 import synth
from oracle import pyref


def test_deterministic_and_seed_sensitive():
    a = synth.uniform_workload(257, 5)
    b = synth.uniform_workload(257, 5)
    c = synth.uniform_workload(257, 6)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0])


def test_prefix_property():
    """A smaller workload with the same seed is a prefix of a larger one."""
    small = synth.uniform_workload(100, 9)
    big = synth.uniform_workload(1000, 9)
    assert np.array_equal(small[0], big[0][:100]) and np.array_equal(small[1], big[1][:100])


def test_uniform_below_r():
    r_vals, k = synth.uniform_workload(4096, 3)
    for arr in (r_vals, k):
        ints = synth.limbs_to_ints(arr)
        assert all(0 <= v < pyref.R for v in ints)
        assert len(set(ints)) == len(ints)
        # top bits are used: the largest draw is close to r
        assert max(ints) > pyref.R * 0.99


def test_adversarial_structure():
    n = 20000
    r_vals, k = synth.adversarial_workload(n, 1005)
    ks = synth.limbs_to_ints(k)
    zero = sum(v == 0 for v in ks) / n
    one = sum(v == 1 for v in ks) / n
    small = sum(1 < v < (1 << 64) for v in ks) / n
    assert abs(zero - 0.125) < 0.02 and abs(one - 0.125) < 0.02 and abs(small - 0.25) < 0.03
    rs = synth.limbs_to_ints(r_vals)
    assert all(0 <= v < pyref.R for v in rs)
    seen = {}
    dup = neg = 0
    for v in rs:
        if v in seen:
            dup += 1
        elif (pyref.R - v) % pyref.R in seen:
            neg += 1
        seen[v] = True
    assert abs(dup / n - 0.05) < 0.015 and abs(neg / n - 0.05) < 0.015


def test_progression():
    r_vals, k = synth.progression_workload(50, 2, scalars="ones")
    rs = synth.limbs_to_ints(r_vals)
    d = rs[1] - rs[0]
    assert all(rs[i + 1] - rs[i] == d for i in range(49))
    assert all(v == 1 for v in synth.limbs_to_ints(k))


def test_u32_layout_roundtrip():
    _, k = synth.uniform_workload(8, 1)
    u32 = synth.scalars_to_u32(k)
    assert u32.shape == (8, 8) and u32.dtype == np.uint32
    assert np.array_equal(u32.view(np.uint64).reshape(8, 4), k)
