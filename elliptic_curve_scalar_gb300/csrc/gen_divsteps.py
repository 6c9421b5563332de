"""Write divstep_table.cuh: the transition of four safegcd divsteps as a table.

One divstep (Bernstein and Yang, "Fast constant-time gcd computation and
modular inversion", TCHES 2019) maps (delta, f, g), f odd, to
    delta > 0 and g odd:  (1 - delta, g, (g - f)/2)
    g odd otherwise:      (1 + delta, f, (g + f)/2)
    g even:               (1 + delta, f, g/2).
Four of them depend only on delta and on f and g mod 16: the decisions of
step i read bit i of values built from the low four bits.  The table maps
(delta, f mod 16, g mod 16) to the 2x2 matrix B with
    16 (f', g') = (u f + v g, q f + r g),   |u| + |v|, |q| + |r| <= 16,
and to delta' = s delta + t.  delta enters clamped to [-4, 4]: every
delta <= -4 takes no swap within four steps (delta' = delta + 4), and every
delta >= 4 swaps at the first odd g and never again (delta' = 4 - delta - 2j
for a swap at step j), so the clamped entry with its (s, t) is exact for the
whole range.

Entry layout (one 32-bit word): bits 0-5 u, 6-11 v, 12-17 q, 18-23 r (6-bit
two's complement), bit 24 s (1: delta' starts from -delta), bits 25-29 t
(5-bit two's complement).  Index: ((clamp(delta) + 4) * 8 + (f mod 16) / 2)
* 16 + g mod 16, 1152 entries.

Run from the repository root: python elliptic_curve_scalar_gb300/csrc/gen_divsteps.py
"""
import os
import random

K = 4


def step(delta, f, g, u, v, q, r):
    """one divstep as inv.cuh applies it, on exact integers, with the row
    matrix (u, v | q, r) kept so that 2^s (f_s, g_s) = (u f_0 + v g_0, q f_0 + r g_0)"""
    c1 = delta > 0
    c2 = g & 1
    if c2:
        if c1:
            g, q, r = g - f, q - u, r - v
        else:
            g, q, r = g + f, q + u, r + v
    swap = c1 and c2
    delta = (1 - delta) if swap else (delta + 1)
    if swap:
        f, u, v = f + g, u + q, v + r
    assert g % 2 == 0
    return delta, f, g // 2, 2 * u, 2 * v, q, r


def entry(dstate, fl, gl):
    """(u, v, q, r, s, t) for delta state dstate in [-4, 4], f mod 16 = fl, g mod 16 = gl"""
    delta, f, g, u, v, q, r = dstate, fl, gl, 1, 0, 0, 1
    swap_at = None
    for j in range(K):
        d0 = delta
        delta, f, g, u, v, q, r = step(delta, f, g, u, v, q, r)
        if d0 > 0 and (delta == 1 - d0) and swap_at is None:
            swap_at = j
    if dstate <= -K:
        s, t = 1, K
    elif dstate >= K:
        s, t = (-1, K - 2 * swap_at) if swap_at is not None else (1, K)
    else:
        s, t = 1, delta - dstate
    return u, v, q, r, s, t


def pack(u, v, q, r, s, t):
    for x in (u, v, q, r):
        assert -32 <= x < 32
    assert -16 <= t < 16
    return ((u & 63) | (v & 63) << 6 | (q & 63) << 12 | (r & 63) << 18 | (1 if s < 0 else 0) << 24
            | (t & 31) << 25)


def table():
    tab = []
    for ds in range(-K, K + 1):
        for fh in range(8):
            for gl in range(16):
                tab.append(entry(ds, 2 * fh + 1, gl))
    return tab


def check(tab, trials=200000, seed=7):
    """every entry against four exact divsteps on random full-size f, g and
    delta anywhere in its clamped range"""
    rng = random.Random(seed)
    for _ in range(trials):
        f = rng.getrandbits(64) | 1
        g = rng.getrandbits(64) - (1 << 63)
        f = f if rng.random() < 0.5 else -f
        delta = rng.choice([rng.randint(-K + 1, K - 1), rng.randint(-1000, -K), rng.randint(K, 1000)])
        ds = max(-K, min(K, delta))
        u, v, q, r, s, t = tab[((ds + K) * 8 + (f % 16) // 2) * 16 + g % 16]
        d, ff, gg, uu, vv, qq, rr = delta, f, g, 1, 0, 0, 1
        for _ in range(K):
            d, ff, gg, uu, vv, qq, rr = step(d, ff, gg, uu, vv, qq, rr)
        assert (uu, vv, qq, rr) == (u, v, q, r), (delta, f, g)
        assert 16 * ff == u * f + v * g and 16 * gg == q * f + r * g
        assert d == s * delta + t, (delta, f, g, d, s, t)


def render(tab):
    words = [pack(*e) for e in tab]
    lines = ["// divstep_table.cuh -- written by gen_divsteps.py; do not edit.",
             "// Four safegcd divsteps per entry: see gen_divsteps.py for the layout.",
             "#pragma once", "#include <stdint.h>", "", "namespace inv {", "",
             "constexpr int kDivTabEntries = %d;" % len(words), "",
             "static __device__ const uint32_t kDivTab[%d] = {" % len(words)]
    for i in range(0, len(words), 8):
        lines.append("    " + ", ".join("0x%08xu" % w for w in words[i:i + 8]) + ",")
    lines += ["};", "", "}  // namespace inv", ""]
    return "\n".join(lines)


if __name__ == "__main__":
    tab = table()
    check(tab)
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "divstep_table.cuh"), "w") as out:
        out.write(render(tab))
