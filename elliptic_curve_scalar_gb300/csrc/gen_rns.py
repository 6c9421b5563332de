"""Write rns_consts.cuh: the constants of the residue number system (RNS) in
which the library runs its long Jacobian chains (the window combination and
the bucket reduction's shifts).

An RNS represents an integer X by its residues modulo pairwise coprime
moduli.  Additions and multiplications act on each residue alone, so 19
lanes of a warp can multiply two field elements with one 32-bit product
each instead of one lane running a 256-bit multi-precision product.  Field
multiplication uses Montgomery's method in RNS form (Bajard, Didier and
Kornerup, "An RNS Montgomery modular multiplication algorithm", IEEE Trans.
Computers 47(7), 1998; the exact second base extension with a redundant
modulus follows Shenoy and Kumaresan, "Fast base extension using a redundant
modulus in RNS", IEEE Trans. Computers 38(2), 1989):

  base B  = 9 primes m_j = 2^32 - c_j,  M  = prod m_j  (~2^288)
  base B' = 9 more primes,              M' = prod m'_j
  redundant modulus m_r = 2^32

  MM(A, B) = A B M^-1 mod p, lazily (see rns.cuh for the bounds).

The product's first step multiplies the two B residues and then by the
constant c1_j = -p^-1 (M/m_j)^-1 mod m_j.  B is chosen (the first set of 9
primes 2^32 - c, in lexicographic order over the 24 smallest c, for which
every c1_j is a square mod m_j) so that the B residues can be stored scaled
by lambda_j = sqrt(c1_j): then x' y' = x y c1 and the step is one product.
Every constant that makes or reads a B residue carries the scale.

A lane of a 10-lane group holds two residue slots: lane j < 9 the B channel
m_j (slot a, scaled by lambda_j) and the B' channel m'_j (slot b); lane 9 the
redundant channel 2^32 in both slots (unscaled).  The per-lane constants are
laid out as struct Lane in rns.cuh, lane j at index j.

Run from the repository root: python elliptic_curve_scalar_gb300/csrc/gen_rns.py
"""
import itertools
import os

P = 0x30644e72e131a029b85045b68181585d97816a916871ca8d3c208c16d87cfd47
R = 1 << 256  # the positional Montgomery radix of fq.cuh
NB = 9


def is_prime(n):
    if n < 2:
        return False
    for q in (2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37):
        if n % q == 0:
            return n == q
    d, s = n - 1, 0
    while d % 2 == 0:
        d //= 2
        s += 1
    for a in (2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37):  # deterministic below 3.3e24
        x = pow(a, d, n)
        if x in (1, n - 1):
            continue
        for _ in range(s - 1):
            x = x * x % n
            if x == n - 1:
                break
        else:
            return False
    return True


def sqrt_mod(a, m):
    """a square root of the quadratic residue a modulo the odd prime m (Tonelli-Shanks)"""
    a %= m
    if a == 0:
        return 0
    assert pow(a, (m - 1) // 2, m) == 1
    q, s = m - 1, 0
    while q % 2 == 0:
        q //= 2
        s += 1
    z = 2
    while pow(z, (m - 1) // 2, m) != m - 1:
        z += 1
    mm, c, t, r = s, pow(z, q, m), pow(a, q, m), pow(a, (q + 1) // 2, m)
    while t != 1:
        i, t2 = 0, t
        while t2 != 1:
            t2 = t2 * t2 % m
            i += 1
        b = pow(c, 1 << (mm - i - 1), m)
        mm, c, t, r = i, b * b % m, t * b * b % m, r * b % m
    assert r * r % m == a
    return r


def c1_of(ms):
    M = 1
    for m in ms:
        M *= m
    return [(-pow(P, -1, m) * pow(M // m, -1, m)) % m for m in ms]


def moduli():
    cs = []
    c = 1
    while len(cs) < 24:
        if is_prime((1 << 32) - c):
            cs.append(c)
        c += 2
    for pick in itertools.combinations(range(24), NB):
        ms = [(1 << 32) - cs[i] for i in pick]
        if all(pow(v, (m - 1) // 2, m) == 1 for v, m in zip(c1_of(ms), ms)):
            ca = [cs[i] for i in pick]
            cb = [c for c in cs if c not in ca][:NB]
            return ca, cb
    raise RuntimeError("no base with square first-step constants")


def lanes():
    ca, cb = moduli()
    ma = [(1 << 32) - c for c in ca]
    mb = [(1 << 32) - c for c in cb]
    assert max(ca + cb) < (1 << 11)  # the folds of rns.cuh assume c < 2^11
    M = 1
    for m in ma:
        M *= m
    Mp = 1
    for m in mb:
        Mp *= m
    mr = 1 << 32
    assert M > 2 ** 287 and Mp > 2 ** 287
    c1 = c1_of(ma)
    out = []
    for j in range(10):
        if j < NB:
            a_m, a_c, b_m, b_c = ma[j], ca[j], mb[j], cb[j]
            lam = sqrt_mod(c1[j], a_m)
        else:
            a_m, a_c, b_m, b_c = mr, 0, mr, 0
            lam = 1
        lami = pow(lam, -1, a_m)
        L = {"ca": a_c, "cb": b_c}
        # fast extension of q from B to the slot-b channel: (M/m_i) mod m_b
        L["e1"] = [(M // ma[i]) % b_m for i in range(NB)]
        # r = (t + q p) M^-1 and xi' = r (M'/m'_j)^-1 in the slot-b channel
        L["pb"] = P % b_m
        L["minv"] = pow(M, -1, b_m)
        L["minvc2"] = (pow(M, -1, b_m) * pow(Mp // b_m, -1, b_m)) % b_m if j < NB else 0
        # exact extension back to the slot-a channel, scaled: (M'/m'_i) lambda, M' lambda
        L["e2"] = [(Mp // mb[i]) * lam % a_m for i in range(NB)]
        L["mpa"] = Mp * lam % a_m
        L["mpinv"] = pow(Mp, -1, mr) if j == NB else 0  # beta in the redundant lane
        # zero test and CRT read the scaled residue: lambda^-1 p^-1, lambda^-1 (M/m_j)^-1
        L["pinv"] = pow(P, -1, a_m) * lami % a_m
        L["crt"] = pow(M // a_m, -1, a_m) * lami % a_m if j < NB else 0
        # p for subtraction offsets (scaled in slot a)
        L["pa"] = P * lam % a_m
        # positional -> residues: 2^(32 k) mod m, k = 0..7 (scaled in slot a)
        L["pow_a"] = [pow(2, 32 * k, a_m) * lam % a_m for k in range(8)]
        L["pow_b"] = [pow(2, 32 * k, b_m) for k in range(8)]
        # domain constants (integers < p): into the RNS Montgomery domain
        # (X = x M mod p from x~ = x R mod p: MM(x~, M^2 R^-1)), out of it (MM(X, R) = x R)
        cin = M * M * pow(R, -1, P) % P
        cout = R % P
        L["cin_a"], L["cin_b"] = cin * lam % a_m, cin % b_m
        L["cout_a"], L["cout_b"] = cout * lam % a_m, cout % b_m
        # moduli for the lazy subtraction offsets
        L["ma"], L["mb"] = a_m & 0xFFFFFFFF, b_m & 0xFFFFFFFF
        out.append(L)
    return out, ma, mb, M, Mp


def words(x, n):
    return [(x >> (32 * i)) & 0xFFFFFFFF for i in range(n)]


def render():
    L, ma, mb, M, Mp = lanes()
    fields = ["ca", "cb", "ma", "mb", "pb", "minv", "minvc2", "mpa", "mpinv", "pinv", "pa", "crt", "cin_a", "cin_b",
              "cout_a", "cout_b"]
    lines = ["// rns_consts.cuh -- written by gen_rns.py; do not edit.",
             "// Residue-number-system constants for rns.cuh: base B c = %s," % ca_str(ma),
             "// base B' c = %s, redundant modulus 2^32." % ca_str(mb),
             "#pragma once", "#include <stdint.h>", "", "namespace rns {", "",
             "constexpr int kChannels = %d;  // moduli per base" % NB, ""]
    lines.append("// per lane of a 10-lane group (struct RnsLane in rns.cuh)")
    lines.append("static __device__ const uint32_t kLane[10][%d] = {" % (len(fields) + 9 + 9 + 8 + 8))
    for j in range(10):
        vals = [L[j][f] for f in fields] + L[j]["e1"] + L[j]["e2"] + L[j]["pow_a"] + L[j]["pow_b"]
        lines.append("    {" + ", ".join("0x%08xu" % v for v in vals) + "},")
    lines.append("};")
    lines.append("")
    lines.append("// M / m_i (i < 9) and M, 10 x 32-bit words each, for the CRT back to positional form")
    lines.append("static __constant__ uint32_t kMdiv[9][10] = {")
    for i in range(NB):
        lines.append("    {" + ", ".join("0x%08xu" % v for v in words(M // ma[i], 10)) + "},")
    lines.append("};")
    lines.append("static __constant__ uint32_t kM[10] = {" + ", ".join("0x%08xu" % v for v in words(M, 10)) + "};")
    lines.append("// 16p, 8p, 4p, 2p, p in 9 words: the final reduction of an integer below 32p")
    lines.append("static __constant__ uint32_t kPmul[5][9] = {")
    for k in (16, 8, 4, 2, 1):
        lines.append("    {" + ", ".join("0x%08xu" % v for v in words(k * P, 9)) + "},")
    lines.append("};")
    lines += ["", "}  // namespace rns", ""]
    return "\n".join(lines)


def ca_str(ms):
    return "{" + ", ".join(str((1 << 32) - m) for m in ms) + "}"


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "rns_consts.cuh"), "w") as f:
        f.write(render())
