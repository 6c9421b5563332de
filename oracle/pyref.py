"""Pure-Python reference for small BN254 G1 multi-scalar multiplications.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Affine coordinates,
Python integers, one modular inversion per group operation via ``pow``.  It is
a second, independent oracle: the C oracle uses Jacobian formulas and Barrett
reduction, this one uses the affine chord-and-tangent law, so agreement between
the two pins both.

The sum it computes is the definition of the MSM, Q = sum_i k_i * P_i, which
the pages' cross-check compares GPU results against (PR #23736, section
"Change (correct, landed)").
"""

# BN254 base-field prime and group order, from the polynomials in
# u = 4965661367192848881 (p = 36u^4+36u^3+24u^2+6u+1, r = 36u^4+36u^3+18u^2+6u+1).
U = 4965661367192848881
P = 36 * U**4 + 36 * U**3 + 24 * U**2 + 6 * U + 1
R = 36 * U**4 + 36 * U**3 + 18 * U**2 + 6 * U + 1
B = 3
G = (1, 2)
INF = None  # the point at infinity


def on_curve(pt):
    if pt is INF:
        return True
    x, y = pt
    return 0 <= x < P and 0 <= y < P and (y * y - x * x * x - B) % P == 0


def neg(pt):
    if pt is INF:
        return INF
    x, y = pt
    return (x, (-y) % P)


def add(p1, p2):
    """Affine chord-and-tangent addition on y^2 = x^3 + 3."""
    if p1 is INF:
        return p2
    if p2 is INF:
        return p1
    x1, y1 = p1
    x2, y2 = p2
    if x1 == x2:
        if (y1 + y2) % P == 0:
            return INF
        lam = (3 * x1 * x1) * pow(2 * y1, P - 2, P) % P
    else:
        lam = (y2 - y1) * pow(x2 - x1, P - 2, P) % P
    x3 = (lam * lam - x1 - x2) % P
    y3 = (lam * (x1 - x3) - y1) % P
    return (x3, y3)


def mul(k, pt):
    """[k]P by right-to-left double and add (k >= 0)."""
    acc = INF
    base = pt
    while k > 0:
        if k & 1:
            acc = add(acc, base)
        base = add(base, base)
        k >>= 1
    return acc


def mul_repeated(k, pt):
    """[k]P by k - 1 plain additions (brute force for tiny k)."""
    acc = INF
    for _ in range(k):
        acc = add(acc, pt)
    return acc


def msm(points, scalars):
    """sum_i [k_i] P_i"""
    acc = INF
    for pt, k in zip(points, scalars):
        acc = add(acc, mul(k, pt))
    return acc


def to_mont(x):
    return x * (1 << 256) % P


def from_mont(x):
    return x * pow(1 << 256, P - 2, P) % P


def jacobian_mont_to_affine(X, Y, Z):
    """Normalise a Jacobian point whose coordinates are Montgomery encoded."""
    X, Y, Z = from_mont(X), from_mont(Y), from_mont(Z)
    if Z == 0:
        return INF
    zi = pow(Z, P - 2, P)
    return (X * zi * zi % P, Y * zi * zi * zi % P)
