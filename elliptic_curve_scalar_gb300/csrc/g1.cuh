// g1.cuh -- BN254 G1 point arithmetic (y^2 = x^3 + 3 over F_p) on sm_103a.
//
// Affine points (x, y) in Montgomery form; the point at infinity is (0, 0).
// No curve point has x = 0 because 3 is not a square mod p, so "x == 0" is the
// infinity test.  Jacobian points (X, Y, Z) represent (X/Z^2, Y/Z^3); Z = 0 is
// infinity.  Formulas are the a = 0 entries of the Explicit-Formulas Database
// (Bernstein-Lange, hyperelliptic.org/EFD): dbl-2009-l, madd-2007-bl and
// add-2007-bl, with the exceptional inputs (equal points, opposite points,
// infinity) handled explicitly because those formulas do not cover them.
#pragma once
#include "fq.cuh"
#include "inv.cuh"

namespace g1 {

using fq::fe;

struct aff {
    fe x, y;
};

struct jac {
    fe X, Y, Z;
};

__device__ __forceinline__ bool is_inf(const aff& p) { return fq::is_zero(p.x); }
__device__ __forceinline__ bool is_inf(const jac& p) { return fq::is_zero(p.Z); }

__device__ __forceinline__ aff aff_inf() { return aff{fq::zero(), fq::zero()}; }
__device__ __forceinline__ jac jac_inf() { return jac{fq::one(), fq::one(), fq::zero()}; }

__device__ __forceinline__ jac to_jac(const aff& p) {
    if (is_inf(p)) return jac_inf();
    return jac{p.x, p.y, fq::one()};
}

// dbl-2009-l: A = X^2, B = Y^2, C = B^2, D = 2((X+B)^2 - A - C), E = 3A,
// F = E^2, X3 = F - 2D, Y3 = E(D - X3) - 8C, Z3 = 2YZ.  Infinity maps to
// infinity (Z3 = 0); no finite point has Y = 0.
__device__ __forceinline__ jac dbl(const jac& p) {
    fe A = fq::sqr(p.X);
    fe B = fq::sqr(p.Y);
    fe C = fq::sqr(B);
    fe D = fq::sub(fq::sub(fq::sqr(fq::add(p.X, B)), A), C);
    D = fq::dbl(D);
    fe E = fq::add(fq::dbl(A), A);
    fe F = fq::sqr(E);
    jac r;
    r.X = fq::sub(F, fq::dbl(D));
    fe C8 = fq::dbl(fq::dbl(fq::dbl(C)));
    r.Y = fq::sub(fq::mul(E, fq::sub(D, r.X)), C8);
    r.Z = fq::dbl(fq::mul(p.Y, p.Z));
    return r;
}

// madd-2007-bl (Jacobian + affine): Z1Z1 = Z1^2, U2 = X2 Z1Z1, S2 = Y2 Z1 Z1Z1,
// H = U2 - X1, HH = H^2, I = 4HH, J = H I, r = 2(S2 - Y1), V = X1 I,
// X3 = r^2 - J - 2V, Y3 = r(V - X3) - 2 Y1 J, Z3 = (Z1 + H)^2 - Z1Z1 - HH.
__device__ __forceinline__ jac add_mixed(const jac& p, const aff& q) {
    if (is_inf(q)) return p;
    if (is_inf(p)) return to_jac(q);
    fe Z1Z1 = fq::sqr(p.Z);
    fe U2 = fq::mul(q.x, Z1Z1);
    fe S2 = fq::mul(q.y, fq::mul(p.Z, Z1Z1));
    fe H = fq::sub(U2, p.X);
    fe rr = fq::sub(S2, p.Y);
    if (fq::is_zero(H)) {
        if (fq::is_zero(rr)) return dbl(p);
        return jac_inf();
    }
    rr = fq::dbl(rr);
    fe HH = fq::sqr(H);
    fe I = fq::dbl(fq::dbl(HH));
    fe J = fq::mul(H, I);
    fe V = fq::mul(p.X, I);
    jac r;
    r.X = fq::sub(fq::sub(fq::sqr(rr), J), fq::dbl(V));
    r.Y = fq::sub(fq::mul(rr, fq::sub(V, r.X)), fq::dbl(fq::mul(p.Y, J)));
    r.Z = fq::sub(fq::sub(fq::sqr(fq::add(p.Z, H)), Z1Z1), HH);
    return r;
}

// mmadd-2007-bl (affine + affine, Z1 = Z2 = 1): H = x2 - x1, HH = H^2,
// I = 4HH, J = H I, r = 2(y2 - y1), V = x1 I, X3 = r^2 - J - 2V,
// Y3 = r(V - X3) - 2 y1 J, Z3 = 2H: 4M + 2S where the mixed addition of the
// second point onto the first takes 7M + 4S.
__device__ __forceinline__ jac add_aff(const aff& p, const aff& q) {
    if (is_inf(p)) return to_jac(q);
    if (is_inf(q)) return to_jac(p);
    fe H = fq::sub(q.x, p.x);
    fe rr = fq::sub(q.y, p.y);
    if (fq::is_zero(H)) {
        if (fq::is_zero(rr)) return dbl(to_jac(p));
        return jac_inf();
    }
    rr = fq::dbl(rr);
    fe I = fq::dbl(fq::dbl(fq::sqr(H)));
    fe J = fq::mul(H, I);
    fe V = fq::mul(p.x, I);
    jac r;
    r.X = fq::sub(fq::sub(fq::sqr(rr), J), fq::dbl(V));
    r.Y = fq::sub(fq::mul(rr, fq::sub(V, r.X)), fq::dbl(fq::mul(p.y, J)));
    r.Z = fq::dbl(H);
    return r;
}

// add-2007-bl (Jacobian + Jacobian): Z1Z1 = Z1^2, Z2Z2 = Z2^2, U1 = X1 Z2Z2,
// U2 = X2 Z1Z1, S1 = Y1 Z2 Z2Z2, S2 = Y2 Z1 Z1Z1, H = U2 - U1, I = (2H)^2,
// J = H I, r = 2(S2 - S1), V = U1 I, X3 = r^2 - J - 2V,
// Y3 = r(V - X3) - 2 S1 J, Z3 = ((Z1 + Z2)^2 - Z1Z1 - Z2Z2) H.
__device__ __forceinline__ jac add(const jac& p, const jac& q) {
    if (is_inf(p)) return q;
    if (is_inf(q)) return p;
    fe Z1Z1 = fq::sqr(p.Z);
    fe Z2Z2 = fq::sqr(q.Z);
    fe U1 = fq::mul(p.X, Z2Z2);
    fe U2 = fq::mul(q.X, Z1Z1);
    fe S1 = fq::mul(p.Y, fq::mul(q.Z, Z2Z2));
    fe S2 = fq::mul(q.Y, fq::mul(p.Z, Z1Z1));
    fe H = fq::sub(U2, U1);
    fe rr = fq::sub(S2, S1);
    if (fq::is_zero(H)) {
        if (fq::is_zero(rr)) return dbl(p);
        return jac_inf();
    }
    fe I = fq::sqr(fq::dbl(H));
    fe J = fq::mul(H, I);
    rr = fq::dbl(rr);
    fe V = fq::mul(U1, I);
    jac r;
    r.X = fq::sub(fq::sub(fq::sqr(rr), J), fq::dbl(V));
    r.Y = fq::sub(fq::mul(rr, fq::sub(V, r.X)), fq::dbl(fq::mul(S1, J)));
    r.Z = fq::mul(fq::sub(fq::sub(fq::sqr(fq::add(p.Z, q.Z)), Z1Z1), Z2Z2), H);
    return r;
}

// Jacobian -> affine with one field inversion (infinity -> (0, 0)).
__device__ __forceinline__ aff to_aff(const jac& p) {
    if (is_inf(p)) return aff_inf();
    fe zi = inv::inv_safegcd(p.Z);
    fe zi2 = fq::sqr(zi);
    return aff{fq::mul(p.X, zi2), fq::mul(p.Y, fq::mul(zi2, zi))};
}

__device__ __forceinline__ aff load_aff(const uint32_t* p) { return aff{fq::load(p), fq::load(p + 8)}; }
__device__ __forceinline__ void store_aff(uint32_t* p, const aff& a) {
    fq::store(p, a.x);
    fq::store(p + 8, a.y);
}
__device__ __forceinline__ jac load_jac(const uint32_t* p) { return jac{fq::load(p), fq::load(p + 8), fq::load(p + 16)}; }
__device__ __forceinline__ void store_jac(uint32_t* p, const jac& a) {
    fq::store(p, a.X);
    fq::store(p + 8, a.Y);
    fq::store(p + 16, a.Z);
}

}  // namespace g1
