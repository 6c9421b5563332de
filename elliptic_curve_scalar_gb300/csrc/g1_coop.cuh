// g1_coop.cuh -- cooperative Jacobian point operations for latency-bound
// chains (the window combination, the bucket reduction).
//
// A group of W lanes (W = 32: the whole warp; W = 8: a quarter of it) calls
// these with the same operands.  The field multiplications of one operation
// are grouped into dependency levels; at each level lane j of the group
// computes the j-th independent multiplication and the results are broadcast
// by shuffles within the group.  SIMT lanes execute the multiplication in
// lockstep anyway, so a level costs one multiplication's latency instead of
// one per product: doubling (dbl-2009-l) takes 3 levels instead of 7
// multiplications in a row, addition (add-2007-bl) and mixed addition
// (madd-2007-bl) 5 levels instead of 16 and 11.  Branches depend only on the
// group's operands, so a group never diverges, and every shuffle names only
// the group's lanes: groups of one warp may take different branches.  The
// multiplications are inlined: these functions run in latency chains, where
// the call's argument moves sit on the critical path (n = 2^10: combination
// 0.395 -> 0.362 ms when inlined).
#pragma once
#include "g1.cuh"

namespace g1c {

using fq::fe;
using g1::jac;

constexpr unsigned FULL = 0xffffffffu;

// the lanes of the calling thread's group of W (a power of two, 8 .. 32)
template <int W>
__device__ __forceinline__ unsigned group_mask() {
    return W == 32 ? FULL : ((1u << W) - 1) << ((threadIdx.x & 31) & ~(W - 1));
}

template <int W = 32>
__device__ __forceinline__ fe bcast(const fe& a, int src) {
    const unsigned m = group_mask<W>();
    fe r;
#pragma unroll
    for (int i = 0; i < 8; i++) r.v[i] = __shfl_sync(m, a.v[i], src, W);
    return r;
}

__device__ __forceinline__ fe sel(int lane, const fe& a0, const fe& a1, const fe& a2, const fe& a3 = fe(),
                                  const fe& a4 = fe()) {
    fe r;
#pragma unroll
    for (int i = 0; i < 8; i++)
        r.v[i] = lane == 0 ? a0.v[i] : lane == 1 ? a1.v[i] : lane == 2 ? a2.v[i] : lane == 3 ? a3.v[i] : a4.v[i];
    return r;
}

// dbl-2009-l, a = 0
template <int W = 32>
__device__ __forceinline__ jac dbl(const jac& p) {
    const int lane = threadIdx.x & (W - 1);
    // level 1: A = X^2, B = Y^2, YZ
    fe m1 = fq::mul_inline(sel(lane, p.X, p.Y, p.Y, p.X, p.X), sel(lane, p.X, p.Y, p.Z, p.X, p.X));
    fe A = bcast<W>(m1, 0), B = bcast<W>(m1, 1), YZ = bcast<W>(m1, 2);
    fe E = fq::add(fq::dbl(A), A);
    fe XB = fq::add(p.X, B);
    // level 2: C = B^2, (X + B)^2, F = E^2
    fe s2 = sel(lane, B, XB, E, B, B);
    fe m2 = fq::mul_inline(s2, s2);
    fe C = bcast<W>(m2, 0), U = bcast<W>(m2, 1), F = bcast<W>(m2, 2);
    fe D = fq::dbl(fq::sub(fq::sub(U, A), C));
    jac r;
    r.X = fq::sub(F, fq::dbl(D));
    // level 3: Y3 = E (D - X3) - 8C
    fe C8 = fq::dbl(fq::dbl(fq::dbl(C)));
    r.Y = fq::sub(fq::mul_inline(E, fq::sub(D, r.X)), C8);
    r.Z = fq::dbl(YZ);
    return r;
}

// add-2007-bl, with equal / opposite / infinite operands handled
template <int W = 32>
__device__ __forceinline__ jac add(const jac& p, const jac& q) {
    if (g1::is_inf(p)) return q;
    if (g1::is_inf(q)) return p;
    const int lane = threadIdx.x & (W - 1);
    // level 1: Z1^2, Z2^2, (Z1 + Z2)^2
    fe ZZ = fq::add(p.Z, q.Z);
    fe s1 = sel(lane, p.Z, q.Z, ZZ, p.Z, p.Z);
    fe m1 = fq::mul_inline(s1, s1);
    fe Z1Z1 = bcast<W>(m1, 0), Z2Z2 = bcast<W>(m1, 1), ZZ2 = bcast<W>(m1, 2);
    // level 2: U1 = X1 Z2Z2, U2 = X2 Z1Z1, Z2 Z2Z2, Z1 Z1Z1
    fe m2 = fq::mul_inline(sel(lane, p.X, q.X, q.Z, p.Z, p.X), sel(lane, Z2Z2, Z1Z1, Z2Z2, Z1Z1, Z2Z2));
    fe U1 = bcast<W>(m2, 0), U2 = bcast<W>(m2, 1), T1 = bcast<W>(m2, 2), T2 = bcast<W>(m2, 3);
    fe H = fq::sub(U2, U1);
    fe H2 = fq::dbl(H);
    // level 3: S1 = Y1 T1, S2 = Y2 T2, I = (2H)^2
    fe m3 = fq::mul_inline(sel(lane, p.Y, q.Y, H2, p.Y, p.Y), sel(lane, T1, T2, H2, T1, T1));
    fe S1 = bcast<W>(m3, 0), S2 = bcast<W>(m3, 1), I = bcast<W>(m3, 2);
    fe rr = fq::sub(S2, S1);
    if (fq::is_zero(H)) {
        if (fq::is_zero(rr)) return g1c::dbl<W>(p);
        return g1::jac_inf();
    }
    rr = fq::dbl(rr);
    fe Zs = fq::sub(fq::sub(ZZ2, Z1Z1), Z2Z2);
    // level 4: J = H I, V = U1 I, r^2, Z3 = (W - Z1Z1 - Z2Z2) H
    fe m4 = fq::mul_inline(sel(lane, H, U1, rr, Zs, H), sel(lane, I, I, rr, H, I));
    fe J = bcast<W>(m4, 0), V = bcast<W>(m4, 1), R2 = bcast<W>(m4, 2);
    jac r;
    r.Z = bcast<W>(m4, 3);
    r.X = fq::sub(fq::sub(R2, J), fq::dbl(V));
    // level 5: r (V - X3), S1 J
    fe m5 = fq::mul_inline(sel(lane, rr, S1, rr, rr, rr), sel(lane, fq::sub(V, r.X), J, J, J, J));
    fe a = bcast<W>(m5, 0), b = bcast<W>(m5, 1);
    r.Y = fq::sub(a, fq::dbl(b));
    return r;
}

// madd-2007-bl (Jacobian + affine), with equal / opposite / infinite operands
// handled; Z3 = (Z1 + H)^2 - Z1Z1 - HH is taken as the product 2 Z1 H.
template <int W = 32>
__device__ __forceinline__ jac add_mixed(const jac& p, const g1::aff& q) {
    if (g1::is_inf(q)) return p;
    if (g1::is_inf(p)) return g1::to_jac(q);
    const int lane = threadIdx.x & (W - 1);
    // level 1: Z1Z1 = Z1^2, Z1 y2
    fe m1 = fq::mul_inline(p.Z, sel(lane, p.Z, q.y, p.Z, p.Z, p.Z));
    const fe Z1Z1 = bcast<W>(m1, 0), Z1y2 = bcast<W>(m1, 1);
    // level 2: U2 = x2 Z1Z1, S2 = Z1 y2 Z1Z1
    fe m2 = fq::mul_inline(sel(lane, q.x, Z1y2, q.x, q.x, q.x), Z1Z1);
    const fe H = fq::sub(bcast<W>(m2, 0), p.X);
    fe rr = fq::sub(bcast<W>(m2, 1), p.Y);
    if (fq::is_zero(H)) {
        if (fq::is_zero(rr)) return g1c::dbl<W>(p);
        return g1::jac_inf();
    }
    rr = fq::dbl(rr);
    // level 3: HH = H^2, Z1 H, r^2
    fe m3 = fq::mul_inline(sel(lane, H, p.Z, rr, H, H), sel(lane, H, H, rr, H, H));
    const fe HH = bcast<W>(m3, 0), Z1H = bcast<W>(m3, 1), R2 = bcast<W>(m3, 2);
    const fe I = fq::dbl(fq::dbl(HH));
    // level 4: J = H I, V = X1 I
    fe m4 = fq::mul_inline(sel(lane, H, p.X, H, H, H), I);
    const fe J = bcast<W>(m4, 0), V = bcast<W>(m4, 1);
    jac r;
    r.X = fq::sub(fq::sub(R2, J), fq::dbl(V));
    r.Z = fq::dbl(Z1H);
    // level 5: r (V - X3), Y1 J
    fe m5 = fq::mul_inline(sel(lane, rr, p.Y, rr, rr, rr), sel(lane, fq::sub(V, r.X), J, J, J, J));
    r.Y = fq::sub(bcast<W>(m5, 0), fq::dbl(bcast<W>(m5, 1)));
    return r;
}

// W = 1 selects the one-thread operations of g1.cuh, W >= 8 the cooperative
// ones: kernels that are latency-bound only when they have few units of work
// take W as a template parameter.
template <int W>
__device__ __forceinline__ jac add_w(const jac& p, const jac& q) {
    if constexpr (W == 1) return g1::add(p, q);
    else return g1c::add<W>(p, q);
}
template <int W>
__device__ __forceinline__ jac add_mixed_w(const jac& p, const g1::aff& q) {
    if constexpr (W == 1) return g1::add_mixed(p, q);
    else return g1c::add_mixed<W>(p, q);
}

}  // namespace g1c
