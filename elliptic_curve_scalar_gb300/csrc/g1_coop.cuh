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

// The operand of lane `lane` among a0 .. a5 (lanes from 5 on take a5), chosen
// by masks: nested conditionals let the compiler branch on the lane, and a
// branch would serialise the lanes' multiplications (probe: 4581 -> 4237
// cycles per cooperative doubling with masks).
__device__ __forceinline__ fe sel(int lane, const fe& a0, const fe& a1, const fe& a2 = fe(), const fe& a3 = fe(),
                                  const fe& a4 = fe(), const fe& a5 = fe()) {
    const uint32_t m0 = 0u - (uint32_t)(lane == 0), m1 = 0u - (uint32_t)(lane == 1);
    const uint32_t m2 = 0u - (uint32_t)(lane == 2), m3 = 0u - (uint32_t)(lane == 3);
    const uint32_t m4 = 0u - (uint32_t)(lane == 4), m5 = 0u - (uint32_t)(lane >= 5);
    fe r;
#pragma unroll
    for (int i = 0; i < 8; i++)
        r.v[i] = (a0.v[i] & m0) | (a1.v[i] & m1) | (a2.v[i] & m2) | (a3.v[i] & m3) | (a4.v[i] & m4) | (a5.v[i] & m5);
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

// n doublings in a row (the Horner chains of the window combination and the
// weighting of the reduction's bit sums), with the constant factors of
// dbl-2009-l moved into the products.  With B = Y^2, D = 4 X B, E = 3 X^2,
// F = E^2 and C = B^2 the doubling is X3 = F - 2D, Y3 = E (3D - F) - 8C,
// Z3 = 2 Y Z; writing 3X^2 = X (3X), 2D = (8X) B, 3D = (12X) B, 2YZ = Y (2Z)
// and 8C = C (8) as products leaves one subtraction between levels 2 and 3
// and none between levels 1 and 2:
//   level 1: E = X (3X), B = Y Y, Z3 = Y (2Z)
//   level 2: C = B B, F = E E, 2D = (8X) B, 3D = (12X) B
//   level 3: E (3D - F), 8C, and the next input's 3 X3, 8 X3, 12 X3, 2 Z3.
// Probe (one warp, 1024 doublings): 3459 cycles per doubling against 4581
// for dbl with its additions between the levels.  The multiples 3, 8, 12 and
// 2 are Montgomery-form constants, so that a product by them is the plain
// multiple.
template <int W = 32>
__device__ __forceinline__ jac dbl_n(jac p, int n) {
    if (n <= 0) return p;
    const int lane = threadIdx.x & (W - 1);
    const fe c2 = {{FQ_MONT2}}, c3 = {{FQ_MONT3}}, c8 = {{FQ_MONT8}}, c12 = {{FQ_MONT12}};
    fe m0 = fq::mul_inline(sel(lane, p.X, p.X, p.X, p.Z), sel(lane, c3, c8, c12, c2));
    fe X3 = bcast<W>(m0, 0), X8 = bcast<W>(m0, 1), X12 = bcast<W>(m0, 2), Z2 = bcast<W>(m0, 3);
    for (int i = 0; i < n; i++) {
        fe m1 = fq::mul_inline(sel(lane, p.X, p.Y, p.Y), sel(lane, X3, p.Y, Z2));
        const fe E = bcast<W>(m1, 0), B = bcast<W>(m1, 1);
        p.Z = bcast<W>(m1, 2);
        fe m2 = fq::mul_inline(sel(lane, B, E, X8, X12), sel(lane, B, E, B, B));
        const fe C = bcast<W>(m2, 0), F = bcast<W>(m2, 1), D2 = bcast<W>(m2, 2), D3 = bcast<W>(m2, 3);
        p.X = fq::sub(F, D2);
        const fe Wd = fq::sub(D3, F);
        fe m3 = fq::mul_inline(sel(lane, E, p.X, p.X, p.X, p.Z, C), sel(lane, Wd, c3, c8, c12, c2, c8));
        X3 = bcast<W>(m3, 1);
        X8 = bcast<W>(m3, 2);
        X12 = bcast<W>(m3, 3);
        Z2 = bcast<W>(m3, 4);
        p.Y = fq::sub(bcast<W>(m3, 0), bcast<W>(m3, 5));
    }
    return p;
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
