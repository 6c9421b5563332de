// g1_coop.cuh -- warp-cooperative Jacobian point operations for latency-bound
// chains (the window combination).
//
// All 32 lanes call these with the same operands.  The field multiplications
// of one operation are grouped into dependency levels; at each level lane j
// computes the j-th independent multiplication and the results are broadcast
// by shuffles.  SIMT lanes execute the multiplication in lockstep anyway, so a
// level costs one multiplication's latency instead of one per product:
// doubling (dbl-2009-l) takes 3 levels instead of 7 multiplications in a row,
// addition (add-2007-bl) 5 levels instead of 16.  Branches depend only on the
// (warp-uniform) operands, so lanes never diverge.  The multiplications are
// inlined: these functions run in single-warp latency chains, where the call's
// argument moves sit on the critical path (n = 2^10: combination 0.395 ->
// 0.362 ms when inlined).
#pragma once
#include "g1.cuh"

namespace g1c {

using fq::fe;
using g1::jac;

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ fe bcast(const fe& a, int src) {
    fe r;
#pragma unroll
    for (int i = 0; i < 8; i++) r.v[i] = __shfl_sync(FULL, a.v[i], src);
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
__device__ __forceinline__ jac dbl(const jac& p) {
    const int lane = threadIdx.x & 31;
    // level 1: A = X^2, B = Y^2, YZ
    fe m1 = fq::mul_inline(sel(lane, p.X, p.Y, p.Y, p.X, p.X), sel(lane, p.X, p.Y, p.Z, p.X, p.X));
    fe A = bcast(m1, 0), B = bcast(m1, 1), YZ = bcast(m1, 2);
    fe E = fq::add(fq::dbl(A), A);
    fe XB = fq::add(p.X, B);
    // level 2: C = B^2, (X + B)^2, F = E^2
    fe s2 = sel(lane, B, XB, E, B, B);
    fe m2 = fq::mul_inline(s2, s2);
    fe C = bcast(m2, 0), U = bcast(m2, 1), F = bcast(m2, 2);
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
__device__ __forceinline__ jac add(const jac& p, const jac& q) {
    if (g1::is_inf(p)) return q;
    if (g1::is_inf(q)) return p;
    const int lane = threadIdx.x & 31;
    // level 1: Z1^2, Z2^2, (Z1 + Z2)^2
    fe ZZ = fq::add(p.Z, q.Z);
    fe s1 = sel(lane, p.Z, q.Z, ZZ, p.Z, p.Z);
    fe m1 = fq::mul_inline(s1, s1);
    fe Z1Z1 = bcast(m1, 0), Z2Z2 = bcast(m1, 1), W = bcast(m1, 2);
    // level 2: U1 = X1 Z2Z2, U2 = X2 Z1Z1, Z2 Z2Z2, Z1 Z1Z1
    fe m2 = fq::mul_inline(sel(lane, p.X, q.X, q.Z, p.Z, p.X), sel(lane, Z2Z2, Z1Z1, Z2Z2, Z1Z1, Z2Z2));
    fe U1 = bcast(m2, 0), U2 = bcast(m2, 1), T1 = bcast(m2, 2), T2 = bcast(m2, 3);
    fe H = fq::sub(U2, U1);
    fe H2 = fq::dbl(H);
    // level 3: S1 = Y1 T1, S2 = Y2 T2, I = (2H)^2
    fe m3 = fq::mul_inline(sel(lane, p.Y, q.Y, H2, p.Y, p.Y), sel(lane, T1, T2, H2, T1, T1));
    fe S1 = bcast(m3, 0), S2 = bcast(m3, 1), I = bcast(m3, 2);
    fe rr = fq::sub(S2, S1);
    if (fq::is_zero(H)) {
        if (fq::is_zero(rr)) return g1c::dbl(p);
        return g1::jac_inf();
    }
    rr = fq::dbl(rr);
    fe Zs = fq::sub(fq::sub(W, Z1Z1), Z2Z2);
    // level 4: J = H I, V = U1 I, r^2, Z3 = (W - Z1Z1 - Z2Z2) H
    fe m4 = fq::mul_inline(sel(lane, H, U1, rr, Zs, H), sel(lane, I, I, rr, H, I));
    fe J = bcast(m4, 0), V = bcast(m4, 1), R2 = bcast(m4, 2);
    jac r;
    r.Z = bcast(m4, 3);
    r.X = fq::sub(fq::sub(R2, J), fq::dbl(V));
    // level 5: r (V - X3), S1 J
    fe m5 = fq::mul_inline(sel(lane, rr, S1, rr, rr, rr), sel(lane, fq::sub(V, r.X), J, J, J, J));
    fe a = bcast(m5, 0), b = bcast(m5, 1);
    r.Y = fq::sub(a, fq::dbl(b));
    return r;
}

}  // namespace g1c
