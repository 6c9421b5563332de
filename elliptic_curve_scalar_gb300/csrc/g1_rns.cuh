// g1_rns.cuh -- Jacobian point chains in the residue number system of
// rns.cuh, for the latency-bound tails of the MSM: the window combination's
// Horner chain (about 115 doublings after the top window's sum is known) and
// the bucket reduction's shifts.
//
// Each dependency level of a point formula is one mm3 round: the warp's
// three 10-lane groups compute three products at once and exchange them.
// A doubling (dbl-2009-l, a = 0) is three rounds, an addition (add-2007-bl)
// six.  Field additions and small multiples act on residues alone.  Values
// keep the bounds rns.cuh requires; each function states its own.
//
// Points enter from positional Jacobian form (fq.cuh, Montgomery radix R)
// and leave in it, canonical, so the rest of the MSM never sees residues.
// Infinity is the caller's business: these functions take finite points.
// An addition whose operands have equal x (P1 = +-P2: H = 0) is reported,
// not computed; the caller then adds the points in positional form.
#pragma once
#include "g1_coop.cuh"
#include "rns.cuh"

namespace g1r {

using rns::Ctx;
using rns::rv;

struct rjac {
    rv X, Y, Z;
};

// positional Jacobian (every lane the same) -> RNS; each coordinate below 20 p
__device__ __forceinline__ rjac to_rns(const Ctx& C, const g1::jac& p) {
    const rv c = rns::cin(C);
    rjac r;
    rns::mm3(C, rns::residues(C, p.X), c, rns::residues(C, p.Y), c, rns::residues(C, p.Z), c, r.X, r.Y, r.Z);
    return r;
}

// RNS (coordinates below 2^14 p) -> positional Jacobian, canonical, every lane the same
__device__ __forceinline__ g1::jac to_jac(const Ctx& C, const rjac& q) {
    const rv c = rns::cout(C);
    rv X, Y, Z;
    rns::mm3(C, q.X, c, q.Y, c, q.Z, c, X, Y, Z);
    return g1::jac{rns::to_positional(C, X), rns::to_positional(C, Y), rns::to_positional(C, Z)};
}

// 2^n q (n >= 0) for a finite q with X < 80 p, Y < 180 p, Z < 20 p; the result
// has X < 60 p, Y < 180 p, Z < 20 p (products are below 20 p).  dbl-2009-l
// with D = 4 X Y^2:
//   E = X (3X), B = Y^2, Z3 = Y (2Z);  F = E^2, C = B^2, D = (4X) B;
//   X3 = F - 2D, Y3 = E (3D - F) - 8C.
// The next doubling's E = X3 (3 X3) rides in the third round beside E (3D - F).
__device__ __forceinline__ rjac dbl_n(const Ctx& C, rjac q, int n) {
    if (n <= 0) return q;
    const rv p20 = rns::kp(C, 20), p40 = rns::kp(C, 40), p160 = rns::kp(C, 160);
    rv E, B, Z3;
    rns::mm3(C, q.X, rns::mul_small(C, q.X, 3), q.Y, q.Y, q.Y, rns::mul_small(C, q.Z, 2), E, B, Z3);
    for (int i = 0;; i++) {
        rv F, Cq, D;
        rns::mm3(C, E, E, B, B, rns::mul_small(C, q.X, 4), B, F, Cq, D);        // all < 20 p
        const rv X3 = rns::sub(C, F, D, p40, 2);                               // F - 2D < 60 p
        const rv T = rns::sub(C, rns::mul_small(C, D, 3), F, p20);             // 3D - F < 80 p
        rv P, En, unused;
        rns::mm3(C, E, T, X3, rns::mul_small(C, X3, 3), E, T, P, En, unused);
        q.X = X3;
        q.Y = rns::sub(C, P, Cq, p160, 8);                                     // P - 8C < 180 p
        q.Z = Z3;
        if (i + 1 == n) return q;
        E = En;
        rns::mm3(C, q.Y, q.Y, q.Y, rns::mul_small(C, q.Z, 2), q.Y, q.Y, B, Z3, unused);
    }
}

// r = p + q for finite p (X < 80 p, Y < 180 p, Z < 20 p) and q (every
// coordinate below 20 p); r has X < 80 p, Y < 60 p, Z < 20 p.  add-2007-bl:
//   Z1Z1 = Z1^2, Z2Z2 = Z2^2, U1 = X1 Z2Z2, U2 = X2 Z1Z1, S1 = Y1 Z2 Z2Z2,
//   S2 = Y2 Z1 Z1Z1, H = U2 - U1, I = (2H)^2, J = H I, r = 2 (S2 - S1),
//   V = U1 I, X3 = r^2 - J - 2V, Y3 = r (V - X3) - 2 S1 J,
//   Z3 = ((Z1 + Z2)^2 - Z1Z1 - Z2Z2) H.
// Returns false, leaving r unset, when H = 0 (equal or opposite points).
__device__ __forceinline__ bool add(const Ctx& C, const rjac& p, const rjac& q, rjac& r) {
    const rv p20 = rns::kp(C, 20), p40 = rns::kp(C, 40), p80 = rns::kp(C, 80);
    rv Z1Z1, Z2Z2, Y1Z2;
    rns::mm3(C, p.Z, p.Z, q.Z, q.Z, p.Y, q.Z, Z1Z1, Z2Z2, Y1Z2);
    rv U1, U2, Z1c;
    rns::mm3(C, p.X, Z2Z2, q.X, Z1Z1, p.Z, Z1Z1, U1, U2, Z1c);
    const rv Zs = rns::add(C, p.Z, q.Z);                                       // < 40 p
    rv S1, S2, ZZ;
    rns::mm3(C, Y1Z2, Z2Z2, q.Y, Z1c, Zs, Zs, S1, S2, ZZ);
    const rv H = rns::sub(C, U2, U1, p20);                                      // < 40 p
    if (rns::is_zero(C, H, 40)) return false;
    const rv H2 = rns::add(C, H, H);                                            // < 80 p
    const rv R = rns::mul_small(C, rns::sub(C, S2, S1, p20), 2);               // < 80 p
    const rv Zt = rns::sub(C, rns::sub(C, ZZ, Z1Z1, p20), Z2Z2, p20);          // < 60 p
    rv I, Z3, R2;
    rns::mm3(C, H2, H2, Zt, H, R, R, I, Z3, R2);
    rv J, V, unused;
    rns::mm3(C, H, I, U1, I, H, I, J, V, unused);
    const rv X3 = rns::sub(C, rns::sub(C, R2, J, p20), V, p40, 2);            // < 80 p
    rv Y, SJ;
    rns::mm3(C, R, rns::sub(C, V, X3, p80), S1, J, R, R, Y, SJ, unused);       // V - X3 < 100 p
    r.X = X3;
    r.Y = rns::sub(C, Y, SJ, p40, 2);                                           // < 60 p
    r.Z = Z3;
    return true;
}

// Horner's rule over the window sums ws[w_hi - 1] .. ws[w_lo] (positional
// Jacobian, 24 words each), starting from q0: q = 2^width_w q + T_w for each
// window w below the start.  Infinite operands and equal-x additions are
// handled in positional form.  Every lane returns the same canonical result.
template <class Width, class Load>
__device__ __forceinline__ g1::jac horner(const Ctx& C, g1::jac q0, int w_from, int w_lo, Width&& width,
                                          Load&& load) {
    bool inf = fq::is_zero(q0.Z);
    rjac q = to_rns(C, q0);
    for (int w = w_from; w >= w_lo; w--) {
        if (!inf) q = dbl_n(C, q, width(w));
        const g1::jac t = load(w);
        if (fq::is_zero(t.Z)) continue;
        const rjac tr = to_rns(C, t);
        if (inf) {
            q = tr;
            inf = false;
            continue;
        }
        rjac s;
        if (add(C, q, tr, s)) {
            q = s;
        } else {  // P1 = +-P2: the positional addition doubles or cancels
            const g1::jac sp = g1c::add(to_jac(C, q), t);
            inf = fq::is_zero(sp.Z);
            q = to_rns(C, sp);
        }
    }
    return inf ? g1::jac_inf() : to_jac(C, q);
}

// 2^n p in positional form through the RNS chain (p may be infinite)
__device__ __forceinline__ g1::jac dbl_n_positional(const Ctx& C, const g1::jac& p, int n) {
    if (n <= 0 || fq::is_zero(p.Z)) return p;
    return to_jac(C, dbl_n(C, to_rns(C, p), n));
}

}  // namespace g1r
