// g1_proj.cuh -- the MSM's long doubling chains on a pair of warps, in the
// residue number system of rns.cuh and homogeneous projective coordinates.
//
// A point (X : Y : Z) stands for the affine (X/Z, Y/Z); (0 : 1 : 0) is the
// identity.  For y^2 = x^3 + 3 the doubling and the addition of Renes,
// Costello and Batina ("Complete addition formulas for prime order elliptic
// curves", EUROCRYPT 2016, the a = 0 formulas with b3 = 3b = 9) are complete:
// no input -- the identity, P = Q, P = -Q -- needs a case of its own, so a
// chain has no branches.  Both are two levels deep in field products: the
// doubling has four products per level, the addition six.  (Jacobian
// doubling is three levels deep, which is what a single warp's three RNS
// groups ran: three products per level.)
//
// A warp holds three 10-lane RNS groups (rns.cuh), so a pair of warps holds
// six: one round computes six independent products, three in each warp, and
// the two warps exchange them through shared memory at a named barrier.  A
// doubling is then two rounds (two slots spare in each, where the next
// window sum is brought into RNS form), an addition two full rounds.
//
// Every function here is called by both warps of the pair -- threads 0..63
// of the block, converged per warp -- with the pair's exchange buffer and
// named barrier; values are the same in both warps.
#pragma once
#include "g1.cuh"
#include "rns.cuh"

namespace g1p {

using rns::Ctx;
using rns::rv;

constexpr int kXchWords = 2 * 6 * 10 * 2;  // two buffers x six products x ten channels x two residues

struct Pair {
    Ctx C;
    int h;          // the warp within the pair: products 3h .. 3h + 2 are this warp's
    uint32_t* xch;  // kXchWords words of shared memory
    int buf;        // the buffer of the next round
};

// threads 0..63 of the block form the pair; named barrier 1 is the pair's
__device__ __forceinline__ Pair make_pair(uint32_t* xch) {
    Pair P;
    P.C = rns::make_ctx();
    P.h = (threadIdx.x >> 5) & 1;
    P.xch = xch;
    P.buf = 0;
    return P;
}

// p[k] = x[k] y[k] M^-1 (rns::mm) for k = 0..5, all six in every lane of both
// warps.  Group g < 3 of warp h computes product 3h + g; lanes 30 and 31
// compute a copy of product 3h and store nothing.  The buffers alternate: a
// warp writes buffer b again two rounds later, after the barrier of the round
// between, which the other warp reaches only once it has read buffer b.
__device__ __forceinline__ void mm6(Pair& P, const rv (&x)[6], const rv (&y)[6], rv (&p)[6]) {
    const int k = P.C.g < 3 ? 3 * P.h + P.C.g : 3 * P.h;
    rv xs = x[0], ys = y[0];
#pragma unroll
    for (int i = 1; i < 6; i++) {
        xs = k == i ? x[i] : xs;
        ys = k == i ? y[i] : ys;
    }
    const rv r = rns::mm(P.C, xs, ys);
    uint32_t* b = P.xch + P.buf * 120 + 2 * P.C.j;
    if (P.C.g < 3) *reinterpret_cast<uint2*>(b + 20 * k) = make_uint2(r.a, r.b);
    asm volatile("bar.sync 1, 64;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 6; i++) {
        const uint2 v = *reinterpret_cast<const uint2*>(b + 20 * i);
        p[i] = rv{v.x, v.y};
    }
    P.buf ^= 1;
}

struct rproj {
    rv X, Y, Z;
};

// The positional Jacobian point t (Montgomery form, every lane the same) on
// its way to projective RNS form (X Z : Y : Z^3), two products per round in a
// doubling's spare slots:
//   step 0: X' = X cin, Y' = Y cin (RNS Montgomery domain, below 20 p)
//   step 1: Z' = Z cin
//   step 2: X' Z', Z'^2
//   step 3: Z'^2 Z'
// The Jacobian identity (Z = 0) becomes (0 : 1 : 0).
struct Side {
    rv a, b;   // residues of X and Y (step 0), Z (step 1); then X', Z'
    rv Xr, Yr, Zr, Z2;
    int stage;
    __device__ __forceinline__ void start(const Ctx& C, const g1::jac& t) {
        const bool inf = fq::is_zero(t.Z);
        a = rns::residues(C, inf ? fq::zero() : t.X);
        b = rns::residues(C, inf ? fq::one() : t.Y);
        Zr = rns::residues(C, inf ? fq::zero() : t.Z);  // held raw until step 1
        stage = 0;
    }
    __device__ __forceinline__ bool done() const { return stage >= 4; }
    // operands of slots 4 and 5 (a spare product where the step needs one)
    __device__ __forceinline__ void operands(const Ctx& C, rv& x4, rv& y4, rv& x5, rv& y5) const {
        const rv cin = rns::cin(C);
        if (stage == 0) { x4 = a; y4 = cin; x5 = b; y5 = cin; }
        else if (stage == 1) { x4 = Zr; y4 = cin; x5 = Zr; y5 = cin; }
        else if (stage == 2) { x4 = Xr; y4 = Zr; x5 = Zr; y5 = Zr; }
        else { x4 = Z2; y4 = Zr; x5 = Z2; y5 = Zr; }
    }
    __device__ __forceinline__ void take(const rv& p4, const rv& p5) {
        if (stage == 0) { Xr = p4; Yr = p5; }
        else if (stage == 1) { Zr = p4; }
        else if (stage == 2) { Xr = p4; Z2 = p5; }
        else if (stage == 3) { Zr = p4; }
        stage++;
    }
    __device__ __forceinline__ rproj point() const { return rproj{Xr, Yr, Zr}; }
};

// 2 q (any q with coordinates below 40 p; the result's below 40 p):
//   level 1: A1 = Y^2, A2 = Z^2, A3 = Y Z, A4 = X Y
//   level 2: B1 = (9 A2)(8 A1), B2 = (A1 - 27 A2)(A1 + 9 A2),
//            B3 = 2 (A1 - 27 A2) A4, B4 = (8 A1) A3
//   X3 = B3, Y3 = B1 + B2, Z3 = B4
// (2 X Y (Y^2 - 27 Z^2), (Y^2 - 27 Z^2)(Y^2 + 9 Z^2) + 72 Y^2 Z^2, 8 Y^3 Z).
// Slots 4 and 5 of both rounds serve the side conversion s.
__device__ __forceinline__ rproj dbl(Pair& P, const rproj& q, Side& s) {
    const Ctx& C = P.C;
    rv x[6], y[6], p[6];
    x[0] = q.Y; y[0] = q.Y;
    x[1] = q.Z; y[1] = q.Z;
    x[2] = q.Y; y[2] = q.Z;
    x[3] = q.X; y[3] = q.Y;
    s.operands(C, x[4], y[4], x[5], y[5]);
    mm6(P, x, y, p);
    if (!s.done()) s.take(p[4], p[5]);
    const rv A1 = p[0], A2 = p[1], A3 = p[2], A4 = p[3];  // all below 20 p
    const rv D = rns::sub(C, A1, A2, rns::kp(C, 540), 27);   // A1 - 27 A2 < 560 p
    x[0] = rns::mul_small(C, A2, 9); y[0] = rns::mul_small(C, A1, 8);  // 180 p, 160 p
    x[1] = D; y[1] = rns::add(C, A1, rns::mul_small(C, A2, 9));       // 560 p, 200 p
    x[2] = rns::add(C, D, D); y[2] = A4;                               // 1120 p, 20 p
    x[3] = y[0]; y[3] = A3;                                            // 160 p, 20 p
    s.operands(C, x[4], y[4], x[5], y[5]);
    mm6(P, x, y, p);
    if (!s.done()) s.take(p[4], p[5]);
    return rproj{p[2], rns::add(C, p[0], p[1]), p[3]};
}

// q1 + q2 for any q1, q2 with coordinates below 40 p (the result's below 40 p):
//   level 1: t0 = X1 X2, t1 = Y1 Y2, t2 = Z1 Z2, t3 = (X1 + Y1)(X2 + Y2),
//            t4 = (Y1 + Z1)(Y2 + Z2), t5 = (X1 + Z1)(X2 + Z2)
//   then u3 = t3 - t0 - t1, u4 = t4 - t1 - t2, u5 = 9 (t5 - t0 - t2),
//        v0 = 3 t0, v2 = 9 t2, w = t1 + v2, d = t1 - v2
//   level 2: X3 = u3 d - u4 u5, Y3 = d w + u5 v0, Z3 = w u4 + v0 u3
__device__ __forceinline__ rproj add(Pair& P, const rproj& q1, const rproj& q2) {
    const Ctx& C = P.C;
    rv x[6], y[6], p[6];
    x[0] = q1.X; y[0] = q2.X;
    x[1] = q1.Y; y[1] = q2.Y;
    x[2] = q1.Z; y[2] = q2.Z;
    x[3] = rns::add(C, q1.X, q1.Y); y[3] = rns::add(C, q2.X, q2.Y);  // below 80 p
    x[4] = rns::add(C, q1.Y, q1.Z); y[4] = rns::add(C, q2.Y, q2.Z);
    x[5] = rns::add(C, q1.X, q1.Z); y[5] = rns::add(C, q2.X, q2.Z);
    mm6(P, x, y, p);  // all below 20 p
    const rv p20 = rns::kp(C, 20), p180 = rns::kp(C, 180);
    const rv u3 = rns::sub(C, rns::sub(C, p[3], p[0], p20), p[1], p20);                       // < 60 p
    const rv u4 = rns::sub(C, rns::sub(C, p[4], p[1], p20), p[2], p20);                       // < 60 p
    const rv u5 = rns::mul_small(C, rns::sub(C, rns::sub(C, p[5], p[0], p20), p[2], p20), 9);  // < 540 p
    const rv v0 = rns::mul_small(C, p[0], 3);                                                  // < 60 p
    const rv v2 = rns::mul_small(C, p[2], 9);                                                  // < 180 p
    const rv w = rns::add(C, p[1], v2);                                                        // < 200 p
    const rv d = rns::sub(C, p[1], v2, p180);                                                  // < 200 p
    x[0] = u3; y[0] = d;
    x[1] = u4; y[1] = u5;
    x[2] = d;  y[2] = w;
    x[3] = u5; y[3] = v0;
    x[4] = w;  y[4] = u4;
    x[5] = v0; y[5] = u3;
    mm6(P, x, y, p);
    return rproj{rns::sub(C, p[0], p[1], p20), rns::add(C, p[2], p[3]), rns::add(C, p[4], p[5])};
}

// Complete a side conversion in rounds of its own (no doubling to ride on).
__device__ __forceinline__ rproj finish(Pair& P, Side& s) {
    rv x[6], y[6], p[6];
    while (!s.done()) {
        s.operands(P.C, x[4], y[4], x[5], y[5]);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            x[i] = x[4];
            y[i] = y[4];
        }
        mm6(P, x, y, p);
        s.take(p[4], p[5]);
    }
    return s.point();
}

__device__ __forceinline__ rproj to_proj(Pair& P, const g1::jac& t) {
    Side s;
    s.start(P.C, t);
    return finish(P, s);
}

// Positional Jacobian (canonical, every lane the same) of a projective RNS
// point with coordinates below 40 p: (X Z, Y Z^2, Z), the identity as
// g1::jac_inf().
__device__ __forceinline__ g1::jac to_jac(Pair& P, const rproj& q) {
    const Ctx& C = P.C;
    const rv cout = rns::cout(C);
    rv x[6], y[6], p[6];
    x[0] = q.X; y[0] = q.Z;
    x[1] = q.Z; y[1] = q.Z;
    x[2] = q.Z; y[2] = cout;
#pragma unroll
    for (int i = 3; i < 6; i++) {
        x[i] = x[0];
        y[i] = y[0];
    }
    mm6(P, x, y, p);
    const rv XZ = p[0], Z2 = p[1], Zo = p[2];
    x[0] = q.Y; y[0] = Z2;
    x[1] = XZ;  y[1] = cout;
    mm6(P, x, y, p);
    const rv Xo = p[1];
    x[0] = p[0]; y[0] = cout;
    mm6(P, x, y, p);
    const g1::jac r{rns::to_positional(C, Xo), rns::to_positional(C, p[0]), rns::to_positional(C, Zo)};
    return fq::is_zero(r.Z) ? g1::jac_inf() : r;
}

// Projective positional form, for values that pass between kernels: (X, Y, Z)
// canonical in Montgomery form (fq.cuh), 24 words, the identity (0, 1, 0).
struct ppos {
    fq::fe X, Y, Z;
};
__device__ __forceinline__ ppos load_ppos(const uint32_t* p) { return ppos{fq::load(p), fq::load(p + 8), fq::load(p + 16)}; }
__device__ __forceinline__ void store_ppos(uint32_t* p, const ppos& q) {
    fq::store(p, q.X);
    fq::store(p + 8, q.Y);
    fq::store(p + 16, q.Z);
}

// Two positional projective points into RNS form in one round.
__device__ __forceinline__ void from_ppos2(Pair& P, const ppos& a, const ppos& b, rproj& ra, rproj& rb) {
    const Ctx& C = P.C;
    const rv cin = rns::cin(C);
    rv x[6], y[6], p[6];
    x[0] = rns::residues(C, a.X);
    x[1] = rns::residues(C, a.Y);
    x[2] = rns::residues(C, a.Z);
    x[3] = rns::residues(C, b.X);
    x[4] = rns::residues(C, b.Y);
    x[5] = rns::residues(C, b.Z);
#pragma unroll
    for (int i = 0; i < 6; i++) y[i] = cin;
    mm6(P, x, y, p);
    ra = rproj{p[0], p[1], p[2]};
    rb = rproj{p[3], p[4], p[5]};
}
__device__ __forceinline__ rproj from_ppos(Pair& P, const ppos& a) {
    rproj r, unused;
    from_ppos2(P, a, a, r, unused);
    return r;
}
// one round and three conversions to positional form (coordinates below 40 p)
__device__ __forceinline__ ppos to_ppos(Pair& P, const rproj& q) {
    const Ctx& C = P.C;
    const rv cout = rns::cout(C);
    rv x[6], y[6], p[6];
    x[0] = q.X;
    x[1] = q.Y;
    x[2] = q.Z;
#pragma unroll
    for (int i = 3; i < 6; i++) x[i] = q.X;
#pragma unroll
    for (int i = 0; i < 6; i++) y[i] = cout;
    mm6(P, x, y, p);
    return ppos{rns::to_positional(C, p[0]), rns::to_positional(C, p[1]), rns::to_positional(C, p[2])};
}

// q doubled n times
__device__ __forceinline__ rproj dbl_n(Pair& P, rproj q, int n) {
    Side idle;
    idle.stage = 4;
    for (int i = 0; i < n; i++) q = dbl(P, q, idle);
    return q;
}

// Horner's rule over the window sums load(w_from) .. load(w_lo) (positional
// Jacobian), from q: q = 2^width(w) q + T_w for w = w_from down to w_lo.
// Each T_w is brought into projective RNS form in the spare slots of the
// doublings before it (two doublings take the four steps; what a narrower
// window leaves runs in rounds of its own).
template <class Width, class Load>
__device__ __forceinline__ rproj horner_proj(Pair& P, rproj q, int w_from, int w_lo, Width&& width, Load&& load) {
    for (int w = w_from; w >= w_lo; w--) {
        Side s;
        s.start(P.C, load(w));
        const int n = width(w);
        for (int i = 0; i < n; i++) q = dbl(P, q, s);
        q = add(P, q, finish(P, s));
    }
    return q;
}

// The same from a positional Jacobian q0 to a positional Jacobian result
// (every lane the same, canonical).
template <class Width, class Load>
__device__ __forceinline__ g1::jac horner(Pair& P, const g1::jac& q0, int w_from, int w_lo, Width&& width,
                                          Load&& load) {
    return to_jac(P, horner_proj(P, to_proj(P, q0), w_from, w_lo, width, load));
}

// 2^n t for a positional Jacobian t (any point, n >= 0), positional out
__device__ __forceinline__ g1::jac dbl_n_positional(Pair& P, const g1::jac& t, int n) {
    if (n <= 0 || fq::is_zero(t.Z)) return t;
    return to_jac(P, dbl_n(P, to_proj(P, t), n));
}

}  // namespace g1p
