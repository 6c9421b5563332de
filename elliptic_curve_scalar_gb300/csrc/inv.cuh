// inv.cuh -- field inversion in F_p by Bernstein-Yang "safegcd" divsteps.
//
// The pages' batched affine additions share one field inversion per batch,
// and the inversion they use is safegcd (PR #23738 "stream-walker S-sweep",
// section "Notes / caveats": "Montgomery/safegcd math"; PR #23736, section
// "Goal & lever", puts it at ~47 % of the accumulate kernel in software).
//
// Algorithm (D. J. Bernstein, B.-Y. Yang, "Fast constant-time gcd computation
// and modular inversion", TCHES 2019): with delta = 1, f = p (odd), g = x,
// one divstep maps
//     delta > 0 and g odd:  (1 - delta, g, (g - f)/2)
//     g odd otherwise:      (1 + delta, f, (g + f)/2)
//     g even:               (1 + delta, f, g/2).
// After 735 divsteps (the paper's bound floor((49 d + 57)/17) for d = 254-bit
// inputs) g = 0 and f = +-gcd(p, x) = +-1.  Divsteps are run 30 at a time on
// the low 32 bits of f and g, which yields a 2x2 transition matrix T with
// entries bounded by 2^30 (|u| + |v| <= 2^30); T is then applied to the full
// f, g and to the cofactors d, e, which keep f = d*x*K^-1 and g = e*x*K^-1
// (mod p).  Starting from d = 0, e = K with K = R^2 mod p gives, at the end,
// d = +-R^2 / x~ for a Montgomery input x~ = x R, i.e. the Montgomery form of
// x^-1 with no extra multiplication.  The division of d, e by 2^30 is made
// exact by adding a multiple of p; adding p*u (p*q) for a negative d and p*v
// (p*r) for a negative e beforehand keeps d, e in (-2p, p) at every batch
// (the bound argument of the libsecp256k1 safegcd write-up, restated).
//
// Numbers are signed, little-endian, 9 limbs of 30 bits in int32 (the top
// limb carries the sign); products are int32 x int32 -> int64.
#pragma once
#include <stdint.h>

#include "divstep_table.cuh"
#include "fq.cuh"

namespace inv {

constexpr int32_t M30 = 0x3FFFFFFF;
constexpr int BATCHES = 25;  // 25 * 30 = 750 >= 735 divsteps

// p in base 2^30
__device__ __forceinline__ int32_t p30(int i) {
    const int32_t P[9] = {0x187cfd47, 0x3082305b, 0x071ca8d3, 0x205aa45a, 0x01585d97,
                          0x0116da06, 0x1a029b85, 0x139cb84c, 0x3064};
    return P[i];
}
constexpr uint32_t PINV30 = 0x1b799c77u;  // p^-1 mod 2^30

struct s9 {
    int32_t v[9];
};

// 30 divsteps on the low words of f and g; returns the transition matrix
// scaled by 2^30: [u v; q r] with 2^30 (f', g') = (u f + v g, q f + r g).
__device__ __forceinline__ int32_t divsteps30(int32_t delta, uint32_t f, uint32_t g, int32_t& u_out, int32_t& v_out,
                                              int32_t& q_out, int32_t& r_out) {
    int32_t u = 1, v = 0, q = 0, r = 1;
#pragma unroll 5
    for (int i = 0; i < 30; i++) {
        // c1: delta > 0; c2: g odd
        int32_t c1 = (-delta) >> 31;
        int32_t c2 = -(int32_t)(g & 1u);
        // if g is odd add (-f, -u, -v) when delta > 0, (f, u, v) otherwise
        int32_t x = ((int32_t)f ^ c1) - c1;
        int32_t y = (u ^ c1) - c1;
        int32_t z = (v ^ c1) - c1;
        g += (uint32_t)(x & c2);
        q += y & c2;
        r += z & c2;
        // swap case (delta > 0 and g odd): f takes the old g, (u, v) the old (q, r)
        c1 &= c2;
        delta = (delta ^ c1) - c1 + 1;
        f += g & (uint32_t)c1;
        u += q & c1;
        v += r & c1;
        g >>= 1;
        u <<= 1;
        v <<= 1;
    }
    u_out = u;
    v_out = v;
    q_out = q;
    r_out = r;
    return delta;
}

// The same 30 divsteps with seven lookups of four steps each in the block's
// copy of kDivTab (divstep_table.cuh, written by gen_divsteps.py), then two
// single steps.  A lookup reads the 2x2 matrix B of four steps from delta and
// the low four bits of f and g, advances f and g by B / 16 on their low words
// and accumulates the batch matrix as B times it; four single steps cost a
// chain of about 30 dependent instructions, a lookup a shared-memory load and
// a few.  tab_sh: shared-memory address of the table (__cvta_generic_to_shared).
__device__ __forceinline__ int32_t divsteps30_tab(int32_t delta, uint32_t f, uint32_t g, int32_t& u_out,
                                                  int32_t& v_out, int32_t& q_out, int32_t& r_out, uint32_t tab_sh) {
    int32_t u = 1, v = 0, q = 0, r = 1;
#pragma unroll
    for (int i = 0; i < 7; i++) {
        const int32_t ds = min(max(delta, -4), 4) + 4;
        const uint32_t idx = ((uint32_t)ds * 8u + ((f >> 1) & 7u)) * 16u + (g & 15u);
        uint32_t e;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(e) : "r"(tab_sh + 4u * idx));
        const int32_t bu = ((int32_t)(e << 26)) >> 26;
        const int32_t bv = ((int32_t)(e << 20)) >> 26;
        const int32_t bq = ((int32_t)(e << 14)) >> 26;
        const int32_t br = ((int32_t)(e << 8)) >> 26;
        const int32_t neg = -(int32_t)((e >> 24) & 1u);
        const int32_t t = ((int32_t)(e << 2)) >> 27;
        delta = ((delta ^ neg) - neg) + t;
        const uint32_t fn = ((uint32_t)bu * f + (uint32_t)bv * g) >> 4;
        const uint32_t gn = ((uint32_t)bq * f + (uint32_t)br * g) >> 4;
        f = fn;
        g = gn;
        const int32_t un = bu * u + bv * q, vn = bu * v + bv * r;
        const int32_t qn = bq * u + br * q, rn = bq * v + br * r;
        u = un;
        v = vn;
        q = qn;
        r = rn;
    }
#pragma unroll
    for (int i = 0; i < 2; i++) {  // steps 29 and 30, as in divsteps30
        int32_t c1 = (-delta) >> 31;
        int32_t c2 = -(int32_t)(g & 1u);
        int32_t x = ((int32_t)f ^ c1) - c1;
        int32_t y = (u ^ c1) - c1;
        int32_t z = (v ^ c1) - c1;
        g += (uint32_t)(x & c2);
        q += y & c2;
        r += z & c2;
        c1 &= c2;
        delta = (delta ^ c1) - c1 + 1;
        f += g & (uint32_t)c1;
        u += q & c1;
        v += r & c1;
        g >>= 1;
        u <<= 1;
        v <<= 1;
    }
    u_out = u;
    v_out = v;
    q_out = q;
    r_out = r;
    return delta;
}

// A block's copy of the divstep table in shared memory; every thread of the
// block calls this before any of them may use the table, and a barrier
// follows before the first lookup.
__device__ __forceinline__ void load_divtab(uint32_t* tab) {
    for (int i = threadIdx.x; i < kDivTabEntries; i += blockDim.x) tab[i] = __ldg(kDivTab + i);
}

// (f, g) := (u f + v g, q f + r g) / 2^30 (exact)
__device__ __forceinline__ void update_fg(s9& f, s9& g, int32_t u, int32_t v, int32_t q, int32_t r) {
    int64_t cf = (int64_t)u * f.v[0] + (int64_t)v * g.v[0];
    int64_t cg = (int64_t)q * f.v[0] + (int64_t)r * g.v[0];
    cf >>= 30;
    cg >>= 30;
#pragma unroll
    for (int i = 1; i < 9; i++) {
        cf += (int64_t)u * f.v[i] + (int64_t)v * g.v[i];
        cg += (int64_t)q * f.v[i] + (int64_t)r * g.v[i];
        f.v[i - 1] = (int32_t)cf & M30;
        g.v[i - 1] = (int32_t)cg & M30;
        cf >>= 30;
        cg >>= 30;
    }
    f.v[8] = (int32_t)cf;
    g.v[8] = (int32_t)cg;
}

// (d, e) := (u d + v e, q d + r e) / 2^30 mod p, kept in (-2p, p)
__device__ __forceinline__ void update_de(s9& d, s9& e, int32_t u, int32_t v, int32_t q, int32_t r) {
    int32_t sd = d.v[8] >> 31, se = e.v[8] >> 31;  // -1 when negative
    int32_t md = (u & sd) + (v & se);
    int32_t me = (q & sd) + (r & se);
    int64_t cd = (int64_t)u * d.v[0] + (int64_t)v * e.v[0];
    int64_t ce = (int64_t)q * d.v[0] + (int64_t)r * e.v[0];
    // make the low 30 bits vanish: subtract k*p with k = (cd + md p0) p^-1 mod 2^30
    md -= (int32_t)(((uint32_t)cd + (uint32_t)md * (uint32_t)p30(0)) * PINV30 & (uint32_t)M30);
    me -= (int32_t)(((uint32_t)ce + (uint32_t)me * (uint32_t)p30(0)) * PINV30 & (uint32_t)M30);
    cd += (int64_t)md * p30(0);
    ce += (int64_t)me * p30(0);
    cd >>= 30;
    ce >>= 30;
#pragma unroll
    for (int i = 1; i < 9; i++) {
        cd += (int64_t)u * d.v[i] + (int64_t)v * e.v[i] + (int64_t)md * p30(i);
        ce += (int64_t)q * d.v[i] + (int64_t)r * e.v[i] + (int64_t)me * p30(i);
        d.v[i - 1] = (int32_t)cd & M30;
        e.v[i - 1] = (int32_t)ce & M30;
        cd >>= 30;
        ce >>= 30;
    }
    d.v[8] = (int32_t)cd;
    e.v[8] = (int32_t)ce;
}

// 8 x 32-bit limbs (< 2^256) -> 9 x 30-bit limbs
__device__ __forceinline__ s9 from_fe(const fq::fe& a) {
    s9 r;
    const uint32_t* w = a.v;
    r.v[0] = (int32_t)(w[0] & M30);
    r.v[1] = (int32_t)(((w[0] >> 30) | (w[1] << 2)) & M30);
    r.v[2] = (int32_t)(((w[1] >> 28) | (w[2] << 4)) & M30);
    r.v[3] = (int32_t)(((w[2] >> 26) | (w[3] << 6)) & M30);
    r.v[4] = (int32_t)(((w[3] >> 24) | (w[4] << 8)) & M30);
    r.v[5] = (int32_t)(((w[4] >> 22) | (w[5] << 10)) & M30);
    r.v[6] = (int32_t)(((w[5] >> 20) | (w[6] << 12)) & M30);
    r.v[7] = (int32_t)(((w[6] >> 18) | (w[7] << 14)) & M30);
    r.v[8] = (int32_t)(w[7] >> 16);
    return r;
}

// 9 x 30-bit limbs of a value in [0, 2^256) -> 8 x 32-bit limbs
__device__ __forceinline__ fq::fe to_fe(const s9& a) {
    fq::fe r;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(a.v);
    r.v[0] = s[0] | (s[1] << 30);
    r.v[1] = (s[1] >> 2) | (s[2] << 28);
    r.v[2] = (s[2] >> 4) | (s[3] << 26);
    r.v[3] = (s[3] >> 6) | (s[4] << 24);
    r.v[4] = (s[4] >> 8) | (s[5] << 22);
    r.v[5] = (s[5] >> 10) | (s[6] << 20);
    r.v[6] = (s[6] >> 12) | (s[7] << 18);
    r.v[7] = (s[7] >> 14) | (s[8] << 16);
    return r;
}

// carry-normalise limbs so that limbs 0..7 lie in [0, 2^30)
__device__ __forceinline__ void normalise(s9& a) {
    int32_t c = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        int32_t t = a.v[i] + c;
        a.v[i] = t & M30;
        c = t >> 30;
    }
    a.v[8] += c;
}

// a := a + (p & mask) limb-wise (mask = 0 or -1), then normalise
__device__ __forceinline__ void add_p_masked(s9& a, int32_t mask) {
#pragma unroll
    for (int i = 0; i < 9; i++) a.v[i] += p30(i) & mask;
    normalise(a);
}

// x~ (Montgomery form of x, < p) -> Montgomery form of x^-1; 0 -> 0.
// tab_sh: shared-memory address of the block's divstep table, or 0 for the
// plain divstep loop (paths without the table in shared memory).
static __device__ __noinline__ fq::fe inv_safegcd_impl(fq::fe xm, uint32_t tab_sh) {
    s9 f, g, d, e;
#pragma unroll
    for (int i = 0; i < 9; i++) f.v[i] = p30(i);
    g = from_fe(xm);
    const int32_t K[9] = {0x138afa89, 0x0cb3f16d, 0x04501fbf, 0x39c64475, 0x017ff6b5,
                          0x2c7bfc29, 0x0351f47a, 0x27dc72ae, 0x6d8};  // R^2 mod p
#pragma unroll
    for (int i = 0; i < 9; i++) {
        d.v[i] = 0;
        e.v[i] = K[i];
    }
    int32_t delta = 1;
#pragma unroll 1
    for (int b = 0; b < BATCHES; b++) {
        int32_t u, v, q, r;
        const uint32_t fl = (uint32_t)f.v[0] | ((uint32_t)f.v[1] << 30), gl = (uint32_t)g.v[0] | ((uint32_t)g.v[1] << 30);
        delta = tab_sh ? divsteps30_tab(delta, fl, gl, u, v, q, r, tab_sh) : divsteps30(delta, fl, gl, u, v, q, r);
        update_fg(f, g, u, v, q, r);
        update_de(d, e, u, v, q, r);
        // once g = 0 everywhere in the warp, further divsteps leave f and d unchanged
        int32_t gz = g.v[0] | g.v[1] | g.v[2] | g.v[3] | g.v[4] | g.v[5] | g.v[6] | g.v[7] | g.v[8];
        if (__all_sync(__activemask(), gz == 0)) break;
    }
    // f = +-1: x^-1 = f * d; bring d from (-2p, p) into [0, p)
    int32_t neg = f.v[8] >> 31;  // -1 when f = -1
#pragma unroll
    for (int i = 0; i < 9; i++) d.v[i] = (d.v[i] ^ neg) - neg;
    normalise(d);                     // d in (-2p, 2p)
    add_p_masked(d, d.v[8] >> 31);    // (-p, 2p)
    add_p_masked(d, d.v[8] >> 31);    // [0, 2p)
    // subtract p if d >= p
    s9 t;
#pragma unroll
    for (int i = 0; i < 9; i++) t.v[i] = d.v[i] - p30(i);
    normalise(t);
    int32_t keep = t.v[8] >> 31;  // -1 when d < p
#pragma unroll
    for (int i = 0; i < 9; i++) d.v[i] = (d.v[i] & keep) | (t.v[i] & ~keep);
    return to_fe(d);
}

// One pass of 32 inversions shared by two warps of a block (both call this,
// converged; blockDim.x >= 64).  Lane i of warp 0 holds the value xm to invert
// and runs the divsteps and the update of f and g -- the chain the next batch
// waits for -- and hands each batch's transition matrix to lane i of warp 1
// through shared memory; warp 1 applies it to the cofactors d and e, one batch
// behind, which takes their 54 limb products off warp 0's path.  The two warps
// meet at a named barrier (id 1, 64 threads) once per batch; the matrices
// alternate between two buffers, so warp 0 rewrites a buffer only after warp 1
// has passed the next meeting and is done with it.  mat: 2 x 6 x 32 words of
// shared memory (u, v, q, r, the sign of f, the end flag).  The inverse is
// returned in warp 1 (lane i: the inverse of warp 0's lane-i value); warp 0's
// return value is unspecified.  tab_sh: the block's divstep table.
__device__ __forceinline__ fq::fe inv_safegcd_pair(const fq::fe& xm, uint32_t* mat, uint32_t tab_sh) {
    const int lane = threadIdx.x & 31;
    const bool lead = (threadIdx.x >> 5) == 0;
    const int32_t K[9] = {0x138afa89, 0x0cb3f16d, 0x04501fbf, 0x39c64475, 0x017ff6b5,
                          0x2c7bfc29, 0x0351f47a, 0x27dc72ae, 0x6d8};  // R^2 mod p
    s9 a, b;  // warp 0: f, g; warp 1: d, e
    if (lead) {
        const s9 g0 = from_fe(xm);
#pragma unroll
        for (int i = 0; i < 9; i++) {
            a.v[i] = p30(i);
            b.v[i] = g0.v[i];
        }
    } else {
#pragma unroll
        for (int i = 0; i < 9; i++) {
            a.v[i] = 0;
            b.v[i] = K[i];
        }
    }
    int32_t delta = 1, fneg = 0;
#pragma unroll 1
    for (int bt = 0; bt < BATCHES; bt++) {
        uint32_t* m = mat + (bt & 1) * 6 * 32 + lane;
        bool fin;
        if (lead) {
            int32_t u, v, q, r;
            const uint32_t fl = (uint32_t)a.v[0] | ((uint32_t)a.v[1] << 30);
            const uint32_t gl = (uint32_t)b.v[0] | ((uint32_t)b.v[1] << 30);
            delta = divsteps30_tab(delta, fl, gl, u, v, q, r, tab_sh);
            m[0] = (uint32_t)u;
            m[32] = (uint32_t)v;
            m[64] = (uint32_t)q;
            m[96] = (uint32_t)r;
            update_fg(a, b, u, v, q, r);
            const int32_t gz = b.v[0] | b.v[1] | b.v[2] | b.v[3] | b.v[4] | b.v[5] | b.v[6] | b.v[7] | b.v[8];
            fin = __all_sync(0xffffffffu, gz == 0);  // g = 0 in every lane: f and d are final
            m[128] = (uint32_t)(a.v[8] >> 31);
            m[160] = fin;
            asm volatile("bar.sync 1, 64;" ::: "memory");
        } else {
            asm volatile("bar.sync 1, 64;" ::: "memory");
            const int32_t u = (int32_t)m[0], v = (int32_t)m[32], q = (int32_t)m[64], r = (int32_t)m[96];
            fneg = (int32_t)m[128];
            fin = m[160] != 0;
            update_de(a, b, u, v, q, r);
        }
        if (fin) break;
    }
    // warp 1: f = +-1, x^-1 = f d; bring d from (-2p, p) into [0, p)
    s9& d = a;
#pragma unroll
    for (int i = 0; i < 9; i++) d.v[i] = (d.v[i] ^ fneg) - fneg;
    normalise(d);
    add_p_masked(d, d.v[8] >> 31);
    add_p_masked(d, d.v[8] >> 31);
    s9 t;
#pragma unroll
    for (int i = 0; i < 9; i++) t.v[i] = d.v[i] - p30(i);
    normalise(t);
    const int32_t keep = t.v[8] >> 31;
#pragma unroll
    for (int i = 0; i < 9; i++) d.v[i] = (d.v[i] & keep) | (t.v[i] & ~keep);
    return to_fe(d);
}

__device__ __forceinline__ fq::fe inv_safegcd(fq::fe xm) { return inv_safegcd_impl(xm, 0u); }
// the same with the block's table (tab: a shared-memory array filled by load_divtab)
__device__ __forceinline__ fq::fe inv_safegcd_tab(fq::fe xm, const uint32_t* tab) {
    return inv_safegcd_impl(xm, (uint32_t)__cvta_generic_to_shared(tab));
}

}  // namespace inv
