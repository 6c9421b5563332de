// msm_core.cuh -- device building blocks shared by the MSM kernels and the
// test hooks: scalar recoding and the batched affine pair addition.
#pragma once
#include <stdint.h>

#include "fq.cuh"
#include "g1.cuh"
#include "glv.cuh"
#include "inv.cuh"

namespace msm {

using fq::fe;
using g1::aff;

constexpr uint32_t HOLE = 0xFFFFFFFFu;  // padding entry: no second operand
constexpr uint32_t SIGN = 0x80000000u;  // entry flag: negate the point

// r = 0x30644e72e131a029b85045b68181585d2833e84879b9709143e1f593f0000001
#define FR_R0 0xf0000001u
#define FR_R1 0x43e1f593u
#define FR_R2 0x79b97091u
#define FR_R3 0x2833e848u
#define FR_R4 0x8181585du
#define FR_R5 0xb85045b6u
#define FR_R6 0xe131a029u
#define FR_R7 0x30644e72u

// k := k mod r for any k < 2^256 (< 6r): subtract r while no borrow results.
__device__ __forceinline__ void reduce_mod_r(uint32_t k[8]) {
#pragma unroll 1
    for (int it = 0; it < 5; it++) {
        uint32_t d0, d1, d2, d3, d4, d5, d6, d7, br;
        asm("sub.cc.u32  %0, %9,  %17;\n\t"
            "subc.cc.u32 %1, %10, %18;\n\t"
            "subc.cc.u32 %2, %11, %19;\n\t"
            "subc.cc.u32 %3, %12, %20;\n\t"
            "subc.cc.u32 %4, %13, %21;\n\t"
            "subc.cc.u32 %5, %14, %22;\n\t"
            "subc.cc.u32 %6, %15, %23;\n\t"
            "subc.cc.u32 %7, %16, %24;\n\t"
            "subc.u32    %8, 0, 0;"
            : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3), "=r"(d4), "=r"(d5), "=r"(d6), "=r"(d7), "=r"(br)
            : "r"(k[0]), "r"(k[1]), "r"(k[2]), "r"(k[3]), "r"(k[4]), "r"(k[5]), "r"(k[6]), "r"(k[7]),
              "n"(FR_R0), "n"(FR_R1), "n"(FR_R2), "n"(FR_R3), "n"(FR_R4), "n"(FR_R5), "n"(FR_R6), "n"(FR_R7));
        if (br) break;  // k < r
        k[0] = d0; k[1] = d1; k[2] = d2; k[3] = d3; k[4] = d4; k[5] = d5; k[6] = d6; k[7] = d7;
    }
}

template <int NL>
__device__ __forceinline__ uint32_t limb_at(const uint32_t (&k)[NL], int i) {
    uint32_t r = 0;
#pragma unroll
    for (int j = 0; j < NL; j++) r = (i == j) ? k[j] : r;
    return r;
}

// c bits of k starting at bit o (bits past the last limb read as zero)
template <int NL>
__device__ __forceinline__ uint32_t window_bits(const uint32_t (&k)[NL], int o, int c) {
    int li = o >> 5;
    uint64_t two = (uint64_t)limb_at(k, li) | ((uint64_t)limb_at(k, li + 1) << 32);
    return (uint32_t)(two >> (o & 31)) & ((1u << c) - 1u);
}

// Window layout: W = ceil(nbits / c) windows cover the nbits bits that a
// signed-digit recoding of the scalars needs (255 for k < r < 2^254; 128 for
// the GLV halves |k_i| < 2^127).  The widths are balanced: the low rr windows
// are q + 1 bits and the rest q bits, q = floor(nbits / W), rr = nbits - q W,
// so that no window is left with only a few bits -- a short top window would
// hold few, very large buckets and deepen the accumulation tree.  Every width
// is at most c.  Window w covers bits [off_w, off_w + width_w).
struct Windows {
    int W, nbits, q, rr;
};
__host__ __device__ __forceinline__ Windows make_windows(int c, int nbits) {
    Windows L;
    L.W = (nbits + c - 1) / c;
    L.nbits = nbits;
    L.q = nbits / L.W;
    L.rr = nbits - L.q * L.W;
    return L;
}
__host__ __device__ __forceinline__ int window_width(const Windows& L, int w) { return w < L.rr ? L.q + 1 : L.q; }
__host__ __device__ __forceinline__ int window_offset(const Windows& L, int w) {
    return w <= L.rr ? w * (L.q + 1) : L.rr * (L.q + 1) + (w - L.rr) * L.q;
}

constexpr int PLAIN_BITS = 255;  // windows of the full scalar
constexpr int GLV_BITS = 128;    // windows of one GLV half

// Signed digit of window w given the carry from window w-1: digits lie in
// (-2^(width-1), 2^(width-1)]; a raw value above 2^(width-1) becomes
// raw - 2^width and carries one into the next window.  The top window never
// carries out: the scalar's top bit (254, resp. 127) is zero.
template <int NL>
__device__ __forceinline__ int signed_digit(const uint32_t (&k)[NL], const Windows& L, int w, uint32_t& carry) {
    const int cw = window_width(L, w);
    uint32_t raw = window_bits(k, window_offset(L, w), cw) + carry;
    uint32_t half = 1u << (cw - 1);
    if (raw > half) {
        carry = 1;
        return (int)raw - (int)(1u << cw);
    }
    carry = 0;
    return (int)raw;
}

__device__ __forceinline__ void load_scalar(const uint32_t* s, uint32_t k[8]) {
    const uint4* q = reinterpret_cast<const uint4*>(s);
    uint4 a = q[0], b = q[1];
    k[0] = a.x; k[1] = a.y; k[2] = a.z; k[3] = a.w;
    k[4] = b.x; k[5] = b.y; k[6] = b.z; k[7] = b.w;
}

// ---------------------------------------------------------------------------
// Small-bucket finish.  A bucket with h level-1 items holds ceil(h / 2^(l-1))
// items at tree level l.  It stays in the affine pair tree while that count
// exceeds T; at the first level where it is at most T its items (stride
// 2^(l-1)) are summed by one thread in Jacobian coordinates instead, which
// needs no inversion and so avoids the per-level inversion latency of the
// tree's narrow tail.  T = 1 keeps every bucket in the tree.
struct FinishPlan {
    uint32_t items;   // items left when the bucket leaves the tree
    uint32_t stride;  // their spacing in the level-1 index space
};

__host__ __device__ __forceinline__ FinishPlan finish_plan(uint32_t h, uint32_t T) {
    uint32_t stride = 1, items = h;
    while (items > T) {
        stride <<= 1;
        items = (h + stride - 1) / stride;
    }
    return FinishPlan{items, stride};
}

// ---------------------------------------------------------------------------
// Batched affine pair addition.
//
// A slot holds one pair (P, Q) and produces P + Q.  The denominator of the
// chord (or tangent) slope is d = x_Q - x_P (d = 2 y_P when P = Q); S slots
// share one inversion through Montgomery's trick: prefix products
// pre_k = d_0 ... d_k on the way forward, one inversion of pre_{S-1}, and on
// the way back d_k^-1 = inv * pre_{k-1}, inv := inv * d_k.  This is the batch
// the pages' stream walker amortises the inversion over ("cost-per-add =
// |inv| / S", PR #23736 "stream-walker -- amortize the field inversion via
// large S + private pref_scratch", section "Goal & lever"); the prefix array is
// their pref_scratch.  Exceptional pairs (a missing second operand, an infinite
// operand, Q = -P) get d = 1 so they cannot poison the shared product -- the
// page records the "affine-add /0" that a colliding x otherwise causes (same
// page, section "Change (correct, landed)").
enum PairCase : int { PC_ADD = 0, PC_DBL = 1, PC_COPY_P = 2, PC_COPY_Q = 3, PC_INF = 4, PC_NONE = 5 };

// Decide the case from the x coordinates; y is only read when x_P == x_Q.
template <class LoadY>
__device__ __forceinline__ int pair_case(bool has_q, const fe& xp, const fe& xq, LoadY&& load_y, fe& yp_out) {
    if (!has_q) return PC_COPY_P;
    if (fq::is_zero(xp)) return PC_COPY_Q;
    if (fq::is_zero(xq)) return PC_COPY_P;
    if (!fq::eq(xp, xq)) return PC_ADD;
    fe yp, yq;
    load_y(yp, yq);
    yp_out = yp;
    return fq::eq(yp, yq) ? PC_DBL : PC_INF;
}

__device__ __forceinline__ fe pair_denominator(int cs, const fe& xp, const fe& xq, const fe& yp) {
    if (cs == PC_ADD) return fq::sub(xq, xp);
    if (cs == PC_DBL) return fq::dbl(yp);
    return fq::one();
}

// P + Q given d^-1 for the pair's denominator
__device__ __forceinline__ aff pair_result(int cs, const aff& p, const aff& q, const fe& dinv) {
    if (cs == PC_COPY_P) return p;
    if (cs == PC_COPY_Q) return q;
    if (cs == PC_INF || cs == PC_NONE) return g1::aff_inf();
    fe num, x2;
    if (cs == PC_ADD) {
        num = fq::sub(q.y, p.y);
        x2 = q.x;
    } else {  // tangent: 3 x^2 / 2y
        fe xx = fq::sqr_fused(p.x);
        num = fq::add(fq::dbl(xx), xx);
        x2 = p.x;
    }
    fe lam = fq::mul(num, dinv);
    aff r;
    r.x = fq::sub(fq::sub(fq::sqr_fused(lam), p.x), x2);
    r.y = fq::sub(fq::mul(lam, fq::sub(p.x, r.x)), p.y);
    return r;
}

// One inversion per block instead of one per warp.  Every thread of the block
// brings one nonzero value a (its batch's product; 1 when it has no batch)
// and receives a^-1.  The block's warps multiply their values pairwise in a
// tree (level s: warp w < s multiplies lane by lane with warp w + s, whose
// values it reads from shared memory), warp 0 inverts the 32 products of all
// warps in one pass of the per-lane inversion, and the tree is walked back
// down (warp w < s hands warp w + s its inverse through shared memory): with
// four warps, two multiplications up and two levels of two independent ones
// down, where a single warp gathering the block's values needed nine in a row.
// The other warps wait at the barriers while warp 0 inverts: the block issues
// one warp's inversion where each warp used to issue its own, which at small
// batches (a launch of one wave, 9 additions per thread at n = 2^16) is a
// quarter of the instructions that dominate (divsteps on the ALU pipe, their
// 64-bit updates on the multiply pipe).  sh: 8 x blockDim.x words, word w of
// thread i's slot at sh[w * blockDim.x + i] (consecutive lanes hit consecutive
// banks).  All threads of the block must call it; blockDim.x is a multiple of
// 32 and at most 256.
__device__ __forceinline__ void sh_store(uint32_t* sh, int i, const fe& a) {
#pragma unroll
    for (int w = 0; w < 8; w++) sh[w * blockDim.x + i] = a.v[w];
}
__device__ __forceinline__ fe sh_load(const uint32_t* sh, int i) {
    fe a;
#pragma unroll
    for (int w = 0; w < 8; w++) a.v[w] = sh[w * blockDim.x + i];
    return a;
}

__device__ __forceinline__ fe block_inverse(const fe& a, uint32_t* sh, int inv_kind, const uint32_t* divtab) {
    const int tid = threadIdx.x, warp = tid >> 5, nw = blockDim.x >> 5;
    fe v = a;
    fe keep[3];  // this warp's values below each level it multiplied at (nw <= 8)
    int lv = 0;
    for (int s = nw >> 1; s >= 1; s >>= 1, lv++) {
        if (warp >= s && warp < 2 * s) sh_store(sh, tid, v);
        __syncthreads();
        if (warp < s) {
            keep[lv] = v;
            v = fq::mul(v, sh_load(sh, tid + 32 * s));
        }
    }
    if (inv_kind == 0 && divtab && nw >= 2) {
        // warps 0 and 1 share the pass (inv_safegcd_pair): warp 0 hands over
        // its 32 values in slots 0..31 of sh (the tree keeps its own values in
        // the slots of warps 1 and up) and warp 1 returns the inverses there
        __shared__ uint32_t pair_mat[2 * 6 * 32];
        if (warp == 0) sh_store(sh, tid, v);
        __syncthreads();
        if (warp < 2) {
            const fe r = inv::inv_safegcd_pair(sh_load(sh, tid & 31), pair_mat,
                                               (uint32_t)__cvta_generic_to_shared(divtab));
            if (warp == 1) sh_store(sh, tid & 31, r);  // warp 0 read its slot before the first meeting
        }
        __syncthreads();
        if (warp == 0) v = sh_load(sh, tid);
    } else if (warp == 0) {
        v = inv_kind ? fq::inv_fermat(v) : divtab ? inv::inv_safegcd_tab(v, divtab) : inv::inv_safegcd(v);
    }
    for (int s = 1; s < nw; s <<= 1) {
        lv--;
        if (warp < s) {
            const fe partner = sh_load(sh, tid + 32 * s);
            sh_store(sh, tid + 32 * s, fq::mul(v, keep[lv]));
            v = fq::mul(v, partner);
        }
        __syncthreads();
        if (warp >= s && warp < 2 * s) v = sh_load(sh, tid);
    }
    return v;
}

// Where a batch keeps its prefix products (the pages' pref_scratch, which they
// move between private and workgroup memory: PR #23738 "stream-walker S-sweep",
// section "What would actually win"):
//  * PLACE_LOCAL: an array in the thread's stack frame.  Its dynamic index puts
//    it in local memory -- device memory (HBM) private to the thread, cached
//    in L1 and L2 -- so this is the HBM-scratch placement; the default.
//  * PLACE_SHARED: the block's dynamic shared memory, word w of product k of
//    thread i at pre[(8 k + w) blockDim.x + i] (consecutive lanes hit
//    consecutive banks); S x 32 bytes per thread.
//  * PLACE_REGS: registers -- both loops fully unrolled so every index is a
//    constant (small S only: S x 8 registers, and S copies of the loop body).
constexpr int PLACE_LOCAL = 0;
constexpr int PLACE_SHARED = 1;
constexpr int PLACE_REGS = 2;

template <int S, int PLACE>
struct PreStore {
    fe v[S];
    __device__ __forceinline__ void set(int k, const fe& a) { v[k] = a; }
    __device__ __forceinline__ fe get(int k) const { return v[k]; }
};
template <int S>
struct PreStore<S, PLACE_SHARED> {
    uint32_t* base;
    __device__ __forceinline__ void set(int k, const fe& a) {
#pragma unroll
        for (int w = 0; w < 8; w++) base[(8 * k + w) * blockDim.x + threadIdx.x] = a.v[w];
    }
    __device__ __forceinline__ fe get(int k) const {
        fe a;
#pragma unroll
        for (int w = 0; w < 8; w++) a.v[w] = base[(8 * k + w) * blockDim.x + threadIdx.x];
        return a;
    }
};

// Run one batch of up to S pair additions.  Src supplies, per slot k < count:
//   bool has_q(k); fe xp(k), xq(k); void ys(k, fe& yp, fe& yq);
//   aff p(k), q(k); void store(k, const aff&).
// Returns the number of slots that were true additions (ADD or DBL).
//
// Except with PLACE_REGS the per-slot loops stay rolled: unrolled, S copies of
// the inlined multiplications overflow the instruction cache (the kernel then
// stalls on instruction fetch) and pin S x 8 registers of prefix products.  The multiplications of Montgomery's
// trick are inlined -- the forward one always, the two backward ones when
// INLINE_BACK -- the others are called: inlined, a multiplication needs no
// moves into and out of the call's argument registers (which occupy the same
// multiply pipe the products do) and leaves the register allocator a global
// view.  Inlining the backward pair pays for large, throughput-bound launches
// (n = 2^22: 12.98 -> 12.79 ms) and for level 0 at any size, and costs the
// tree's latency-bound narrow levels through the larger loop body (the
// accumulation kernels choose); inlining all six was slower still.
// inv_kind selects the batch inversion: 0 = safegcd divsteps (the default),
// 1 = Fermat (a^(p-2), 4-bit windows) -- kept for the measured comparison.
// The three products of Montgomery's trick (the prefix, and the backward pair)
// skip the final conditional subtraction (fq::mul_lazy_inline): the chain's
// values stay below 2p, which every product of the chain and the slope's
// multiplication accept, and both inversions take any representative.  This
// is the lighter-reduction lever for the batch inversion that the pages list
// as a next direction (PR #23736 "stream-walker -- amortize the field
// inversion via large S + private pref_scratch", section "Honest status --
// NOT done").
// With sh (shared scratch of 8 x blockDim.x words) the block's threads share
// one inversion (block_inverse): then every thread of the block must call,
// those without pairs with count = 0.  pre_sh is the block's prefix-product
// area for PLACE_SHARED (S x 8 x blockDim.x words), unused otherwise.
// divtab: the block's shared-memory copy of the divstep table (inv.cuh,
// load_divtab), or null for the plain divstep loop.
template <int S, bool INLINE_BACK, int PLACE = PLACE_LOCAL, class Src>
__device__ __forceinline__ int batch_pairs(Src& src, int count, int inv_kind = 0, uint32_t* sh = nullptr,
                                           uint32_t* pre_sh = nullptr, const uint32_t* divtab = nullptr) {
    PreStore<S, PLACE> pre;
    if constexpr (PLACE == PLACE_SHARED) pre.base = pre_sh;
    fe acc = fq::one();
    int adds = 0;
    auto forward = [&](int k) {
        bool hq = src.has_q(k);
        fe xp = src.xp(k);
        fe xq = hq ? src.xq(k) : fq::zero();
        fe yp = fq::zero();
        int cs = pair_case(hq, xp, xq, [&](fe& a, fe& b) { src.ys(k, a, b); }, yp);
        fe d = pair_denominator(cs, xp, xq, yp);
        adds += (cs == PC_ADD || cs == PC_DBL);
        acc = (k == 0) ? d : fq::mul_lazy_inline(acc, d);
        pre.set(k, acc);
    };
    if constexpr (PLACE == PLACE_REGS) {
#pragma unroll
        for (int k = 0; k < S; k++)
            if (k < count) forward(k);
    } else {
#pragma unroll 1
        for (int k = 0; k < count; k++) forward(k);
    }
    fe inv = sh ? block_inverse(acc, sh, inv_kind, divtab)
                : inv_kind ? fq::inv_fermat(acc) : divtab ? inv::inv_safegcd_tab(acc, divtab) : inv::inv_safegcd(acc);
    auto backward = [&](int k) {
        aff p = src.p(k);
        bool hq = src.has_q(k);
        aff q = hq ? src.q(k) : g1::aff_inf();
        fe yp_unused = p.y;
        int cs = pair_case(hq, p.x, q.x, [&](fe& a, fe& b) { a = p.y; b = q.y; }, yp_unused);
        fe d = pair_denominator(cs, p.x, q.x, p.y);
        fe dinv = inv;
        if (k > 0) {
            if (INLINE_BACK) {
                dinv = fq::mul_lazy_inline(inv, pre.get(k - 1));
                inv = fq::mul_lazy_inline(inv, d);
            } else {
                dinv = fq::mul_lazy(inv, pre.get(k - 1));
                inv = fq::mul_lazy(inv, d);
            }
        }
        src.store(k, pair_result(cs, p, q, dinv));
    };
    if constexpr (PLACE == PLACE_REGS) {
#pragma unroll
        for (int j = 0; j < S; j++)
            if (S - 1 - j < count) backward(S - 1 - j);
    } else {
#pragma unroll 1
        for (int k = count - 1; k >= 0; k--) backward(k);
    }
    return adds;
}

}  // namespace msm
