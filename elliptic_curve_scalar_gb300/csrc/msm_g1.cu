// msm_g1.cu -- the BN254 G1 bucket-method MSM on sm_103a and its C ABI.
//
// Pipeline per call (all on the caller's stream, no host synchronisation):
//   1. digits+histogram: each scalar is reduced mod r and recoded into signed
//      c-bit digits; every non-zero digit d of window w counts one entry for
//      bucket g = w*B + |d| - 1 (B = 2^(c-1)).  The window size c is the knob
//      the pages fix at 13 for n = 2^16 (PR #23520 "cache dx + idx in
//      ba_fused_super pref_scratch", section "Measurements").
//   2. scan: exclusive prefix of the bucket counts, each padded to even, into
//      the bucket offsets (the pages' sorted_count_list, PR #23738
//      "stream-walker S-sweep", section "What would actually win").
//   3. scatter: a counting sort writes, per bucket, the point indices with a
//      negate flag (the sorted_bucket_list of the same section); odd buckets
//      get one padding entry.
//   4. accumulation, level 0: entries (2u, 2u+1) form pair u; every pair is
//      one affine addition, batched S per thread with one shared inversion.
//   5. accumulation, levels l >= 1: the pair tree halves each bucket's items
//      in place until every bucket holds one point, its bucket sum.  (This is
//      the pages' other accumulator, the level-wise pair tree "ba_fused_super"
//      of PR #23520, section "Summary", rather than their sequential stream
//      walker: on a 152-SM part every level offers n*W/2^(l+1) independent
//      additions, enough to fill the GPU, where a walker's per-thread streams
//      would have to be cut into pieces shorter than a bucket.)
//   6. bucket reduction: per window T_w = sum_b b * S_b by running sums over
//      short chunks, then a per-window tree sum.
//   7. window combination: Q = sum_w 2^(c w) T_w by Horner's rule.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "../../include/msm_g1.h"
#include "g1_coop.cuh"
#include "g1_proj.cuh"
#include "msm_internal.cuh"

using fq::fe;
using g1::aff;
using g1::jac;

namespace msm {

constexpr int SCAN_TPB = 256;
constexpr int SCAN_ITEMS = 8;
constexpr int SCAN_TILE = SCAN_TPB * SCAN_ITEMS;
constexpr int REDUCE_TPB = 256;
constexpr uint32_t MAX_REDUCE_JOBS = 16;  // 1 + log2 G, G <= 2^12 (one warp per job)
constexpr uint32_t REDUCE_MAX_PARTS = 8;  // partial blocks per reduction job
constexpr uint64_t MAX_BATCH_WINDOWS = 4096;  // windows of all MSMs of one batch pass

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// exclusive block scan; blockDim.x multiple of 32 and <= 1024
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sm, uint32_t& total) {
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t inc = warp_incl_scan(v);
    if (lane == 31) sm[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < nw ? sm[lane] : 0;
        uint32_t wi = warp_incl_scan(w);
        if (lane < nw) sm[lane] = wi - w;
        if (lane == 31) sm[32] = wi;
    }
    __syncthreads();
    uint32_t r = sm[warp] + inc - v;
    total = sm[32];
    __syncthreads();
    return r;
}

// ------------------------------------------------------ 1. digits + histogram

// Visit every window digit of scalar i (k mod r; a dead lane sees k = 0 and
// only zero digits): f(d, g, e) gets the digit, its bucket g = w B + |d| - 1
// (HOLE for d = 0 or a dead lane) and its entry e, the point index with SIGN
// set when the point enters negated.  With GLV, k P = k1 P + k2 phi(P): the
// digits of |k1| go with point i, those of |k2| with point n + i (phi(P_i)),
// each negated when its half is negative.  All lanes call f the same number
// of times, so f may use warp collectives.
// Batches: MSM m of a batch of `count` owns terms [off[m], off[m+1]) and the
// windows [m W, (m + 1) W); the MSM of term i is found by binary search.
struct BatchMap {
    const uint32_t* off;  // count + 1 term offsets (device), or null for one MSM
    int count;
};

__device__ __forceinline__ uint32_t msm_of(const BatchMap& bm, uint32_t i) {
    if (!bm.off) return 0;
    uint32_t lo = 0, hi = (uint32_t)bm.count;
    while (hi - lo > 1) {  // the last m with off[m] <= i (empty MSMs are skipped)
        const uint32_t mid = (lo + hi) >> 1;
        if (__ldg(bm.off + mid) <= i) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <bool GLV, class F>
__device__ __forceinline__ void scalar_digits(const uint32_t* __restrict__ scalars, size_t n, size_t i, bool live,
                                              int c, const Windows& L, const BatchMap& bm, F&& f) {
    uint32_t k[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (live) {
        load_scalar(scalars + 8 * i, k);
        reduce_mod_r(k);
    }
    const uint32_t B = 1u << (c - 1);
    const uint32_t wbase = live ? msm_of(bm, (uint32_t)i) * (uint32_t)L.W : 0;
    auto visit = [&](auto& half, uint32_t e_base, uint32_t neg) {
        uint32_t carry = 0;
        for (int w = 0; w < L.W; w++) {
            const int d = signed_digit(half, L, w, carry);
            const uint32_t g = (live && d != 0) ? (wbase + (uint32_t)w) * B + (uint32_t)(d < 0 ? -d : d) - 1u : HOLE;
            f(g, e_base | (((uint32_t)(d < 0) ^ neg) ? SIGN : 0u));
        }
    };
    if constexpr (GLV) {
        uint32_t k1[4], k2[4], neg1, neg2;
        glv::split(k, k1, k2, neg1, neg2);
        visit(k1, (uint32_t)i, neg1);
        visit(k2, (uint32_t)(n + i), neg2);
    } else {
        visit(k, (uint32_t)i, 0u);
    }
}

// One thread per scalar; the lanes of a warp hitting the same bucket share one
// atomic.
template <bool GLV>
__global__ void k_digits_hist(const uint32_t* __restrict__ scalars, size_t n, int c, Windows L, BatchMap bm,
                              uint32_t* __restrict__ counts) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = i < n;
    const int lane = threadIdx.x & 31;
    scalar_digits<GLV>(scalars, n, i, live, c, L, bm, [&](uint32_t g, uint32_t) {
        const uint32_t peers = __match_any_sync(0xffffffffu, g);
        if (g != HOLE && lane == __ffs(peers) - 1) atomicAdd(&counts[g], (uint32_t)__popc(peers));
    });
}

// GLV images phi(P_i) = (beta x_i, y_i); one thread per point.  Needs only the
// points, so it runs beside the sort (which needs only the scalars).
__global__ void k_phi(const uint32_t* __restrict__ points, size_t n, uint32_t* __restrict__ phi) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const fe beta = {{GLV_BETA_MONT}};
    aff p = g1::load_aff(points + 16 * i);
    p.x = fq::mul(p.x, beta);  // the point at infinity (0, 0) stays (0, 0)
    g1::store_aff(phi + 16 * i, p);
}

// ---------------------------------------------------------------- 2. scan

// per tile: sum of counts padded to even; also the statistics
__global__ void k_scan_reduce(const uint32_t* __restrict__ counts, uint32_t nb, uint32_t* __restrict__ tile_sums,
                              ctl_t* ctl) {
    __shared__ uint32_t sm[33];
    uint32_t base = blockIdx.x * SCAN_TILE;
    uint32_t s = 0, mx = 0, ne = 0, ent = 0;
#pragma unroll
    for (int j = 0; j < SCAN_ITEMS; j++) {
        uint32_t g = base + j * SCAN_TPB + threadIdx.x;
        uint32_t m = g < nb ? counts[g] : 0;
        s += m + (m & 1);
        mx = max(mx, m);
        ne += m != 0;
        ent += m;
    }
    uint32_t tot;
    block_excl_scan(s, sm, tot);
    if (threadIdx.x == 0) tile_sums[blockIdx.x] = tot;
    mx = __reduce_max_sync(0xffffffffu, mx);
    ne = __reduce_add_sync(0xffffffffu, ne);
    ent = __reduce_add_sync(0xffffffffu, ent);
    if ((threadIdx.x & 31) == 0) {
        if (mx) atomicMax(&ctl->max_count, mx);
        if (ne) atomicAdd(&ctl->nonempty, ne);
        if (ent) atomicAdd(&ctl->entries, ent);
    }
}

// single block: exclusive scan of the tile sums in place; total -> ctl
__global__ void k_scan_tiles(uint32_t* __restrict__ tile_sums, uint32_t ntiles, ctl_t* ctl) {
    __shared__ uint32_t sm[33];
    uint32_t carry = 0;
    for (uint32_t base = 0; base < ntiles; base += blockDim.x) {
        uint32_t i = base + threadIdx.x;
        uint32_t v = i < ntiles ? tile_sums[i] : 0;
        uint32_t tot;
        uint32_t ex = block_excl_scan(v, sm, tot);
        if (i < ntiles) tile_sums[i] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) ctl->total = carry;
}

// per tile: offsets, scatter cursors and the padding entry of odd buckets
__global__ void k_scan_apply(const uint32_t* __restrict__ counts, uint32_t nb, const uint32_t* __restrict__ tile_sums,
                             uint32_t* __restrict__ offsets, uint32_t* __restrict__ cursor,
                             uint32_t* __restrict__ entries, const ctl_t* __restrict__ ctl) {
    __shared__ uint32_t sm[33];
    uint32_t base = blockIdx.x * SCAN_TILE + threadIdx.x * SCAN_ITEMS;  // contiguous run per thread
    uint32_t m[SCAN_ITEMS];
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < SCAN_ITEMS; j++) {
        uint32_t g = base + j;
        m[j] = g < nb ? counts[g] : 0;
        s += m[j] + (m[j] & 1);
    }
    uint32_t tot;
    uint32_t off = tile_sums[blockIdx.x] + block_excl_scan(s, sm, tot);
#pragma unroll
    for (int j = 0; j < SCAN_ITEMS; j++) {
        uint32_t g = base + j;
        if (g < nb) {
            offsets[g] = off;
            cursor[g] = off;
            if (m[j] & 1) entries[off + m[j]] = HOLE;
        }
        off += m[j] + (m[j] & 1);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) offsets[nb] = ctl->total;
}

// Small bucket counts (nb <= SCAN_SMALL_MAX): the three passes above in one
// block of 1024 threads -- thread t takes the run of buckets [t r, (t + 1) r),
// r = ceil(nb / 1024) -- which saves two launches and their gaps (n = 2^10,
// c = 8, 2048 buckets: scan phase 21 -> 11 us).  Runs of more than a few
// buckets make the block's loads uncoalesced and the single SM the bottleneck
// (n = 2^16, 40960 buckets: 27 -> 85 us), so larger counts keep three passes.
constexpr uint32_t SCAN_SMALL_MAX = 1u << 12;
__global__ void __launch_bounds__(1024) k_scan_small(const uint32_t* __restrict__ counts, uint32_t nb,
                                                     uint32_t* __restrict__ offsets, uint32_t* __restrict__ cursor,
                                                     uint32_t* __restrict__ entries, ctl_t* ctl) {
    __shared__ uint32_t sm[33];
    const uint32_t r = (nb + blockDim.x - 1) / blockDim.x;
    const uint32_t b0 = threadIdx.x * r, b1 = min(b0 + r, nb);
    uint32_t s = 0, mx = 0, ne = 0, ent = 0;
    for (uint32_t g = b0; g < b1; g++) {
        const uint32_t m = counts[g];
        s += m + (m & 1);
        mx = max(mx, m);
        ne += m != 0;
        ent += m;
    }
    uint32_t tot;
    uint32_t off = block_excl_scan(s, sm, tot);
    for (uint32_t g = b0; g < b1; g++) {
        const uint32_t m = counts[g];
        offsets[g] = off;
        cursor[g] = off;
        if (m & 1) entries[off + m] = HOLE;
        off += m + (m & 1);
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    ne = __reduce_add_sync(0xffffffffu, ne);
    ent = __reduce_add_sync(0xffffffffu, ent);
    if ((threadIdx.x & 31) == 0) {
        if (mx) atomicMax(&ctl->max_count, mx);
        if (ne) atomicAdd(&ctl->nonempty, ne);
        if (ent) atomicAdd(&ctl->entries, ent);
    }
    if (threadIdx.x == 0) {
        offsets[nb] = tot;
        ctl->total = tot;
    }
}

// ------------------------------------------------------------- 3. scatter

template <bool GLV>
__global__ void k_scatter(const uint32_t* __restrict__ scalars, size_t n, int c, Windows L, BatchMap bm,
                          uint32_t* __restrict__ cursor, uint32_t* __restrict__ entries) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    scalar_digits<GLV>(scalars, n, i, i < n, c, L, bm, [&](uint32_t g, uint32_t e) {
        const uint32_t peers = __match_any_sync(0xffffffffu, g);
        const int leader = __ffs(peers) - 1;
        uint32_t pos = 0;
        if (g != HOLE && lane == leader) pos = atomicAdd(&cursor[g], (uint32_t)__popc(peers));
        pos = __shfl_sync(0xffffffffu, pos, leader);
        if (g != HOLE) entries[pos + __popc(peers & lt_mask)] = e;
    });
}

// ------------------------------------------ 3'. sort of large single MSMs
//
// With 2^23 terms and 8 windows the two passes above issue 67 M global atomics
// each, and the scalar split runs twice.  For large single MSMs (window width
// at most 16, so a window's B counters fit in shared memory) the digits are
// formed once into a code matrix, and every block counts one slice of one
// window's codes in shared memory: one global atomic per bucket and block
// instead of one per digit, and the scatter writes one window's region of
// the entry list at a time, which stays in L2.  The order of the entries
// within a bucket is whatever the shared atomics give: a bucket's sum does
// not depend on it.

// code of one (term, window): NO_DIGIT for digit 0, else (|d| - 1) | negate << 31.
// (32-bit codes: with 16-bit windows the 2^15 buckets and the sign fill 16
// bits, and no 16-bit value would be left for "no digit".)
constexpr uint32_t NO_DIGIT = 0xFFFFFFFFu;

// One thread per scalar: its W codes per half, codes[w * tstride + t] for term t
// (t = i, and n + i for the GLV half on phi(P_i)).
template <bool GLV>
__global__ void k_digit_codes(const uint32_t* __restrict__ scalars, size_t n, Windows L, size_t tstride,
                              uint32_t* __restrict__ codes) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t k[8];
    load_scalar(scalars + 8 * i, k);
    reduce_mod_r(k);
    auto emit = [&](auto& half, size_t t, uint32_t neg) {
        uint32_t carry = 0;
        for (int w = 0; w < L.W; w++) {
            const int d = signed_digit(half, L, w, carry);
            const uint32_t mag = (uint32_t)(d < 0 ? -d : d);
            codes[(size_t)w * tstride + t] = d == 0 ? NO_DIGIT : (mag - 1u) | ((((uint32_t)(d < 0)) ^ neg) << 31);
        }
    };
    if constexpr (GLV) {
        uint32_t k1[4], k2[4], neg1, neg2;
        glv::split(k, k1, k2, neg1, neg2);
        emit(k1, i, neg1);
        emit(k2, n + i, neg2);
    } else {
        emit(k, i, 0u);
    }
}

// Block b: window b / S, terms [s T, min((s + 1) T, nterms)) with s = b % S and
// T a multiple of 4 (codes read 4 at a time; the row stride is a multiple of 4
// and its padding is read but ignored).  sh: B shared counters.
__device__ __forceinline__ void slice_counts(const uint32_t* __restrict__ row, size_t t0, size_t t1, uint32_t* sh) {
    for (size_t t = t0 + 4 * (size_t)threadIdx.x; t < t1; t += 4 * (size_t)blockDim.x) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + t);
        const uint32_t cd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; j++)
            if (cd[j] != NO_DIGIT && t + j < t1) atomicAdd(&sh[cd[j] & ~SIGN], 1u);
    }
}

__global__ void __launch_bounds__(1024) k_hist_slices(const uint32_t* __restrict__ codes, size_t tstride,
                                                      size_t nterms, uint32_t S, size_t T, uint32_t B,
                                                      uint32_t* __restrict__ counts) {
    extern __shared__ uint32_t sh[];
    const uint32_t w = blockIdx.x / S, s = blockIdx.x % S;
    const size_t t0 = (size_t)s * T, t1 = min(t0 + T, nterms);
    for (uint32_t b = threadIdx.x; b < B; b += blockDim.x) sh[b] = 0;
    __syncthreads();
    if (t0 < t1) slice_counts(codes + (size_t)w * tstride, t0, t1, sh);
    __syncthreads();
    for (uint32_t b = threadIdx.x; b < B; b += blockDim.x)
        if (sh[b]) atomicAdd(&counts[(size_t)w * B + b], sh[b]);
}

// The same slices again: count, reserve each bucket's run in the entry list
// with one global atomic on its cursor, then place every entry at the
// reservation's next free slot (a shared atomic).
__global__ void __launch_bounds__(1024) k_scatter_slices(const uint32_t* __restrict__ codes, size_t tstride,
                                                         size_t nterms, uint32_t S, size_t T, uint32_t B,
                                                         uint32_t* __restrict__ cursor,
                                                         uint32_t* __restrict__ entries) {
    extern __shared__ uint32_t sh[];
    const uint32_t w = blockIdx.x / S, s = blockIdx.x % S;
    const size_t t0 = (size_t)s * T, t1 = min(t0 + T, nterms);
    const uint32_t* row = codes + (size_t)w * tstride;
    for (uint32_t b = threadIdx.x; b < B; b += blockDim.x) sh[b] = 0;
    __syncthreads();
    if (t0 < t1) slice_counts(row, t0, t1, sh);
    __syncthreads();
    for (uint32_t b = threadIdx.x; b < B; b += blockDim.x)
        if (sh[b]) sh[b] = atomicAdd(&cursor[(size_t)w * B + b], sh[b]);
    __syncthreads();
    for (size_t t = t0 + 4 * (size_t)threadIdx.x; t < t1; t += 4 * (size_t)blockDim.x) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + t);
        const uint32_t cd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (cd[j] != NO_DIGIT && t + j < t1) {
                const uint32_t pos = atomicAdd(&sh[cd[j] & ~SIGN], 1u);
                entries[pos] = (uint32_t)(t + j) | (cd[j] & SIGN);
            }
        }
    }
}

// The scatter of the codes in term order, one thread per term and window row,
// the lanes of a warp that hit the same bucket sharing one atomic (like
// k_scatter, without recomputing the digits).  Every bucket then fills from
// its start in term order: one partial sector per bucket is being written at
// any time, which L2 holds even when the entry list does not fit (n = 2^22:
// 268 MB of entries; the slices' per-block runs, 152 write fronts per bucket,
// thrashed L2: 0.75 -> 2.0 ms).
__global__ void k_scatter_codes(const uint32_t* __restrict__ codes, size_t tstride, size_t nterms, int W,
                                uint32_t B, uint32_t* __restrict__ cursor, uint32_t* __restrict__ entries) {
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int w = 0; w < W; w++) {
        const uint32_t cd = t < nterms ? codes[(size_t)w * tstride + t] : NO_DIGIT;
        const uint32_t g = cd == NO_DIGIT ? HOLE : (uint32_t)w * B + (cd & ~SIGN);
        const uint32_t peers = __match_any_sync(0xffffffffu, g);
        const int leader = __ffs(peers) - 1;
        uint32_t pos = 0;
        if (g != HOLE && lane == leader) pos = atomicAdd(&cursor[g], (uint32_t)__popc(peers));
        pos = __shfl_sync(0xffffffffu, pos, leader);
        if (g != HOLE) entries[pos + __popc(peers & lt_mask)] = (uint32_t)t | (cd & SIGN);
    }
}

// ---------------------------------------------------------- 6. reduction
//
// T_w = sum_{b<B} (b + 1) S_b per window, without a per-chunk scalar multiple.
// Buckets are cut into G = B / L chunks of L; chunk j yields its plain sum
// R_j and its local weighted sum C_j = sum_{i<L} (i + 1) S_{jL+i}, so that
//     T_w = sum_j C_j + L sum_j j R_j,   sum_j j R_j = sum_t 2^t V_t,
// V_t = sum of the R_j whose index j has bit t set.  The 1 + log2 G plain sums
// (sum C_j and every V_t) are wide tree reductions; only a log2 G-step Horner
// pass (one doubling and one addition per bit) and log2 L doublings remain
// sequential, run by one warp with the warp-cooperative point operations.

// One thread per chunk: running sums from the chunk's top bucket give
// run = R_j and sum = C_j (bucket jL + i is added into run at steps i .. 0).
template <int W>
__global__ void k_reduce_chunks(const uint32_t* __restrict__ items, const uint32_t* __restrict__ counts,
                                const uint32_t* __restrict__ offsets, const uint32_t* __restrict__ jsum,
                                uint32_t finish_t, int w_lo, int nwin, uint32_t B, uint32_t L, uint32_t G,
                                uint32_t* __restrict__ chunks) {
    // one thread (W = 1) or one group of W lanes per chunk, whose additions
    // are then cooperative: 5 multiplication latencies each instead of 11 or
    // 16, for 2.5 times the multiply-pipe work (idle lanes multiply too)
    uint32_t t = (blockIdx.x * blockDim.x + threadIdx.x) / W;
    if (t >= (uint32_t)nwin * G) return;
    uint32_t w = (uint32_t)w_lo + t / G, j = t % G;
    uint32_t b0 = j * L;
    uint32_t b1 = min(b0 + L, B);
    jac run = g1::jac_inf(), sum = g1::jac_inf();
    for (uint32_t b = b1; b-- > b0;) {
        uint32_t g = w * B + b;
        if (counts[g]) {
            const uint32_t og = offsets[g] >> 1;
            if (finish_plan((offsets[g + 1] >> 1) - og, finish_t).items >= 2)
                run = g1c::add_w<W>(run, g1::load_jac(jsum + (size_t)g * 24));  // finished in Jacobian
            else
                run = g1c::add_mixed_w<W>(run, g1::load_aff(items + (size_t)og * 16));
        }
        sum = g1c::add_w<W>(sum, run);
    }
    if ((threadIdx.x & (W - 1)) == 0) {
        uint32_t* dst = chunks + ((size_t)w * G + j) * 48;
        g1::store_jac(dst, sum);
        g1::store_jac(dst + 24, run);
    }
}

// Small MSMs (T >= 2, buckets that leave the tree with 2..T items are summed
// in Jacobian form): the small-bucket finish and the chunk sums in one launch.
// A group of W lanes per point operation (W = 1: one thread; W = 8:
// cooperative additions), H groups per bucket and L buckets per chunk.  The
// H groups of a bucket add its items i = r, r + H, ... (mixed additions) and
// then each other's sums, so that a bucket's chain is about T / H + log2 H
// additions long; group r = 0 then holds the bucket's sum S_k (or its single
// tree item, or infinity).  The chunk's buckets form the suffix sums
// U_k = S_k + ... + S_{L-1} by a scan (log2 L additions deep, where one
// thread's running sum was L long) and sum_k U_k by a tree (log2 L more),
// and bucket 0 stores (sum_k U_k, U_0) -- what k_reduce_chunks stores -- with
// no Jacobian bucket sums going through memory.  A warp holds whole chunks.
__device__ __forceinline__ jac shfl_down_jac(const jac& p, int d) {
    jac r;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        r.X.v[i] = __shfl_down_sync(0xffffffffu, p.X.v[i], d);
        r.Y.v[i] = __shfl_down_sync(0xffffffffu, p.Y.v[i], d);
        r.Z.v[i] = __shfl_down_sync(0xffffffffu, p.Z.v[i], d);
    }
    return r;
}

template <int W, int H, int L>
__global__ void k_finish_chunks(const uint32_t* __restrict__ items, const uint32_t* __restrict__ offsets,
                                uint32_t finish_t, int w_lo, int nwin, uint32_t B, uint32_t G,
                                uint32_t* __restrict__ chunks) {
    static_assert(W * H * L <= 32 && 32 % (W * H * L) == 0, "a warp holds whole chunks");
    const uint32_t gt = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t t = gt / (W * H * L), k = (gt / (W * H)) % L, r = (gt / W) % H;
    const bool live = t < (uint32_t)nwin * G;  // dead lanes add infinities and store nothing
    const uint32_t w = (uint32_t)w_lo + t / G, j = t % G;
    jac S = g1::jac_inf();
    if (live) {
        const uint32_t g = w * B + j * L + k;
        const uint32_t og = offsets[g] >> 1, h = (offsets[g + 1] >> 1) - og;
        const FinishPlan fp = finish_plan(h, finish_t);
        if (fp.items >= 2) {
            auto item = [&](uint32_t i) { return g1::load_aff(items + (size_t)(og + i * fp.stride) * 16); };
            uint32_t i = r;
            if constexpr (W == 1) {  // the chain's first two items by the affine-affine addition
                if (i + H < fp.items) {
                    S = g1::add_aff(item(i), item(i + H));
                    i += 2 * H;
                }
            }
            for (; i < fp.items; i += H) S = g1c::add_mixed_w<W>(S, item(i));
        } else if (h && r == 0) {
            S = g1::to_jac(g1::load_aff(items + (size_t)og * 16));
        }
    }
#pragma unroll
    for (int d = 1; d < H; d <<= 1) {  // the bucket's groups, into group 0
        const jac o = shfl_down_jac(S, d * W);
        if ((r & (2 * d - 1)) == 0 && r + d < (uint32_t)H) S = g1c::add_w<W>(S, o);
    }
#pragma unroll
    for (int d = 1; d < L; d <<= 1) {  // suffix sums over the chunk's buckets
        const jac o = shfl_down_jac(S, d * W * H);
        if (r == 0 && k + d < (uint32_t)L) S = g1c::add_w<W>(S, o);
    }
    const jac run = S;
#pragma unroll
    for (int d = 1; d < L; d <<= 1) {  // their sum, into bucket 0
        const jac o = shfl_down_jac(S, d * W * H);
        if (r == 0 && (k & (2 * d - 1)) == 0 && k + d < (uint32_t)L) S = g1c::add_w<W>(S, o);
    }
    if (live && k == 0 && r == 0 && (threadIdx.x & (W - 1)) == 0) {
        uint32_t* dst = chunks + ((size_t)w * G + j) * 48;
        g1::store_jac(dst, S);
        g1::store_jac(dst + 24, run);
    }
}

// Sum of the n Jacobian points in sm[0 .. n) (n a power of two, n <= blockDim.x
// <= 256, one point per thread slot); the result lands in sm[0].  Wide levels
// use one thread per addition; once a level has at most one addition per warp,
// a whole warp takes each addition (its latency is a third of one thread's).
__device__ void block_tree_sum(uint32_t* sm, uint32_t n) {
    const uint32_t tid = threadIdx.x, warp = tid >> 5, nwarps = blockDim.x >> 5;
    uint32_t s = n;
    for (; (s >> 1) > nwarps; s >>= 1) {
        const uint32_t h = s >> 1;
        if (tid < h) g1::store_jac(sm + tid * 24, g1::add(g1::load_jac(sm + tid * 24), g1::load_jac(sm + (tid + h) * 24)));
        __syncthreads();
    }
    for (; s > 1; s >>= 1) {
        const uint32_t h = s >> 1;
        for (uint32_t q = warp; q < h; q += nwarps) {
            jac r = g1c::add(g1::load_jac(sm + q * 24), g1::load_jac(sm + (q + h) * 24));
            __syncwarp();
            if ((tid & 31) == 0) g1::store_jac(sm + q * 24, r);
        }
        __syncthreads();
    }
}

// Job 0 of a window sums every C_j; job 1 + t sums the R_j with bit t of j set.
// Block (w, job, part) of T threads (a power of two, 32 .. 256) sums the
// job's terms [part T m, (part + 1) T m), m per thread.
__global__ void __launch_bounds__(REDUCE_TPB) k_reduce_jobs(const uint32_t* __restrict__ chunks, int w_lo, uint32_t G,
                                                            uint32_t jobs, uint32_t parts, uint32_t m,
                                                            uint32_t* __restrict__ partials) {
    __shared__ uint32_t sm[REDUCE_TPB * 24];
    const uint32_t part = blockIdx.x % parts, job = (blockIdx.x / parts) % jobs;
    const uint32_t w = (uint32_t)w_lo + blockIdx.x / (parts * jobs);
    const uint32_t terms = job == 0 ? G : G >> 1;
    const uint32_t tb = job == 0 ? 0 : job - 1;  // the bit of job 1 + tb
    jac acc = g1::jac_inf();
    const uint32_t k0 = (part * blockDim.x + threadIdx.x) * m;
    for (uint32_t k = k0; k < k0 + m && k < terms; k++) {
        uint32_t jdx, half;
        if (job == 0) {
            jdx = k;
            half = 0;  // C_j
        } else {  // the k-th index with bit tb set
            jdx = ((k >> tb) << (tb + 1)) | (1u << tb) | (k & ((1u << tb) - 1u));
            half = 24;  // R_j
        }
        acc = g1::add(acc, g1::load_jac(chunks + ((size_t)w * G + jdx) * 48 + half));
    }
    g1::store_jac(sm + threadIdx.x * 24, acc);
    __syncthreads();
    block_tree_sum(sm, blockDim.x);
    if (threadIdx.x < 24) partials[((size_t)(w * jobs + job) * parts + part) * 24 + threadIdx.x] = sm[threadIdx.x];
}

// One block of two warps per (window, job): it sums the job's partial sums
// and shifts the result to its weight -- V_t by 2^t L (t + log2 L
// doublings), the sum of C_j not at all -- so that the bits are weighted in
// parallel rather than by a sequential Horner pass.  The doublings run on the
// warp pair in residue arithmetic (g1_proj.cuh): a chain of them is
// latency-bound, and there a doubling costs two rounds of RNS products
// (about 400 cycles each, six products to a round) instead of three levels of
// positional ones (about 870).  The shifted value replaces the job's first
// partial sum.
__global__ void __launch_bounds__(64) k_reduce_shift(uint32_t* __restrict__ partials, int w_lo, uint32_t jobs,
                                                     uint32_t parts, uint32_t log2L) {
    __shared__ __align__(16) uint32_t xch[g1p::kXchWords];
    const uint32_t w = (uint32_t)w_lo + blockIdx.x / jobs, q = blockIdx.x % jobs;
    uint32_t* src = partials + (size_t)(w * jobs + q) * parts * 24;
    jac acc = g1::load_jac(src);  // both warps sum the parts (cooperatively within each)
    for (uint32_t p = 1; p < parts; p++) acc = g1c::add(acc, g1::load_jac(src + p * 24));
    const uint32_t shift = q == 0 ? 0 : q - 1 + log2L;
    if (shift) {
        g1p::Pair P = g1p::make_pair(xch);
        acc = g1p::dbl_n_positional(P, acc, (int)shift);
    }
    __syncthreads();
    if (threadIdx.x == 0) g1::store_jac(src, acc);
}

// One block per window, one warp per job: a tree over the jobs' shifted
// values gives T_w = sum C_j + L sum_t 2^t V_t.
__global__ void __launch_bounds__(32 * MAX_REDUCE_JOBS) k_reduce_final(const uint32_t* __restrict__ partials, int w_lo,
                                                                       uint32_t jobs, uint32_t parts,
                                                                       uint32_t* __restrict__ wsums) {
    __shared__ uint32_t sm[MAX_REDUCE_JOBS * 24];
    const uint32_t w = (uint32_t)w_lo + blockIdx.x;
    const uint32_t q = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t span = 1;
    while (span < jobs) span <<= 1;
    // the tree runs over span = 2^k >= jobs values; the block has one warp per
    // job, so its first threads set the span - jobs padding values to infinity
    if (threadIdx.x < span - jobs) g1::store_jac(sm + (jobs + threadIdx.x) * 24, g1::jac_inf());
    if (q < jobs && lane < 24) sm[q * 24 + lane] = partials[(size_t)(w * jobs + q) * parts * 24 + lane];
    __syncthreads();
    for (uint32_t h = span >> 1; h >= 1; h >>= 1) {
        if (q < h) {
            jac r = g1c::add(g1::load_jac(sm + q * 24), g1::load_jac(sm + (q + h) * 24));
            __syncwarp();
            if (lane == 0) g1::store_jac(sm + q * 24, r);
        }
        __syncthreads();
    }
    if (threadIdx.x < 24) wsums[(size_t)w * 24 + threadIdx.x] = sm[threadIdx.x];
}

// ---------------------------------------------------------- 7. combination

// Two warps: Horner's rule over windows w_hi-1 .. w_lo (the chain of about
// nbits - c doublings is the latency floor of the whole MSM), run in residue
// arithmetic and projective coordinates (g1_proj.cuh): six groups of ten
// lanes compute a round of six products at once, each a 32-bit product per
// residue and two short base extensions, about 400 cycles where a positional
// product is about 870; a doubling is two rounds, an addition two.  The first
// group starts from its top window, a later one from the running value in acc
// (projective positional form, g1p::ppos); the result is doubled shift_after
// more times (a later group's bits, in the pipelined schedule) and goes to
// acc, or, from the last group, to out as a Jacobian point.
__global__ void __launch_bounds__(64) k_combine_part(const uint32_t* __restrict__ wsums, int w_hi, int w_lo,
                                                     Windows L, uint32_t* __restrict__ acc,
                                                     uint32_t* __restrict__ out, int first, int last,
                                                     int shift_after) {
    __shared__ __align__(16) uint32_t xch[g1p::kXchWords];
    if (blockIdx.x != 0 || threadIdx.x >= 64) return;
    g1p::Pair P = g1p::make_pair(xch);
    const g1p::rproj q0 = first ? g1p::to_proj(P, g1::load_jac(wsums + (size_t)(w_hi - 1) * 24))
                                : g1p::from_ppos(P, g1p::load_ppos(acc));
    // Q = 2^(off_{w+1} - off_w) Q + T_w, the shift being window w's width
    g1p::rproj q = g1p::horner_proj(
        P, q0, first ? w_hi - 2 : w_hi - 1, w_lo, [&](int w) { return window_width(L, w); },
        [&](int w) { return g1::load_jac(wsums + (size_t)w * 24); });
    q = g1p::dbl_n(P, q, shift_after);
    if (last) {
        const jac r = g1p::to_jac(P, q);
        if (threadIdx.x == 0) g1::store_jac(out, r);
    } else {
        const g1p::ppos r = g1p::to_ppos(P, q);
        if (threadIdx.x == 0) g1p::store_ppos(acc, r);
    }
}

// In the pipelined schedule a later group's windows w_lo .. w_hi-1 enter the
// running value Q as Q' = 2^(off_hi - off_lo) Q + L, where L is the group's
// own Horner value (k_combine_part with first = 1 into loc, on the group's
// stream).  The shift depends on the earlier groups only: the chain kernel
// before this one applies it (shift_after) while the group still
// accumulates, so the group's sums leave only L's shorter chain and this
// addition on the critical path; the join then applies the next group's
// shift.  acc and loc hold projective positional points.
__global__ void __launch_bounds__(64) k_combine_join(uint32_t* __restrict__ acc, const uint32_t* __restrict__ loc,
                                                     uint32_t* __restrict__ out, int last, int shift_after) {
    __shared__ __align__(16) uint32_t xch[g1p::kXchWords];
    if (blockIdx.x != 0 || threadIdx.x >= 64) return;
    g1p::Pair P = g1p::make_pair(xch);
    g1p::rproj a, b;
    g1p::from_ppos2(P, g1p::load_ppos(acc), g1p::load_ppos(loc), a, b);
    const g1p::rproj q = g1p::dbl_n(P, g1p::add(P, a, b), shift_after);
    if (last) {
        const jac r = g1p::to_jac(P, q);
        if (threadIdx.x == 0) g1::store_jac(out, r);
    } else {
        const g1p::ppos r = g1p::to_ppos(P, q);
        if (threadIdx.x == 0) g1p::store_ppos(acc, r);
    }
}

// Batches: one warp pair per MSM m, Horner's rule over its windows [m W, (m + 1) W).
__global__ void __launch_bounds__(64) k_combine_batch(const uint32_t* __restrict__ wsums, Windows L,
                                                      uint32_t* __restrict__ out) {
    __shared__ __align__(16) uint32_t xch[g1p::kXchWords];
    const uint32_t m = blockIdx.x;
    const uint32_t* ws = wsums + (size_t)m * L.W * 24;
    g1p::Pair P = g1p::make_pair(xch);
    const jac q = g1p::horner(
        P, g1::load_jac(ws + (size_t)(L.W - 1) * 24), L.W - 2, 0, [&](int w) { return window_width(L, w); },
        [&](int w) { return g1::load_jac(ws + (size_t)w * 24); });
    if (threadIdx.x == 0) g1::store_jac(out + (size_t)m * 24, q);
}

// infinity into out[blockIdx.x] (one block per result)
__global__ void k_write_inf(uint32_t* out) {
    if (threadIdx.x == 0) g1::store_jac(out + (size_t)blockIdx.x * 24, g1::jac_inf());
}

// ------------------------------------------------------ generator multiples

// table[j] = [2^j]G, affine Montgomery; one thread doubles, then all normalise
__global__ void k_gen_table_jac(uint32_t* __restrict__ tj) {
    if (threadIdx.x != 0) return;
    jac g{fq::one(), fq::one(), fq::one()};
    g.Y = fq::dbl(g.Y);  // (1, 2, 1) in Montgomery form
    for (int j = 0; j < 256; j++) {
        g1::store_jac(tj + j * 24, g);
        g = g1::dbl(g);
    }
}

__global__ void k_gen_table_norm(const uint32_t* __restrict__ tj, uint32_t* __restrict__ table) {
    int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < 256) g1::store_aff(table + j * 16, g1::to_aff(g1::load_jac(tj + j * 24)));
}

__global__ void k_mul_generator(const uint32_t* __restrict__ scalars, size_t n, const uint32_t* __restrict__ table,
                                uint32_t* __restrict__ out) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t k[8];
    load_scalar(scalars + 8 * i, k);
    jac acc = g1::jac_inf();
    for (int j = 0; j < 256; j++)
        if ((k[j >> 5] >> (j & 31)) & 1) acc = g1::add_mixed(acc, g1::load_aff(table + j * 16));
    g1::store_aff(out + i * 16, g1::to_aff(acc));
}

}  // namespace msm

// ============================================================== host side

using namespace msm;

static const int kPhases = 7;

struct msm_g1_ctx {
    int device;
    size_t max_n;
    int max_c;
    uint64_t cap_entries;  // padded entries
    uint64_t cap_buckets;  // W * B
    uint64_t cap_chunks;   // W * G
    uint64_t cap_pairs;    // pair-list entries over all tree levels
    size_t scratch_bytes;
    char* scratch;
    uint32_t *counts, *offsets, *cursor, *tile_sums, *entries, *items, *chunks, *wsums, *gen_table, *gen_tj;
    uint32_t* partials;    // partial sums of the bucket-reduction jobs
    uint32_t* msm_off;     // term offsets of the MSMs of a batch (device)
    uint64_t cap_windows, cap_partials;
    uint32_t* pairs;
    uint32_t* qacc;        // running value of the window combination, then one value per window group
    uint32_t* jsum;        // Jacobian bucket sums of buckets finished outside the tree
    uint32_t* phi;         // phi(P_i) = (beta x_i, y_i) for the GLV split
    int glv;               // 1: split scalars by the endomorphism (default)
    int inv_kind;          // batch inversion: 0 safegcd (default), 1 Fermat
    int finish_t;          // 0: automatic
    Resident resident[3];  // resident accumulation threads for tpb = 64, 128, 256
    int groups;            // window groups of the pipelined schedule (1 = serial)
    bool streams_ok;       // the context's own streams and events exist
    bool slice_sort_ok;    // the shared-memory sort kernels may take 128 KB of shared memory
    bool shared_place_ok;  // the accumulation kernels may keep prefix products in shared memory
    // graph replay of small MSMs: the last captured run and its arguments
    int graph_on;                 // MSM_G1_PARAM_GRAPH
    cudaStream_t cap_stream;      // where runs are captured and replayed
    cudaEvent_t ev_in, ev_out;    // the caller's stream -> cap_stream -> the caller's stream
    cudaGraphExec_t gexec;
    const void* gkey_ptr[4];      // points, scalars, out, and 1 for the host-buffer entry
    size_t gkey_n;
    int gkey_c;
    int sms;               // streaming multiprocessors of the device
    cudaStream_t acc_stream[MAX_GROUPS], chain_stream;
    cudaEvent_t ev_fork, ev_group[MAX_GROUPS], ev_chain;
    cudaStream_t side_stream;    // points upload and phi beside the sort
    cudaEvent_t ev_side, ev_points;
    uint32_t* stage;             // host-buffer entry: device copies of points, scalars and the result
    size_t stage_n;
    ctl_t* ctl;
    bool gen_ready;
    int batch_s, tpb, timing, stats;
    int acc_place;         // MSM_G1_PARAM_ACC_PLACEMENT
    int grid;              // MSM_G1_PARAM_GRID (0: automatic)
    int last_launches;
    cudaEvent_t ev[kPhases + 1];
    bool events_made;
    bool have_timing;
    int last_levels;
    // plan of the last run: small-bucket threshold, buckets per reduction chunk, window groups
    uint32_t last_finish_t, last_chunk_len, last_groups;
};

static int window_count(int c) { return make_windows(c, PLAIN_BITS).W; }
static int glv_window_count(int c) { return make_windows(c, GLV_BITS).W; }
static uint32_t reduce_chunk_len(uint32_t B) {
    // L = 4 (2 for windows of at most 8 bits) keeps each chunk's running sum
    // short (2L additions); from B = 2^13
    // on, L grows so that G = B / L stays <= 2^12 and the subset sums of the
    // reduction ((1 + log2 G) G / 2 additions per window) stay small
    // (measured at n = 2^22, c = 16: G = 8192 made the subset sums 0.36 ms)
    // (n = 2^10, c = 8, B = 128: L = 2 made the MSM 0.400 -> 0.388 ms; at
    // n = 2^16, c = 13, B = 4096 it was slower, 0.698 -> 0.729 ms)
    uint32_t L = B <= 128 ? 2 : 4;
    while ((uint64_t)L * 4096 < B) L <<= 1;
    return std::min(L, B);
}

static uint32_t ilog2(uint32_t x) {
    uint32_t r = 0;
    while ((1u << (r + 1)) <= x) r++;
    return r;
}

// Reduction jobs of one window (sum of C_j, and one V_t per bit of the chunk
// index) and their split into partial blocks of 256 threads x m terms.
struct ReducePlan {
    uint32_t L, G, jobs, parts, m, tpb;
};
// m, the terms each thread adds before the block tree, is the smallest power
// of two that keeps parts <= REDUCE_MAX_PARTS (a longer per-thread chain cost
// more than a second wave of blocks when measured).
static ReducePlan reduce_plan(uint32_t B) {
    ReducePlan r;
    r.L = reduce_chunk_len(B);
    r.G = B / r.L;
    r.jobs = 1 + ilog2(r.G);
    r.m = 1;
    // blocks of the next power of two >= G threads, 32 .. 256: a small job
    // (G = 32 at c = 8) would leave most of a 256-thread block adding infinities
    r.tpb = 32;
    while (r.tpb < 256 && r.tpb < r.G) r.tpb <<= 1;
    auto parts_for = [&](uint32_t m) { return (r.G + r.tpb * m - 1) / (r.tpb * m); };
    while (parts_for(r.m) > REDUCE_MAX_PARTS) r.m <<= 1;
    r.parts = parts_for(r.m);
    return r;
}

struct sizing {
    uint64_t points, entries, buckets, chunks, pairs, partials, windows;
};

// Level pair-list capacities for at most h_ub level-1 items in nb buckets:
// level l lists at most h_ub / 2^l + min(nb, h_ub / 2^(l-1)) / 2 pairs (a bucket
// contributes floor(ceil(h / 2^(l-1)) / 2) <= h / 2^l + 1/2, and only buckets
// with h > 2^(l-1) contribute).
static uint64_t level_cap(uint64_t h_ub, uint64_t nb, int l) {
    uint64_t live = std::min(nb, (h_ub >> (l - 1)) + 1);
    return (h_ub >> l) + 1 + (live + 1) / 2;
}

// Automatic small-bucket threshold: small MSMs are latency-bound in the
// narrow tail of the pair tree, large ones are throughput-bound throughout
// (GB300 with the cooperative reduction: n = 2^16, T = 2 / 4 / 8 / 16: 0.912 /
// 0.926 / 0.898 / 0.977 ms; 2^10, T = 4 / 8 / 16: 0.549 / 0.545 / 0.538 ms;
// from 2^20 every T >= 2 was slower).
static int auto_finish(uint64_t n, int W, uint32_t B, uint64_t resident) {
    const uint64_t pairs1 = n * (uint64_t)W / 4;  // about the level-1 pairs
    if (pairs1 >= 8 * resident) return 1;
    if (pairs1 >= 2 * resident) return 8;
    // buckets so few that four threads share each finish chain (k_finish_chunks):
    // no tree level beyond level 0 (n = 2^10, c = 8: 0.341 ms at T = 16,
    // 0.333 at T = 20 ... 48)
    if ((uint64_t)W * B * 8 <= resident / 4) return 32;
    return 16;
}

// The tree levels worth a launch of their own for terms_pw terms per window
// over B buckets: a bucket's level-1 item count h is about terms / (2 B) for
// uniform scalars (Poisson-like), so the largest one is below
// h_max = h + 6 sqrt(h) + 8, and level l has pairs while
// ceil(h_max / 2^(l-1)) > T.  Deeper levels are left to the deep-level
// launch, which normally finds them empty (n = 2^22: 9 levels instead of 22
// per window group).
static int dense_levels(uint64_t terms_pw, uint32_t B, uint32_t finish_t) {
    const double h = (double)terms_pw / (2.0 * (double)B);
    const double hmax = h + 6.0 * sqrt(h) + 8.0;
    const double t = finish_t > 1 ? (double)finish_t : 1.0;
    int l = 1;
    while (l < MAX_LEVELS && hmax / (double)(1ull << (l - 1)) > t) l++;
    return l - 1 < 1 ? 1 : l - 1;
}

// Window groups (top windows first) and their pair-list layout.  Two groups
// (small MSMs) split unevenly: the top group takes about a quarter of the
// windows, floor((W + 2) / 4).  Its sums then exist earlier, and the
// doublings that must follow them -- about all the bits below the top window --
// start earlier, while the larger lower group's own Horner chain is shorter
// than that (GB300, n = 2^16, W = 10: top 3 0.790 ms, even split 0.810, top 2
// 0.817; n = 2^10, W = 16: top 4 0.450, 5 0.452, 6 0.456, even 0.457).
static PairLayout make_layout(uint64_t n, int W, uint32_t B, int groups, uint64_t* total) {
    PairLayout lay;
    memset(&lay, 0, sizeof(lay));
    groups = std::max(1, std::min(groups, std::min(W, MAX_GROUPS)));
    lay.groups = groups;
    lay.B = B;
    const int per = (W + groups - 1) / groups;
    const int top = groups == 2 ? std::max(1, (W + 2) / 4) : per;
    uint64_t base = 0;
    for (int j = 0; j < groups; j++) {
        lay.w_hi[j] = std::max(0, j == 0 ? W : W - top - (j - 1) * per);
        lay.w_lo[j] = std::max(0, W - top - j * per);
        if (j == groups - 1) lay.w_lo[j] = 0;
        const uint64_t nw = (uint64_t)(lay.w_hi[j] - lay.w_lo[j]);
        const uint64_t nbj = nw * B;
        const uint64_t h_ub = (n * nw + nbj + 1) / 2;
        for (int l = 1; l < MAX_LEVELS; l++) {
            uint64_t cap = nw ? level_cap(h_ub, nbj, l) : 0;
            lay.base[j][l] = (uint32_t)base;
            lay.cap[j][l] = (uint32_t)cap;
            base += cap;
        }
    }
    if (total) *total = base;
    return lay;
}

// max_batch: MSMs fused in one pass (their per-bucket and per-window
// buffers scale with it; max_n bounds the terms of the whole pass)
static sizing size_for(size_t max_n, int max_c, int max_batch = 1) {
    sizing s{max_n, 0, 0, 0, 0, 0, 0};
    const uint64_t kb = (uint64_t)std::max(1, max_batch);
    // entries for windows down to 8 bits (smaller windows fit smaller n); the
    // GLV split doubles the terms and about halves the windows
    const int cmin = std::min(max_c, 8);
    s.entries = (uint64_t)max_n * std::max(window_count(cmin), 2 * glv_window_count(cmin));
    for (int c = 1; c <= max_c; c++) {
        uint64_t B = 1ull << (c - 1);
        uint64_t wb = (uint64_t)window_count(c) * B;
        const ReducePlan rp = reduce_plan((uint32_t)B);
        const uint64_t wg = (uint64_t)window_count(c) * rp.G;
        s.buckets = std::max(s.buckets, wb * kb);
        s.chunks = std::max(s.chunks, wg * kb);
        s.partials = std::max(s.partials, (uint64_t)window_count(c) * rp.jobs * rp.parts * kb);
    }
    s.windows = std::max<uint64_t>(256, std::min<uint64_t>(MAX_BATCH_WINDOWS, s.buckets));
    s.entries += s.buckets;  // one padding entry per bucket at most
    s.entries += 2;
    // pair lists: the largest grouped layout over the windows this context allows
    for (int c = 1; c <= max_c; c++) {
        for (int glv = 0; glv <= 1; glv++) {
            const int W = glv ? glv_window_count(c) : window_count(c);
            const uint64_t terms = std::min<uint64_t>((uint64_t)max_n << glv, (s.entries - s.buckets) / W);
            for (int groups = 1; groups <= MAX_GROUPS; groups++) {
                uint64_t t = 0;
                make_layout(terms, W, 1u << (c - 1), groups, &t);
                s.pairs = std::max(s.pairs, t);
            }
            if (kb > 1) {  // a fused batch: one group over kb W windows
                uint64_t t = 0;
                make_layout((terms + kb - 1) / kb, (int)(W * kb), 1u << (c - 1), 1, &t);
                s.pairs = std::max(s.pairs, t);
            }
        }
    }
    return s;
}

static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

static size_t layout(msm_g1_ctx* c, const sizing& s, bool assign) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align_up(bytes);
        return o;
    };
    size_t o_ctl = take(sizeof(ctl_t));
    size_t o_counts = take(4 * s.buckets);
    size_t o_offsets = take(4 * (s.buckets + 1));
    size_t o_cursor = take(4 * s.buckets);
    size_t o_tiles = take(4 * (s.buckets / SCAN_TILE + 2));
    size_t o_entries = take(4 * s.entries);
    size_t o_items = take((size_t)64 * ((s.entries + 1) / 2));
    size_t o_chunks = take((size_t)192 * s.chunks);  // C_j, R_j per chunk
    size_t o_partials = take((size_t)96 * s.partials);
    size_t o_wsums = take((size_t)96 * s.windows);
    size_t o_msm_off = take((size_t)4 * (s.windows + 1));
    size_t o_table = take((size_t)64 * 256);
    size_t o_tj = take((size_t)96 * 256);
    size_t o_pairs = take((size_t)4 * s.pairs);
    size_t o_qacc = take((size_t)96 * (1 + MAX_GROUPS));  // running value, one local value per group
    size_t o_jsum = take((size_t)96 * s.buckets);
    size_t o_phi = take((size_t)64 * s.points);
    if (assign) {
        c->phi = (uint32_t*)(c->scratch + o_phi);
        c->jsum = (uint32_t*)(c->scratch + o_jsum);
        c->pairs = (uint32_t*)(c->scratch + o_pairs);
        c->qacc = (uint32_t*)(c->scratch + o_qacc);
        c->ctl = (ctl_t*)(c->scratch + o_ctl);
        c->counts = (uint32_t*)(c->scratch + o_counts);
        c->offsets = (uint32_t*)(c->scratch + o_offsets);
        c->cursor = (uint32_t*)(c->scratch + o_cursor);
        c->tile_sums = (uint32_t*)(c->scratch + o_tiles);
        c->entries = (uint32_t*)(c->scratch + o_entries);
        c->items = (uint32_t*)(c->scratch + o_items);
        c->chunks = (uint32_t*)(c->scratch + o_chunks);
        c->partials = (uint32_t*)(c->scratch + o_partials);
        c->msm_off = (uint32_t*)(c->scratch + o_msm_off);
        c->wsums = (uint32_t*)(c->scratch + o_wsums);
        c->gen_table = (uint32_t*)(c->scratch + o_table);
        c->gen_tj = (uint32_t*)(c->scratch + o_tj);
    }
    return off;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// Makes a context's device current for one entry point and gives the caller
// back its own current device on return, so a call never moves the caller's
// thread to another GPU.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            prev = -1;
            return;
        }
        ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
    DeviceGuard(const DeviceGuard&) = delete;
    DeviceGuard& operator=(const DeviceGuard&) = delete;
};

#define CK(call)                                  \
    do {                                          \
        if ((call) != cudaSuccess) return MSM_G1_ERR_CUDA; \
    } while (0)

extern "C" {

int msm_g1_window_count(int c) {
    if (c < 1 || c > MSM_G1_MAX_WINDOW) return MSM_G1_ERR_INVALID_ARG;
    return window_count(c);
}

int msm_g1_auto_window(size_t n) {
    if (n < 2) return 4;
    double lg = 0;
    while (((size_t)1 << (int)(lg + 1)) <= n && lg < 62) lg += 1;
    int c = (int)(0.8 * lg + 0.5);
    return std::max(4, std::min(18, c));
}

int msm_g1_create(msm_g1_ctx** out, size_t max_n, int max_c) { return msm_g1_create_batch(out, max_n, max_c, 1); }

size_t msm_g1_scratch_bytes(size_t max_n, int max_c) {
    if (max_n < 1 || max_c < 1 || max_c > MSM_G1_MAX_WINDOW) return 0;
    return layout(nullptr, size_for(max_n, max_c), false);
}

const char* msm_g1_strerror(int code) {
    switch (code) {
        case MSM_G1_OK: return "ok";
        case MSM_G1_ERR_INVALID_ARG: return "invalid argument";
        case MSM_G1_ERR_CUDA: return "CUDA error";
        case MSM_G1_ERR_CAPACITY: return "context capacity exceeded";
        case MSM_G1_ERR_ALLOC: return "allocation failed";
        case MSM_G1_ERR_NO_DEVICE: return "no usable CUDA device (compute capability 10.3 required)";
        default: return "unknown error";
    }
}

int msm_g1_create_batch(msm_g1_ctx** out, size_t max_n, int max_c, int max_batch) {
    if (!out) return MSM_G1_ERR_INVALID_ARG;
    *out = nullptr;
    if (max_n < 1 || max_n > (1ull << 30) || max_c < 1 || max_c > MSM_G1_MAX_WINDOW) return MSM_G1_ERR_INVALID_ARG;
    if (max_batch < 1 || max_batch > (int)MAX_BATCH_WINDOWS) return MSM_G1_ERR_INVALID_ARG;
    sizing s = size_for(max_n, max_c, max_batch);
    if (s.entries >= (1ull << 31) || s.pairs >= (1ull << 32)) return MSM_G1_ERR_INVALID_ARG;  // 32-bit offsets
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MSM_G1_ERR_NO_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MSM_G1_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return MSM_G1_ERR_NO_DEVICE;
    msm_g1_ctx* c = (msm_g1_ctx*)calloc(1, sizeof(msm_g1_ctx));
    if (!c) return MSM_G1_ERR_ALLOC;
    c->device = dev;
    c->sms = prop.multiProcessorCount;
    c->max_n = max_n;
    c->max_c = max_c;
    c->cap_entries = s.entries;
    c->cap_buckets = s.buckets;
    c->cap_chunks = s.chunks;
    c->cap_pairs = s.pairs;
    c->cap_windows = s.windows;
    c->cap_partials = s.partials;
    c->scratch_bytes = layout(nullptr, s, false);
    if (cudaMalloc((void**)&c->scratch, c->scratch_bytes) != cudaSuccess) {
        cudaGetLastError();
        free(c);
        return MSM_G1_ERR_ALLOC;
    }
    layout(c, s, true);
    c->batch_s = 0;
    c->tpb = 0;
    c->timing = 0;
    c->glv = 1;
    c->resident[0] = accum_resident_threads(64);
    c->resident[1] = accum_resident_threads(128);
    c->resident[2] = accum_resident_threads(256);
    c->groups = 0;
    c->graph_on = 1;
    {
        int lo = 0, hi = 0;
        bool ok = cudaDeviceGetStreamPriorityRange(&lo, &hi) == cudaSuccess;
        // accumulation streams at the lowest priority, the combination chain at
        // the greatest, so its single-warp kernels start as soon as they may
        // (graded priorities per group were measured slower at n = 2^22)
        for (int j = 0; j < MAX_GROUPS; j++)
            ok = ok && cudaStreamCreateWithPriority(&c->acc_stream[j], cudaStreamNonBlocking, lo) == cudaSuccess;
        ok = ok && cudaStreamCreateWithPriority(&c->chain_stream, cudaStreamNonBlocking, hi) == cudaSuccess;
        ok = ok && cudaStreamCreateWithPriority(&c->side_stream, cudaStreamNonBlocking, hi) == cudaSuccess;
        ok = ok && cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->ev_in, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->ev_out, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->ev_side, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->ev_points, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->ev_chain, cudaEventDisableTiming) == cudaSuccess;
        for (int j = 0; j < MAX_GROUPS; j++)
            ok = ok && cudaEventCreateWithFlags(&c->ev_group[j], cudaEventDisableTiming) == cudaSuccess;
        cudaGetLastError();
        c->streams_ok = ok;  // without them every run takes the serial schedule
        const int smem = 4 << 15;  // B = 2^15 counters, window width 16
        c->slice_sort_ok =
            cudaFuncSetAttribute(k_hist_slices, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
            cudaFuncSetAttribute(k_scatter_slices, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
        cudaGetLastError();
        c->shared_place_ok = accum_prepare_device();
    }
    *out = c;
    return MSM_G1_OK;
}

void msm_g1_destroy(msm_g1_ctx* c) {
    if (!c) return;
    const DeviceGuard dg(c->device);
    cudaDeviceSynchronize();
    if (c->events_made)
        for (int i = 0; i <= kPhases; i++) cudaEventDestroy(c->ev[i]);
    for (int j = 0; j < MAX_GROUPS; j++)
        if (c->acc_stream[j]) cudaStreamDestroy(c->acc_stream[j]);
    if (c->chain_stream) cudaStreamDestroy(c->chain_stream);
    if (c->side_stream) cudaStreamDestroy(c->side_stream);
    if (c->gexec) cudaGraphExecDestroy(c->gexec);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    if (c->ev_in) cudaEventDestroy(c->ev_in);
    if (c->ev_out) cudaEventDestroy(c->ev_out);
    if (c->ev_side) cudaEventDestroy(c->ev_side);
    if (c->ev_points) cudaEventDestroy(c->ev_points);
    if (c->stage) cudaFree(c->stage);
    if (c->ev_fork) cudaEventDestroy(c->ev_fork);
    if (c->ev_chain) cudaEventDestroy(c->ev_chain);
    for (int j = 0; j < MAX_GROUPS; j++)
        if (c->ev_group[j]) cudaEventDestroy(c->ev_group[j]);
    cudaFree(c->scratch);
    free(c);
}

// Every parameter shapes the captured launches: a change drops the graph
// (after the replays in flight).
static void drop_graph(msm_g1_ctx* c) {
    if (!c->gexec) return;
    cudaStreamSynchronize(c->cap_stream);
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
}

int msm_g1_set_param(msm_g1_ctx* c, int key, int value) {
    if (!c) return MSM_G1_ERR_INVALID_ARG;
    drop_graph(c);
    switch (key) {
        case MSM_G1_PARAM_BATCH_S:
            if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8 && value != 16 && value != 32 &&
                value != 64)
                return MSM_G1_ERR_INVALID_ARG;
            c->batch_s = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_TPB:
            if (value != 0 && value != 64 && value != 128 && value != 256) return MSM_G1_ERR_INVALID_ARG;
            c->tpb = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_TIMING:
            if (value != 0 && value != 1) return MSM_G1_ERR_INVALID_ARG;
            c->timing = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_STATS:
            if (value != 0 && value != 1) return MSM_G1_ERR_INVALID_ARG;
            c->stats = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_GROUPS:
            if (value < 0 || value > MAX_GROUPS) return MSM_G1_ERR_INVALID_ARG;
            c->groups = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_FINISH:
            if (value < 0 || value > 64) return MSM_G1_ERR_INVALID_ARG;
            c->finish_t = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_GLV:
            if (value != 0 && value != 1) return MSM_G1_ERR_INVALID_ARG;
            c->glv = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_INVERSION:
            if (value != 0 && value != 1) return MSM_G1_ERR_INVALID_ARG;
            c->inv_kind = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_GRAPH:
            if (value != 0 && value != 1) return MSM_G1_ERR_INVALID_ARG;
            c->graph_on = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_GRID:
            if (value < 0) return MSM_G1_ERR_INVALID_ARG;
            c->grid = value;
            return MSM_G1_OK;
        case MSM_G1_PARAM_ACC_PLACEMENT:
            if (value != MSM_G1_ACC_LOCAL && value != MSM_G1_ACC_SHARED && value != MSM_G1_ACC_REGISTERS)
                return MSM_G1_ERR_INVALID_ARG;
            if (value == MSM_G1_ACC_SHARED && !c->shared_place_ok) return MSM_G1_ERR_INVALID_ARG;
            c->acc_place = value;
            return MSM_G1_OK;
        default:
            return MSM_G1_ERR_INVALID_ARG;
    }
}

int msm_g1_get_param(const msm_g1_ctx* c, int key, int* value) {
    if (!c || !value) return MSM_G1_ERR_INVALID_ARG;
    switch (key) {
        case MSM_G1_PARAM_BATCH_S: *value = c->batch_s; return MSM_G1_OK;
        case MSM_G1_PARAM_TPB: *value = c->tpb; return MSM_G1_OK;
        case MSM_G1_PARAM_TIMING: *value = c->timing; return MSM_G1_OK;
        case MSM_G1_PARAM_STATS: *value = c->stats; return MSM_G1_OK;
        case MSM_G1_PARAM_GROUPS: *value = c->groups; return MSM_G1_OK;
        case MSM_G1_PARAM_FINISH: *value = c->finish_t; return MSM_G1_OK;
        case MSM_G1_PARAM_GLV: *value = c->glv; return MSM_G1_OK;
        case MSM_G1_PARAM_INVERSION: *value = c->inv_kind; return MSM_G1_OK;
        case MSM_G1_PARAM_GRAPH: *value = c->graph_on; return MSM_G1_OK;
        case MSM_G1_PARAM_GRID: *value = c->grid; return MSM_G1_OK;
        case MSM_G1_PARAM_ACC_PLACEMENT: *value = c->acc_place; return MSM_G1_OK;
        default: return MSM_G1_ERR_INVALID_ARG;
    }
}

}  // extern "C"

// The MSM.  points_host: when non-null, the points are copied from this host
// buffer into `points` (device) on the side stream while the sort runs.
static int run_core(msm_g1_ctx* c, const uint32_t* points, const uint32_t* scalars, size_t n, int window_c,
                    uint32_t* out, cudaStream_t st, const uint32_t* points_host, int count = 1,
                    const uint32_t* d_off = nullptr) {
    int cw = window_c == 0 ? std::min(msm_g1_auto_window(n), c->max_c) : window_c;
    if (cw < 1 || cw > MSM_G1_MAX_WINDOW) return MSM_G1_ERR_INVALID_ARG;
    if (cw > c->max_c || n > c->max_n) return MSM_G1_ERR_CAPACITY;
    // With GLV the MSM runs over 2n terms (P_i and phi(P_i)) with 128-bit windows.
    const bool glv = c->glv != 0;
    const Windows win = make_windows(cw, glv ? GLV_BITS : PLAIN_BITS);
    const int W = win.W;
    const uint64_t terms = glv ? 2 * (uint64_t)n : (uint64_t)n;
    const uint32_t nsplit = glv ? (uint32_t)n : HOLE;  // entry indices >= nsplit address phi
    const uint32_t B = 1u << (cw - 1);
    // a batch of `count` MSMs runs as one MSM over count W windows, MSM m
    // owning windows [m W, (m + 1) W)
    const int Wall = W * count;
    const uint32_t nb = (uint32_t)Wall * B;
    if (terms * W + nb + 2 > c->cap_entries || nb > c->cap_buckets) return MSM_G1_ERR_CAPACITY;
    {
        const ReducePlan rp0 = reduce_plan(B);
        if ((uint64_t)Wall > c->cap_windows || (uint64_t)Wall * rp0.G > c->cap_chunks ||
            (uint64_t)Wall * rp0.jobs * rp0.parts > c->cap_partials)
            return MSM_G1_ERR_CAPACITY;
    }
    const BatchMap bm{count > 1 ? d_off : nullptr, count};
    c->have_timing = false;
    if (c->timing && !c->events_made) {
        for (int i = 0; i <= kPhases; i++) CK(cudaEventCreate(&c->ev[i]));
        c->events_made = true;
    }
    auto mark = [&](int i) {
        if (c->timing) cudaEventRecord(c->ev[i], st);
    };
    if (n == 0) {
        CK(cudaMemsetAsync(c->ctl, 0, sizeof(ctl_t), st));
        k_write_inf<<<count, 32, 0, st>>>(out);
        c->last_launches = 1;
        return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
    }
    const int stats = c->stats;
    int launches = 0;
    // threads per accumulation block: automatic (0) takes 256 from 2^19 points
    // (GB300: n = 2^20 3.474 -> 3.430 ms, 2^22 11.14 -> 10.95 ms) and 128 below
    // (n = 2^16: 0.882 against 0.927 ms at 256)
    const int tpb = c->tpb ? c->tpb : (n >= ((size_t)1 << 19) ? 256 : 128);
    // Points side: upload (host-buffer entry) and phi need only the points and
    // run on the side stream beside the sort, which needs only the scalars;
    // level 0 waits for them.  With phase timing (or without context streams)
    // they run in order on the calling stream, inside the first phase.
    const bool side = c->streams_ok && !c->timing;
    auto points_side = [&](cudaStream_t s) -> int {
        if (points_host) CK(cudaMemcpyAsync((void*)points, points_host, 64ull * n, cudaMemcpyHostToDevice, s));
        if (glv) {
            k_phi<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(points, n, c->phi);
            launches++;
        }
        return MSM_G1_OK;
    };
    mark(0);
    if (side) {
        CK(cudaEventRecord(c->ev_side, st));
        CK(cudaStreamWaitEvent(c->side_stream, c->ev_side, 0));
        if (points_side(c->side_stream) != MSM_G1_OK) return MSM_G1_ERR_CUDA;
        CK(cudaEventRecord(c->ev_points, c->side_stream));
    } else if (points_side(st) != MSM_G1_OK) {
        return MSM_G1_ERR_CUDA;
    }
    CK(cudaMemsetAsync(c->ctl, 0, sizeof(ctl_t), st));
    CK(cudaMemsetAsync(c->counts, 0, 4ull * nb, st));
    // single MSMs with windows of at most 16 bits and 2^12 or more digits take
    // the shared-memory sort (digit codes once, slices of one window per
    // block); its code matrix lives in the item buffer, which the accumulation
    // fills only afterwards (against the per-term digits and scatter: n = 2^16,
    // c = 13, 0.698 -> 0.672 ms; n = 2^10, c = 8, 0.381 -> 0.359 ms)
    const bool slice_sort = c->slice_sort_ok && count == 1 && cw <= 16 && terms * W >= ((uint64_t)1 << 12);
    const size_t tstride = (size_t)((terms + 3) & ~(uint64_t)3);
    uint32_t* codes = c->items;
    const uint32_t slices = (uint32_t)std::max(1, c->sms / W);
    const size_t slice_t = (size_t)(((terms + slices - 1) / slices + 3) & ~(uint64_t)3);
    if (slice_sort) {
        unsigned blocks = (unsigned)((n + 255) / 256);
        if (glv) k_digit_codes<true><<<blocks, 256, 0, st>>>(scalars, n, win, tstride, codes);
        else k_digit_codes<false><<<blocks, 256, 0, st>>>(scalars, n, win, tstride, codes);
        k_hist_slices<<<(unsigned)W * slices, 1024, 4 * B, st>>>(codes, tstride, terms, slices, slice_t, B, c->counts);
        launches += 2;
    } else {
        unsigned blocks = (unsigned)((n + 255) / 256);
        if (glv) k_digits_hist<true><<<blocks, 256, 0, st>>>(scalars, n, cw, win, bm, c->counts);
        else k_digits_hist<false><<<blocks, 256, 0, st>>>(scalars, n, cw, win, bm, c->counts);
        launches++;
    }
    mark(1);
    const uint32_t ntiles = (nb + SCAN_TILE - 1) / SCAN_TILE;
    if (nb <= SCAN_SMALL_MAX) {
        k_scan_small<<<1, 1024, 0, st>>>(c->counts, nb, c->offsets, c->cursor, c->entries, c->ctl);
        launches -= 2;  // counted below as three
    } else {
        k_scan_reduce<<<ntiles, SCAN_TPB, 0, st>>>(c->counts, nb, c->tile_sums, c->ctl);
        k_scan_tiles<<<1, 1024, 0, st>>>(c->tile_sums, ntiles, c->ctl);
        k_scan_apply<<<ntiles, SCAN_TPB, 0, st>>>(c->counts, nb, c->tile_sums, c->offsets, c->cursor, c->entries,
                                                  c->ctl);
    }
    // Serial schedule (one stream, one window group) when phase timing is on --
    // the phase events then delimit whole phases -- or when the context has no
    // streams of its own; otherwise window groups are pipelined (below).
    // two groups for small MSMs, three from 2^19 points (GB300: n = 2^20 4.10 ->
    // 4.00 ms, 2^22 12.13 -> 12.07 ms; at 2^16 three were 3 % slower, four
    // slower everywhere)
    const int groups = c->groups ? c->groups : (n >= ((size_t)1 << 19) ? 3 : 2);
    const bool split_combine = n < ((size_t)1 << 19);
    const bool pipelined = c->streams_ok && !c->timing && groups > 1 && W > 1 && count == 1;
    uint64_t pairs_total = 0;
    // (a batch's windows hold only their own MSM's terms: ceil(terms / count)
    // per window bounds the entries of all of them together)
    const uint64_t terms_pw = (terms + count - 1) / count;
    PairLayout lay = make_layout(terms_pw, Wall, B, pipelined ? groups : 1, &pairs_total);
    lay.finish_t = (uint32_t)(c->finish_t ? c->finish_t : auto_finish(terms, W, B, c->resident[1].narrow));
    if (pairs_total > c->cap_pairs) return MSM_G1_ERR_CAPACITY;
    launch_build_pairs(c->offsets, nb, c->pairs, lay, c->ctl, st);
    launches += 4;
    mark(2);
    if (slice_sort) {
        // per-slice runs while the entry list fits in L2, else term order
        if (terms * W * 4 <= ((uint64_t)64 << 20))
            k_scatter_slices<<<(unsigned)W * slices, 1024, 4 * B, st>>>(codes, tstride, terms, slices, slice_t, B,
                                                                        c->cursor, c->entries);
        else
            k_scatter_codes<<<(unsigned)((terms + 255) / 256), 256, 0, st>>>(codes, tstride, terms, W, B, c->cursor,
                                                                             c->entries);
        launches++;
    } else {
        unsigned blocks = (unsigned)((n + 255) / 256);
        if (glv) k_scatter<true><<<blocks, 256, 0, st>>>(scalars, n, cw, win, bm, c->cursor, c->entries);
        else k_scatter<false><<<blocks, 256, 0, st>>>(scalars, n, cw, win, bm, c->cursor, c->entries);
        launches++;
    }
    mark(3);
    // the groups share the GPU in the pipelined schedule: size each grid for a share of it
    Resident resident = c->resident[tpb == 64 ? 0 : tpb == 128 ? 1 : 2];
    if (pipelined) {
        resident.narrow /= 2;
        resident.wide /= 2;
    }
    const ReducePlan rp = reduce_plan(B);
    const uint32_t L = rp.L, G = rp.G;
    if (rp.jobs > MAX_REDUCE_JOBS) return MSM_G1_ERR_INVALID_ARG;  // unreachable for c <= 20
    const AccumKnobs knobs{c->batch_s, tpb, c->acc_place, c->grid};
    c->last_finish_t = lay.finish_t;
    c->last_chunk_len = L;
    c->last_groups = (uint32_t)lay.groups;
    // one window group: level 0, the tree levels, the bucket reduction
    auto level0 = [&](int j, cudaStream_t s) {
        if (side) cudaStreamWaitEvent(s, c->ev_points, 0);
        const int nw = lay.w_hi[j] - lay.w_lo[j];
        launches += launch_accum_level0(knobs, resident, points, c->phi, nsplit, c->entries, c->offsets,
                                        (uint32_t)lay.w_lo[j] * B, (uint32_t)lay.w_hi[j] * B, c->items, c->ctl,
                                        (terms_pw * nw + (uint64_t)nw * B + 1) / 2, stats, c->inv_kind, s);
    };
    // Tree levels launched one by one: those uniform data fills (dense_levels);
    // the rest, usually empty, go to one deep-level launch.
    const int dense = dense_levels(terms_pw, B, lay.finish_t);
    auto tree = [&](int j, cudaStream_t s) {
        // levels while some bucket may still hold two items: 2^level < max bucket <= terms
        int level = 1;
        for (; level <= dense && level < MAX_LEVELS && ((uint64_t)1 << level) < terms; level++) {
            launches += launch_accum_level(knobs, resident, c->items, c->pairs, lay, c->ctl, j, level, stats,
                                           c->inv_kind, s);
        }
        if (level < MAX_LEVELS && ((uint64_t)1 << level) < terms) {
            launch_accum_deep(c->items, c->pairs, lay, c->ctl, j, level, stats, c->inv_kind, s);
            launches++;
        }
    };
    auto reduce = [&](int j, cudaStream_t s) {
        const int nw = lay.w_hi[j] - lay.w_lo[j];
        const uint32_t threads = (uint32_t)nw * G;
        // small MSMs: the finish and the chunk sums in one launch.  While the
        // buckets fill a quarter of the GPU at most, four threads share each
        // bucket's chain (n = 2^10: 0.355 -> 0.349 ms; eight-lane cooperative
        // additions on one chain took 0.355); above that the launch is bound by
        // issue slots and one thread per bucket is fastest (n = 2^16: 0.650 ms,
        // two threads 0.763, four 0.889).
        const bool small = (uint64_t)nw * B * 8 <= c->resident[1].narrow / 4;
        bool fused = lay.finish_t >= 2;
        if (fused) {
            const unsigned lanes = (unsigned)nw * B * (small ? 4 : 1);
            const unsigned blocks = (lanes + 127) / 128;
#define FC(HH, LL) k_finish_chunks<1, HH, LL><<<blocks, 128, 0, s>>>(c->items, c->offsets, lay.finish_t, \
                                                                    lay.w_lo[j], nw, B, G, c->chunks)
            if (small && L == 1) FC(4, 1);
            else if (small && L == 2) FC(4, 2);
            else if (small && L == 4) FC(4, 4);
            else if (small && L == 8) FC(4, 8);
            else if (L == 1) FC(1, 1);
            else if (L == 2) FC(1, 2);
            else if (L == 4) FC(1, 4);
            else if (L == 8) FC(1, 8);
            else fused = false;
#undef FC
        }
        if (!fused && lay.finish_t >= 2) {
            launch_finish(c->items, c->offsets, (uint32_t)lay.w_lo[j] * B, (uint32_t)lay.w_hi[j] * B, lay.finish_t,
                          c->jsum, c->resident[1].narrow, s);
            launches++;
        }
        if (!fused) {
            // cooperative groups while the chunks fill a quarter of the GPU at most
            // (n = 2^10, 512 chunks: reduction 0.22 -> 0.18 ms; at 2^16, with 5 k
            // chunks per group, they made the MSM 2 % slower: idle lanes multiply)
            if ((uint64_t)threads * 8 <= c->resident[1].narrow / 4)
                k_reduce_chunks<8><<<(threads * 8 + 127) / 128, 128, 0, s>>>(
                    c->items, c->counts, c->offsets, c->jsum, lay.finish_t, lay.w_lo[j], nw, B, L, G, c->chunks);
            else
                k_reduce_chunks<1><<<(threads + 127) / 128, 128, 0, s>>>(c->items, c->counts, c->offsets, c->jsum,
                                                                        lay.finish_t, lay.w_lo[j], nw, B, L, G,
                                                                        c->chunks);
        }
        k_reduce_jobs<<<(unsigned)nw * rp.jobs * rp.parts, rp.tpb, 0, s>>>(c->chunks, lay.w_lo[j], G, rp.jobs,
                                                                          rp.parts, rp.m, c->partials);
        k_reduce_shift<<<(unsigned)nw * rp.jobs, 64, 0, s>>>(c->partials, lay.w_lo[j], rp.jobs, rp.parts, ilog2(L));
        k_reduce_final<<<nw, 32 * rp.jobs, 0, s>>>(c->partials, lay.w_lo[j], rp.jobs, rp.parts, c->wsums);
        launches += 4;
    };
    // the bits of window group j (the shift a later group's own Horner value
    // needs before it joins the running value)
    auto group_bits = [&](int j) { return window_offset(win, lay.w_hi[j]) - window_offset(win, lay.w_lo[j]); };
    auto combine = [&](int j, cudaStream_t s, int shift_after) {
        if (count > 1)  // one warp pair per MSM of the batch
            k_combine_batch<<<count, 64, 0, s>>>(c->wsums, win, out);
        else
            k_combine_part<<<1, 64, 0, s>>>(c->wsums, lay.w_hi[j], lay.w_lo[j], win, c->qacc, out, j == 0,
                                            j == lay.groups - 1, shift_after);
        launches++;
    };
    if (!pipelined) {
        level0(0, st);
        mark(4);
        tree(0, st);
        mark(5);
        reduce(0, st);
        mark(6);
        combine(0, st, 0);
        mark(7);
    } else {
        // Window groups, top windows first, each on its own accumulation
        // stream; the combination chain runs on a high-priority stream and
        // takes each group's window sums as soon as that group is done, so the
        // long doubling chain overlaps the accumulation of the lower windows and
        // the latency-bound tail of one group overlaps the next group's work.
        CK(cudaEventRecord(c->ev_fork, st));
        for (int j = 0; j < lay.groups; j++) CK(cudaStreamWaitEvent(c->acc_stream[j], c->ev_fork, 0));
        CK(cudaStreamWaitEvent(c->chain_stream, c->ev_fork, 0));
        for (int j = 0; j < lay.groups; j++) {
            cudaStream_t s = c->acc_stream[j];
            level0(j, s);
            tree(j, s);
            reduce(j, s);
            // below 2^19 points the later groups' combination is split (n = 2^10:
            // 0.714 -> 0.675 ms, 2^16: 1.071 -> 1.048 ms); for larger MSMs, with
            // three groups, the group's own Horner chain on its low-priority
            // stream waited behind the accumulation (2^20: 3.84 -> 3.91 ms)
            // (with the split, each chain kernel also shifts the running value
            // past the next group's windows while that group accumulates)
            const int shift_next = split_combine && j + 1 < lay.groups ? group_bits(j + 1) : 0;
            if (j == 0 || !split_combine) {
                CK(cudaEventRecord(c->ev_group[j], s));
                CK(cudaStreamWaitEvent(c->chain_stream, c->ev_group[j], 0));
                combine(j, c->chain_stream, shift_next);
                continue;
            }
            // the group's own Horner value on its stream; on the chain the join
            // with the running value, already shifted past the group's windows
            uint32_t* loc = c->qacc + 24 * (1 + j);
            k_combine_part<<<1, 64, 0, s>>>(c->wsums, lay.w_hi[j], lay.w_lo[j], win, loc, out, 1, 0, 0);
            CK(cudaEventRecord(c->ev_group[j], s));
            CK(cudaStreamWaitEvent(c->chain_stream, c->ev_group[j], 0));
            k_combine_join<<<1, 64, 0, c->chain_stream>>>(c->qacc, loc, out, j == lay.groups - 1, shift_next);
            launches += 2;
        }
        CK(cudaEventRecord(c->ev_chain, c->chain_stream));
        CK(cudaStreamWaitEvent(st, c->ev_chain, 0));
    }
    c->last_launches = launches;
    if (cudaGetLastError() != cudaSuccess) return MSM_G1_ERR_CUDA;
    c->have_timing = c->timing != 0;
    return MSM_G1_OK;
}

// Small MSMs are a few dozen short, latency-bound launches; replayed as one
// CUDA graph they start back to back (GB300: n = 2^10 0.655 -> 0.592 ms, 2^16
// 1.057 -> 0.992 ms per MSM; at 2^20 the graph was 2 % slower, so larger
// MSMs launch eagerly).  A call of msm_g1_run (or of msm_g1_run_host, with its
// copies, when its host buffers are page-locked) is captured on the context's
// capture stream the first time a (points, scalars, out, n, c) combination is seen -- an
// existing executable graph is updated in place when the launches keep their
// shape -- and replayed while the arguments and the parameters stay the same;
// the buffers' contents may change between calls, since the kernels read them
// when they run.  Not while the caller's own stream is being captured (the run
// then becomes part of the caller's graph as usual).
static bool pinned(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

static bool graph_eligible(const msm_g1_ctx* c, size_t n, cudaStream_t st) {
    if (!c->graph_on || !c->streams_ok || c->timing || n == 0 || n >= ((size_t)1 << 19)) return false;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs == cudaStreamCaptureStatusNone;
}

// body(stream) enqueues the whole call on `stream`; key names its arguments.
template <class Body>
static int run_graph(msm_g1_ctx* c, const void* const (&key)[4], size_t n, int window_c, cudaStream_t st,
                     Body&& body) {
    bool hit = c->gexec && c->gkey_n == n && c->gkey_c == window_c;
    for (int i = 0; i < 4; i++) hit = hit && c->gkey_ptr[i] == key[i];
    if (!hit) {
        if (cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            cudaGetLastError();
            return body(st);
        }
        const int rc = body(c->cap_stream);
        cudaGraph_t g = nullptr;
        const cudaError_t ec = cudaStreamEndCapture(c->cap_stream, &g);
        if (rc != MSM_G1_OK || ec != cudaSuccess || !g) {
            if (g) cudaGraphDestroy(g);
            cudaGetLastError();
            return rc != MSM_G1_OK ? rc : MSM_G1_ERR_CUDA;
        }
        if (c->gexec) {
            cudaGraphExecUpdateResultInfo info;
            if (cudaGraphExecUpdate(c->gexec, g, &info) != cudaSuccess) {
                cudaGetLastError();
                drop_graph(c);
            }
        }
        if (!c->gexec && cudaGraphInstantiate(&c->gexec, g, 0) != cudaSuccess) {
            cudaGetLastError();
            c->gexec = nullptr;
            cudaGraphDestroy(g);
            return MSM_G1_ERR_CUDA;
        }
        cudaGraphDestroy(g);
        for (int i = 0; i < 4; i++) c->gkey_ptr[i] = key[i];
        c->gkey_n = n;
        c->gkey_c = window_c;
    }
    CK(cudaEventRecord(c->ev_in, st));
    CK(cudaStreamWaitEvent(c->cap_stream, c->ev_in, 0));
    CK(cudaGraphLaunch(c->gexec, c->cap_stream));
    CK(cudaEventRecord(c->ev_out, c->cap_stream));
    CK(cudaStreamWaitEvent(st, c->ev_out, 0));
    return MSM_G1_OK;
}

extern "C" int msm_g1_run(msm_g1_ctx* c, const uint32_t* points, const uint32_t* scalars, size_t n, int window_c,
                          uint32_t* out, cudaStream_t st) {
    if (!c || !out || !aligned16(out)) return MSM_G1_ERR_INVALID_ARG;
    if (n > 0 && (!points || !scalars || !aligned16(points) || !aligned16(scalars))) return MSM_G1_ERR_INVALID_ARG;
    const DeviceGuard dg(c->device);
    if (!dg.ok) return MSM_G1_ERR_CUDA;
    auto body = [&](cudaStream_t s) { return run_core(c, points, scalars, n, window_c, out, s, nullptr); };
    if (graph_eligible(c, n, st)) {
        const void* const key[4] = {points, scalars, out, nullptr};
        return run_graph(c, key, n, window_c, st, body);
    }
    return body(st);
}

extern "C" int msm_g1_run_batch(msm_g1_ctx* c, const uint32_t* points, const uint32_t* scalars, const size_t* offsets,
                                int count, int window_c, uint32_t* out, cudaStream_t st) {
    if (!c || !out || !aligned16(out) || !offsets || count < 1) return MSM_G1_ERR_INVALID_ARG;
    if (offsets[0] != 0) return MSM_G1_ERR_INVALID_ARG;
    size_t largest = 0;
    for (int m = 0; m < count; m++) {
        if (offsets[m + 1] < offsets[m]) return MSM_G1_ERR_INVALID_ARG;
        largest = std::max(largest, offsets[m + 1] - offsets[m]);
    }
    const size_t total = offsets[count];
    if (total > 0 && (!points || !scalars || !aligned16(points) || !aligned16(scalars))) return MSM_G1_ERR_INVALID_ARG;
    if (largest > c->max_n) return MSM_G1_ERR_CAPACITY;
    const int cw = window_c == 0 ? std::min(msm_g1_auto_window(largest), c->max_c) : window_c;
    if (cw < 1 || cw > MSM_G1_MAX_WINDOW) return MSM_G1_ERR_INVALID_ARG;
    if (cw > c->max_c) return MSM_G1_ERR_CAPACITY;
    const int glv = c->glv != 0;
    const int W = make_windows(cw, glv ? GLV_BITS : PLAIN_BITS).W;
    const uint64_t B = 1ull << (cw - 1);
    const ReducePlan rp = reduce_plan((uint32_t)B);
    const DeviceGuard dg(c->device);
    if (!dg.ok) return MSM_G1_ERR_CUDA;
    // Greedy passes: as many consecutive MSMs as the context's buffers hold.
    int m0 = 0;
    while (m0 < count) {
        int cnt = 0;
        uint64_t terms = 0;
        while (m0 + cnt < count) {
            const uint64_t t2 = terms + (offsets[m0 + cnt + 1] - offsets[m0 + cnt]);
            const uint64_t k = (uint64_t)cnt + 1;
            const uint64_t wall = k * W;
            uint64_t pairs = 0;
            make_layout(((t2 << glv) + k - 1) / k, (int)std::min<uint64_t>(wall, 1u << 30), (uint32_t)B, 1, &pairs);
            const bool fits = t2 <= c->max_n && wall <= c->cap_windows && wall * B <= c->cap_buckets &&
                              (t2 << glv) * W + wall * B + 2 <= c->cap_entries && wall * rp.G <= c->cap_chunks &&
                              wall * rp.jobs * rp.parts <= c->cap_partials && pairs <= c->cap_pairs;
            if (!fits) break;
            terms = t2;
            cnt++;
        }
        if (cnt == 0) return MSM_G1_ERR_CAPACITY;  // one MSM always fits a context made for it
        uint32_t off[MAX_BATCH_WINDOWS + 1];
        for (int m = 0; m <= cnt; m++) off[m] = (uint32_t)(offsets[m0 + m] - offsets[m0]);
        // from pageable memory: the copy is staged before the call returns
        CK(cudaMemcpyAsync(c->msm_off, off, 4ull * (cnt + 1), cudaMemcpyHostToDevice, st));
        const size_t base = offsets[m0];
        int rc = run_core(c, points ? points + 16 * base : nullptr, scalars ? scalars + 8 * base : nullptr, terms, cw,
                          out + 24 * (size_t)m0, st, nullptr, cnt, c->msm_off);
        if (rc != MSM_G1_OK) return rc;
        m0 += cnt;
    }
    return MSM_G1_OK;
}

extern "C" int msm_g1_run_host(msm_g1_ctx* c, const uint32_t* points_host, const uint32_t* scalars_host, size_t n,
                               int window_c, uint32_t* out_host, cudaStream_t st) {
    if (!c || !out_host) return MSM_G1_ERR_INVALID_ARG;
    if (n > 0 && (!points_host || !scalars_host)) return MSM_G1_ERR_INVALID_ARG;
    if (n > c->max_n) return MSM_G1_ERR_CAPACITY;
    const DeviceGuard dg(c->device);
    if (!dg.ok) return MSM_G1_ERR_CUDA;
    if (!c->stage) {  // first call: device copies of points, scalars and the result, for max_n
        size_t bytes = 96 * c->max_n + 256;
        if (cudaMalloc((void**)&c->stage, bytes) != cudaSuccess) {
            cudaGetLastError();
            c->stage = nullptr;
            return MSM_G1_ERR_ALLOC;
        }
        c->stage_n = c->max_n;
    }
    uint32_t* pts = c->stage;
    uint32_t* sc = c->stage + 16 * c->stage_n;
    uint32_t* res = c->stage + 24 * c->stage_n;  // 96 B, 16-byte aligned (offset 96 max_n)
    auto body = [&](cudaStream_t s) -> int {
        if (n > 0) CK(cudaMemcpyAsync(sc, scalars_host, 32ull * n, cudaMemcpyHostToDevice, s));
        // the points are copied by run_core beside the sort (in order on s when
        // the context has no streams or times phases)
        int rc = run_core(c, pts, sc, n, window_c, res, s, n > 0 ? points_host : nullptr);
        if (rc != MSM_G1_OK) return rc;
        CK(cudaMemcpyAsync(out_host, res, 96, cudaMemcpyDeviceToHost, s));
        return MSM_G1_OK;
    };
    // replayed as a graph like msm_g1_run, when all three host buffers are
    // page-locked (copies of pageable memory cannot be captured)
    if (graph_eligible(c, n, st) && pinned(points_host) && pinned(scalars_host) && pinned(out_host)) {
        const void* const key[4] = {points_host, scalars_host, out_host, (const void*)1};
        return run_graph(c, key, n, window_c, st, body);
    }
    return body(st);
}

extern "C" int msm_g1_last_phase_ms(msm_g1_ctx* c, float* ms, int nphase) {
    if (!c || !ms || nphase < 0) return MSM_G1_ERR_INVALID_ARG;
    if (!c->have_timing) return 0;
    CK(cudaEventSynchronize(c->ev[kPhases]));
    int k = std::min(nphase, kPhases);
    for (int i = 0; i < k; i++) CK(cudaEventElapsedTime(&ms[i], c->ev[i], c->ev[i + 1]));
    return k;
}

extern "C" int msm_g1_last_stats(msm_g1_ctx* c, uint64_t* out, int nout) {
    if (!c || !out || nout < 0) return MSM_G1_ERR_INVALID_ARG;
    ctl_t h;
    const DeviceGuard dg(c->device);
    if (!dg.ok) return MSM_G1_ERR_CUDA;
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(&h, c->ctl, sizeof(h), cudaMemcpyDeviceToHost));
    uint64_t v[11] = {h.entries, h.nonempty, h.max_count, h.adds, h.inversions, h.levels,
                      (uint64_t)c->last_launches, h.error, c->last_finish_t, c->last_chunk_len, c->last_groups};
    int k = std::min(nout, 11);
    for (int i = 0; i < k; i++) out[i] = v[i];
    return k;
}

extern "C" int msm_g1_mul_generator(msm_g1_ctx* c, const uint32_t* scalars, size_t n, uint32_t* out,
                                    cudaStream_t st) {
    if (!c) return MSM_G1_ERR_INVALID_ARG;
    if (n == 0) return MSM_G1_OK;
    if (!scalars || !out || !aligned16(scalars) || !aligned16(out)) return MSM_G1_ERR_INVALID_ARG;
    const DeviceGuard dg(c->device);
    if (!dg.ok) return MSM_G1_ERR_CUDA;
    if (!c->gen_ready) {
        k_gen_table_jac<<<1, 32, 0, st>>>(c->gen_tj);
        k_gen_table_norm<<<2, 128, 0, st>>>(c->gen_tj, c->gen_table);
        c->gen_ready = true;
    }
    k_mul_generator<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(scalars, n, c->gen_table, out);
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_debug_read(msm_g1_ctx* c, int which, void* dst, size_t max_bytes, size_t* bytes) {
    if (!c || !dst || !bytes) return MSM_G1_ERR_INVALID_ARG;
    const DeviceGuard dg(c->device);
    if (!dg.ok) return MSM_G1_ERR_CUDA;
    CK(cudaDeviceSynchronize());
    ctl_t h;
    CK(cudaMemcpy(&h, c->ctl, sizeof(h), cudaMemcpyDeviceToHost));
    (void)h;
    const void* src = nullptr;
    size_t sz = 0;
    // sizes come from the last run's window: recover nb from the offsets buffer length is not
    // stored, so the caller passes max_bytes and reads what it needs
    switch (which) {
        case 0: src = c->counts; sz = 4 * c->cap_buckets; break;
        case 1: src = c->offsets; sz = 4 * (c->cap_buckets + 1); break;
        case 2: src = c->entries; sz = 4 * (size_t)h.total; break;
        default: return MSM_G1_ERR_INVALID_ARG;
    }
    *bytes = sz;
    size_t k = std::min(sz, max_bytes);
    if (k) CK(cudaMemcpy(dst, src, k, cudaMemcpyDeviceToHost));
    return MSM_G1_OK;
}

// ====================================================== allocation-free entry
//
// msm_g1_run_noalloc serves callers that must not allocate device memory
// themselves -- code whose device heap is owned by another allocator (a
// framework's caching allocator that accounts for every byte), services with a
// fixed memory budget, or hot paths that cannot afford cudaMalloc's implicit
// device-wide synchronisation.  It runs the same kernels as msm_g1_run, with
// all scratch carved from one fixed array in device global memory that every
// GPU loading this library holds until the process exits.
//
// Host code must not take the array's name as a device address: the device
// address of each GPU's copy is fetched once per device with
// cudaGetSymbolAddress, with that device current, on the first call.

#define NOALLOC_MAX_N 4096
#define NOALLOC_MAX_C 10
#define NOALLOC_SCRATCH_BYTES (8u << 20)

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoallocDevices = 64;
std::mutex g_noalloc_lock;
void* g_noalloc_ptr[kNoallocDevices];
Resident g_noalloc_resident[kNoallocDevices][3];
}  // namespace

extern "C" int msm_g1_run_noalloc(const uint32_t* points, const uint32_t* scalars, size_t n, int window_c,
                                  uint32_t* out, cudaStream_t stream) {
    if (n > NOALLOC_MAX_N) return MSM_G1_ERR_CAPACITY;
    int cw = window_c == 0 ? std::min(msm_g1_auto_window(n), NOALLOC_MAX_C) : window_c;
    if (cw < 1 || cw > MSM_G1_MAX_WINDOW) return MSM_G1_ERR_INVALID_ARG;
    if (cw > NOALLOC_MAX_C) return MSM_G1_ERR_CAPACITY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocDevices) return MSM_G1_ERR_NO_DEVICE;
    const sizing s = size_for(NOALLOC_MAX_N, NOALLOC_MAX_C);
    if (layout(nullptr, s, false) > NOALLOC_SCRATCH_BYTES) return MSM_G1_ERR_CAPACITY;
    {
        std::lock_guard<std::mutex> guard(g_noalloc_lock);
        if (!g_noalloc_ptr[dev]) {
            cudaDeviceProp prop;
            if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MSM_G1_ERR_NO_DEVICE;
            if (prop.major != 10 || prop.minor != 3) return MSM_G1_ERR_NO_DEVICE;
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
                cudaGetLastError();
                return MSM_G1_ERR_CUDA;
            }
            g_noalloc_resident[dev][0] = accum_resident_threads(64);
            g_noalloc_resident[dev][1] = accum_resident_threads(128);
            g_noalloc_resident[dev][2] = accum_resident_threads(256);
            g_noalloc_ptr[dev] = ptr;
        }
    }
    // a context on the host stack whose buffers all point into the fixed array
    msm_g1_ctx c;
    memset(&c, 0, sizeof(c));
    c.device = dev;
    c.max_n = NOALLOC_MAX_N;
    c.max_c = NOALLOC_MAX_C;
    c.cap_entries = s.entries;
    c.cap_buckets = s.buckets;
    c.cap_chunks = s.chunks;
    c.cap_pairs = s.pairs;
    c.cap_windows = s.windows;
    c.cap_partials = s.partials;
    c.scratch = (char*)g_noalloc_ptr[dev];
    c.scratch_bytes = NOALLOC_SCRATCH_BYTES;
    layout(&c, s, true);
    c.batch_s = 0;
    c.tpb = 128;
    c.glv = 1;
    for (int i = 0; i < 3; i++) c.resident[i] = g_noalloc_resident[dev][i];
    return msm_g1_run(&c, points, scalars, n, cw, out, stream);
}
