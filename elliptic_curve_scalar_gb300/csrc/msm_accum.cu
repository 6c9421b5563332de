// msm_accum.cu -- bucket accumulation by batched affine pair additions.
//
// Level 0 adds the two points of each even-aligned entry pair of the sorted
// bucket list; level l >= 1 halves every bucket's remaining items in place.
// Each thread runs its pairs in batches of S that share one field inversion
// (Montgomery's trick, see batch_pairs in msm_core.cuh), the amortisation the
// pages study as "walkerS" (PR #23736 "stream-walker -- amortize the field
// inversion via large S + private pref_scratch", section "Goal & lever").
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "msm_internal.cuh"

using fq::fe;
using g1::aff;

namespace msm {

__device__ __forceinline__ void warp_stats(ctl_t* ctl, int adds, int invs) {
    unsigned a = __reduce_add_sync(__activemask(), (unsigned)adds);
    unsigned v = __reduce_add_sync(__activemask(), (unsigned)invs);
    if ((threadIdx.x & 31) == __ffs(__activemask()) - 1) {
        if (a) atomicAdd(&ctl->adds, (unsigned long long)a);
        if (v) atomicAdd(&ctl->inversions, (unsigned long long)v);
    }
}

// level 0: pair u = entries (2u, 2u+1) of the sorted list; operands are input
// points gathered by index, negated when the entry's flag says so.
template <int S>
struct Level0Src {
    const uint32_t* points;
    uint32_t* items;
    uint32_t e0[S], e1[S];
    uint32_t u0;
    __device__ __forceinline__ const uint32_t* pt(uint32_t e) const { return points + (size_t)(e & ~SIGN) * 16; }
    __device__ __forceinline__ bool has_q(int k) const { return e1[k] != HOLE; }
    __device__ __forceinline__ fe xp(int k) const { return fq::load(pt(e0[k])); }
    __device__ __forceinline__ fe xq(int k) const { return fq::load(pt(e1[k])); }
    __device__ __forceinline__ fe yof(uint32_t e) const {
        fe y = fq::load(pt(e) + 8);
        return (e & SIGN) ? fq::neg(y) : y;
    }
    __device__ __forceinline__ void ys(int k, fe& a, fe& b) const {
        a = yof(e0[k]);
        b = yof(e1[k]);
    }
    __device__ __forceinline__ aff p(int k) const { return aff{xp(k), yof(e0[k])}; }
    __device__ __forceinline__ aff q(int k) const { return aff{xq(k), yof(e1[k])}; }
    __device__ __forceinline__ void store(int k, const aff& r) { g1::store_aff(items + (size_t)(u0 + k) * 16, r); }
};

template <int S>
__global__ void __launch_bounds__(256) k_accum_level0(const uint32_t* __restrict__ points,
                                                      const uint32_t* __restrict__ entries,
                                                      uint32_t* __restrict__ items, ctl_t* ctl, int stats) {
    const uint32_t units = ctl->total >> 1;
    size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t u0 = t * S;
    if (u0 >= units) return;
    int count = (int)min((size_t)S, (size_t)units - u0);
    Level0Src<S> src;
    src.points = points;
    src.items = items;
    src.u0 = (uint32_t)u0;
#pragma unroll
    for (int k = 0; k < S; k++) {
        uint2 e = k < count ? reinterpret_cast<const uint2*>(entries)[u0 + k] : make_uint2(HOLE, HOLE);
        src.e0[k] = e.x;
        src.e1[k] = e.y;
    }
    int adds = batch_pairs<S>(src, count);
    if (stats) warp_stats(ctl, adds, 1);
}

// level l >= 1: items of bucket g sit at o_g + i*2^(l-1) (o_g = offset_g / 2);
// pair j is (o_g + j*2^l, o_g + j*2^l + 2^(l-1)) and its sum replaces the first.
template <int S>
struct LevelSrc {
    uint32_t* items;
    uint32_t half;
    uint32_t qi[S];  // index of each pair's first item
    __device__ __forceinline__ const uint32_t* a(int k) const { return items + (size_t)qi[k] * 16; }
    __device__ __forceinline__ const uint32_t* b(int k) const { return items + (size_t)(qi[k] + half) * 16; }
    __device__ __forceinline__ bool has_q(int) const { return true; }
    __device__ __forceinline__ fe xp(int k) const { return fq::load(a(k)); }
    __device__ __forceinline__ fe xq(int k) const { return fq::load(b(k)); }
    __device__ __forceinline__ void ys(int k, fe& ya, fe& yb) const {
        ya = fq::load(a(k) + 8);
        yb = fq::load(b(k) + 8);
    }
    __device__ __forceinline__ aff p(int k) const { return g1::load_aff(a(k)); }
    __device__ __forceinline__ aff q(int k) const { return g1::load_aff(b(k)); }
    __device__ __forceinline__ void store(int k, const aff& r) { g1::store_aff(items + (size_t)qi[k] * 16, r); }
};

template <int S>
__global__ void __launch_bounds__(256) k_accum_level(uint32_t* __restrict__ items, const uint32_t* __restrict__ offsets,
                                                     uint32_t nb, ctl_t* ctl, int level, int stats) {
    const uint32_t step = 1u << level;
    if (ctl->max_count <= step) return;  // every bucket already holds at most one item
    const uint32_t H = ctl->total >> 1;  // level-1 index space
    const uint64_t K = (uint64_t)S * step;
    uint64_t q0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * K;
    if (q0 >= H) return;
    uint64_t q1 = min(q0 + K, (uint64_t)H);
    const uint32_t half = step >> 1;
    const int sh = level - 1;
    // last bucket g with o_g <= q0
    uint32_t lo = 0, hi = nb;  // invariant: o_lo <= q0 < o_hi (o_nb = H)
    while (hi - lo > 1) {
        uint32_t mid = (lo + hi) >> 1;
        if ((offsets[mid] >> 1) <= q0) lo = mid; else hi = mid;
    }
    LevelSrc<S> src;
    src.items = items;
    src.half = half;
    int adds = 0, invs = 0;
    // iterator over the pairs whose first item lies in [q0, q1): bucket g, next
    // pair j in [j, jhi).  Batches are filled here and run below at one
    // program point per round, so the lanes of a warp execute each batch (and
    // its inversion) together instead of one divergent group after another.
    const unsigned live = __activemask();
    uint32_t g = lo;
    uint32_t og = offsets[g] >> 1;
    uint64_t j = 0, jhi = 0;
    bool more = true;
    auto enter_bucket = [&]() {
        uint32_t on = offsets[g + 1] >> 1;
        uint32_t h = on - og;                                  // level-1 items of bucket g
        uint32_t np = ((h + (1u << sh) - 1) >> sh) >> 1;       // pairs at this level
        j = q0 > og ? (q0 - og + step - 1) >> level : 0;
        jhi = min((uint64_t)np, (q1 - og + step - 1) >> level);
        return on;
    };
    uint32_t on = enter_bucket();
    for (;;) {
        int count = 0;
        while (count < S && more) {
            if (j < jhi) {
                src.qi[count++] = og + (uint32_t)(j << level);
                j++;
            } else {
                g++;
                og = on;
                if (g >= nb || og >= q1) {
                    more = false;
                } else {
                    on = enter_bucket();
                }
            }
        }
        if (__ballot_sync(live, count > 0) == 0) break;
        if (count > 0) {
            adds += batch_pairs<S>(src, count);
            invs++;
        }
    }
    if (stats) {
        warp_stats(ctl, adds, invs);
        if (invs && threadIdx.x == 0) atomicMax(&ctl->levels, (uint32_t)level + 1);
    }
}


template <int S>
static void level0_t(int tpb, const uint32_t* points, const uint32_t* entries, uint32_t* items, ctl_t* ctl,
                     uint64_t units_ub, int stats, cudaStream_t st) {
    uint64_t threads = (units_ub + S - 1) / S;
    uint64_t blocks = std::max<uint64_t>(1, (threads + tpb - 1) / tpb);
    k_accum_level0<S><<<(unsigned)blocks, tpb, 0, st>>>(points, entries, items, ctl, stats);
}

template <int S>
static void level_t(int tpb, uint32_t* items, const uint32_t* offsets, uint32_t nb, ctl_t* ctl, uint64_t h_ub,
                    int level, int stats, cudaStream_t st) {
    uint64_t K = (uint64_t)S << level;
    uint64_t threads = (h_ub + K - 1) / K;
    uint64_t blocks = std::max<uint64_t>(1, (threads + tpb - 1) / tpb);
    k_accum_level<S><<<(unsigned)blocks, tpb, 0, st>>>(items, offsets, nb, ctl, level, stats);
}

void launch_accum_level0(int batch_s, int tpb, const uint32_t* points, const uint32_t* entries, uint32_t* items,
                         ctl_t* ctl, uint64_t units_ub, int stats, cudaStream_t st) {
    switch (batch_s) {
        case 1: level0_t<1>(tpb, points, entries, items, ctl, units_ub, stats, st); break;
        case 2: level0_t<2>(tpb, points, entries, items, ctl, units_ub, stats, st); break;
        case 4: level0_t<4>(tpb, points, entries, items, ctl, units_ub, stats, st); break;
        case 16: level0_t<16>(tpb, points, entries, items, ctl, units_ub, stats, st); break;
        case 32: level0_t<32>(tpb, points, entries, items, ctl, units_ub, stats, st); break;
        default: level0_t<8>(tpb, points, entries, items, ctl, units_ub, stats, st); break;
    }
}

void launch_accum_level(int batch_s, int tpb, uint32_t* items, const uint32_t* offsets, uint32_t nb, ctl_t* ctl,
                        uint64_t h_ub, int level, int stats, cudaStream_t st) {
    switch (batch_s) {
        case 1: level_t<1>(tpb, items, offsets, nb, ctl, h_ub, level, stats, st); break;
        case 2: level_t<2>(tpb, items, offsets, nb, ctl, h_ub, level, stats, st); break;
        case 4: level_t<4>(tpb, items, offsets, nb, ctl, h_ub, level, stats, st); break;
        case 16: level_t<16>(tpb, items, offsets, nb, ctl, h_ub, level, stats, st); break;
        case 32: level_t<32>(tpb, items, offsets, nb, ctl, h_ub, level, stats, st); break;
        default: level_t<8>(tpb, items, offsets, nb, ctl, h_ub, level, stats, st); break;
    }
}

}  // namespace msm
