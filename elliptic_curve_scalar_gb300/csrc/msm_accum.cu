// msm_accum.cu -- bucket accumulation by batched affine pair additions.
//
// The buckets are reduced by a pair tree, the pages' level-wise accumulator
// ("ba_fused_super", "the bin-packed pair-tree bucket-accumulate that runs for
// every level of the MSM, with level 0 being the largest single dispatch",
// PR #23520 "cache dx + idx in ba_fused_super pref_scratch", section "Summary"):
//
//  * level 0 adds the two entries of every even-aligned pair (2u, 2u+1) of the
//    sorted bucket list (buckets are padded to even length, so a pair never
//    straddles two buckets) and writes the sum to item u;
//  * level l >= 1 adds items (q, q + 2^(l-1)) into q, halving every bucket's
//    items in place until each bucket holds one point, its bucket sum.
//
// Which pairs exist at each level depends only on the bucket sizes, so one
// kernel lists them for all levels up front (the pages' chunk_plan plays the
// same role).  Every thread then takes a contiguous chunk of a level's list
// and adds its pairs in batches that share one field inversion (Montgomery's
// trick, batch_pairs in msm_core.cuh) -- the amortisation the pages study as
// "walkerS" (PR #23736 "stream-walker -- amortize the field inversion via large
// S + private pref_scratch", section "Goal & lever").  The chunk is
// min(S, ceil(pairs / threads)): wide levels fill batches of S, narrow levels
// spread their few pairs one per thread for the shortest latency.
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

// ------------------------------------------------------------------ level 0

// pair u = entries (2u, 2u+1); operands are input points gathered by index,
// negated when the entry's flag says so; a padding second entry means "copy".
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
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t chunk = min((uint64_t)S, ((uint64_t)units + nthreads - 1) / nthreads);
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t u0 = t * chunk;
    if (u0 >= units) return;
    const int count = (int)min(chunk, (uint64_t)units - u0);
    Level0Src<S> src;
    src.points = points;
    src.items = items;
    src.u0 = (uint32_t)u0;
    for (int k = 0; k < count; k++) {
        uint2 e = reinterpret_cast<const uint2*>(entries)[u0 + k];
        src.e0[k] = e.x;
        src.e1[k] = e.y;
    }
    int adds = batch_pairs<S>(src, count);
    if (stats) warp_stats(ctl, adds, 1);
}

// ------------------------------------------------------- pair lists per level

// Bucket g's level-1 items occupy [o_g, o_g + h_g) with o_g = offset_g / 2;
// at level l it holds n_l = ceil(h_g / 2^(l-1)) items at stride 2^(l-1), which
// form floor(n_l / 2) pairs, pair j starting at o_g + j 2^l.  One thread per
// bucket; the lanes of a warp reserve list space with one atomic per level.
__global__ void k_build_pairs(const uint32_t* __restrict__ offsets, uint32_t nb, uint32_t* __restrict__ pairs,
                              PairLayout lay, ctl_t* ctl) {
    const uint32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    uint32_t og = 0, h = 0;
    if (g < nb) {
        og = offsets[g] >> 1;
        h = (offsets[g + 1] >> 1) - og;
    }
    for (int level = 1; level < MAX_LEVELS; level++) {
        const int sh = level - 1;
        uint32_t nl = h ? ((h - 1) >> sh) + 1 : 0;
        uint32_t np = nl >> 1;
        if (!__any_sync(0xffffffffu, np != 0)) break;
        uint32_t incl = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t base = 0;
        if (lane == 31) base = atomicAdd(&ctl->pair_count[level], total);
        base = __shfl_sync(0xffffffffu, base, 31);
        uint32_t off = base + incl - np;
        uint32_t* list = pairs + lay.base[level];
        const uint32_t cap = lay.cap[level];
        for (uint32_t j = 0; j < np; j++) {
            uint32_t idx = off + j;
            if (idx < cap) list[idx] = og + (j << level);
            else atomicOr(&ctl->error, 1u);  // capacity bound violated (never expected)
        }
    }
}

// ------------------------------------------------------------- levels >= 1

// pair (q, q + 2^(l-1)) of the level's list; its sum replaces the first item
template <int S>
struct ListSrc {
    uint32_t* items;
    uint32_t half;
    uint32_t qi[S];
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
__global__ void __launch_bounds__(256) k_accum_list(uint32_t* __restrict__ items, const uint32_t* __restrict__ list,
                                                    ctl_t* ctl, int level, int stats) {
    const uint32_t cnt = ctl->pair_count[level];
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t chunk = min((uint64_t)S, ((uint64_t)cnt + nthreads - 1) / nthreads);
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t i0 = t * chunk;
    if (i0 >= cnt) return;
    const int count = (int)min(chunk, (uint64_t)cnt - i0);
    ListSrc<S> src;
    src.items = items;
    src.half = 1u << (level - 1);
    for (int k = 0; k < count; k++) src.qi[k] = list[i0 + k];
    int adds = batch_pairs<S>(src, count);
    if (stats) {
        warp_stats(ctl, adds, 1);
        if (threadIdx.x == 0) atomicMax(&ctl->levels, (uint32_t)level + 1);
    }
}

// ----------------------------------------------------------------- launchers

static unsigned grid_for(uint64_t work, int S, int tpb, uint64_t resident) {
    // enough threads for chunks of S, but at least one resident wave when the
    // level may hold that much work
    uint64_t threads = std::max((work + S - 1) / S, std::min(work, resident));
    return (unsigned)std::max<uint64_t>(1, (threads + tpb - 1) / tpb);
}

template <int S>
static void level0_t(int tpb, uint64_t resident, const uint32_t* points, const uint32_t* entries, uint32_t* items,
                     ctl_t* ctl, uint64_t units_ub, int stats, cudaStream_t st) {
    k_accum_level0<S><<<grid_for(units_ub, S, tpb, resident), tpb, 0, st>>>(points, entries, items, ctl, stats);
}

template <int S>
static void list_t(int tpb, uint64_t resident, uint32_t* items, const uint32_t* list, ctl_t* ctl, uint64_t cap,
                   int level, int stats, cudaStream_t st) {
    k_accum_list<S><<<grid_for(cap, S, tpb, resident), tpb, 0, st>>>(items, list, ctl, level, stats);
}

void launch_accum_level0(int batch_s, int tpb, uint64_t resident, const uint32_t* points, const uint32_t* entries,
                         uint32_t* items, ctl_t* ctl, uint64_t units_ub, int stats, cudaStream_t st) {
    switch (batch_s) {
        case 1: level0_t<1>(tpb, resident, points, entries, items, ctl, units_ub, stats, st); break;
        case 2: level0_t<2>(tpb, resident, points, entries, items, ctl, units_ub, stats, st); break;
        case 4: level0_t<4>(tpb, resident, points, entries, items, ctl, units_ub, stats, st); break;
        case 8: level0_t<8>(tpb, resident, points, entries, items, ctl, units_ub, stats, st); break;
        case 16: level0_t<16>(tpb, resident, points, entries, items, ctl, units_ub, stats, st); break;
        default: level0_t<32>(tpb, resident, points, entries, items, ctl, units_ub, stats, st); break;
    }
}

void launch_build_pairs(const uint32_t* offsets, uint32_t nb, uint32_t* pairs, const PairLayout& lay, ctl_t* ctl,
                        cudaStream_t st) {
    k_build_pairs<<<(nb + 255) / 256, 256, 0, st>>>(offsets, nb, pairs, lay, ctl);
}

void launch_accum_level(int batch_s, int tpb, uint64_t resident, uint32_t* items, const uint32_t* pairs,
                        const PairLayout& lay, ctl_t* ctl, int level, int stats, cudaStream_t st) {
    const uint32_t* list = pairs + lay.base[level];
    uint64_t cap = lay.cap[level];
    switch (batch_s) {
        case 1: list_t<1>(tpb, resident, items, list, ctl, cap, level, stats, st); break;
        case 2: list_t<2>(tpb, resident, items, list, ctl, cap, level, stats, st); break;
        case 4: list_t<4>(tpb, resident, items, list, ctl, cap, level, stats, st); break;
        case 8: list_t<8>(tpb, resident, items, list, ctl, cap, level, stats, st); break;
        case 16: list_t<16>(tpb, resident, items, list, ctl, cap, level, stats, st); break;
        default: list_t<32>(tpb, resident, items, list, ctl, cap, level, stats, st); break;
    }
}

}  // namespace msm

namespace msm {

uint64_t accum_resident_threads(int tpb) {
    int dev = 0, sms = 0, b0 = 0, b1 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, k_accum_level0<32>, tpb, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, k_accum_list<32>, tpb, 0);
    return (uint64_t)sms * (uint64_t)std::max(1, std::min(b0, b1)) * (uint64_t)tpb;
}

}  // namespace msm
