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

#include "g1_coop.cuh"
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
// Indices from nsplit on address the GLV images phi(P_i) instead of P_i.
template <int S>
struct Level0Src {
    const uint32_t* points;
    const uint32_t* phi;
    uint32_t nsplit;
    uint32_t* items;
    uint32_t e0[S], e1[S];
    uint32_t u0;
    __device__ __forceinline__ const uint32_t* pt(uint32_t e) const {
        const uint32_t i = e & ~SIGN;
        return i < nsplit ? points + (size_t)i * 16 : phi + (size_t)(i - nsplit) * 16;
    }
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

// Each accumulation kernel comes in two builds of one body: at its natural
// register count (about 100), and capped at 80 registers ("wide": 6 blocks of
// 128 threads per SM instead of 4; it spilled a few words when introduced).  The wide build
// is used for launches with enough work per resident thread (wide() below),
// where the extra warps hide latency (n = 2^22 on GB300: 14.17 -> 13.29 ms per
// MSM; caps of 96, 88, 72 and 64 were slower); small launches are
// latency-bound and the cap only adds latency there (n = 2^16: 1.27 vs 1.32 ms
// when introduced).
#define LEVEL0_PARAMS                                                                                     \
    const uint32_t *__restrict__ points, const uint32_t *__restrict__ phi, uint32_t nsplit,                \
        const uint32_t *__restrict__ entries, const uint32_t *__restrict__ offsets, uint32_t g0, uint32_t g1, \
        uint32_t *__restrict__ items, ctl_t *ctl, int stats, int inv_kind, uint32_t base
#define LEVEL0_ARGS points, phi, nsplit, entries, offsets, g0, g1, items, ctl, stats, inv_kind, base

template <int S, bool WIDE, int PLACE>
__device__ __forceinline__ void accum_level0(LEVEL0_PARAMS) {
    // units of buckets [g0, g1): pairs (2u, 2u+1) for u in [offset_g0 / 2, offset_g1 / 2);
    // this launch takes those from `base` on (a grid capped below the work,
    // MSM_G1_PARAM_GRID, runs as several launches with increasing base)
    const uint32_t ubeg = offsets[g0] >> 1;
    const uint32_t all = (offsets[g1] >> 1) - ubeg;
    if (base >= all) return;
    const uint32_t units = all - base;
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t chunk = min((uint64_t)S, ((uint64_t)units + nthreads - 1) / nthreads);
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t u0 = (uint64_t)ubeg + base + t * chunk;
    // the block may share one inversion: a block with work keeps all its threads
    if ((uint64_t)blockIdx.x * blockDim.x * chunk >= units) return;
    const int count = t * chunk < units ? (int)min(chunk, (uint64_t)units - t * chunk) : 0;
    // narrow launches (one pair per thread) keep per-thread inversions: the
    // block's shared one would add warp 0's group products to their latency
    const bool share = chunk >= 2;
    __shared__ uint32_t divtab[inv::kDivTabEntries];
    inv::load_divtab(divtab);
    __syncthreads();
    if (!share && count == 0) return;
    __shared__ uint32_t sh[8 * 256];
    extern __shared__ uint32_t pre_sh[];  // prefix products with PLACE_SHARED
    Level0Src<S> src;
    src.points = points;
    src.phi = phi;
    src.nsplit = nsplit;
    src.items = items;
    src.u0 = (uint32_t)u0;
    if constexpr (PLACE == PLACE_REGS) {
#pragma unroll
        for (int k = 0; k < S; k++) {
            uint2 e = k < count ? reinterpret_cast<const uint2*>(entries)[u0 + k] : make_uint2(0, 0);
            src.e0[k] = e.x;
            src.e1[k] = e.y;
        }
    } else {
        for (int k = 0; k < count; k++) {
            uint2 e = reinterpret_cast<const uint2*>(entries)[u0 + k];
            src.e0[k] = e.x;
            src.e1[k] = e.y;
        }
    }
    // the backward multiplications inlined in both builds of level 0 (n = 2^16,
    // natural build: 131 -> 127 us); the tree's narrow levels keep them called
    int adds = batch_pairs<S, true, PLACE>(src, count, inv_kind, share ? sh : nullptr, pre_sh, divtab);
    if (stats) warp_stats(ctl, adds, share ? threadIdx.x < 32 : 1);
}

template <int S, int PLACE>
__global__ void __launch_bounds__(256) k_accum_level0(LEVEL0_PARAMS) {
    accum_level0<S, false, PLACE>(LEVEL0_ARGS);
}
template <int S, int PLACE>
__global__ void __maxnreg__(80) k_accum_level0_wide(LEVEL0_PARAMS) {
    accum_level0<S, true, PLACE>(LEVEL0_ARGS);
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
    int grp = 0;
    if (g < nb) {
        og = offsets[g] >> 1;
        h = (offsets[g + 1] >> 1) - og;
        const int w = (int)(g / lay.B);
        while (grp + 1 < lay.groups && w < lay.w_lo[grp]) grp++;
    }
    // lanes of one group share one atomic per level; a warp spanning two groups
    // (only when B < 32) reserves per lane
    const bool uniform = __match_any_sync(0xffffffffu, grp) == 0xffffffffu;
    for (int level = 1; level < MAX_LEVELS; level++) {
        const int sh = level - 1;
        uint32_t nl = h ? ((h - 1) >> sh) + 1 : 0;
        uint32_t np = nl > lay.finish_t ? nl >> 1 : 0;  // small buckets are finished in Jacobian
        if (!__any_sync(0xffffffffu, np != 0)) break;
        uint32_t off;
        if (uniform) {
            uint32_t incl = np;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
            uint32_t base = 0;
            if (lane == 31 && total) base = atomicAdd(&ctl->pair_count[grp][level], total);
            base = __shfl_sync(0xffffffffu, base, 31);
            off = base + incl - np;
        } else {
            off = np ? atomicAdd(&ctl->pair_count[grp][level], np) : 0;
        }
        uint32_t* list = pairs + lay.base[grp][level];
        const uint32_t cap = lay.cap[grp][level];
        // long lists (a giant bucket) are written by the whole warp, short ones by their lane
        constexpr uint32_t kLong = 64;
        unsigned longs = __ballot_sync(0xffffffffu, np > kLong);
        while (longs) {
            const int src = __ffs(longs) - 1;
            longs &= longs - 1;
            const uint32_t nps = __shfl_sync(0xffffffffu, np, src);
            const uint32_t offs = __shfl_sync(0xffffffffu, off, src);
            const uint32_t ogs = __shfl_sync(0xffffffffu, og, src);
            uint32_t* ls = pairs + lay.base[__shfl_sync(0xffffffffu, grp, src)][level];
            const uint32_t caps = lay.cap[__shfl_sync(0xffffffffu, grp, src)][level];
            for (uint32_t j = lane; j < nps; j += 32) {
                if (offs + j < caps) ls[offs + j] = ogs + (j << level);
                else atomicOr(&ctl->error, 1u);
            }
        }
        if (np <= kLong) {
            for (uint32_t j = 0; j < np; j++) {
                uint32_t idx = off + j;
                if (idx < cap) list[idx] = og + (j << level);
                else atomicOr(&ctl->error, 1u);  // capacity bound violated (never expected)
            }
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

template <int S, bool WIDE, int PLACE>
__device__ __forceinline__ void accum_list(uint32_t* __restrict__ items, const uint32_t* __restrict__ list,
                                           ctl_t* ctl, int grp, int level, int stats, int inv_kind, uint32_t base) {
    const uint32_t all = ctl->pair_count[grp][level];
    if (base >= all) return;  // pairs from `base` on, as in accum_level0
    const uint32_t cnt = all - base;
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t chunk = min((uint64_t)S, ((uint64_t)cnt + nthreads - 1) / nthreads);
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t i0 = t * chunk;
    // the block may share one inversion: a block with work keeps all its threads
    if ((uint64_t)blockIdx.x * blockDim.x * chunk >= cnt) return;
    const int count = i0 < cnt ? (int)min(chunk, (uint64_t)cnt - i0) : 0;
    const bool share = chunk >= 2;  // as in accum_level0
    __shared__ uint32_t divtab[inv::kDivTabEntries];
    inv::load_divtab(divtab);
    __syncthreads();
    if (!share && count == 0) return;
    __shared__ uint32_t sh[8 * 256];
    extern __shared__ uint32_t pre_sh[];
    ListSrc<S> src;
    src.items = items;
    src.half = 1u << (level - 1);
    const uint32_t* lst = list + base;
    if constexpr (PLACE == PLACE_REGS) {
#pragma unroll
        for (int k = 0; k < S; k++) src.qi[k] = k < count ? lst[i0 + k] : 0u;
    } else {
        for (int k = 0; k < count; k++) src.qi[k] = lst[i0 + k];
    }
    int adds = batch_pairs<S, WIDE, PLACE>(src, count, inv_kind, share ? sh : nullptr, pre_sh, divtab);
    if (stats) {
        warp_stats(ctl, adds, share ? threadIdx.x < 32 : 1);
        if (threadIdx.x == 0) atomicMax(&ctl->levels, (uint32_t)level + 1);
    }
}

template <int S, int PLACE>
__global__ void __launch_bounds__(256) k_accum_list(uint32_t* __restrict__ items, const uint32_t* __restrict__ list,
                                                    ctl_t* ctl, int grp, int level, int stats, int inv_kind,
                                                    uint32_t base) {
    accum_list<S, false, PLACE>(items, list, ctl, grp, level, stats, inv_kind, base);
}
template <int S, int PLACE>
__global__ void __maxnreg__(80) k_accum_list_wide(uint32_t* __restrict__ items, const uint32_t* __restrict__ list,
                                                  ctl_t* ctl, int grp, int level, int stats, int inv_kind,
                                                  uint32_t base) {
    accum_list<S, true, PLACE>(items, list, ctl, grp, level, stats, inv_kind, base);
}

// ------------------------------------------------------------ deep levels

// The tree levels past those the host launches one by one: one block works
// through level `first` and every later level whose list is non-empty, in
// rounds of blockDim x S pairs, with a barrier between rounds and levels (a
// level's pairs read the items the previous level wrote).  The host sizes its
// per-level launches for the bucket sizes uniform data gives, so this launch
// usually finds its first level empty and returns at once -- one launch
// instead of one per possible level; an unusually deep bucket (e.g. many
// equal scalars) is still summed, by this block.
template <int S>
__global__ void __launch_bounds__(256) k_accum_deep(uint32_t* __restrict__ items, const uint32_t* __restrict__ pairs,
                                                    PairLayout lay, ctl_t* ctl, int grp, int first, int stats,
                                                    int inv_kind) {
    __shared__ uint32_t sh[8 * 256];
    __shared__ uint32_t divtab[inv::kDivTabEntries];
    inv::load_divtab(divtab);
    __syncthreads();
    int adds = 0, invs = 0;
    for (int level = first; level < MAX_LEVELS; level++) {
        const uint32_t cnt = ctl->pair_count[grp][level];
        if (cnt == 0) break;  // deeper levels are empty too
        const uint32_t* list = pairs + lay.base[grp][level];
        const uint32_t chunk = min((uint32_t)S, (cnt + blockDim.x - 1) / blockDim.x);
        for (uint32_t base = 0; base < cnt; base += blockDim.x * chunk) {
            const uint32_t i0 = base + threadIdx.x * chunk;
            const int count = i0 < cnt ? (int)min(chunk, cnt - i0) : 0;
            ListSrc<S> src;
            src.items = items;
            src.half = 1u << (level - 1);
            for (int k = 0; k < count; k++) src.qi[k] = list[i0 + k];
            // every thread of the block takes part in the shared inversion
            adds += batch_pairs<S, false>(src, count, inv_kind, sh, nullptr, divtab);
            invs += threadIdx.x < 32;
            __syncthreads();  // the next round reuses sh; the next level reads these items
        }
        if (stats && threadIdx.x == 0) atomicMax(&ctl->levels, (uint32_t)level + 1);
    }
    if (stats) warp_stats(ctl, adds, invs);
}

// ------------------------------------------------------------ small buckets

// One thread (W = 1) or one group of W lanes (cooperative additions) per bucket:
// buckets that left the tree with 2..T items get their sum by Jacobian mixed
// additions (see finish_plan in msm_core.cuh).
template <int W>
__global__ void k_finish(const uint32_t* __restrict__ items, const uint32_t* __restrict__ offsets, uint32_t g0,
                         uint32_t g1, uint32_t finish_t, uint32_t* __restrict__ jsum) {
    const uint32_t g = g0 + (blockIdx.x * blockDim.x + threadIdx.x) / W;
    if (g >= g1) return;
    const uint32_t og = offsets[g] >> 1;
    const uint32_t h = (offsets[g + 1] >> 1) - og;
    const FinishPlan fp = finish_plan(h, finish_t);
    if (fp.items < 2) return;
    g1::jac acc = g1::jac_inf();
    for (uint32_t i = 0; i < fp.items; i++)
        acc = g1c::add_mixed_w<W>(acc, g1::load_aff(items + (size_t)(og + i * fp.stride) * 16));
    if ((threadIdx.x & (W - 1)) == 0) g1::store_jac(jsum + (size_t)g * 24, acc);
}

void launch_finish(const uint32_t* items, const uint32_t* offsets, uint32_t g0, uint32_t g1, uint32_t finish_t,
                   uint32_t* jsum, uint64_t resident, cudaStream_t st) {
    if (finish_t < 2 || g1 <= g0) return;
    // cooperative groups of 8 lanes while the buckets fill a quarter of the GPU
    // at most (the chunk reduction's rule)
    if ((uint64_t)(g1 - g0) * 8 <= resident / 4)
        k_finish<8><<<((g1 - g0) * 8 + 127) / 128, 128, 0, st>>>(items, offsets, g0, g1, finish_t, jsum);
    else
        k_finish<1><<<(g1 - g0 + 127) / 128, 128, 0, st>>>(items, offsets, g0, g1, finish_t, jsum);
}

// ----------------------------------------------------------------- launchers

static unsigned grid_for(uint64_t work, int S, int tpb, uint64_t resident) {
    // Chunks of S, except that a launch of fewer than four resident waves
    // takes whole waves, the units spread evenly over them (the kernels take
    // chunks of ceil(units / threads)): 2.25 waves of full chunks would leave
    // the last wave three quarters empty while it still pays a whole batch's
    // latency (n = 2^20, level 0: 1.40 -> 1.35 ms).  From four waves on the
    // blocks' staggered finish already hides the partial wave, and the
    // rounding only adds inversions (n = 2^22, level 0: 4.95 -> 5.01 ms).
    // Below one wave of single units, one thread per unit.
    uint64_t threads = work;
    if (work > resident) {
        const uint64_t per_wave = (uint64_t)S * resident;
        threads = work >= 4 * per_wave ? (work + S - 1) / S : (work + per_wave - 1) / per_wave * resident;
    }
    return (unsigned)std::max<uint64_t>(1, (threads + tpb - 1) / tpb);
}

// the register-capped build once the work fills a resident wave of the other
// in chunks of min(S, per); tree levels switch from 8 pairs per resident
// thread on (n = 2^20: 3.67 -> 3.63 ms, adversarial 2.81 -> 2.79 ms), level 0
// from 32 (the single wave of level 0 at n = 2^16 was 5 % slower wide)
static bool wide(uint64_t work, int S, const Resident& res, int per) {
    const uint64_t s = (uint64_t)std::min(S, per);
    return (work + s - 1) / s >= res.narrow;
}

// batch_s = 0 (automatic): at most 64 additions per inversion.  With whole
// waves for small launches, a larger cap never adds a wave; it only halves the
// inversions of the launches that have more than 32 units per resident thread
// (a cap of 32 was 4 % slower at n = 2^20 and 6 % at 2^22).
static int auto_batch(int batch_s) { return batch_s ? batch_s : 64; }

// Prefix products in shared memory take S x 32 bytes per thread; a block may
// use at most this much for them (the rest of the SM's 228 KB holds the
// block-inversion buffer and at least one more block's static use).
constexpr int kPreSharedMax = 200 << 10;

// The batch size a placement runs with: the request (automatic = 64), clamped
// to the instantiated sizes -- PLACE_LOCAL 1..64, PLACE_SHARED 4..32 and
// S x 32 x tpb within kPreSharedMax, PLACE_REGS 2..8.
int placed_batch(int batch_s, int place, int tpb) {
    int S = auto_batch(batch_s);
    if (place == PLACE_SHARED) {
        S = std::max(4, std::min(S, 32));
        while (S > 4 && S * 32 * tpb > kPreSharedMax) S >>= 1;
    } else if (place == PLACE_REGS) {
        S = std::max(2, std::min(S, 8));
    }
    return S;
}

// One accumulation step: the natural or the register-capped build of the
// placement's kernel over `work` units (an upper bound; the kernels read the
// exact count on the device), with a grid from grid_for and dynamic shared
// memory for PLACE_SHARED (whose resident threads follow from that memory).
// A grid cap (MSM_G1_PARAM_GRID) below that grid splits the work into
// consecutive launches of cap x tpb x S units each, the kernel's last
// argument giving each launch's first unit.
template <class KN, class KW, class... Args>
static int launch_placed(KN kn, KW kw, int place, int S, int per, int tpb, const Resident& res, uint64_t work,
                          int grid_cap, cudaStream_t st, Args... args) {
    const size_t dyn = place == PLACE_SHARED ? (size_t)S * 32 * tpb : 0;
    Resident r = res;
    if (place == PLACE_SHARED) {
        int dev = 0, sms = 0, bn = 0, bw = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bn, kn, tpb, dyn);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bw, kw, tpb, dyn);
        r.narrow = (uint64_t)sms * std::max(1, bn) * tpb;
        r.wide = (uint64_t)sms * std::max(1, bw) * tpb;
    }
    // register-resident prefix products have no capped build: the cap would spill them
    const bool use_wide = place != PLACE_REGS && wide(work, S, r, per);
    const unsigned blocks = grid_for(work, S, tpb, use_wide ? r.wide : r.narrow);
    if (grid_cap <= 0 || blocks <= (unsigned)grid_cap) {
        if (use_wide) kw<<<blocks, tpb, dyn, st>>>(args..., 0u);
        else kn<<<blocks, tpb, dyn, st>>>(args..., 0u);
        return 1;
    }
    const uint64_t per_launch = (uint64_t)grid_cap * tpb * S;
    int launches = 0;
    for (uint64_t base = 0; base < work; base += per_launch, launches++) {
        if (use_wide) kw<<<grid_cap, tpb, dyn, st>>>(args..., (uint32_t)base);
        else kn<<<grid_cap, tpb, dyn, st>>>(args..., (uint32_t)base);
    }
    return launches;
}

template <int S, int PLACE>
static int level0_t(int tpb, const Resident& res, int grid_cap, const uint32_t* points, const uint32_t* phi,
                     uint32_t nsplit, const uint32_t* entries, const uint32_t* offsets, uint32_t g0, uint32_t g1,
                     uint32_t* items, ctl_t* ctl, uint64_t units_ub, int stats, int inv_kind, cudaStream_t st) {
    return launch_placed(k_accum_level0<S, PLACE>, k_accum_level0_wide<S, PLACE>, PLACE, S, 32, tpb, res, units_ub,
                  grid_cap, st, points, phi, nsplit, entries, offsets, g0, g1, items, ctl, stats, inv_kind);
}

template <int S, int PLACE>
static int list_t(int tpb, const Resident& res, int grid_cap, uint32_t* items, const uint32_t* list, ctl_t* ctl,
                   uint64_t cap, int grp, int level, int stats, int inv_kind, cudaStream_t st) {
    return launch_placed(k_accum_list<S, PLACE>, k_accum_list_wide<S, PLACE>, PLACE, S, 8, tpb, res, cap, grid_cap, st,
                  items, list, ctl, grp, level, stats, inv_kind);
}

// Dispatch on (placement, batch size) to the instantiated kernels.
#define ACCUM_DISPATCH(F)                               \
    switch (place) {                                    \
        case PLACE_SHARED:                              \
            switch (S) {                                \
                case 4: F(4, PLACE_SHARED); break;      \
                case 8: F(8, PLACE_SHARED); break;      \
                case 16: F(16, PLACE_SHARED); break;    \
                default: F(32, PLACE_SHARED); break;    \
            }                                           \
            break;                                      \
        case PLACE_REGS:                                \
            switch (S) {                                \
                case 2: F(2, PLACE_REGS); break;        \
                case 4: F(4, PLACE_REGS); break;        \
                default: F(8, PLACE_REGS); break;       \
            }                                           \
            break;                                      \
        default:                                        \
            switch (S) {                                \
                case 1: F(1, PLACE_LOCAL); break;       \
                case 2: F(2, PLACE_LOCAL); break;       \
                case 4: F(4, PLACE_LOCAL); break;       \
                case 8: F(8, PLACE_LOCAL); break;       \
                case 16: F(16, PLACE_LOCAL); break;     \
                case 32: F(32, PLACE_LOCAL); break;     \
                default: F(64, PLACE_LOCAL); break;     \
            }                                           \
    }

int launch_accum_level0(const AccumKnobs& kb, const Resident& res, const uint32_t* points, const uint32_t* phi,
                        uint32_t nsplit, const uint32_t* entries, const uint32_t* offsets, uint32_t g0, uint32_t g1,
                        uint32_t* items, ctl_t* ctl, uint64_t units_ub, int stats, int inv_kind, cudaStream_t st) {
    const int place = kb.place, S = placed_batch(kb.batch_s, kb.place, kb.tpb);
    int launches = 0;
#define L0(SS, PP)                                                                                              \
    launches = level0_t<SS, PP>(kb.tpb, res, kb.grid, points, phi, nsplit, entries, offsets, g0, g1, items, ctl, \
                                units_ub, stats, inv_kind, st)
    ACCUM_DISPATCH(L0)
#undef L0
    return launches;
}

void launch_build_pairs(const uint32_t* offsets, uint32_t nb, uint32_t* pairs, const PairLayout& lay, ctl_t* ctl,
                        cudaStream_t st) {
    k_build_pairs<<<(nb + 255) / 256, 256, 0, st>>>(offsets, nb, pairs, lay, ctl);
}

int launch_accum_level(const AccumKnobs& kb, const Resident& res, uint32_t* items, const uint32_t* pairs,
                       const PairLayout& lay, ctl_t* ctl, int grp, int level, int stats, int inv_kind,
                       cudaStream_t st) {
    const uint32_t* list = pairs + lay.base[grp][level];
    uint64_t cap = lay.cap[grp][level];
    const int place = kb.place, S = placed_batch(kb.batch_s, kb.place, kb.tpb);
    int launches = 0;
#define LV(SS, PP) \
    launches = list_t<SS, PP>(kb.tpb, res, kb.grid, items, list, ctl, cap, grp, level, stats, inv_kind, st)
    ACCUM_DISPATCH(LV)
#undef LV
    return launches;
}

void launch_accum_deep(uint32_t* items, const uint32_t* pairs, const PairLayout& lay, ctl_t* ctl, int grp, int first,
                       int stats, int inv_kind, cudaStream_t st) {
    k_accum_deep<16><<<1, 256, 0, st>>>(items, pairs, lay, ctl, grp, first, stats, inv_kind);
}

// The shared-memory placement's kernels may take up to kPreSharedMax bytes of
// dynamic shared memory; returns false if the device refuses.
static bool set_shared_limit() {
    bool ok = true;
#define SETMAX(SS, PP)                                                                                             \
    ok = ok && cudaFuncSetAttribute(k_accum_level0<SS, PP>, cudaFuncAttributeMaxDynamicSharedMemorySize,          \
                                    kPreSharedMax) == cudaSuccess;                                              \
    ok = ok && cudaFuncSetAttribute(k_accum_level0_wide<SS, PP>, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                    kPreSharedMax) == cudaSuccess;                                              \
    ok = ok && cudaFuncSetAttribute(k_accum_list<SS, PP>, cudaFuncAttributeMaxDynamicSharedMemorySize,            \
                                    kPreSharedMax) == cudaSuccess;                                              \
    ok = ok && cudaFuncSetAttribute(k_accum_list_wide<SS, PP>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                    kPreSharedMax) == cudaSuccess;
    SETMAX(4, PLACE_SHARED)
    SETMAX(8, PLACE_SHARED)
    SETMAX(16, PLACE_SHARED)
    SETMAX(32, PLACE_SHARED)
#undef SETMAX
    cudaGetLastError();
    return ok;
}

bool accum_prepare_device() { return set_shared_limit(); }

}  // namespace msm

namespace msm {

Resident accum_resident_threads(int tpb) {
    int dev = 0, sms = 0, b0 = 0, b1 = 0, w0 = 0, w1 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, k_accum_level0<32, PLACE_LOCAL>, tpb, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, k_accum_list<32, PLACE_LOCAL>, tpb, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&w0, k_accum_level0_wide<32, PLACE_LOCAL>, tpb, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&w1, k_accum_list_wide<32, PLACE_LOCAL>, tpb, 0);
    Resident r;
    r.narrow = (uint64_t)sms * (uint64_t)std::max(1, std::min(b0, b1)) * (uint64_t)tpb;
    r.wide = (uint64_t)sms * (uint64_t)std::max(1, std::min(w0, w1)) * (uint64_t)tpb;
    return r;
}

}  // namespace msm
