// msm_internal.cuh -- declarations shared by the MSM translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "msm_core.cuh"

namespace msm {

// device-side control block of one run (zeroed at the start of every run)
struct ctl_t {
    uint32_t max_count;  // largest bucket
    uint32_t total;      // padded entries
    uint32_t entries;    // non-zero digits
    uint32_t nonempty;   // buckets with at least one entry
    unsigned long long adds;
    unsigned long long inversions;
    uint32_t levels;
    uint32_t error;       // non-zero if a device-side capacity check failed
    uint32_t pad[6];
    uint32_t pair_count[4][32];  // pairs listed per window group and tree level
};

constexpr int MAX_LEVELS = 32;
constexpr int MAX_GROUPS = 4;

// Window groups: group j (j = 0 is the top) covers windows [w_lo[j], w_hi[j]);
// each group's pair list for tree level l starts at base[j][l] in the pair
// buffer and holds at most cap[j][l] entries.
struct PairLayout {
    int groups;
    uint32_t B;
    uint32_t finish_t;  // buckets leave the affine tree once they hold <= finish_t items
    int w_lo[MAX_GROUPS], w_hi[MAX_GROUPS];
    uint32_t base[MAX_GROUPS][MAX_LEVELS];
    uint32_t cap[MAX_GROUPS][MAX_LEVELS];
};


// resident threads of the accumulation kernels in their natural and their
// register-capped ("wide") builds
struct Resident {
    uint64_t narrow, wide;
};

// The accumulation knobs: batch_s in {1, 2, 4, 8, 16, 32, 64} (0: automatic)
// is the largest number of pairs a thread shares one inversion across; tpb
// the threads per block; place where a batch keeps its prefix products
// (PLACE_LOCAL, PLACE_SHARED, PLACE_REGS in msm_core.cuh); grid the most
// blocks a launch may use (0: automatic).
struct AccumKnobs {
    int batch_s, tpb, place, grid;
};

// accumulation launchers (msm_accum.cu):
// level 0 over the units of buckets [g0, g1); levels >= 1 over group grp's list;
// inv_kind: 0 = safegcd, 1 = Fermat
// (entry indices below nsplit address points, the others phi - nsplit);
// each returns the number of kernels it launched
int launch_accum_level0(const AccumKnobs& kb, const Resident& res, const uint32_t* points, const uint32_t* phi,
                        uint32_t nsplit, const uint32_t* entries, const uint32_t* offsets, uint32_t g0, uint32_t g1,
                        uint32_t* items, ctl_t* ctl, uint64_t units_ub, int stats, int inv_kind, cudaStream_t st);
void launch_build_pairs(const uint32_t* offsets, uint32_t nb, uint32_t* pairs, const PairLayout& lay, ctl_t* ctl,
                        cudaStream_t st);
int launch_accum_level(const AccumKnobs& kb, const Resident& res, uint32_t* items, const uint32_t* pairs,
                       const PairLayout& lay, ctl_t* ctl, int grp, int level, int stats, int inv_kind,
                       cudaStream_t st);
// one block over tree levels first, first + 1, ... of group grp while their lists are non-empty
void launch_accum_deep(uint32_t* items, const uint32_t* pairs, const PairLayout& lay, ctl_t* ctl, int grp, int first,
                       int stats, int inv_kind, cudaStream_t st);
Resident accum_resident_threads(int tpb);
// the batch size a launch with these knobs runs with
int placed_batch(int batch_s, int place, int tpb);
// per-device set-up of the accumulation kernels (shared-memory limits); false on failure
bool accum_prepare_device();
// Jacobian sums of the buckets of [g0, g1) that left the tree with >= 2 items
void launch_finish(const uint32_t* items, const uint32_t* offsets, uint32_t g0, uint32_t g1, uint32_t finish_t,
                   uint32_t* jsum, uint64_t resident, cudaStream_t st);

}  // namespace msm
