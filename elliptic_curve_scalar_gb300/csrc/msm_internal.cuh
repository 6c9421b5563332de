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
    uint32_t pair_count[32];  // pairs listed per tree level (index = level)
};

constexpr int MAX_LEVELS = 32;

// where each tree level's pair list starts in the pair buffer, and its capacity
struct PairLayout {
    uint32_t base[MAX_LEVELS];
    uint32_t cap[MAX_LEVELS];
};


// accumulation launchers (msm_accum.cu); batch_s in {1, 2, 4, 8, 16, 32} is the
// largest number of pairs a thread shares one inversion across
void launch_accum_level0(int batch_s, int tpb, uint64_t resident, const uint32_t* points, const uint32_t* entries,
                         uint32_t* items, ctl_t* ctl, uint64_t units_ub, int stats, cudaStream_t st);
void launch_build_pairs(const uint32_t* offsets, uint32_t nb, uint32_t* pairs, const PairLayout& lay, ctl_t* ctl,
                        cudaStream_t st);
void launch_accum_level(int batch_s, int tpb, uint64_t resident, uint32_t* items, const uint32_t* pairs,
                        const PairLayout& lay, ctl_t* ctl, int level, int stats, cudaStream_t st);
uint64_t accum_resident_threads(int tpb);

}  // namespace msm
