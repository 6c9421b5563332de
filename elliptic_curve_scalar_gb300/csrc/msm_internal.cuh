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
    uint32_t pad[7];
};


// accumulation launchers (msm_accum.cu); batch_s in {1, 2, 4, 8, 16, 32}
void launch_accum_level0(int batch_s, int tpb, const uint32_t* points, const uint32_t* entries, uint32_t* items,
                         ctl_t* ctl, uint64_t units_ub, int stats, cudaStream_t st);
void launch_accum_level(int batch_s, int tpb, uint32_t* items, const uint32_t* offsets, uint32_t nb, ctl_t* ctl,
                        uint64_t h_ub, int level, int stats, cudaStream_t st);

}  // namespace msm
