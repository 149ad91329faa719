// Host-visible entry points of the fused decode kernel.
#pragma once

#include <cuda_runtime.h>

#include "plan.h"

namespace moe {

constexpr int DECODE_THREADS = 384;  // 11 consumer warps + 1 producer warp

// Launches the decode kernel for one token (grid = a.p.nc CTAs).
cudaError_t decode_launch(const DecodeArgs& a, int qtype, int maxb, uint32_t smem, cudaStream_t st,
                          bool pdl);
// Resident CTAs per SM of the decode kernel at this dynamic shared memory size.
cudaError_t decode_occupancy(int qtype, int maxb, uint32_t smem, int* blocks);
// Dynamic shared memory the decode kernel needs for this plan.
uint32_t decode_smem_bytes(const DecodePlan& p);

}  // namespace moe
