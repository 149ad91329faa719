// Host-visible entry point of the decode chain (router, gate/up, down kernels).
#pragma once

#include <cuda_runtime.h>

#include "plan.h"

namespace moe {

// Enqueues the decode chain for up to DEC_TMAX tokens on `st` (with programmatic dependent
// launch when `pdl`). `maxb` = blocks per lane of a gate/up row: ceil(H / 1024). `fx`: the
// block dots take 16-bit block fixed-point activations instead of f32.
// The plan's shared-memory sizes and rows per CTA must come from the host planner.
// With a trace, CTAs with index below `trows` record their timeline.
cudaError_t decode_launch(const DecodeArgs& a, int maxb, cudaStream_t st, bool pdl, bool fx, int trows);

}  // namespace moe
