// Shape and arguments of the decode pipeline (one token through three kernels):
//   router   logits = Wr x; the last CTA done picks the top-k and their weights
//   gate/up  one CTA per 32 intermediate values of a slot (a pick or the shared expert):
//            their 32 gate and 32 up rows against x -> SwiGLU -> one activation block
//   down     one warp per output row: the row's blocks of every slot's down matrix
//            against the activation blocks, each weighted by its slot -> out
// Slots in activation order: the shared expert first (it needs no routing), then the
// k picks in selection order.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

struct DecodePlan {
  // layer shape
  int H, E, K, F, Fs, G, Gu, qtype;
  // bytes
  uint32_t blk;         // bytes per 32-value block (18 or 20)
  uint32_t rb_h;        // bytes per gate/up row (H values)
  uint32_t rb_f;        // bytes per routed down row (F values)
  uint32_t rb_fs;       // bytes per shared down row (Fs values)
  uint64_t rec_bytes;   // bytes per routed expert record
  // blocks
  int nbH, nbF, nbFs;   // blocks per gate/up row, routed down row, shared down row
  int nact;             // activation blocks: (K * F + Fs) / 32 (shared expert's first)
  int act_smem;         // the down kernel stages the activation planes in shared memory
};

MOE_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

constexpr uint32_t FLAG_ACCUMULATE = 1u;  // out = out + contribution
constexpr uint32_t FLAG_RESIDUAL = 2u;    // out = x + contribution

// Arguments of the three decode kernels (one token).
struct DecodeArgs {
  const float* x;             // [H]
  const float* router_w;      // [E][H]
  const float* bias;          // [E] or null
  const uint8_t* experts;     // E packed records
  const uint8_t* shared;      // shared record or null
  float* out;                 // [H]
  int32_t* topk_ids;          // [K] or null
  float* topk_w;              // [K] or null
  uint32_t* ctrl;             // control block: [1] router CTAs done (the last resets it)
  unsigned long long* trace;  // timeline (MOE_TRACE) or null
  float* logits;              // [E]
  int32_t* ids;               // [K] picks
  float* wts;                 // [K] their weights
  uint8_t* aplanes;           // [nact][96] activation blocks: byte planes
  float2* ainfo;              // [nact] {2^-k scale, sum of the block's integers}
  float scale, norm_min;
  uint32_t flags;
  DecodePlan p;
};

}  // namespace moe
