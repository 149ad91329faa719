// Shape and arguments of the decode pipeline (one token through three kernels):
//   router   logits = Wr x
//   gate/up  one CTA per 16 intermediate values of a slot (a pick or the shared expert):
//            the picks from the logits, the slot's 16 gate and 16 up rows copied into
//            shared memory, dotted with x -> SwiGLU -> f32 activations
//   down     R output rows per CTA: the picks from the logits, the rows' blocks of every
//            slot's down matrix copied into shared memory, dotted with the activations
//            (quantised per 32-block in shared memory), each slot weighted -> out
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
  int H, E, K, F, Fs, G, Gu;
  int qtype, qtype_dn;  // block types of the gate/up rows and of the down rows (ggml ids)
  // bytes
  uint32_t rb_h;        // bytes per gate/up row (H values)
  uint32_t rb_f;        // bytes per routed down row (F values)
  uint32_t rb_fs;       // bytes per shared down row (Fs values)
  uint64_t rec_bytes;   // bytes per routed expert record
  // blocks
  int nbH, nbF, nbFs;   // blocks per gate/up row, routed down row, shared down row
  int nact;             // activation blocks: (K * F + Fs) / 32 (shared expert's first)
  int act_stride;       // floats from one token's activations to the next (K * F + Fs)
  int rep;              // copies of the arrays many CTAs read (logits, activations); a CTA
                        // reads copy blockIdx.x % rep, so no L2 line serves every CTA
  // gate/up kernel: two chunks of 8 values, each a gate and an up window of 8 rows
  uint32_t gu_win;      // bytes of one window (8 rows rounded out to 16-byte bounds)
  uint32_t gu_smem;     // dynamic shared memory
  // down kernel
  int dn_rows;          // output rows per CTA (1, 2, 4 or 8)
  int dn_piece;         // activation blocks quantised at a time (all, or a multiple of 256)
  int dn_rg;            // row groups of the down CTA's threads (1, 2, 4 or 8; divides dn_rows)
  uint32_t dn_win_f;    // bytes of a routed window (dn_rows rows rounded out)
  uint32_t dn_win_fs;   // bytes of the shared window (0 without a shared expert)
  uint32_t dn_smem;     // dynamic shared memory
};

constexpr int GU_VALUES = 16;  // intermediate values per gate/up CTA
// Shared-memory bytes per 32-value activation block: f32 chunks (128) and the block sum (4),
// or the 16-bit fixed-point form: planes (64) and each half's scale and sum (16).
constexpr uint32_t ACT_BLOCK_SMEM = 132;
constexpr uint32_t ACT_BLOCK_SMEM_FX = 80;  // 64 B of planes, {s0, X0, s1, X1}
constexpr int DEC_TMAX = 16;   // tokens per decode call (the chain takes up to this many at once)

MOE_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }
MOE_HD uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

// A window holding `bytes` bytes that start anywhere: the copy is rounded out to
// 16-byte bounds, so it can take up to 16 more bytes than align16(bytes).
MOE_HD uint32_t window_bytes(uint32_t bytes) { return align16(bytes) + 16u; }

// Dynamic shared memory of the selection: probabilities and keys of every expert,
// then 256 candidate keys and 256 candidate experts.
MOE_HD uint32_t select_smem(int E) { return align16((uint32_t)E * 8u) + 2048u; }


constexpr unsigned long long PUB_EMPTY = ~0ull;  // an entry not (yet) published in this call
constexpr int DEC_REP = 8;                        // copies of the broadcast arrays (at most)

constexpr uint32_t FLAG_ACCUMULATE = 1u;  // out = out + contribution
constexpr uint32_t FLAG_RESIDUAL = 2u;    // out = x + contribution

// Arguments of the three decode kernels (one token).
struct DecodeArgs {
  const float* x;             // [T][H]
  const float* router_w;      // [E][H]
  const float* bias;          // [E] or null
  const uint8_t* experts;     // E packed records
  const uint8_t* shared;      // shared record or null
  float* out;                 // [T][H]
  int32_t* topk_ids;          // [T][K] or null
  float* topk_w;              // [T][K] or null
  uint32_t* ctrl;             // control block (status word)
  unsigned long long* trace;  // timeline (MOE_TRACE) or null
  float* logits;              // [rep][T][E]
  float* act;                 // [rep][T][act_stride] SwiGLU activations, shared expert's first
  size_t lg_copy, act_copy;   // floats from one copy of the logits (activations) to the next
  int32_t* ids;               // [T][K] picks (calls of T > 1: made by the selection kernel)
  float* wts;                 // [T][K] their weights
  unsigned long long* pub;    // [K] a single-token call's picks as the gate/up kernel publishes
                              // them: id | weight bits << 32, or PUB_EMPTY
  int T;                      // tokens of this call, 1 .. DEC_TMAX
  float scale, norm_min;
  float lim, lim_s;           // SwiGLU clamp limits of the routed and shared experts (0: none)
  const float* norm;          // [H] prologue norm weights, or null (x enters as is)
  float eps;                  // the prologue's epsilon
  uint32_t flags;
  DecodePlan p;
};

}  // namespace moe
