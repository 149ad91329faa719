// Batched (prefill) MoE-FFN step: arguments and host-visible launcher.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

constexpr int PREFILL_MIN_T = 44;     // calls of at least this many tokens take the batched path
                                      // (measured crossover with the multi-token decode chain)
constexpr int PREFILL_CHUNK_T = 512;  // tokens per prefill pass (larger batches run in passes)
constexpr int PREFILL_NMAX = 64;      // tokens (or pairs) per GEMM work unit (general path)
constexpr int PREFILL_TILE_NMAX = 64; // tokens (or pairs) per GEMM work unit (tile pipeline)
constexpr int PREFILL_RT_SLICES = 4;  // tile router: K slices at most
constexpr int PREFILL_THREADS = 256;

// One token-chunk of a GEMM: `slot` = expert id (or n_experts for the shared expert),
// rows [row0, row0 + n) of the expert-sorted pair list (or of the tokens, shared).
// `prow`: rows of the earlier chunks of its kind, each rounded up to 16 (the chunk's
// first row in the tiled operand images of the tile pipeline).
struct GemmChunk {
  int slot, row0, n, prow;
};

struct PrefillArgs {
  // caller's buffers (device)
  const float* x;           // [T][H]
  const float* router_w;    // [E][H]
  const float* bias;        // [E] or null
  const uint8_t* experts;   // E records
  const uint8_t* shared;    // shared record or null
  float* out;               // [T][H]
  int32_t* topk_ids;        // [T][K] or null
  float* topk_w;            // [T][K] or null
  // workspace
  float* logits;            // [T][E]
  int32_t* ids;             // [T][K]
  float* wts;               // [T][K]
  uint32_t* offsets;        // [E + 1] first sorted position of each expert
  uint32_t* perm;           // [P] pair (t * K + j) at each sorted position
  float* wsorted;           // [P] routing weight at each sorted position
  uint32_t* pos_of;         // [P] sorted position of each pair
  GemmChunk* chunks;        // routed chunks (expert order), then shared chunks
  uint32_t* nchunks;        // [2]: routed chunks, all chunks
  __half* x16;              // [T][2][H] f16 hi and lo parts, K order permuted within 32-blocks
  // tile pipeline: operand images, each chunk's rows tiled as its MMA B operand
  // ([chunk][128-value K block][rows/8][8 rows x 16 bytes] per 8 K values)
  uint8_t* ximg;            // x hi/lo: token chunks, then routed chunks from ximg_routed
  uint8_t* ximg_routed;
  uint8_t* aimg;            // routed activations (sorted-pair chunks)
  uint8_t* aimg_s;          // shared-expert activations (token chunks)
  __half* act16;            // [P][F] f16 (sorted-pair rows), permuted K order
  __half* act16s;           // [T][Fs] f16, permuted K order
  float* ybuf;              // [P][H] weighted down outputs (sorted-pair rows)
  float* sbuf;              // [T][H] shared-expert down outputs
  uint32_t* status;         // device error bits
  // shape
  int T, H, E, K, F, Fs, G, Gu;
  int qtype, qtype_dn;      // block types of the gate/up rows and of the down rows (ggml ids)
  float scale, norm_min;
  float lim, lim_s;         // SwiGLU clamp limits of the routed and shared experts (0: none)
  const float* norm;        // [H] prologue norm weights, or null
  float eps;                // the prologue's epsilon
  const float* xres;        // [T][H] the raw tokens (the residual form adds these)
  float* xn;                // [T][H] workspace for the normalised tokens (with a norm)
  uint32_t flags;
  uint32_t rb_h, rb_f, rb_fs;
  uint64_t rec_bytes;
  int nc;                   // CTAs of the persistent GEMM kernels
  int nmax;                 // rows per chunk: PREFILL_NMAX or PREFILL_TILE_NMAX
  int tile;                 // 1: tile pipeline (prefill_tile_ok), 0: general path
  int rt_slices, rt_ups;    // tile router: K slices (logits = the sum of rt_slices partial
                            // arrays [T][E], in slice order) of rt_ups 128-value units; 1 elsewhere
};

// Bytes of each prefill workspace region for a pass of T tokens (host).
struct PrefillWs {
  size_t logits, ids, wts, offsets, perm, wsorted, pos_of, chunks, nchunks, x16, act16, act16s,
      ybuf, sbuf, ximg, ximg_routed, aimg, aimg_s, total;
};
PrefillWs prefill_ws_layout(int T, int H, int E, int K, int F, int Fs, bool tile);

// True when the layer's rows suit the tile pipeline's copies: all three matrices Q4_0 or all
// Q4_1, with K dimensions in whole pipeline chunks (128 values for Q4_1, 256 for Q4_0), so
// every weight-row segment a chunk copies starts and ends on a 16-byte boundary; or Q4_K
// gate/up rows with Q4_K or Q6_K down rows and H, F, Fs multiples of 256 (Q4_K: one 144-byte
// super-block per row segment; Q6_K: F, Fs <= 768, a stage holds 128 whole down rows, whose
// span is a multiple of 16 bytes). Other layers take the general contractions.
bool prefill_tile_ok(int H, int F, int Fs, int qtype, int qtype_dn);

// Tile pipeline launches (prefill_tc.cu).
cudaError_t tile_router_launch(const PrefillArgs& a, cudaStream_t st);
cudaError_t tile_images_launch(const PrefillArgs& a, bool routed, cudaStream_t st);
cudaError_t tile_gemm_launch(const PrefillArgs& a, int mode, cudaStream_t st);
// The down contraction with tokens as A and 256 down rows per tile (needs H % 256 == 0).
cudaError_t swap_down_launch(const PrefillArgs& a, cudaStream_t st);

// Enqueues the whole prefill pass on `st`. Returns the first launch error.
cudaError_t prefill_launch(const PrefillArgs& a, cudaStream_t st);

}  // namespace moe
