/*
 * moeffn.h - C ABI of the routed MoE-FFN step on GB300 (sm_103a).
 *
 * The step, for each token t (diskformer engine modules, as shown by diffend.io):
 *   logit_e = sum_h Wr[e][h] x[t][h]                      router, F32 "ffn_gate_inp"
 *                                                          (lfm2_moe_ssd.js, initBuffers: router binding)
 *   p_e = 1 / (1 + exp(-logit_e)); s_e = p_e + bias_e      bias only selects
 *                                                          (lfm2_moe_ssd.js, TOPK_SIG_BODY and its comment)
 *   groups (n_groups > 1): group score = the two largest s of the group summed;
 *   keep the groups_used best groups, lowest group on ties  (ling_moe_ssd.js, routeLing)
 *   picks: top_k rounds of argmax over the kept s, lowest index on ties, in
 *   selection order                                         (TOPK_SIG_BODY)
 *   w_j = p_pick_j / max(sum_j p_pick_j, norm_min) * weights_scale   (TOPK_SIG_BODY, routeLing)
 *   expert: [g; u] = W_gu x (gate rows then up rows), y = W_down (silu(g) * u), or with a
 *   clamp limit L > 0, y = W_down (min(silu(g), L) * clamp(u, -L, L))
 *                                                          (ling_moe_ssd.js, swiglu;
 *                                                           flint_moe_ssd.js, planLayoutFlint record)
 *   shared expert: the same SwiGLU with weight 1, no gate  (flint_moe_ssd.js, file header)
 *   out[t] = sum_j w_j y_j + shared                         (ling_moe_ssd.js, moeAccum)
 * Weights are ggml 4-bit blocks of 32 values (flint_moe_ssd.js, WGSL section,
 * comment above Q41DOT): Q4_1 = f16 d, f16 m, 16 nibble bytes, value d*q + m;
 * Q4_0 = f16 d, 16 nibble bytes, value d*(q - 8). In a block the low nibble of
 * byte i is value i and its high nibble is value 16 + i.
 * K-quant super-blocks of 256 values, the types the Ling store keeps (ling_moe_ssd.js,
 * file header and planLayoutLing: Q4_K gate/up rows, Q6_K or Q4_K down rows); the pages
 * name these types without their layouts, which are ggml's:
 *   Q4_K, 144 bytes: f16 d, f16 dmin, 12 bytes of packed 6-bit scales sc_j and mins mn_j
 *     of the eight 32-value sub-blocks, then four runs of 32 nibble bytes (run c: values
 *     64c .. in the low nibbles, 64c + 32 .. in the high nibbles); value = d sc_j q - dmin mn_j.
 *   Q6_K, 210 bytes: 128 bytes of low nibbles, 64 bytes of 2-bit high parts, 16 int8
 *     scales (one per 16 values), f16 d; value = d * scale * (q - 32).
 *
 * Layouts (all row-major, little-endian):
 *   x, out         [n_tokens][hidden] f32
 *   router_w       [n_experts][hidden] f32 (row e = expert e)
 *   router_bias    [n_experts] f32, or NULL for no selection bias
 *   expert_blocks  n_experts records back to back; record = gate [expert_ff rows of hidden
 *                  values], up [expert_ff rows], both in qtype, then down [hidden rows of
 *                  expert_ff values] in the down type (qtype_down, or qtype when it is 0);
 *                  a row of n values takes n/32 blocks (Q4_0 18, Q4_1 20 bytes) or n/256
 *                  super-blocks (Q4_K 144, Q6_K 210 bytes)
 *   shared_blocks  one record of the same form with shared_ff, or NULL when shared_ff == 0
 *   topk_ids       [n_tokens][top_k] int32 picks in selection order (optional output)
 *   topk_w         [n_tokens][top_k] f32 weights (optional output)
 *
 * Ownership: the caller owns every buffer; the library never frees caller memory.
 * Device pointers unless MOE_HOST_IO is set. Weights must not change while a call
 * that reads them is in flight: calls read weights before the previous kernel on
 * the stream has finished (programmatic dependent launch) unless MOE_NO_PDL is set.
 * x and out must not overlap.
 *
 * Errors: every entry point returns MOE_OK (0) or a negative MOE_ERR_* code and
 * sets a thread-local message (moe_last_error). Configurations and pointers are
 * checked on the host before anything is launched. Kernels never trap: a device
 * wait that runs out of time sets a status word in the workspace, which
 * moe_workspace_status reports as MOE_ERR_TIMEOUT.
 */
#ifndef MOEFFN_H
#define MOEFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ggml block type ids (flint_moe_ssd.js: GGML_Q4_1 = 3). */
#define MOE_Q4_0 2
#define MOE_Q4_1 3
#define MOE_Q4_K 12
#define MOE_Q6_K 14

/* moe_cfg.flags */
#define MOE_ACCUMULATE 1u /* out = out + contribution (the pages' x += ...)          */
#define MOE_RESIDUAL 2u   /* out = x + contribution                                 */
#define MOE_HOST_IO 4u    /* x, out, topk_ids, topk_w are host pointers: x is copied in;
                           * outputs in page-locked memory mapped into the device's address
                           * space are written in place, other outputs are staged */
#define MOE_NO_PDL 8u     /* launch without programmatic dependent launch             */
#define MOE_TRACE 16u     /* record a per-CTA timeline in the workspace (see below)   */
#define MOE_BATCHED 32u   /* take the batched path whatever the token count           */
#define MOE_F32_ACT 64u   /* decode chain: f32 activations in the block dots (the pages'
                           * arithmetic) instead of 16-bit block fixed point (see below) */
#define MOE_GRAPH 128u    /* replay a captured CUDA graph for an argument set seen before
                           * (see moe_ffn_forward_ex)                                  */

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_CFG = -1,
  MOE_ERR_NULL_PTR = -2,
  MOE_ERR_ALIGNMENT = -3,
  MOE_ERR_UNSUPPORTED = -4,
  MOE_ERR_CUDA = -5,
  MOE_ERR_TIMEOUT = -6,
  MOE_ERR_WORKSPACE = -7
};

/* One MoE layer and one batch of tokens. The knobs are the layer's GGUF keys
 * (expert_count, expert_used_count, expert_feed_forward_length,
 * expert_shared_feed_forward_length, expert_group_count, expert_group_used_count,
 * expert_weights_scale; flint_moe_ssd.js configFromGgufFlint, ling_moe_ssd.js
 * configFromGgufLing). Limits checked by every entry point:
 *   hidden, expert_ff, shared_ff multiples of 32 (shared_ff may be 0), at most 3072;
 *   1 <= top_k <= min(n_experts, 32); n_experts <= 1024;
 *   n_groups divides n_experts; n_groups > 1 needs n_experts / n_groups >= 2,
 *   n_groups <= 64, 1 <= groups_used <= n_groups, top_k <= groups_used * n_experts / n_groups;
 *   n_tokens >= 0 (0: nothing is launched); qtype MOE_Q4_0, MOE_Q4_1 or MOE_Q4_K;
 *   qtype_down 0 (the same as qtype), MOE_Q4_0, MOE_Q4_1, MOE_Q4_K or MOE_Q6_K;
 *   K-quant gate/up rows need hidden % 256 == 0, K-quant down rows expert_ff and
 *   shared_ff multiples of 256;
 *   norm_min >= 0 (the pages use 2^-14 = 6.103515625e-5). */
typedef struct moe_cfg {
  int32_t hidden;
  int32_t n_experts;
  int32_t top_k;
  int32_t expert_ff;
  int32_t shared_ff;
  int32_t n_groups;    /* 1 = plain top-k */
  int32_t groups_used; /* ignored when n_groups == 1 */
  int32_t n_tokens;
  int32_t qtype;
  float weights_scale; /* 1.0 unless the layer says otherwise */
  float norm_min;      /* clamp on the sum of the picked sigmoids */
  uint32_t flags;      /* MOE_* flags above */
  /* SwiGLU clamp limits L, >= 0 (ling_moe_ssd.js, the swiglu kernel and its comment:
   * act = min(silu(g), L) * clamp(u, -L, L); L = 0 means no clamp). The routed experts
   * and the shared expert take separate per-layer limits, as the page's
   * swiglu_clamp_exp / swiglu_clamp_shexp arrays do. */
  float swiglu_limit;
  float swiglu_limit_shared;
  /* Optional layer prologue: with ffn_norm (a device vector [hidden] f32, 16-byte
   * aligned) the step's input is rms_norm(x) * ffn_norm, rms_norm(x) = x /
   * sqrt(mean(x^2) + rms_eps) (flint_moe_ssd.js / lfm2_moe_ssd.js headers: x +=
   * ffn(rms_norm(x) * ffn_norm)); MOE_RESIDUAL then adds the raw x, giving the whole
   * FFN block. NULL: x enters as is. */
  float rms_eps;
  const float* ffn_norm;
  /* Block type of the down rows (routed and shared), or 0 for qtype: the Ling store
   * types its down rows per layer, apart from the gate/up rows (ling_moe_ssd.js,
   * planLayoutLing). */
  int32_t qtype_down;
} moe_cfg;

/* Two execution paths, chosen by n_tokens (both are exact restatements of the step
 * above; they differ in arithmetic only):
 *   n_tokens < 44  the decode chain, up to 16 tokens per launch: a router kernel,
 *                  (with several tokens) a selection kernel, a gate/up kernel and a
 *                  down kernel with the weighted sum. The router is an f32 dot. By
 *                  default the 4-bit blocks meet activations held in 16-bit block
 *                  fixed point (a power-of-two scale per 16 values, error at most
 *                  2^-15 of the largest magnitude among those 16), so each block dot is an
 *                  exact int32 sum (dp4a), scaled and accumulated in f32. With
 *                  MOE_F32_ACT the activations stay f32 and each block contributes
 *                  d * sum(q x) + m * sum(x) by f32 fused multiply-adds (the pages'
 *                  arithmetic); it runs about 12% slower on the Flint-shaped layer.
 *   n_tokens >= 44 (or MOE_BATCHED) the batched path, in passes of at most 512
 *                  tokens. A router contraction accumulated in f32 (on the tile pipeline
 *                  from f16 hi + lo parts of the f32 rows and tokens, in up to four K
 *                  slices summed in order); one warp per token for the selection; a stable
 *                  counting sort of the (token, pick) pairs by expert; grouped
 *                  contractions on the tensor cores. The 4-bit blocks are dequantised
 *                  exactly to f16 before a single rounding; K-quant values on the tile
 *                  pipeline below take their f16-rounded scale and offset (up to three
 *                  roundings of 2^-11). x enters as an f16 hi + lo pair (22 bits). The
 *                  SwiGLU activations are rounded once to f16. Products accumulate in
 *                  f32. Requires |x| and every activation to stay below 65504 (the f16
 *                  range).
 *   The batched contractions run as warp-specialised TMA/TMEM pipelines for layers whose
 *   three matrices are all Q4_1 (or all Q4_0) with hidden, expert_ff and shared_ff whole
 *   multiples of 128 (Q4_1) or 256 (Q4_0), and for Q4_K gate/up rows with Q4_K or Q6_K down
 *   rows with all three multiples of 256 (Q6_K down rows of at most 768 values); other
 *   layers run a general form of the same contractions.
 * Both paths give the same picks; outputs agree to the tolerance of their arithmetic
 * (relative L2 well under 2e-3 against a float64 evaluation). */

/* The step on the default stream with a library-owned workspace (one per
 * device, grown on demand, freed by moe_shutdown). Blocks until the step is
 * done and returns device-side errors directly. Pointer alignment: x, out,
 * router_w, expert_blocks, shared_blocks 16 bytes; router_bias 4 bytes. */
int moe_ffn_forward(const float* x, const float* router_w, const float* router_bias,
                    const void* expert_blocks, const void* shared_blocks, const moe_cfg* cfg,
                    float* out);

/* The step enqueued on `stream` (a cudaStream_t, NULL = legacy default stream)
 * with a caller-owned device workspace of at least moe_workspace_size(cfg) bytes,
 * 256-byte aligned. A workspace must be zero-filled before its first use and then
 * only touched by this library: its first 512 bytes are control words (the
 * status word that moe_workspace_status reads). Calls sharing one workspace must
 * be ordered (same stream, or synchronised); calls with different configurations
 * may share one.
 * Asynchronous: device-side errors surface through moe_workspace_status.
 * topk_ids / topk_w may be NULL.
 * With MOE_GRAPH the library remembers the 64 argument sets (every pointer, the sizes and
 * the cfg) used most recently in the process. The second call with a set captures all of
 * its work into a CUDA graph on a library-owned stream, and every later call with that set
 * is one launch of the graph on `stream`: the same kernels and arguments, so the same
 * results, with less host time per call. The buffers of a remembered set must stay
 * allocated, and host buffers page-locked, until moe_shutdown or until 64 other sets have
 * been used since. A call made while `stream` is being captured, a MOE_TRACE call, and a
 * set whose capture fails run directly. */
int moe_ffn_forward_ex(const float* x, const float* router_w, const float* router_bias,
                       const void* expert_blocks, const void* shared_blocks, const moe_cfg* cfg,
                       float* out, void* workspace, size_t workspace_bytes, void* stream,
                       int32_t* topk_ids, float* topk_w);

/* Workspace bytes a call with this configuration needs (0 for an invalid cfg). */
size_t moe_workspace_size(const moe_cfg* cfg);

/* Byte offset of the MOE_TRACE timeline in the workspace (0 when cfg is invalid or
 * has no MOE_TRACE). The timeline holds 24 u64 words for each of the first
 * n_SM CTA indices: %globaltimer readings in nanoseconds, written by thread 0 of
 * the CTA with that index in each of the three decode kernels of the last token:
 * router kernel 0 start, 1 x ready (previous kernel done), 2 logits written;
 * gate/up kernel 4 start, 5 x quantised, 6 logits ready, 7 picks made, 8 the CTA's
 * first rows in shared memory, 9 activation block written, and within its selection
 * (single-token calls) 3 keys made, 19 candidates gathered, 22 picks ranked; down kernel 12 start,
 * 13 picks made, 14 row copies issued, 15 activation blocks ready, 16 activation
 * blocks staged, 17 rows in shared memory, 18 output rows written. Unused words
 * stay 0. */
size_t moe_trace_offset(const moe_cfg* cfg);

/* Waits for `stream`, then reads and clears the workspace's status word:
 * MOE_OK, or MOE_ERR_TIMEOUT when a device-side wait ran out of time (the
 * workspace's control block is zeroed again so it can be reused). */
int moe_workspace_status(void* workspace, void* stream);

/* Exercises the error path above without a fault: one kernel waits on an mbarrier that
 * nothing completes, through the same bounded wait the step's kernels use, gives up after
 * its time limit (0.5 s) and sets the timeout bit in the workspace's status word, as a
 * stalled copy would. A following moe_workspace_status reports MOE_ERR_TIMEOUT and clears
 * it; the context stays usable. `workspace` is any workspace of at least 512 bytes;
 * asynchronous on `stream`. Returns MOE_OK or MOE_ERR_NULL_PTR / MOE_ERR_CUDA. */
int moe_selftest_timeout(void* workspace, void* stream);

/* The step for callers that cannot allocate memory: the call makes no cudaMalloc,
 * cudaFree or other allocating call, on the device or on the host. Such callers include
 * code that runs where an allocator may not be entered (inside another allocator's hooks,
 * in a real-time or signal context, under a memory budget that has already been handed
 * out) or that has no allocator of its own to lend a workspace. The pages have no
 * counterpart: their engines own every buffer.
 * The scratch lives in a fixed device array of 512 KiB compiled into the library; every
 * device that loads the library holds it until the process exits, and every call on a
 * device shares it, so calls whose work overlaps on the GPU (other streams, other
 * threads) race and must not be made. Each call looks the array's device address up
 * afresh. CUDA loads the library's kernels and this array onto a device on first use,
 * and that loading may itself allocate device memory: make the first call on each device
 * before the stretch in which nothing may be allocated, and before any stream capture.
 * Up to 16 tokens are decoded per launch, as many as the array holds the scratch of
 * (control block, logits and SwiGLU activations); one token of the largest layer the
 * configuration checks admit needs about 401 KiB, so every admitted layer runs, and a
 * layer that needed more would be rejected with MOE_ERR_UNSUPPORTED. Device buffers
 * only: MOE_HOST_IO and MOE_TRACE are rejected. Blocking: returns after the step has
 * finished on `stream` (a cudaStream_t, NULL = legacy default stream), with device-side
 * errors reported directly. Arguments otherwise as moe_ffn_forward. */
int moe_ffn_forward_noalloc(const float* x, const float* router_w, const float* router_bias,
                            const void* expert_blocks, const void* shared_blocks, const moe_cfg* cfg,
                            float* out, void* stream);

/* Text of the last error on the calling thread ("" if none). */
const char* moe_last_error(void);

/* Frees the library-owned workspaces. Returns MOE_OK or MOE_ERR_CUDA. */
int moe_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEFFN_H */
