// Batched MoE-FFN step (prefill: T tokens at once) for sm_103a: the general form of its
// contractions, for every shape and block type, and the passes both forms share. Layers
// whose three matrices are all Q4_1 (or all Q4_0), with K dimensions in whole 128 (256)
// value chunks, run the contractions and the router as the TMA/TMEM tile pipeline in
// prefill_tc.cu instead.
//
// Passes, each a kernel on the caller's stream:
//   router      logits[T][E] = X Wr^T                       (f32, tiled SIMT)
//   top-k       per token: sigmoid, bias, (group) top-k, weights; expert histogram
//   sort        stable counting sort of the T*K (token, pick) pairs by expert, and
//               the GEMM chunk lists (at most PREFILL_NMAX rows a chunk)
//   x16         X -> two f16 rows per token, hi = f16(x) and lo = f16(x - hi), with
//               the K order permuted inside every 32-value block
//   gate/up     grouped GEMM on the tensor cores: per (chunk, 64 pairs of rows)
//               D[128 x 2N] = W_gu (dequantised to f16 in shared memory) * [X_hi X_lo]^T,
//               accumulated in TMEM; the epilogue adds the hi and lo columns and
//               applies SwiGLU -> act16
//   down        grouped GEMM: per (chunk, 128 output rows) D = W_down * act_chunk^T,
//               epilogue scales by the pair's routing weight -> ybuf (shared: sbuf)
//   combine     out[t] = sum_j ybuf[pos(t, j)] + sbuf[t] (fixed order: deterministic)
//
// Weights are the MMA's A operand (M = 128 rows), tokens the B operand (N = the
// chunk's rows rounded up to 16), so a work unit streams its expert's rows once
// whatever the number of tokens that picked it. The token rows enter the gate/up
// GEMM as hi + lo f16 pairs: the rounding of x to f16 is the same for every row of
// W, so its error would add up coherently over the down projection; the pair
// carries x to 22 bits. The activations (one rounding per value, independent
// across rows) and the weights go in as single f16 values. The 4-bit blocks are dequantised
// exactly (nibble -> f16 integer, then d*q + m rounded once) into f16; the
// products are summed in f32 in TMEM. K-quant sub-blocks (Q4_K, Q6_K) are dequantised in
// f32, where their scale products are exact, and rounded once to f16. Each 128-value K
// step copies the token rows by cp.async and has its weight loads issued one step ahead,
// so a step waits on one round trip rather than one per operand piece. Inside each
// 32-value block the K order is
// permuted so that one 32-bit nibble word fills one 16-byte row of a core matrix:
// slot 8w + (0..7) holds values 4w, 4w+2, 4w+1, 4w+3, 16+4w, 16+4w+2, 16+4w+1,
// 16+4w+3. Every operand uses the same order, so the dot products are unchanged.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "plan.h"
#include "prefill_host.h"
#include "select.cuh"
#include "tc.cuh"

namespace moe {

// Slot of value e (0..31) of a block in the permuted K order.
__host__ __device__ __forceinline__ int kslot(int e) {
  const int hi = e >> 4, r = e & 15, w = r >> 2, j = r & 3;
  const int jj = (j == 1) ? 2 : (j == 2 ? 1 : j);  // 0, 2, 1, 3
  return 8 * w + 4 * hi + jj;
}
__host__ __device__ __forceinline__ int kpos(int k) { return (k & ~31) | kslot(k & 31); }

// ---------------------------------------------------------------------------
// router: logits[t][e] = sum_h x[t][h] * Wr[e][h]
// ---------------------------------------------------------------------------
// CTA tile: 64 tokens x 64 experts, thread (ty, tx) = (tid / 16, tid % 16) owns tokens
// 4 ty .. 4 ty + 3 and experts 4 tx .. 4 tx + 3. K goes in slices of 32 staged in shared
// memory K-major (row stride RT_LD floats, 16-byte aligned), so each k costs two 16-byte
// shared loads for 16 FMAs; the next slice's global loads are held in registers while the
// current slice is multiplied. Each logit is one f32 sum in a fixed order.
constexpr int RT_TILE = 64, RT_KS = 32, RT_LD = 68;
__global__ void __launch_bounds__(256) prefill_router(const PrefillArgs a) {
  __shared__ __align__(16) float xs[RT_KS][RT_LD], ws[RT_KS][RT_LD];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.y * RT_TILE, e0 = blockIdx.x * RT_TILE;
  // global loads of a slice: 64 rows x 8 float4 of each matrix, two of each per thread
  float4 gx[2], gw[2];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int idx = tid + 256 * q, row = idx >> 3, c4 = idx & 7;
      const int t = t0 + row, e = e0 + row;
      gx[q] = t < a.T ? __ldg(reinterpret_cast<const float4*>(a.x + (size_t)t * a.H + k0) + c4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      gw[q] = e < a.E ? __ldg(reinterpret_cast<const float4*>(a.router_w + (size_t)e * a.H + k0) + c4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int idx = tid + 256 * q, row = idx >> 3, k = 4 * (idx & 7);
      xs[k][row] = gx[q].x; xs[k + 1][row] = gx[q].y; xs[k + 2][row] = gx[q].z; xs[k + 3][row] = gx[q].w;
      ws[k][row] = gw[q].x; ws[k + 1][row] = gw[q].y; ws[k + 2][row] = gw[q].z; ws[k + 3][row] = gw[q].w;
    }
  };
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  load(0);
  for (int k0 = 0; k0 < a.H; k0 += RT_KS) {
    stash();
    __syncthreads();
    if (k0 + RT_KS < a.H) load(k0 + RT_KS);
#pragma unroll 8
    for (int k = 0; k < RT_KS; ++k) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[k][4 * ty]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[k][4 * tx]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * ty + i;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * tx + j;
      if (t < a.T && e < a.E) a.logits[(size_t)t * a.E + e] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// top-k: one warp per token
// ---------------------------------------------------------------------------
// One warp per token, TOPK_WARPS tokens a CTA: few warps a CTA spread a batch's tokens over
// every SM (a token's work is a serial chain of warp steps, so SMs, not warps per SM, set
// the pace). Lane l holds the keys of experts l + 32 i (i < EPL) in registers; every logit
// and bias is loaded before the first is used, so the token waits on one round trip.
constexpr int TOPK_WARPS = 2;
template <int EPL>
__device__ __forceinline__ void topk_token(const PrefillArgs& a, int t, int lane, uint8_t* base) {
  float* probs = reinterpret_cast<float*>(base);                            // [E]
  uint32_t* keys = reinterpret_cast<uint32_t*>(base + (size_t)a.E * 4);    // [E] (groups only)
  float* gscore = reinterpret_cast<float*>(base + (size_t)a.E * 8);        // [64]
  int* picks = reinterpret_cast<int*>(base + (size_t)a.E * 8 + 64 * 4);    // [32]
  float lg[EPL], bs[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    // the logit: the router's partial sums over its K slices, in slice order. Every slice
    // array is read (the workspace holds PREFILL_RT_SLICES of them) so that the loads issue
    // together, unpredicated; the unused ones drop out of the sum.
    const int ec = min(e, a.E - 1);
    float pk[PREFILL_RT_SLICES];
#pragma unroll
    for (int k = 0; k < PREFILL_RT_SLICES; ++k) pk[k] = __ldcg(a.logits + ((size_t)k * a.T + t) * a.E + ec);
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < PREFILL_RT_SLICES; ++k) l = k < a.rt_slices ? l + pk[k] : l;
    lg[i] = e < a.E ? l : 0.f;
    bs[i] = (a.bias && e < a.E) ? __ldg(a.bias + e) : 0.f;
  }
  uint32_t kv[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    kv[i] = 0u;
    if (e < a.E) {
      const float pr = 1.f / (1.f + expf(-lg[i]));
      probs[e] = pr;
      kv[i] = order_key(pr + bs[i]);
      if (a.G > 1) keys[e] = kv[i];
    }
  }
  __syncwarp();
  if (a.G > 1) {
    // group score: the two largest s of the group, summed (multiset top-2): each lane's two
    // largest over its experts of the group, then a butterfly that keeps the two largest
    const int per = a.E / a.G;
#pragma unroll 1
    for (int g = 0; g < a.G; ++g) {
      float x1 = -INFINITY, x2 = -INFINITY;
#pragma unroll 1
      for (int e = g * per + lane; e < (g + 1) * per; e += 32) {
        const uint32_t k = keys[e];
        const float v = __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
        if (v > x1) { x2 = x1; x1 = v; } else if (v > x2) { x2 = v; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ox1 = __shfl_xor_sync(0xffffffffu, x1, o);
        const float ox2 = __shfl_xor_sync(0xffffffffu, x2, o);
        const float hi = fmaxf(x1, ox1), lo = fminf(x1, ox1);
        x2 = fmaxf(lo, fmaxf(x2, ox2));
        x1 = hi;
      }
      if (lane == 0) gscore[g] = x1 + x2;
    }
    __syncwarp();
    // kept groups: groups_used rounds of the largest score, lowest group on ties. Lane l
    // offers groups l and l + 32, the larger first (a score's key is never 0: only a NaN's is)
    uint32_t gk0 = lane < a.G ? order_key(gscore[lane]) : 0u;
    uint32_t gk1 = lane + 32 < a.G ? order_key(gscore[lane + 32]) : 0u;
    int gi0 = lane, gi1 = lane + 32;
    if (gk1 > gk0) {
      const uint32_t tk = gk0; gk0 = gk1; gk1 = tk;
      gi0 = lane + 32; gi1 = lane;
    }
    unsigned long long kept = 0ull;
#pragma unroll 1
    for (int j = 0; j < a.Gu; ++j) {
      const uint32_t mk = __reduce_max_sync(0xffffffffu, gk0);
      const int win = (int)__reduce_min_sync(0xffffffffu, gk0 == mk && mk != 0u ? (unsigned)gi0 : 0xffffffffu);
      kept |= 1ull << (win & 63);
      if (gk0 == mk && gi0 == win) {
        gk0 = gk1; gi0 = gi1; gk1 = 0u;
      }
    }
    // experts of dropped groups take key 0
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E && !((kept >> (e / per)) & 1ull)) kv[i] = 0u;
    }
  }
  topk_rounds_kv<EPL>(kv, a.E, a.K, picks, lane);
  __syncwarp();
  const float pj = lane < a.K ? probs[picks[lane]] : 0.f;
  const float wsum = fmaxf(warp_sum(pj), a.norm_min);
  if (lane < a.K) {
    const int id = picks[lane];
    const float wj = pj / wsum * a.scale;
    a.ids[(size_t)t * a.K + lane] = id;
    a.wts[(size_t)t * a.K + lane] = wj;
    if (a.topk_ids) a.topk_ids[(size_t)t * a.K + lane] = id;
    if (a.topk_w) a.topk_w[(size_t)t * a.K + lane] = wj;
  }
}

__global__ void __launch_bounds__(32 * TOPK_WARPS) prefill_topk(const PrefillArgs a) {
  extern __shared__ __align__(16) uint8_t tsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * TOPK_WARPS + warp;
  if (t >= a.T) return;  // whole warp
  uint8_t* base = tsm + (size_t)warp * ((size_t)a.E * 8 + 64 * 4 + 32 * 4);
  if (a.E <= 256) topk_token<8>(a, t, lane, base);
  else if (a.E <= 512) topk_token<16>(a, t, lane, base);
  else topk_token<32>(a, t, lane, base);
}

// ---------------------------------------------------------------------------
// sort: one CTA of 1024 threads (E <= 1024: thread e owns expert e)
// ---------------------------------------------------------------------------
// Warp w owns the contiguous pair range of 32-pair chunks w * nc .. w * nc + nc - 1 (nc =
// ceil(P / 1024)), held in registers: MAXC >= nc is a template bound, the smallest of 4, 8, 16
// that fits (short straight-line code for the common sizes); a pass of T <= PREFILL_CHUNK_T
// tokens with K <= 32 has P <= 16384 pairs, so nc <= 16.
constexpr int SORT_WARPS = 32, SORT_MAXC = 16;
static_assert(SORT_WARPS * 32 * SORT_MAXC >= PREFILL_CHUNK_T * 32, "a pass's pairs fit the sort's chunks");

// Exclusive prefix sums over the CTA of three values at once; `tot` gets their sums.
__device__ __forceinline__ void cta_excl_scan3(uint32_t v[3], uint32_t (*wsum)[SORT_WARPS], uint32_t tot[3]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, inc[c], o);
      if (lane >= o) inc[c] += y;
    }
  }
  if (lane == 31)
    for (int c = 0; c < 3; ++c) wsum[c][warp] = inc[c];
  __syncthreads();
  if (warp < 3) {
    uint32_t w = wsum[warp][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[warp][lane] = w;  // inclusive over warps
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    tot[c] = wsum[c][SORT_WARPS - 1];
    v[c] = inc[c] - v[c] + (warp ? wsum[c][warp - 1] : 0u);
  }
}

// Dynamic shared memory of the sort for P pairs and E experts: the per-warp count table
// [SORT_WARPS][E] (u16), then the sorted pair ids and weights [P] (u32, f32), written out in
// order at the end (one coalesced pass instead of scattered stores from one SM).
__host__ __device__ __forceinline__ int sort_table_bytes(int E) { return (SORT_WARPS * E * 2 + 15) & ~15; }
__host__ __device__ __forceinline__ int sort_smem(int P, int E) { return sort_table_bytes(E) + P * 8; }

template <int MAXC>
__global__ void __launch_bounds__(1024) prefill_sort(const PrefillArgs a) {
  extern __shared__ __align__(16) uint8_t ssm[];
  __shared__ uint32_t offs[1024];
  __shared__ uint32_t wsum[3][SORT_WARPS];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = a.T * a.K, E = a.E, nc = (P + SORT_WARPS * 32 - 1) / (SORT_WARPS * 32);
  uint16_t* cnt_w = reinterpret_cast<uint16_t*>(ssm);
  uint32_t* s_perm = reinterpret_cast<uint32_t*>(ssm + sort_table_bytes(E));
  float* s_w = reinterpret_cast<float*>(s_perm + P);
  const uint32_t lt = (1u << lane) - 1u;
  // every pick and weight of this warp's range, loaded at once
  uint32_t pk[MAXC];  // the pick (E: none), then its rank in bits 16..31
  float wv[MAXC];
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    if (i >= nc) break;
    const int p = (warp * nc + i) * 32 + lane;
    pk[i] = p < P ? (uint32_t)__ldg(a.ids + p) : (uint32_t)E;
    wv[i] = p < P ? __ldg(a.wts + p) : 0.f;
  }
  for (int i = tid; i < SORT_WARPS * E; i += 1024) cnt_w[i] = 0;
  __syncthreads();
  // (a) the warp's count of each expert over its range; each pair's rank among the range's
  // pairs of its expert (earlier chunks, then earlier lanes)
  uint16_t* row = cnt_w + (size_t)warp * E;
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    if (i >= nc) break;
    const int e = (int)pk[i];
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    if (e < E) pk[i] |= (uint32_t)(row[e] + __popc(m & lt)) << 16;
    __syncwarp();
    if (e < E && (m & lt) == 0) row[e] = (uint16_t)(row[e] + __popc(m));
    __syncwarp();
  }
  __syncthreads();
  // (b) per expert: the counts of the earlier warps (in place), and the total
  uint32_t cnt = 0;
  if (tid < E) {
#pragma unroll
    for (int w0 = 0; w0 < SORT_WARPS; w0 += 8) {
      uint16_t c[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) c[w] = cnt_w[(w0 + w) * E + tid];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        cnt_w[(w0 + w) * E + tid] = (uint16_t)cnt;
        cnt += c[w];
      }
    }
  }
  // (c) first sorted position, first chunk and first padded row of each expert
  const int nmax = a.nmax;
  const uint32_t nck = (cnt + nmax - 1) / nmax;
  const uint32_t prows = nck ? (nck - 1) * nmax + ((cnt - (nck - 1) * nmax + 15) & ~15u) : 0u;
  uint32_t v[3] = {cnt, nck, prows}, tot[3];
  cta_excl_scan3(v, wsum, tot);
  const uint32_t off = v[0], cbase = v[1], pbase = v[2], nrouted = tot[1];
  if (tid < E) {
    offs[tid] = off;
    a.offsets[tid] = off;
    for (uint32_t r = 0; r < nck; ++r) {
      const int row0 = (int)(off + r * nmax), n = (int)min(cnt - r * nmax, (uint32_t)nmax);
      a.chunks[cbase + r] = GemmChunk{tid, row0, n, (int)(pbase + r * nmax)};
    }
  }
  if (tid == 0) a.offsets[E] = tot[0];
  // shared-expert chunks (token chunks) follow the routed ones
  const int nsh = a.Fs ? (a.T + nmax - 1) / nmax : 0;
  if (tid < nsh) a.chunks[nrouted + tid] = GemmChunk{E, tid * nmax, min(a.T - tid * nmax, nmax), tid * nmax};
  if (tid == 0) {
    a.nchunks[0] = nrouted;
    a.nchunks[1] = nrouted + (uint32_t)nsh;
  }
  __syncthreads();
  // (d) stable positions: expert's first position + earlier warps + rank in the range
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    if (i >= nc) break;
    const int e = (int)(pk[i] & 0xffffu);
    if (e < E) {
      const int p = (warp * nc + i) * 32 + lane;
      const uint32_t pos = offs[e] + row[e] + (pk[i] >> 16);
      s_perm[pos] = (uint32_t)p;
      s_w[pos] = wv[i];
      a.pos_of[p] = pos;
    }
  }
  __syncthreads();
  for (int i = tid; i < P; i += 1024) {
    a.perm[i] = s_perm[i];
    a.wsorted[i] = s_w[i];
  }
}

// ---------------------------------------------------------------------------
// x16: X -> hi and lo f16 rows in the permuted K order (row 2t: hi, row 2t + 1: lo)
// ---------------------------------------------------------------------------
__global__ void prefill_x16(const PrefillArgs a) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t n = (size_t)a.T * a.H;
  if (i >= n) return;
  const int k = (int)(i % a.H);
  const size_t t = i / a.H;
  const float v = __ldg(a.x + i);
  const __half hi = __float2half_rn(v);
  a.x16[(2 * t) * a.H + kpos(k)] = hi;
  a.x16[(2 * t + 1) * a.H + kpos(k)] = __float2half_rn(v - __half2float(hi));
}

// ---------------------------------------------------------------------------
// grouped Q4 GEMM on the tensor cores (MODE 0: gate/up + SwiGLU, 1: down + weight)
// ---------------------------------------------------------------------------
constexpr int KC = 128;                      // K values per pipeline chunk (4 blocks)
constexpr int A_STAGE = 128 * KC * 2;        // 32 KB f16
// B stage: up to 2 * PREFILL_NMAX rows (gate/up: hi and lo rows of each token)
constexpr int B_STAGE_GU = 2 * PREFILL_NMAX * KC * 2;  // 32 KB f16
constexpr int B_STAGE_DN = PREFILL_NMAX * KC * 2;      // 16 KB f16
constexpr uint32_t TMEM_COLS = 256;
constexpr int NSTAGE = 3;                    // pipeline stages (A and B buffers)

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}
__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// One nibble word (values 4w..4w+3 and 16+4w..16+4w+3 of a block) -> the 16-byte
// core-matrix row of slots 8w .. 8w+7, value = d*q + m (Q4_1) or d*(q - 8) (Q4_0).
template <int QT>
__device__ __forceinline__ uint4 dequant_word(uint32_t qw, __half2 d2, __half2 m2) {
  const uint32_t MAGIC = 0x64006400u;  // f16 1024 in both halves
  const uint32_t sh = qw >> 8;
  __half2 lo02 = bits2h(lop3_and_or(qw, 0x000F000Fu, MAGIC));  // 1024 + q
  __half2 lo13 = bits2h(lop3_and_or(sh, 0x000F000Fu, MAGIC));
  __half2 hi02 = bits2h(lop3_and_or(qw, 0x00F000F0u, MAGIC));  // 1024 + 16 q
  __half2 hi13 = bits2h(lop3_and_or(sh, 0x00F000F0u, MAGIC));
  const __half2 k16 = __float2half2_rn(0.0625f);
  if constexpr (QT == 3) {
    const __half2 b1024 = __float2half2_rn(1024.f), b64 = __float2half2_rn(-64.f);
    lo02 = __hfma2(__hsub2(lo02, b1024), d2, m2);
    lo13 = __hfma2(__hsub2(lo13, b1024), d2, m2);
    hi02 = __hfma2(__hfma2(hi02, k16, b64), d2, m2);
    hi13 = __hfma2(__hfma2(hi13, k16, b64), d2, m2);
  } else {
    const __half2 b1032 = __float2half2_rn(1032.f), b72 = __float2half2_rn(-72.f);
    lo02 = __hmul2(__hsub2(lo02, b1032), d2);
    lo13 = __hmul2(__hsub2(lo13, b1032), d2);
    hi02 = __hmul2(__hfma2(hi02, k16, b72), d2);
    hi13 = __hmul2(__hfma2(hi13, k16, b72), d2);
  }
  return make_uint4(h2bits(lo02), h2bits(lo13), h2bits(hi02), h2bits(hi13));
}

// Values 4w .. 4w + 3 (bytes of qa) and 16 + 4w .. 16 + 4w + 3 (bytes of qb) of a 32-value
// block, each v = df * q + mf in f32 (exact for the K-quant scales) and rounded once to f16,
// as the core-matrix row of slots 8w .. 8w + 7 (slot order: kslot).
__device__ __forceinline__ uint4 core_row_f32(uint32_t qa, uint32_t qb, float df, float mf) {
  float v[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[k] = fmaf(df, (float)((qa >> (8 * k)) & 0xFFu), mf);
    v[4 + k] = fmaf(df, (float)((qb >> (8 * k)) & 0xFFu), mf);
  }
  return make_uint4(h2bits(__floats2half2_rn(v[0], v[2])), h2bits(__floats2half2_rn(v[1], v[3])),
                    h2bits(__floats2half2_rn(v[4], v[6])), h2bits(__floats2half2_rn(v[5], v[7])));
}

// Block `blk` (32 values) of a weight row in global memory, dequantised into the four core
// rows of its slots, in two steps so that a thread can have several blocks' loads in
// flight before it uses them: load_raw issues the loads, dequant_raw does the arithmetic.
// Q4_0/Q4_1: one block. K-quants (ggml layouts, as the Ling store keeps them; the pages name
// the types only): sub-block blk % 8 of super-block blk / 8.
//   Q4_K (144 bytes, rows on 16-byte bounds): f16 d, f16 dmin, 12 packed scale bytes S,
//   four runs of 32 nibble bytes (run c: sub-block 2c low nibbles, 2c + 1 high nibbles);
//   sub-block j < 4: sc = S[j] & 63, mn = S[j + 4] & 63; j >= 4: low 4 bits from S[j + 4],
//   top 2 bits from S[j - 4] (sc) and S[j] (mn); value = d sc q - dmin mn.
//   Q6_K (210 bytes, rows on 2-byte bounds): ql[128], qh[64], 16 int8 scales, f16 d;
//   sub-block j = (n = j / 4, r = j % 4), value i: nibble (low for r < 2) of
//   ql[64n + 32 (r % 2) + i], high bits 2r, 2r + 1 of qh[32n + i], scale[8n + 2r + i / 16];
//   value = d * scale * (q - 32).
struct RawBlk {
  uint32_t w[18];
};

template <int QT>
__device__ __forceinline__ void load_raw(const uint8_t* row, int blk, RawBlk& r) {
  if constexpr (QT == 12) {
    const uint8_t* sb = row + 144 * (blk >> 3);
    const int j = blk & 7;
    const uint4 hd = __ldg(reinterpret_cast<const uint4*>(sb));
    const uint4 n0 = __ldg(reinterpret_cast<const uint4*>(sb + 16 + 32 * (j >> 1)));
    const uint4 n1 = __ldg(reinterpret_cast<const uint4*>(sb + 32 + 32 * (j >> 1)));
    r.w[0] = hd.x; r.w[1] = hd.y; r.w[2] = hd.z; r.w[3] = hd.w;
    r.w[4] = n0.x; r.w[5] = n0.y; r.w[6] = n0.z; r.w[7] = n0.w;
    r.w[8] = n1.x; r.w[9] = n1.y; r.w[10] = n1.z; r.w[11] = n1.w;
  } else if constexpr (QT == 14) {
    const uint8_t* sb = row + 210 * (blk >> 3);
    const int j = blk & 7, n = j >> 2, q = j & 3;
    // each 32-byte run as nine aligned words, shifted by the run's 2-byte offset (the run ends
    // at least 4 bytes before its super-block does, so the ninth word stays inside it)
    const uint8_t* ql = sb + 64 * n + 32 * (q & 1);
    const uint8_t* qh = sb + 128 + 32 * n;
    const uint32_t* wl = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(ql) & ~uintptr_t(3));
    const uint32_t* wh = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(qh) & ~uintptr_t(3));
    const uint32_t sl = (uint32_t)(reinterpret_cast<uintptr_t>(ql) & 3u) * 8u;  // 0 or 16
    uint32_t tl[9], th[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      tl[i] = __ldg(wl + i);
      th[i] = __ldg(wh + i);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r.w[i] = __funnelshift_r(tl[i], tl[i + 1], sl);
      r.w[8 + i] = __funnelshift_r(th[i], th[i + 1], sl);
    }
    r.w[16] = __ldg(reinterpret_cast<const unsigned short*>(sb + 192 + 8 * n + 2 * q));
    r.w[17] = __ldg(reinterpret_cast<const unsigned short*>(sb + 208));
  } else if constexpr (QT == 3) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(row + 20 * blk);
#pragma unroll
    for (int i = 0; i < 5; ++i) r.w[i] = __ldg(w + i);
  } else {
    const unsigned short* h = reinterpret_cast<const unsigned short*>(row + 18 * blk);
    unsigned short u[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) u[i] = __ldg(h + i);
    r.w[0] = u[0];
#pragma unroll
    for (int i = 0; i < 4; ++i) r.w[1 + i] = (uint32_t)u[1 + 2 * i] | ((uint32_t)u[2 + 2 * i] << 16);
  }
}

template <int QT>
__device__ __forceinline__ void dequant_raw(const RawBlk& r, int blk, uint4 (&o)[4]) {
  if constexpr (QT == 12) {
    const int j = blk & 7, sh = 8 * (j & 3);
    const uint32_t by = (r.w[1] >> sh) & 0xFFu, bz = (r.w[2] >> sh) & 0xFFu, bw = (r.w[3] >> sh) & 0xFFu;
    const uint32_t sc = j < 4 ? (by & 63u) : ((bw & 15u) | ((by >> 6) << 4));
    const uint32_t mn = j < 4 ? (bz & 63u) : ((bw >> 4) | ((bz >> 6) << 4));
    const float2 f = __half22float2(bits2h(r.w[0]));
    const float df = f.x * (float)sc, mf = -(f.y * (float)mn);
    const int ns = 4 * (j & 1);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      o[c] = core_row_f32((r.w[4 + c] >> ns) & 0x0F0F0F0Fu, (r.w[8 + c] >> ns) & 0x0F0F0F0Fu, df, mf);
  } else if constexpr (QT == 14) {
    const int q = blk & 3;
    const float d = __half2float(__ushort_as_half((unsigned short)r.w[17]));
    const uint32_t scp = r.w[16];
    const float df0 = d * (float)(int)(int8_t)(scp & 0xFFu), df1 = d * (float)(int)(int8_t)(scp >> 8);
    const int ls = 4 * (q >> 1), hs = 2 * q;
    uint32_t u[8];  // q of values 4i .. 4i + 3, 0 .. 63
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = ((r.w[i] >> ls) & 0x0F0F0F0Fu) | (((r.w[8 + i] >> hs) & 0x03030303u) << 4);
    // values 0 .. 15 take scale 0 and 16 .. 31 scale 1: core row c holds 4c .. (first half)
    // and 16 + 4c .. (second half), so each half has its own scale; q - 32 enters as the offset
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 lo = core_row_f32(u[c], 0u, df0, -32.f * df0);
      const uint4 hi = core_row_f32(u[4 + c], 0u, df1, -32.f * df1);
      o[c] = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  } else {
    __half2 d2, m2;
    if constexpr (QT == 3) {
      const __half2 h = bits2h(r.w[0]);
      d2 = __low2half2(h);
      m2 = __high2half2(h);
    } else {
      d2 = __half2half2(__ushort_as_half((unsigned short)r.w[0]));
      m2 = d2;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) o[w] = dequant_word<QT>(r.w[1 + w], d2, m2);
  }
}

// The two blocks (rows m = i % 128, blocks b = i / 128 of the chunk, i = tid and
// tid + 256) that thread `tid` dequantises for pipeline chunk kc: their loads are issued.
template <int QT, typename RowFn>
__device__ __forceinline__ void issue_raw(RawBlk (&r)[2], bool (&v)[2], int kc, int nbk, int mrows, int tid,
                                          const RowFn& wrow) {
  const int kb = min(KC / 32, nbk - kc * (KC / 32));
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int i = pass * PREFILL_THREADS + tid, m = i & 127, b = i >> 7;
    v[pass] = m < mrows && b < kb;
    if (v[pass]) load_raw<QT>(wrow(m), kc * (KC / 32) + b, r[pass]);
  }
}

// 16 bytes from global to shared memory without a register round trip; with !valid the
// destination is zero-filled (nothing is read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most one (wait_group1) or none (wait_group0) of the committed groups of the
// thread's asynchronous copies is still in flight.
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_group0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// L2 prefetch of the 16-byte-aligned part of [p, p + bytes).
__device__ __forceinline__ void prefetch_span(const void* p, uint32_t bytes) {
  const uintptr_t lo = (reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15);
  const uintptr_t hi = (reinterpret_cast<uintptr_t>(p) + bytes) & ~uintptr_t(15);
  if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo));
}

template <int QT, int MODE>
__global__ void __launch_bounds__(PREFILL_THREADS, 1) prefill_gemm(const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t gsm[];
  uint8_t* As = gsm;                      // [NSTAGE][A_STAGE]
  constexpr int B_STAGE = MODE == 0 ? B_STAGE_GU : B_STAGE_DN;
  uint8_t* Bs = gsm + NSTAGE * A_STAGE;   // [NSTAGE][B_STAGE]
  __shared__ __align__(8) uint64_t mma_bar[NSTAGE];
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t rowsrc[PREFILL_NMAX];  // B source row of each chunk row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) tmem_alloc(&tmem_base, TMEM_COLS);
  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(&mma_bar[i], 1);
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;

  const int nr = (int)a.nchunks[0], ntot = (int)a.nchunks[1];
  // M tiles per chunk: gate/up 64 pairs (128 rows) a tile, down 128 output rows a tile
  const int mt_r = MODE == 0 ? ceil_div(a.F, 64) : ceil_div(a.H, 128);
  const int mt_s = MODE == 0 ? ceil_div(a.Fs > 0 ? a.Fs : 1, 64) : ceil_div(a.H, 128);
  const int units = nr * mt_r + (ntot - nr) * mt_s;
  uint32_t g = 0;  // pipeline chunks so far (stage = g % NSTAGE, use = g / NSTAGE)
  bool ok = true;

  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    int ci, mt;
    if (u < nr * mt_r) { ci = u / mt_r; mt = u % mt_r; }
    else { ci = nr + (u - nr * mt_r) / mt_s; mt = (u - nr * mt_r) % mt_s; }
    const GemmChunk ch = a.chunks[ci];
    const bool sh = ch.slot >= a.E;
    const int ff = sh ? a.Fs : a.F;
    const uint8_t* rec = sh ? a.shared : a.experts + (size_t)ch.slot * a.rec_bytes;
    const int Kdim = MODE == 0 ? a.H : ff;       // reduction length
    const int nbk = Kdim / 32;                   // blocks per weight row
    const int nkc = ceil_div(nbk, KC / 32);      // pipeline chunks
    const int npad = (ch.n + 15) & ~15;      // chunk rows, rounded up for the MMA
    const int nb = MODE == 0 ? 2 * npad : npad;  // B rows: gate/up takes hi then lo rows
    // weight rows of this tile
    const uint32_t rb = MODE == 0 ? a.rb_h : (sh ? a.rb_fs : a.rb_f);
    int mrows;  // valid M rows of the tile
    if (MODE == 0) mrows = 2 * min(64, ff - 64 * mt);
    else mrows = min(128, a.H - 128 * mt);
    auto wrow = [&](int m) -> const uint8_t* {
      if (MODE == 0) {
        const int f = 64 * mt + (m >> 1);
        return rec + (size_t)((m & 1) ? ff + f : f) * rb;  // even rows gate, odd rows up
      }
      return rec + (size_t)2 * ff * a.rb_h + (size_t)(128 * mt + m) * rb;
    };
    if (tid == 0) {  // bring this tile's rows into L2 ahead of the loads
      if (MODE == 0) {
        const uint32_t bytes = (uint32_t)(mrows / 2) * rb;
        prefetch_span(wrow(0), bytes);
        prefetch_span(wrow(1), bytes);
      } else {
        prefetch_span(wrow(0), (uint32_t)mrows * rb);
      }
    }
    // B rows: the chunk's tokens (gate/up) or sorted pairs (down)
    for (int r = tid; r < ch.n; r += PREFILL_THREADS) {
      if (MODE == 0) rowsrc[r] = sh ? (uint32_t)(ch.row0 + r) : a.perm[ch.row0 + r] / (uint32_t)a.K;
      else rowsrc[r] = (uint32_t)(ch.row0 + r);
    }
    __syncthreads();
    const __half* bsrc = MODE == 0 ? a.x16 : (sh ? a.act16s : a.act16);
    const int bld = MODE == 0 ? a.H : ff;  // B row length (values)
    // Three stages, each an A and a B buffer that the MMAs of one chunk read. Chunk kc takes
    // stage g % NSTAGE; its B rows are copied one chunk ahead (into the stage once the MMAs of
    // its previous use are done), and its A blocks are loaded two chunks ahead into registers.
    auto stage_free = [&](uint32_t gs) {  // the MMAs of stage use gs - NSTAGE are done
      if (gs >= (uint32_t)NSTAGE && !mbar_wait(&mma_bar[gs % NSTAGE], ((gs / NSTAGE) - 1) & 1u)) ok = false;
    };
    auto copy_b = [&](int kc, uint32_t gs) {  // rows past the chunk are zero-filled
      uint8_t* B = Bs + (gs % NSTAGE) * B_STAGE;
      const int kb = min(KC / 32, nbk - kc * (KC / 32));
      const int pieces = kb * 4;  // 8 values a piece
      for (int i = tid; i < nb * pieces; i += PREFILL_THREADS) {
        const int r = i / pieces, pc = i % pieces;
        const int rr = r < npad ? r : r - npad;  // chunk row (lo rows: second half)
        const bool valid = rr < ch.n;
        const size_t src = !valid ? 0 : MODE == 0 ? 2 * (size_t)rowsrc[rr] + (r >= npad) : (size_t)rowsrc[rr];
        cp_async16(B + (pc * (nb / 8) + (r >> 3)) * 128 + 16 * (r & 7), bsrc + src * bld + kc * KC + pc * 8, valid);
      }
      cp_async_commit();
    };
    RawBlk r0[2], r1[2], r2[2];
    bool v0[2], v1[2] = {false, false}, v2[2] = {false, false};
    issue_raw<QT>(r0, v0, 0, nbk, mrows, tid, wrow);
    if (nkc > 1) issue_raw<QT>(r1, v1, 1, nbk, mrows, tid, wrow);
    stage_free(g);
    copy_b(0, g);

    for (int kc = 0; kc < nkc; ++kc, ++g) {
      const int s = (int)(g % NSTAGE);
      const bool more = kc + 1 < nkc;
      if (more) {  // the next chunk's B rows, into the next stage once its last MMAs are done
        stage_free(g + 1);
        copy_b(kc + 1, g + 1);
      }
      if (kc + 2 < nkc) issue_raw<QT>(r2, v2, kc + 2, nbk, mrows, tid, wrow);
      // A: 128 rows x 4 blocks, two per thread; a warp takes 32 consecutive rows of one
      // block, so its 16-byte shared stores of one core row cover all banks
      uint8_t* A = As + s * A_STAGE;
      const int kb = min(KC / 32, nbk - kc * (KC / 32));  // blocks in this chunk
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const int i = pass * PREFILL_THREADS + tid, m = i & 127, b = i >> 7;
        if (v0[pass]) {
          uint4 o[4];
          dequant_raw<QT>(r0[pass], kc * (KC / 32) + b, o);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int kcore = 4 * b + w, mcore = m >> 3;
            *reinterpret_cast<uint4*>(A + (kcore * 16 + mcore) * 128 + 16 * (m & 7)) = o[w];
          }
        }
      }
      if (more) cp_async_wait_group1();  // this chunk's B rows (the next chunk's may still fly)
      else cp_async_wait_group0();
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        r0[pass] = r1[pass];
        v0[pass] = v1[pass];
        r1[pass] = r2[pass];
        v1[pass] = v2[pass];
        v2[pass] = false;
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after_sync();
        const uint8_t* B = Bs + s * B_STAGE;
        const uint32_t idesc = idesc_f16_f32(128, nb);
        for (int j = 0; j < 2 * kb; ++j) {  // K = 16 per MMA: two core matrices along K
          const uint64_t ad = smem_desc(A + 2 * j * 2048, 2048, 128);
          const uint64_t bd = smem_desc(B + 2 * j * 16 * nb, 16 * nb, 128);
          mma_f16(tmem, ad, bd, idesc, kc > 0 || j > 0);
        }
        mma_commit(&mma_bar[s]);
      }
    }
    // epilogue: the last commit covers every MMA of the tile
    {
      const uint32_t gl = g - 1;
      if (!mbar_wait(&mma_bar[gl % NSTAGE], (gl / NSTAGE) & 1u)) ok = false;
    }
    tc_fence_after_sync();
    if (warp < 4) {
      const int m = 32 * warp + lane;  // this thread's TMEM lane = tile row
      for (int c0 = 0; c0 < npad; c0 += 16) {
        uint32_t r[16];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        tmem_ld16(lane_base + (uint32_t)c0, r);
        if (MODE == 0) {
          uint32_t rl[16];
          tmem_ld16(lane_base + (uint32_t)(npad + c0), rl);
          tmem_ld_wait();
          const int f = 64 * mt + (m >> 1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float v = __uint_as_float(r[i]) + __uint_as_float(rl[i]);  // x_hi + x_lo parts
            const float other = __shfl_xor_sync(0xffffffffu, v, 1);
            const int c = c0 + i;
            if (!(m & 1) && m < mrows && c < ch.n) {
              const float act = swiglu_act(v, other, sh ? a.lim_s : a.lim);  // silu(gate) * up, clamped
              __half* dst = sh ? a.act16s + (size_t)(ch.row0 + c) * ff : a.act16 + (size_t)(ch.row0 + c) * ff;
              dst[kpos(f)] = __float2half_rn(act);
            }
          }
        } else {
          tmem_ld_wait();
          const int h = 128 * mt + m;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (m < mrows && c < ch.n) {
              const float y = __uint_as_float(r[i]);
              if (sh) a.sbuf[(size_t)(ch.row0 + c) * a.H + h] = y;
              else a.ybuf[(size_t)(ch.row0 + c) * a.H + h] = a.wsorted[ch.row0 + c] * y;
            }
          }
        }
      }
    }
    tc_fence_before_sync();
    // TMEM read and rowsrc used before the next tile reuses them; a timed-out wait
    // anywhere in the CTA ends its loop
    const bool failed = __syncthreads_or(!ok);
    tc_fence_after_sync();
    if (failed) {
      ok = false;
      break;
    }
  }
  if (!ok && tid == 0) atomicOr(a.status, DEV_ERR_MBAR_TIMEOUT);
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// combine: out[t][h] = sum_j ybuf[pos(t, j)][h] + sbuf[t][h] (+ x | + out)
// ---------------------------------------------------------------------------
__global__ void prefill_combine(const PrefillArgs a) {
  // four consecutive outputs a thread (H is a multiple of 32); the sum order per output is
  // unchanged: the picks in order, then the shared row, then the residual or out
  const size_t i4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i4 * 4 >= (size_t)a.T * a.H) return;
  const size_t i = i4 * 4;
  const int t = (int)(i / a.H), h = (int)(i % a.H);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.K; ++j) {
    const uint32_t pj = __ldg(a.pos_of + (size_t)t * a.K + j);
    const float4 y = __ldcs(reinterpret_cast<const float4*>(a.ybuf + (size_t)pj * a.H + h));
    acc.x += y.x;
    acc.y += y.y;
    acc.z += y.z;
    acc.w += y.w;
  }
  if (a.Fs) {
    const float4 sv = __ldcs(reinterpret_cast<const float4*>(a.sbuf + i));
    acc.x += sv.x;
    acc.y += sv.y;
    acc.z += sv.z;
    acc.w += sv.w;
  }
  if (a.flags & FLAG_RESIDUAL) {
    const float4 xv = *reinterpret_cast<const float4*>(a.xres + i);
    acc.x = xv.x + acc.x;
    acc.y = xv.y + acc.y;
    acc.z = xv.z + acc.z;
    acc.w = xv.w + acc.w;
  }
  if (a.flags & FLAG_ACCUMULATE) {
    const float4 ov = *reinterpret_cast<const float4*>(a.out + i);
    acc.x = ov.x + acc.x;
    acc.y = ov.y + acc.y;
    acc.z = ov.z + acc.z;
    acc.w = ov.w + acc.w;
  }
  *reinterpret_cast<float4*>(a.out + i) = acc;
}

// The layer prologue: xn[t] = x[t] / sqrt(mean(x[t]^2) + eps) * norm, one CTA per token.
__global__ void __launch_bounds__(256) prefill_rmsnorm(const PrefillArgs a) {
  __shared__ float red[32];
  const int t = blockIdx.x;
  const float* xr = a.x + (size_t)t * a.H;
  const float r = block_rms_scale(xr, a.H, a.eps, red);
  for (int h = 4 * threadIdx.x; h < a.H; h += 4 * blockDim.x) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(xr + h));
    const float4 n = __ldg(reinterpret_cast<const float4*>(a.norm + h));
    *reinterpret_cast<float4*>(a.xn + (size_t)t * a.H + h) =
        make_float4(v.x * r * n.x, v.y * r * n.y, v.z * r * n.z, v.w * r * n.w);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static size_t up256(size_t v) { return (v + 255) / 256 * 256; }

bool prefill_tile_ok(int H, int F, int Fs, int qtype, int qtype_dn) {
  if (qtype == 12 && (qtype_dn == 12 || qtype_dn == 14)) {
    // Q4_K gate/up rows in 256-value super-blocks; Q6_K down rows as whole rows in one stage
    if (H % 256 || F % 256 || Fs % 256) return false;
    return qtype_dn == 12 || (F <= 768 && Fs <= 768);
  }
  if (qtype != qtype_dn || (qtype != 2 && qtype != 3)) return false;
  const int kc = qtype == 3 ? 128 : 256;
  return H % kc == 0 && F % kc == 0 && Fs % kc == 0;
}

PrefillWs prefill_ws_layout(int T, int H, int E, int K, int F, int Fs, bool tile) {
  PrefillWs w{};
  const size_t P = (size_t)T * K;
  const size_t nmax = tile ? PREFILL_TILE_NMAX : PREFILL_NMAX;
  const size_t max_routed = (P + nmax - 1) / nmax + (size_t)E;  // routed chunks at most
  const size_t tok_chunks = ((size_t)T + nmax - 1) / nmax;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = up256(o + bytes); return at; };
  w.logits = take((size_t)T * E * 4 * PREFILL_RT_SLICES);  // the tile router's partial sums (top-k reads all)
  w.ids = take(P * 4);
  w.wts = take(P * 4);
  w.offsets = take((size_t)(E + 1) * 4);
  w.perm = take(P * 4);
  w.wsorted = take(P * 4);
  w.pos_of = take(P * 4);
  w.chunks = take((max_routed + tok_chunks + 1) * sizeof(GemmChunk));
  w.nchunks = take(8);
  w.ybuf = take(P * H * 4);
  w.sbuf = take((size_t)T * H * 4);
  if (!tile) {
    w.x16 = take((size_t)T * H * 4);
    w.act16 = take(P * F * 2);
    w.act16s = take((size_t)T * (Fs ? Fs : 1) * 2);
  } else {
    const size_t prow_routed = P + 15 * max_routed;  // padded rows of all routed chunks, at most
    const size_t prow_tok = tok_chunks * nmax;
    w.ximg = take(2 * prow_tok * H * 2);
    w.ximg_routed = take(2 * prow_routed * H * 2);
    w.aimg = take(prow_routed * F * 2);
    w.aimg_s = take(prow_tok * (Fs ? Fs : 32) * 2);
  }
  w.total = o;
  return w;
}

template <int QT, int MODE>
static cudaError_t launch_gemm(const PrefillArgs& a, cudaStream_t st) {
  auto kern = prefill_gemm<QT, MODE>;
  const int smem = NSTAGE * (A_STAGE + (MODE == 0 ? B_STAGE_GU : B_STAGE_DN));
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<a.nc, PREFILL_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t prefill_launch(const PrefillArgs& a_in, cudaStream_t st) {
  cudaError_t e;
  PrefillArgs a = a_in;
  const size_t nx = (size_t)a.T * a.H;
  if (a.norm) {
    // the prologue: every kernel below reads the normalised tokens, the combine's
    // residual the raw ones (a.xres)
    prefill_rmsnorm<<<(unsigned)a.T, 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    a.x = a.xn;
  }
  a.rt_slices = a.rt_ups = 1;
  if (a.tile) {
    // the router's (token chunk, 64 experts) tiles are cut into up to PREFILL_RT_SLICES K slices
    // while the tiles still fit one wave of the persistent grid
    const int nkh = a.H / 128, tiles = ((a.T + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX) * ((a.E + 63) / 64);
    const int s = std::max(1, std::min(std::min(PREFILL_RT_SLICES, nkh), a.nc / tiles));
    a.rt_ups = (nkh + s - 1) / s;
    a.rt_slices = (nkh + a.rt_ups - 1) / a.rt_ups;
    // token-chunk images first: the router and the shared expert read them
    if ((e = tile_images_launch(a, false, st)) != cudaSuccess) return e;
    if ((e = tile_router_launch(a, st)) != cudaSuccess) return e;
  } else {
    prefill_router<<<dim3((a.E + RT_TILE - 1) / RT_TILE, (a.T + RT_TILE - 1) / RT_TILE), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t topk_smem = (size_t)TOPK_WARPS * ((size_t)a.E * 8 + 64 * 4 + 32 * 4);
  e = ensure_smem(reinterpret_cast<const void*>(prefill_topk), (int)topk_smem);
  if (e != cudaSuccess) return e;
  prefill_topk<<<(a.T + TOPK_WARPS - 1) / TOPK_WARPS, 32 * TOPK_WARPS, topk_smem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    const int sbytes = sort_smem(a.T * a.K, a.E);
    const int nc = (a.T * a.K + SORT_WARPS * 32 - 1) / (SORT_WARPS * 32);
    auto kern = nc <= 4 ? prefill_sort<4> : nc <= 8 ? prefill_sort<8> : prefill_sort<SORT_MAXC>;
    if ((e = ensure_smem(reinterpret_cast<const void*>(kern), sbytes)) != cudaSuccess) return e;
    kern<<<1, 1024, sbytes, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.tile) {
    if ((e = tile_images_launch(a, true, st)) != cudaSuccess) return e;
    // gate/up runs weights-as-A; the down contraction runs tokens-as-A when its
    // 256-row weight tiles cover H exactly (the faster of the two layouts for each)
    if ((e = tile_gemm_launch(a, 0, st)) != cudaSuccess) return e;
    const bool swap = a.H % 256 == 0 && (a.qtype_dn == 2 || a.qtype_dn == 3);
    if ((e = swap ? swap_down_launch(a, st) : tile_gemm_launch(a, 1, st)) != cudaSuccess) return e;
  } else {
    prefill_x16<<<(unsigned)((nx + 255) / 256), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    switch (a.qtype) {  // gate/up in the gate/up rows' block type
      case 2: e = launch_gemm<2, 0>(a, st); break;
      case 3: e = launch_gemm<3, 0>(a, st); break;
      case 12: e = launch_gemm<12, 0>(a, st); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    switch (a.qtype_dn) {  // down in the down rows' block type
      case 2: e = launch_gemm<2, 1>(a, st); break;
      case 3: e = launch_gemm<3, 1>(a, st); break;
      case 12: e = launch_gemm<12, 1>(a, st); break;
      case 14: e = launch_gemm<14, 1>(a, st); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  prefill_combine<<<(unsigned)((nx / 4 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
