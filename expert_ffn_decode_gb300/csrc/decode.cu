// Single-token MoE-FFN step (decode, T = 1) for sm_103a: three kernels in a chain.
//
//   dec_router    one router row per 4 warps (each a quarter of H), f32 dot with x
//                 -> logits; the last CTA to finish (counted with a device-scope
//                 atomic after a fence) turns them into sigmoid probabilities and
//                 selection scores, runs the (group-limited) top-k and writes the
//                 picks and their normalised weights
//   dec_gate_up   one CTA per activation block: 32 intermediate values of a slot (the
//                 shared expert's blocks first, then the picks'). Two values a warp:
//                 their gate and up rows against x -> SwiGLU -> the block, held as
//                 22-bit block fixed point (byte planes), written out
//   dec_down      one warp per output row: the row's block of every slot's down
//                 matrix against the activation blocks, each weighted by its slot's
//                 routing weight (1 for the shared expert), summed in a fixed order
//
// The kernels run with programmatic dependent launch, and each requests the bytes it
// can before waiting on its predecessor:
//   - the router kernel loads its router rows before the wait for x;
//   - the gate/up kernel quantises x, and computes the shared expert's blocks, while
//     the router kernel runs;
//   - the down kernel loads its rows' weight blocks while the gate/up kernel runs
//     (the picks are known by then).
// There are no grid-wide spin waits: kernel boundaries order every exchange.
//
// Dequant-dot: a 4-bit block (ggml Q4_0/Q4_1, 32 values) times 32 activations.
// Activations are held per 32-block as integers v = x * 2^k with |v| <= 2^22
// (power-of-two block scale; error at most 2^-22 of the block's largest
// magnitude), split into byte planes; dp4a forms sum(q * v) exactly in int32,
// the block result d * s * sum(q v) (+ m * s * sum(v) for Q4_1, - 8 d s sum(v)
// for Q4_0) is accumulated in fp32. The block formats and the per-block dot
// identity follow flint_moe_ssd.js (WGSL section, Q41DOT and its comment).
#include <cstdint>
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_host.h"
#include "plan.h"
#include "select.cuh"

namespace moe {

constexpr int RT_THREADS = 256;  // router: 8 warps, two rows a CTA
constexpr int GU_THREADS = 512;  // gate/up: 16 warps, two intermediate values each
constexpr int DN_THREADS = 256;  // down: 8 warps, one output row each
constexpr int DN_PRE = 8;        // down blocks a lane loads before the wait (rows of up to 256 blocks)

// ---------------------------------------------------------------------------
// Activation blocks
// ---------------------------------------------------------------------------

// Quantise blocks [0, nb) of an f32 vector (global memory, or shared memory when
// kShared). Four consecutive threads share a block (8 values each); the block's 32
// values v_i become integers q_i = v_i * 2^k, |q_i| <= 2^22, the power of two
// chosen from the block's largest magnitude; plane P holds byte P of every q_i
// (value i at byte P*32 + i) and info[b] = {2^-k, sum q_i}. A block whose values
// are all below 2^-97 in magnitude is taken as zero. Whole warps call it (the
// groups use shuffles) and every thread runs the same number of rounds.
template <bool kShared = false>
__device__ __forceinline__ void quant_blocks(const float* src, int nb, uint8_t* planes, float2* info, int t,
                                             int nthreads) {
  for (int base = 0; base < 4 * nb; base += nthreads) {
    const int idx = base + t, b = idx >> 2, qq = idx & 3;
    const bool active = idx < 4 * nb;
    float v[8];
    if (active) {
      const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)b * 32 + qq * 8);
      const float4 a = kShared ? s4[0] : __ldcg(s4), c = kShared ? s4[1] : __ldcg(s4 + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFF);  // amax < 2^(eb - 126)
    float inv = 0.f, sc = 0.f;
    if (eb >= 30) {
      inv = __uint_as_float((uint32_t)(148 - eb + 127) << 23);  // 2^(148 - eb)
      sc = __uint_as_float((uint32_t)(eb - 148 + 127) << 23);   // 2^(eb - 148)
    }
    int q[8];
    int X = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      q[i] = round_small(v[i] * inv);
      X += q[i];
    }
    X += __shfl_xor_sync(0xffffffffu, X, 1);
    X += __shfl_xor_sync(0xffffffffu, X, 2);
    if (active) {
#pragma unroll
      for (int P = 0; P < 3; ++P) {
        uint32_t w[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t lo = __byte_perm(q[4 * k], q[4 * k + 1], P | ((4 + P) << 4));
          const uint32_t hi = __byte_perm(q[4 * k + 2], q[4 * k + 3], P | ((4 + P) << 4));
          w[k] = __byte_perm(lo, hi, 0x5410);
        }
        *reinterpret_cast<uint2*>(planes + (size_t)b * 96 + P * 32 + qq * 8) = make_uint2(w[0], w[1]);
      }
      if (qq == 0) info[b] = make_float2(sc, (float)X);
    }
  }
}

struct ActBlock {
  uint32_t p[24];  // planes: [0,8) low bytes, [8,16) middle bytes, [16,24) signed high bytes
  float s, X;
};

__device__ __forceinline__ void load_act_block(ActBlock& a, const uint8_t* planes, const float2* info,
                                               int b) {
  const uint4* src = reinterpret_cast<const uint4*>(planes + (size_t)b * 96);
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    uint4 v = src[i];
    a.p[4 * i + 0] = v.x;
    a.p[4 * i + 1] = v.y;
    a.p[4 * i + 2] = v.z;
    a.p[4 * i + 3] = v.w;
  }
  float2 f = info[b];
  a.s = f.x;
  a.X = f.y;
}

// sum(q * v) over the block for the four nibble words.
__device__ __forceinline__ float nibble_dot(const uint32_t (&qw)[4], const ActBlock& a) {
  int a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo = qw[i] & 0x0F0F0F0Fu;         // values 4i .. 4i+3
    uint32_t hi = (qw[i] >> 4) & 0x0F0F0F0Fu;  // values 16+4i .. 16+4i+3
    a0 = dp4a_uu(lo, a.p[i], a0);
    a0 = dp4a_uu(hi, a.p[4 + i], a0);
    a1 = dp4a_uu(lo, a.p[8 + i], a1);
    a1 = dp4a_uu(hi, a.p[12 + i], a1);
    a2 = dp4a_us(lo, a.p[16 + i], a2);
    a2 = dp4a_us(hi, a.p[20 + i], a2);
  }
  // sum = a2 * 2^16 + a1 * 2^8 + a0; a2 * 2^8 + a1 is exact in fp32 (< 2^24)
  return fmaf((float)(a2 * 256 + a1), 256.f, (float)a0);
}

// A block of a row in global memory as five 32-bit words read from the 4-byte
// boundary at or below it. Q4_1 blocks are 4-byte aligned. A Q4_0 block is 2-byte
// aligned and its 18 bytes lie inside the 20 read; a read past a block's end stays
// inside the next block, and the last block of the expert array (or of the shared
// record) starts 2 bytes past a 4-byte boundary, since both byte counts are
// multiples of 4 (F * H / 32 is a multiple of 32), so no read leaves the buffer.
struct RawBlock {
  uint32_t w[5];
  uint32_t sh;  // Q4_0: 0 or 16, the block's bit offset in w
};
template <int QT>
__device__ __forceinline__ void load_block_g(const uint8_t* row, int b, RawBlock& r) {
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row) + (uintptr_t)(QT == 3 ? 20 : 18) * (uint32_t)b;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(addr & ~uintptr_t(3));
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = __ldg(w + i);
  r.sh = (uint32_t)(addr & 3u) * 8u;
}
template <int QT>
__device__ __forceinline__ float raw_block_dot(const RawBlock& r, const ActBlock& a) {
  if constexpr (QT == 3) {
    const uint32_t qw[4] = {r.w[1], r.w[2], r.w[3], r.w[4]};
    const float S = nibble_dot(qw, a);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r.w[0]));
    return a.s * fmaf(f.x, S, f.y * a.X);
  } else {
    const uint32_t dbits = __funnelshift_rc(r.w[0], r.w[1], r.sh) & 0xFFFFu;
    const uint32_t qw[4] = {__funnelshift_rc(r.w[0], r.w[1], 16 + r.sh), __funnelshift_rc(r.w[1], r.w[2], 16 + r.sh),
                            __funnelshift_rc(r.w[2], r.w[3], 16 + r.sh), __funnelshift_rc(r.w[3], r.w[4], 16 + r.sh)};
    const float S = nibble_dot(qw, a);
    const float d = __half2float(__ushort_as_half((unsigned short)dbits));
    return a.s * d * fmaf(-8.f, a.X, S);
  }
}

// Lane mapping of a row of nb blocks over a warp: LPR lanes per row (a power
// of two, at most 32), so 32/LPR rows per step; lane l takes blocks
// (l % LPR) + LPR*i.
struct RowMap {
  int lpr, sub, rsub, rps;
};
__device__ __forceinline__ RowMap row_map(int nb, int lane) {
  int lpr = 1;
  while (lpr < nb && lpr < 32) lpr *= 2;
  return RowMap{lpr, lane % lpr, lane / lpr, 32 / lpr};
}
// group sums of N values at once over lpr-lane groups (their shuffles interleave)
template <int N>
__device__ __forceinline__ void group_sum_n(float (&v)[N], int lpr) {
  for (int o = lpr / 2; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Timeline points (MOE_TRACE): %globaltimer readings per CTA index (CTAs below the
// trace's row count), written by thread 0.
enum TracePoint : int {
  TR_RT_START = 0, TR_RT_X, TR_RT_DONE, TR_RT_PICKED, TR_GU_START, TR_GU_XQ, TR_GU_WAITED, TR_GU_END,
  TR_DN_START, TR_DN_LOADED, TR_DN_WAITED, TR_DN_END, TR_POINTS = 24
};
__device__ __forceinline__ void tr(const DecodeArgs& a, int point, int rows) {
  if (a.trace && threadIdx.x == 0 && (int)blockIdx.x < rows) a.trace[(size_t)blockIdx.x * TR_POINTS + point] = globaltimer();
}

// ===========================================================================
// Router: logits, then (last CTA) the picks and their weights
// ===========================================================================
__global__ void __launch_bounds__(RT_THREADS) dec_router(const DecodeArgs a, int trows) {
  extern __shared__ __align__(16) uint8_t rsm[];  // probs [E], keys [E]
  __shared__ float part[RT_THREADS / 32];
  __shared__ float gscore[64];
  __shared__ int rids[32];
  __shared__ int is_last;
  const DecodePlan& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tr(a, TR_RT_START, trows);
  const int row = blockIdx.x * 2 + (warp >> 2), q = warp & 3;
  const int nq4 = p.H / 16;  // float4s in a quarter row
  const bool has = row < p.E;
  // this warp's quarter of its router row, before the wait (weights do not change)
  float4 wv[6];
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    const int j = lane + 32 * i;
    wv[i] = (has && j < nq4) ? __ldg(reinterpret_cast<const float4*>(a.router_w + (size_t)row * p.H + q * (p.H / 4)) + j)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait_prior_grids();  // x may come from the previous kernel
  pdl_launch_dependents();
  tr(a, TR_RT_X, trows);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    const int j = lane + 32 * i;
    if (has && j < nq4) {
      const float4 xv = __ldcg(reinterpret_cast<const float4*>(a.x + q * (p.H / 4)) + j);
      acc = fmaf(wv[i].x, xv.x, acc);
      acc = fmaf(wv[i].y, xv.y, acc);
      acc = fmaf(wv[i].z, xv.z, acc);
      acc = fmaf(wv[i].w, xv.w, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) part[warp] = acc;
  __syncthreads();
  if (tid < 2) {
    const int r = blockIdx.x * 2 + tid;
    if (r < p.E) a.logits[r] = ((part[4 * tid] + part[4 * tid + 1]) + part[4 * tid + 2]) + part[4 * tid + 3];
  }
  // ---- the last CTA to finish selects ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();  // this CTA's logits are visible device-wide before it is counted
    const uint32_t t = atomicAdd(a.ctrl + CTRL_ROUTER, 1u);
    is_last = t == gridDim.x - 1u;
  }
  __syncthreads();
  tr(a, TR_RT_DONE, trows);
  if (!is_last) return;
  __threadfence();
  float* probs = reinterpret_cast<float*>(rsm);
  uint32_t* keys = reinterpret_cast<uint32_t*>(rsm + (size_t)p.E * 4);
  for (int e = tid; e < p.E; e += RT_THREADS) {
    const float l = __ldcg(a.logits + e);
    const float pr = 1.f / (1.f + expf(-l));
    probs[e] = pr;
    keys[e] = order_key(pr + (a.bias ? __ldg(a.bias + e) : 0.f));
  }
  __syncthreads();
  if (p.G > 1) {
    // group score: the two largest s of the group, summed (multiset top-2)
    const int per = p.E / p.G;
    for (int g = warp; g < p.G; g += RT_THREADS / 32) {
      float x1 = -INFINITY, x2 = -INFINITY;
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
    __syncthreads();
  }
  if (warp == 0) {
    // kept groups: groups_used rounds of the largest group score, lowest group on ties;
    // experts of dropped groups get key 0 (below every real key)
    if (p.G > 1) {
      uint32_t keep_lo = 0, keep_hi = 0;  // groups 0..63
      for (int j = 0; j < p.Gu; ++j) {
        int best = -1;
        float bv = 0.f;
        for (int g = 0; g < p.G; ++g) {
          const bool kept = g < 32 ? ((keep_lo >> g) & 1u) : ((keep_hi >> (g - 32)) & 1u);
          if (!kept && (best < 0 || gscore[g] > bv)) { best = g; bv = gscore[g]; }
        }
        if (best < 32) keep_lo |= 1u << best; else keep_hi |= 1u << (best - 32);
      }
      const int per = p.E / p.G;
      for (int e = lane; e < p.E; e += 32) {
        const int g = e / per;
        const bool kept = g < 32 ? ((keep_lo >> g) & 1u) : ((keep_hi >> (g - 32)) & 1u);
        if (!kept) keys[e] = 0u;
      }
      __syncwarp();
    }
    // k rounds of the largest key, lowest index among equals (keys in registers)
    if (p.E <= 256) topk_rounds<8>(keys, p.E, p.K, rids, lane);
    else if (p.E <= 512) topk_rounds<16>(keys, p.E, p.K, rids, lane);
    else topk_rounds<32>(keys, p.E, p.K, rids, lane);
    __syncwarp();
    // weights from the picked sigmoids
    const float pj = lane < p.K ? probs[rids[lane]] : 0.f;
    const float wsum = fmaxf(warp_sum(pj), a.norm_min);
    if (lane < p.K) {
      const float wj = pj / wsum * a.scale;
      a.ids[lane] = rids[lane];
      a.wts[lane] = wj;
      if (a.topk_ids) a.topk_ids[lane] = rids[lane];
      if (a.topk_w) a.topk_w[lane] = wj;
    }
    if (lane == 0) a.ctrl[CTRL_ROUTER] = 0;  // the next call counts from zero
  }
  tr(a, TR_RT_PICKED, trows);
}

// ===========================================================================
// Gate/up: one activation block (32 intermediate values of a slot) per CTA
// ===========================================================================
template <int QT, int MAXB>
__global__ void __launch_bounds__(GU_THREADS) dec_gate_up(const DecodeArgs a, int trows) {
  extern __shared__ __align__(16) uint8_t gsm[];  // x planes [nbH][96], then x info [nbH]
  __shared__ float rowdot[GU_THREADS / 32][4];
  __shared__ __align__(16) float colact[32];
  const DecodePlan& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x;
  const bool shared = blk < p.nbFs;  // the shared expert's blocks need no routing
  tr(a, TR_GU_START, trows);
  uint8_t* xplanes = gsm;
  float2* xinfo = reinterpret_cast<float2*>(gsm + (size_t)p.nbH * 96);
  // x -> activation blocks (x is complete: the router kernel waited for it before this
  // launch was triggered)
  quant_blocks(a.x, p.nbH, xplanes, xinfo, tid, GU_THREADS);
  __syncthreads();
  tr(a, TR_GU_XQ, trows);
  const RowMap mh = row_map(p.nbH, lane);
  ActBlock xc[MAXB];
#pragma unroll
  for (int i = 0; i < MAXB; ++i) {
    const int b = mh.sub + mh.lpr * i;
    if (b < p.nbH) load_act_block(xc[i], xplanes, xinfo, b);
  }
  if (!shared) pdl_wait_prior_grids();  // the picks
  pdl_launch_dependents();
  tr(a, TR_GU_WAITED, trows);
  const int slot = shared ? p.K : (blk - p.nbFs) / p.nbF;
  const uint8_t* rec = shared ? a.shared : a.experts + (size_t)__ldcg(a.ids + slot) * p.rec_bytes;
  const int ff = shared ? p.Fs : p.F;
  const int f0 = (shared ? blk : (blk - p.nbFs) % p.nbF) * 32 + 2 * warp;
  // the warp's rows: 0 gate(f0), 1 up(f0), 2 gate(f0 + 1), 3 up(f0 + 1); lane group
  // rsub takes rows rsub + rps * s
  auto row_ptr = [&](int r) -> const uint8_t* {
    const int f = f0 + (r >> 1);
    return rec + (size_t)((r & 1) ? ff + f : f) * p.rb_h;
  };
  float dots[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (MAXB <= 2) {
    RawBlock rb[4][MAXB];  // every row's blocks requested before any is used
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int r = mh.rsub + mh.rps * s;
#pragma unroll
      for (int i = 0; i < MAXB; ++i) {
        const int b = mh.sub + mh.lpr * i;
        if (r < 4 && b < p.nbH) load_block_g<QT>(row_ptr(r), b, rb[s][i]);
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int r = mh.rsub + mh.rps * s;
#pragma unroll
      for (int i = 0; i < MAXB; ++i) {
        const int b = mh.sub + mh.lpr * i;
        if (r < 4 && b < p.nbH) dots[s] += raw_block_dot<QT>(rb[s][i], xc[i]);
      }
    }
  } else {
#pragma unroll
    for (int s = 0; s < 4; ++s) {  // one row's blocks at a time (registers)
      const int r = mh.rsub + mh.rps * s;
      RawBlock rb[MAXB];
#pragma unroll
      for (int i = 0; i < MAXB; ++i) {
        const int b = mh.sub + mh.lpr * i;
        if (r < 4 && b < p.nbH) load_block_g<QT>(row_ptr(r), b, rb[i]);
      }
#pragma unroll
      for (int i = 0; i < MAXB; ++i) {
        const int b = mh.sub + mh.lpr * i;
        if (r < 4 && b < p.nbH) dots[s] += raw_block_dot<QT>(rb[i], xc[i]);
      }
    }
  }
  group_sum_n(dots, mh.lpr);
  if (mh.sub == 0) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int r = mh.rsub + mh.rps * s;
      if (r < 4) rowdot[warp][r] = dots[s];
    }
  }
  __syncwarp();
  if (lane < 2) colact[2 * warp + lane] = silu_mul(rowdot[warp][2 * lane], rowdot[warp][2 * lane + 1]);
  __syncthreads();
  if (warp == 0) quant_blocks<true>(colact, 1, a.aplanes + (size_t)blk * 96, a.ainfo + blk, lane, 32);
  tr(a, TR_GU_END, trows);
}

// ===========================================================================
// Down: one output row per warp over every slot, weighted, in a fixed order
// ===========================================================================
template <int QT>
__global__ void __launch_bounds__(DN_THREADS) dec_down(const DecodeArgs a, int trows) {
  extern __shared__ __align__(16) uint8_t dsm[];  // activation planes [nact][96], info [nact]
  __shared__ int sids[32];
  __shared__ float swts[32];
  const DecodePlan& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x * (DN_THREADS / 32) + warp;
  tr(a, TR_DN_START, trows);
  // the picks (the router kernel is complete: every gate/up CTA waited for it before
  // this launch was triggered)
  if (tid < p.K) {
    sids[tid] = __ldcg(a.ids + tid);
    swts[tid] = __ldcg(a.wts + tid);
  }
  __syncthreads();
  // blocks of the row in activation order: the shared expert's, then each pick's
  const int nblk = p.nbFs + p.K * p.nbF;
  auto block_src = [&](int cb, int& b) -> const uint8_t* {
    if (cb < p.nbFs) {
      b = cb;
      return a.shared + (size_t)2 * p.Fs * p.rb_h + (size_t)h * p.rb_fs;
    }
    const int j = (cb - p.nbFs) / p.nbF;
    b = (cb - p.nbFs) % p.nbF;
    return a.experts + (size_t)sids[j] * p.rec_bytes + (size_t)2 * p.F * p.rb_h + (size_t)h * p.rb_f;
  };
  auto block_w = [&](int cb) -> float { return cb < p.nbFs ? 1.f : swts[(cb - p.nbFs) / p.nbF]; };
  // the row's first blocks, requested before the wait
  RawBlock rb[DN_PRE];
#pragma unroll
  for (int i = 0; i < DN_PRE; ++i) {
    const int cb = lane + 32 * i;
    if (h < p.H && cb < nblk) {
      int b;
      const uint8_t* row = block_src(cb, b);
      load_block_g<QT>(row, b, rb[i]);
    }
  }
  tr(a, TR_DN_LOADED, trows);
  pdl_wait_prior_grids();  // the activation blocks
  pdl_launch_dependents();
  tr(a, TR_DN_WAITED, trows);
  const uint8_t* aplanes = a.aplanes;
  const float2* ainfo = a.ainfo;
  if (p.act_smem) {
    // stage the activation blocks in shared memory (read by every warp)
    const int n16 = p.nact * 96 / 16;
    uint4* d16 = reinterpret_cast<uint4*>(dsm);
    for (int i = tid; i < n16; i += DN_THREADS) d16[i] = __ldcg(reinterpret_cast<const uint4*>(a.aplanes) + i);
    float2* dinfo = reinterpret_cast<float2*>(dsm + (size_t)p.nact * 96);
    for (int i = tid; i < p.nact; i += DN_THREADS) dinfo[i] = __ldcg(a.ainfo + i);
    __syncthreads();
    aplanes = dsm;
    ainfo = dinfo;
  }
  float acc = 0.f;
  if (h < p.H) {
#pragma unroll
    for (int i = 0; i < DN_PRE; ++i) {
      const int cb = lane + 32 * i;
      if (cb < nblk) {
        ActBlock ab;
        load_act_block(ab, aplanes, ainfo, cb);
        acc = fmaf(block_w(cb), raw_block_dot<QT>(rb[i], ab), acc);
      }
    }
    for (int cb = lane + 32 * DN_PRE; cb < nblk; cb += 32) {  // rows of more than 256 blocks
      int b;
      const uint8_t* row = block_src(cb, b);
      RawBlock r;
      load_block_g<QT>(row, b, r);
      ActBlock ab;
      load_act_block(ab, aplanes, ainfo, cb);
      acc = fmaf(block_w(cb), raw_block_dot<QT>(r, ab), acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0 && h < p.H) {
    if (a.flags & FLAG_RESIDUAL) acc = __ldcg(a.x + h) + acc;
    if (a.flags & FLAG_ACCUMULATE) acc = __ldcg(a.out + h) + acc;
    a.out[h] = acc;
  }
  tr(a, TR_DN_END, trows);
}

// ===========================================================================
// Host side
// ===========================================================================
template <typename... Args>
static cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, int threads, size_t smem, cudaStream_t st, bool pdl,
                              Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int QT, int MAXB>
static cudaError_t launch_chain(const DecodeArgs& a, cudaStream_t st, bool pdl, int trows) {
  const DecodePlan& p = a.p;
  cudaError_t e = launch_pdl(dec_router, dim3((unsigned)ceil_div(p.E, 2)), RT_THREADS, (size_t)p.E * 8, st, pdl, a,
                             trows);
  if (e != cudaSuccess) return e;
  e = launch_pdl(dec_gate_up<QT, MAXB>, dim3((unsigned)p.nact), GU_THREADS, (size_t)p.nbH * 104, st, pdl, a, trows);
  if (e != cudaSuccess) return e;
  return launch_pdl(dec_down<QT>, dim3((unsigned)ceil_div(p.H, DN_THREADS / 32)), DN_THREADS,
                    p.act_smem ? (size_t)p.nact * 104 : (size_t)0, st, pdl, a, trows);
}

cudaError_t decode_launch(const DecodeArgs& a, int maxb, cudaStream_t st, bool pdl, int trows) {
  switch (a.p.qtype * 8 + maxb) {
    case 2 * 8 + 1: return launch_chain<2, 1>(a, st, pdl, trows);
    case 2 * 8 + 2: return launch_chain<2, 2>(a, st, pdl, trows);
    case 2 * 8 + 3: return launch_chain<2, 3>(a, st, pdl, trows);
    case 3 * 8 + 1: return launch_chain<3, 1>(a, st, pdl, trows);
    case 3 * 8 + 2: return launch_chain<3, 2>(a, st, pdl, trows);
    case 3 * 8 + 3: return launch_chain<3, 3>(a, st, pdl, trows);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
