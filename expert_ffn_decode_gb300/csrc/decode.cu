// Single-token MoE-FFN step (decode, T = 1) for sm_103a: three kernels in a chain.
//
//   dec_router    one router row per 4 warps (each a quarter of H), f32 dot with x
//                 -> logits
//   dec_gate_up   one CTA per 16 intermediate values of a slot (the shared expert's
//                 first, then the picks'). The CTA makes the picks from the logits,
//                 copies its 16 gate and 16 up rows into shared memory (bulk async
//                 copies, two chunks of 8 values) and dots them with x -> SwiGLU -> the
//                 f32 activations
//   dec_down      R output rows per CTA: the picks again, the rows' blocks of every
//                 slot's down matrix copied into shared memory, the activations
//                 quantised into shared memory, the dots each weighted by the slot's
//                 routing weight (1 for the shared expert), summed in a fixed order
//
// The kernels run with programmatic dependent launch, and each requests the bytes it
// can before waiting on its predecessor:
//   - the router kernel loads its router rows before the wait for x;
//   - the gate/up kernel quantises x, and copies and computes the shared expert's
//     values, while the router kernel runs;
//   - the down kernel makes the picks and copies its weight rows while the gate/up
//     kernel runs.
// The router is complete once any routed gate/up CTA has waited, and every routed
// gate/up CTA has waited before the down kernel starts, so both consumers read the
// logits straight away. There are no grid-wide spin waits: kernel boundaries order
// every exchange, and every mbarrier wait is bounded in time.
//
// Dequant-dot: a 4-bit block (ggml Q4_0/Q4_1, 32 values) times 32 activations.
// Activations are held per 16 values (half a block) as 16-bit integers v = x * 2^k with
// |v| <= 2^14 (a power-of-two scale per half; error at most 2^-15 of the half's largest
// magnitude), split into a low (unsigned) and a high (signed) byte plane; dp4a forms
// sum(q * v) of each half exactly in int32, and the block result d * (s0 S0 + s1 S1)
// (+ m * sum(x) for Q4_1, - 8 d sum(x) for Q4_0) is accumulated in fp32. The block formats and the
// per-block dot identity follow flint_moe_ssd.js (WGSL section, Q41DOT and its
// comment). K-quant rows (256-value super-blocks: Q4_K gate/up, Q6_K or Q4_K down, as
// the Ling store holds them) are walked in the same 32-value blocks: a Q4_K sub-block
// dots like a Q4_1 block with d*sc and -dmin*mn, a Q6_K sub-block as two 16-value halves
// of signed 6-bit values, each with its own int8 scale. The gate/up kernel takes the
// gate/up rows' type and the down kernel the down rows' type.
#include <cstdint>
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_host.h"
#include "plan.h"
#include "select.cuh"

namespace moe {

constexpr int RT_THREADS = 256;  // router: 8 warps, two rows a CTA
constexpr int GU_THREADS = 256;  // gate/up: 8 warps, two intermediate values each
constexpr int DN_THREADS = 256;  // down: 8 warps

// ---------------------------------------------------------------------------
// Activation blocks
// ---------------------------------------------------------------------------

// One quantisation task: 8 consecutive values (part qq of block b) of a block whose
// four tasks sit in four consecutive lanes. Each half of the block (values 0..15: tasks
// 0, 1; values 16..31: tasks 2, 3) becomes integers q_i = v_i * 2^k, |q_i| <= 2^14, the
// power of two chosen from the half's largest magnitude; a half whose values are all below
// 2^-97 in magnitude is taken as zero. Plane P (0: low byte, 1: signed high byte) of the
// block holds byte P of every q_i; the planes' 16 words are stored as 4 chunks of 4 words
// (chunk 2P + h: plane P of half h), chunk c of block b at planes + (c * stride + b) * 16,
// so that lanes reading consecutive blocks hit consecutive 16-byte words;
// info[b] = {2^-k0, sum of half 0's q_i, 2^-k1, sum of half 1's q_i}.
__device__ __forceinline__ void quant_task(const float (&v)[8], bool active, int b, int qq, int stride,
                                           uint8_t* planes, float4* info) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the half's other task
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFF);  // amax < 2^(eb - 126)
  float inv = 0.f, sc = 0.f;
  if (eb >= 30) {
    inv = __uint_as_float((uint32_t)(140 - eb + 127) << 23);  // 2^(140 - eb): |v| * inv < 2^14
    sc = __uint_as_float((uint32_t)(eb - 140 + 127) << 23);   // 2^(eb - 140)
  }
  int q[8];
  int X = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    q[i] = round_small(v[i] * inv);
    X += q[i];
  }
  X += __shfl_xor_sync(0xffffffffu, X, 1);
  if (active) {
#pragma unroll
    for (int P = 0; P < 2; ++P) {
      uint32_t w[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t lo = __byte_perm(q[4 * k], q[4 * k + 1], P | ((4 + P) << 4));
        const uint32_t hi = __byte_perm(q[4 * k + 2], q[4 * k + 3], P | ((4 + P) << 4));
        w[k] = __byte_perm(lo, hi, 0x5410);
      }
      // plane words 8P + 2qq, 8P + 2qq + 1: chunk 2P + qq / 2, words 2 (qq & 1) + 0, 1
      const int c = 2 * P + (qq >> 1);
      *reinterpret_cast<uint2*>(planes + ((size_t)c * stride + b) * 16 + 8 * (qq & 1)) = make_uint2(w[0], w[1]);
    }
    if ((qq & 1) == 0) reinterpret_cast<float2*>(info + b)[qq >> 1] = make_float2(sc, (float)X);
  }
}

// Quantise blocks [0, nb) of an f32 vector (global memory, or shared memory when
// kShared) as quant_task describes; with `mul`, value i is first multiplied by
// scal * mul[i]. With `ss`, the thread adds the squares of the values it loaded (before
// any multiplication) to *ss. Each thread takes TPR tasks a round and loads all of them
// before computing; every thread runs the same number of rounds and whole warps call it
// (the groups use shuffles). TPR: tasks a thread loads per round.
template <int TPR, bool kShared = false>
__device__ __forceinline__ void quant_blocks(const float* src, int nb, int stride, uint8_t* planes, float4* info,
                                             int t, int nthreads, const float* mul = nullptr, float scal = 1.f,
                                             float* ss = nullptr) {
  #pragma unroll 1
  for (int base = 0; base < 4 * nb; base += TPR * nthreads) {
    float4 va[TPR], vc[TPR], ma[TPR], mc[TPR];
    int idx[TPR];
#pragma unroll
    for (int h = 0; h < TPR; ++h) {
      idx[h] = base + h * nthreads + t;
      const bool ok = idx[h] < 4 * nb;
      const size_t off = (size_t)(idx[h] >> 2) * 32 + (idx[h] & 3) * 8;
      const float4* s4 = reinterpret_cast<const float4*>(src + off);
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f), one = make_float4(1.f, 1.f, 1.f, 1.f);
      va[h] = ok ? (kShared ? s4[0] : __ldcg(s4)) : z;
      vc[h] = ok ? (kShared ? s4[1] : __ldcg(s4 + 1)) : z;
      ma[h] = (mul && ok) ? __ldg(reinterpret_cast<const float4*>(mul + off)) : one;
      mc[h] = (mul && ok) ? __ldg(reinterpret_cast<const float4*>(mul + off) + 1) : one;
    }
    // one task a pass, the rest moved down a slot: a single copy of the task's code
    #pragma unroll 1
    for (int h = 0; h < TPR; ++h) {
      float v[8] = {va[0].x, va[0].y, va[0].z, va[0].w, vc[0].x, vc[0].y, vc[0].z, vc[0].w};
      if (ss) {
#pragma unroll
        for (int i = 0; i < 8; ++i) *ss = fmaf(v[i], v[i], *ss);
      }
      if (mul) {
        const float mm[8] = {ma[0].x, ma[0].y, ma[0].z, ma[0].w, mc[0].x, mc[0].y, mc[0].z, mc[0].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = v[i] * scal * mm[i];
      }
      quant_task(v, idx[0] < 4 * nb, idx[0] >> 2, idx[0] & 3, stride, planes, info);
#pragma unroll
      for (int k = 0; k + 1 < TPR; ++k) {
        va[k] = va[k + 1];
        vc[k] = vc[k + 1];
        ma[k] = ma[k + 1];
        mc[k] = mc[k + 1];
        idx[k] = idx[k + 1];
      }
    }
  }
}

struct ActBlock {
  uint32_t p[16];  // planes: [0,8) low bytes, [8,16) signed high bytes (words 0-3, 8-11: half 0)
  float s0, s1;    // the halves' scales 2^-k
  float XS;        // s0 X0 + s1 X1: the block's sum of activations
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// Block b of a transposed activation array (chunk stride `stride` blocks) in shared
// memory, planes and info given as shared addresses.
__device__ __forceinline__ void load_act_block_s(ActBlock& a, uint32_t planes, uint32_t info, int b, int stride) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = lds128(planes + (uint32_t)(c * stride + b) * 16u);
    a.p[4 * c + 0] = v.x;
    a.p[4 * c + 1] = v.y;
    a.p[4 * c + 2] = v.z;
    a.p[4 * c + 3] = v.w;
  }
  const uint4 f = lds128(info + (uint32_t)b * 16u);
  a.s0 = __uint_as_float(f.x);
  a.s1 = __uint_as_float(f.z);
  a.XS = fmaf(a.s0, __uint_as_float(f.y), a.s1 * __uint_as_float(f.w));
}

// s0 S0 + s1 S1, S_h = sum(q * v) over half h of the block for the four nibble words (exact:
// |S_h| < 2^24): the low nibbles hold half 0, the high nibbles half 1.
__device__ __forceinline__ float nibble_dot(const uint32_t (&qw)[4], const ActBlock& a) {
  int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = qw[i] & 0x0F0F0F0Fu;         // values 4i .. 4i+3
    const uint32_t hi = (qw[i] >> 4) & 0x0F0F0F0Fu;  // values 16+4i .. 16+4i+3
    a0 = dp4a_uu(lo, a.p[i], a0);
    a1 = dp4a_us(lo, a.p[8 + i], a1);
    b0 = dp4a_uu(hi, a.p[4 + i], b0);
    b1 = dp4a_us(hi, a.p[12 + i], b1);
  }
  return fmaf(a.s0, (float)(a1 * 256 + a0), a.s1 * (float)(b1 * 256 + b0));
}

// A block of a row as five 32-bit words read from the 4-byte boundary at or below
// it. Q4_1 blocks are 4-byte aligned. A Q4_0 block is 2-byte aligned and its 18
// bytes lie inside the 20 read; a read past a block's end stays inside the copied
// window (windows are rounded out to 16-byte bounds).
struct RawBlock {
  uint32_t w[5];
  uint32_t sh;  // Q4_0: 0 or 16, the block's bit offset in w
};
template <int QT>
__device__ __forceinline__ void load_block_s(uint32_t row, int b, RawBlock& r) {  // row: a shared address
  const uint32_t addr = row + (uint32_t)(QT == 3 ? 20 : 18) * (uint32_t)b;
  const uint32_t w = addr & ~3u;
#pragma unroll
  for (int i = 0; i < 5; ++i) r.w[i] = lds32(w + 4u * i);
  r.sh = (addr & 3u) * 8u;
}
template <int QT>
__device__ __forceinline__ float raw_block_dot(const RawBlock& r, const ActBlock& a) {
  if constexpr (QT == 3) {
    const uint32_t qw[4] = {r.w[1], r.w[2], r.w[3], r.w[4]};
    const float S = nibble_dot(qw, a);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r.w[0]));
    return fmaf(f.x, S, f.y * a.XS);
  } else {
    const uint32_t dbits = __funnelshift_rc(r.w[0], r.w[1], r.sh) & 0xFFFFu;
    const uint32_t qw[4] = {__funnelshift_rc(r.w[0], r.w[1], 16 + r.sh), __funnelshift_rc(r.w[1], r.w[2], 16 + r.sh),
                            __funnelshift_rc(r.w[2], r.w[3], 16 + r.sh), __funnelshift_rc(r.w[3], r.w[4], 16 + r.sh)};
    const float S = nibble_dot(qw, a);
    const float d = __half2float(__ushort_as_half((unsigned short)dbits));
    return d * fmaf(-8.f, a.XS, S);
  }
}

// ---- K-quant super-blocks (256 values). Each 32-value sub-block meets one activation
// block, so a row is still walked in 32-value blocks b: super-block b / 8, sub-block b % 8.
// The layouts are ggml's (the Ling store's Q4_K gate/up and Q6_K down rows, ling_moe_ssd.js
// header; the pages name the types only).

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Q4_K, 144 bytes: f16 d, f16 dmin, 12 bytes S of packed 6-bit scales and mins, four runs
// of 32 nibble bytes (run c: sub-block 2c in the low nibbles, 2c + 1 in the high nibbles).
// Sub-block j < 4: sc = S[j] & 63, mn = S[j + 4] & 63; j >= 4: the low 4 bits of both from
// S[j + 4], the top 2 bits from S[j - 4] (sc) and S[j] (mn). Value = d sc q - dmin mn.
// Q4_K rows are whole 16-byte multiples and start on 16-byte bounds, here and in shared memory.
__device__ __forceinline__ float q4k_sub_dot(uint32_t row, int b, const ActBlock& a) {
  const uint32_t sb = row + 144u * (uint32_t)(b >> 3);
  const int j = b & 7, sh = 8 * (j & 3);
  const uint4 hd = lds128(sb);
  const uint4 n0 = lds128(sb + 16u + 32u * (uint32_t)(j >> 1));
  const uint4 n1 = lds128(sb + 32u + 32u * (uint32_t)(j >> 1));
  const uint32_t by = (hd.y >> sh) & 0xFFu, bz = (hd.z >> sh) & 0xFFu, bw = (hd.w >> sh) & 0xFFu;
  const uint32_t sc = j < 4 ? (by & 63u) : ((bw & 15u) | ((by >> 6) << 4));
  const uint32_t mn = j < 4 ? (bz & 63u) : ((bw >> 4) | ((bz >> 6) << 4));
  const int ns = 4 * (j & 1);  // the run's low or high nibbles
  const uint32_t w[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
  int s0[2] = {0, 0}, s1[2] = {0, 0};  // per half
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t q = (w[i] >> ns) & 0x0F0F0F0Fu;  // values 4i .. 4i + 3
    s0[i >> 2] = dp4a_uu(q, a.p[i], s0[i >> 2]);
    s1[i >> 2] = dp4a_us(q, a.p[8 + i], s1[i >> 2]);
  }
  const float S = fmaf(a.s0, (float)(s1[0] * 256 + s0[0]), a.s1 * (float)(s1[1] * 256 + s0[1]));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));  // d, dmin
  return fmaf(f.x * (float)sc, S, -(f.y * (float)mn) * a.XS);
}

// 32 bytes from a 2-byte aligned shared address as 8 words (9 aligned words read; the run
// ends at least 4 bytes before its super-block does, so the ninth word stays inside it).
__device__ __forceinline__ void lds_run32(uint32_t addr, uint32_t (&w)[8]) {
  const uint32_t base = addr & ~3u, sh = (addr & 3u) * 8u;
  uint32_t t[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) t[i] = lds32(base + 4u * i);
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

// Q6_K, 210 bytes: ql[128], qh[64], 16 int8 scales, f16 d. Sub-block j = (half n = j / 4,
// quarter r = j % 4): value i takes its low 4 bits from ql[64n + 32 (r % 2) + i] (the low
// nibble for r < 2, the high one for r >= 2) and its high 2 bits from bits 2r, 2r + 1 of
// qh[32n + i]; value = d * scale[8n + 2r + i / 16] * (q - 32). Rows start on 2-byte bounds.
__device__ __forceinline__ float q6k_sub_dot(uint32_t row, int b, const ActBlock& a) {
  const uint32_t sb = row + 210u * (uint32_t)(b >> 3);
  const int j = b & 7, n = j >> 2, r = j & 3;
  uint32_t L[8], Hh[8];
  lds_run32(sb + 64u * n + 32u * (r & 1), L);
  lds_run32(sb + 128u + 32u * n, Hh);
  const uint32_t scp = lds16(sb + 192u + 8u * n + 2u * r);  // the quarter's two scales
  const float d = __half2float(__ushort_as_half((unsigned short)lds16(sb + 208u)));
  const int ls = 4 * (r >> 1), hs = 2 * r;
  int s0[2] = {0, 0}, s1[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = ((L[i] >> ls) & 0x0F0F0F0Fu) | (((Hh[i] >> hs) & 0x03030303u) << 4);  // 0..63
    // q - 32 as signed bytes: flip bit 5, and set bits 6, 7 where bit 5 was clear (q < 32)
    const uint32_t t = ~u & 0x20202020u;
    const uint32_t q = (u ^ 0x20202020u) | (t << 1) | (t << 2);
    s0[i >> 2] = dp4a_su(q, a.p[i], s0[i >> 2]);
    s1[i >> 2] = dp4a_ss(q, a.p[8 + i], s1[i >> 2]);
  }
  const float sc0 = (float)(int)(int8_t)(scp & 0xFFu), sc1 = (float)(int)(int8_t)(scp >> 8);
  const float S0 = (float)(s1[0] * 256 + s0[0]), S1 = (float)(s1[1] * 256 + s0[1]);
  return d * fmaf(sc1 * a.s1, S1, (sc0 * a.s0) * S0);
}

// ---- f32 activations (the default) -------------------------------------------------
// Activations stay f32, the pages' arithmetic (flint_moe_ssd.js, WGSL section, Q41DOT and its
// comment: a Q4_1 block contributes d * sum(q x) + m * sum(x), in f32). In shared memory an
// activation array of nb blocks is stored as 8 chunks of 4 floats per block, chunk c (values
// 4c .. 4c+3) of block b at (c * nb + b) * 16 bytes, so that lanes reading consecutive blocks
// hit consecutive 16-byte words; the block sums sum(x) sit in a float array [nb].

// Stores blocks [0, nb) of an f32 vector (global memory) as above, with chunk stride `stride`
// blocks (>= nb); with `mul`, value i is first multiplied by mul[i]. With `ss`, the thread
// adds the squares of the values it loaded (before any multiplication) to *ss. Each thread
// takes U chunks a round and loads all of them (and their `mul` chunks) before storing any;
// every thread runs the same number of rounds and whole warps call it (the block sums use
// shuffles over the 8 lanes of a block).
template <int U>
__device__ __forceinline__ void store_blocks_f32(const float* src, int nb, int stride, float4* xs, float* xsum,
                                                 int t, int nthreads, const float* mul = nullptr,
                                                 float* ss = nullptr) {
  #pragma unroll 1
  for (int base = 0; base < 8 * nb; base += U * nthreads) {
    float4 v[U], m[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int u = base + j * nthreads + t;  // chunk u & 7 of block u >> 3
      const bool ok = u < 8 * nb;
      v[j] = ok ? __ldcg(reinterpret_cast<const float4*>(src) + u) : make_float4(0.f, 0.f, 0.f, 0.f);
      m[j] = (mul && ok) ? __ldg(reinterpret_cast<const float4*>(mul) + u) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int u = base + j * nthreads + t;
      float4 w = v[j];
      if (ss) *ss = fmaf(w.x, w.x, fmaf(w.y, w.y, fmaf(w.z, w.z, fmaf(w.w, w.w, *ss))));
      if (mul) {
        w.x *= m[j].x; w.y *= m[j].y; w.z *= m[j].z; w.w *= m[j].w;
      }
      float s = (w.x + w.y) + (w.z + w.w);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      if (u < 8 * nb) {
        xs[(size_t)(u & 7) * stride + (u >> 3)] = w;
        if ((u & 7) == 0) xsum[u >> 3] = s;
      }
    }
  }
}

struct XBlock {
  float4 c[8];  // values 4k .. 4k+3 in c[k]
  float s;      // their sum
};
__device__ __forceinline__ void load_xblock(XBlock& x, uint32_t xs, uint32_t xsum, int b, int nb) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = lds128(xs + (uint32_t)(k * nb + b) * 16u);
    x.c[k] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
  }
  x.s = __uint_as_float(lds32(xsum + (uint32_t)b * 4u));
}

// sum over the block of (q_i - off) x_i for the four nibble words of a Q4_0/Q4_1 block (word k:
// low nibbles = values 4k .. 4k+3, high nibbles = values 16+4k ..), in f32
__device__ __forceinline__ float nibble_dot_f32(const uint32_t (&qw)[4], const XBlock& x, float off) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    word_dot_f32(qw[k] & 0x0F0F0F0Fu, x.c[k], off, a0, a1);
    word_dot_f32((qw[k] >> 4) & 0x0F0F0F0Fu, x.c[4 + k], off, a2, a3);
  }
  return (a0 + a1) + (a2 + a3);
}

// Q4_1: d * sum(q x) + m * sum(x); Q4_0: d * sum((q - 8) x), the 8 taken off each q exactly.
template <int QT>
__device__ __forceinline__ float raw_block_dot_f32(const RawBlock& r, const XBlock& x) {
  if constexpr (QT == 3) {
    const uint32_t qw[4] = {r.w[1], r.w[2], r.w[3], r.w[4]};
    const float S = nibble_dot_f32(qw, x, MAGIC_2P23);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r.w[0]));
    return fmaf(f.x, S, f.y * x.s);
  } else {
    const uint32_t dbits = __funnelshift_rc(r.w[0], r.w[1], r.sh) & 0xFFFFu;
    const uint32_t qw[4] = {__funnelshift_rc(r.w[0], r.w[1], 16 + r.sh), __funnelshift_rc(r.w[1], r.w[2], 16 + r.sh),
                            __funnelshift_rc(r.w[2], r.w[3], 16 + r.sh), __funnelshift_rc(r.w[3], r.w[4], 16 + r.sh)};
    const float S = nibble_dot_f32(qw, x, MAGIC_2P23 + 8.f);
    return __half2float(__ushort_as_half((unsigned short)dbits)) * S;
  }
}

// Q4_K sub-block b % 8 of super-block b / 8 (layout as q4k_sub_dot): d sc sum(q x) - dmin mn sum(x).
__device__ __forceinline__ float q4k_sub_dot_f32(uint32_t row, int b, const XBlock& x) {
  const uint32_t sb = row + 144u * (uint32_t)(b >> 3);
  const int j = b & 7, sh = 8 * (j & 3);
  const uint4 hd = lds128(sb);
  const uint4 n0 = lds128(sb + 16u + 32u * (uint32_t)(j >> 1));
  const uint4 n1 = lds128(sb + 32u + 32u * (uint32_t)(j >> 1));
  const uint32_t by = (hd.y >> sh) & 0xFFu, bz = (hd.z >> sh) & 0xFFu, bw = (hd.w >> sh) & 0xFFu;
  const uint32_t sc = j < 4 ? (by & 63u) : ((bw & 15u) | ((by >> 6) << 4));
  const uint32_t mn = j < 4 ? (bz & 63u) : ((bw >> 4) | ((bz >> 6) << 4));
  const int ns = 4 * (j & 1);
  const uint32_t w[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    word_dot_f32((w[i] >> ns) & 0x0F0F0F0Fu, x.c[i], MAGIC_2P23, a0, a1);
    word_dot_f32((w[i + 1] >> ns) & 0x0F0F0F0Fu, x.c[i + 1], MAGIC_2P23, a2, a3);
  }
  const float S = (a0 + a1) + (a2 + a3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));  // d, dmin
  return fmaf(f.x * (float)sc, S, -(f.y * (float)mn) * x.s);
}

// Q6_K sub-block (layout as q6k_sub_dot): d (sc0 sum_{i<16} (q_i - 32) x_i + sc1 sum_{i>=16} ...).
__device__ __forceinline__ float q6k_sub_dot_f32(uint32_t row, int b, const XBlock& x) {
  const uint32_t sb = row + 210u * (uint32_t)(b >> 3);
  const int j = b & 7, n = j >> 2, r = j & 3;
  uint32_t L[8], Hh[8];
  lds_run32(sb + 64u * n + 32u * (r & 1), L);
  lds_run32(sb + 128u + 32u * n, Hh);
  const uint32_t scp = lds16(sb + 192u + 8u * n + 2u * r);
  const float d = __half2float(__ushort_as_half((unsigned short)lds16(sb + 208u)));
  const int ls = 4 * (r >> 1), hs = 2 * r;
  float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = ((L[i] >> ls) & 0x0F0F0F0Fu) | (((Hh[i] >> hs) & 0x03030303u) << 4);  // 0..63
    word_dot_f32(u, x.c[i], MAGIC_2P23 + 32.f, a[i >> 2][0], a[i >> 2][1]);
  }
  const float sc0 = (float)(int)(int8_t)(scp & 0xFFu), sc1 = (float)(int)(int8_t)(scp >> 8);
  return d * fmaf(sc1, a[1][0] + a[1][1], sc0 * (a[0][0] + a[0][1]));
}

// Block b of a row in shared memory times f32 activation block x.
template <int QT>
__device__ __forceinline__ float row_block_dot_f32(uint32_t row, int b, const XBlock& x) {
  if constexpr (QT == 12) {
    return q4k_sub_dot_f32(row, b, x);
  } else if constexpr (QT == 14) {
    return q6k_sub_dot_f32(row, b, x);
  } else {
    RawBlock r;
    load_block_s<QT>(row, b, r);
    return raw_block_dot_f32<QT>(r, x);
  }
}

// Block b of a row in shared memory times activation block a.
template <int QT>
__device__ __forceinline__ float row_block_dot(uint32_t row, int b, const ActBlock& a) {
  if constexpr (QT == 12) {
    return q4k_sub_dot(row, b, a);
  } else if constexpr (QT == 14) {
    return q6k_sub_dot(row, b, a);
  } else {
    RawBlock r;
    load_block_s<QT>(row, b, r);
    return raw_block_dot<QT>(r, a);
  }
}

// Bulk copy of [src, src + bytes) rounded out to 16-byte bounds into the 16-byte
// aligned shared window `dst`, completing on `bar`; the data starts at
// dst + (src & 15). The buffers the windows come from start on a 16-byte boundary
// and hold a multiple of 16 bytes, so a rounded-out window never leaves them.
__device__ __forceinline__ uint32_t window_span(const uint8_t* src, uint32_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
  const uintptr_t hi = (reinterpret_cast<uintptr_t>(src) + bytes + 15) & ~uintptr_t(15);
  return (uint32_t)(hi - lo);
}
__device__ __forceinline__ void copy_window(uint8_t* dst, const uint8_t* src, uint32_t bytes, uint64_t* bar,
                                            uint64_t pol) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
  bulk_g2s(dst, reinterpret_cast<const void*>(lo), window_span(src, bytes), bar, pol);
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



// Timeline points (MOE_TRACE): %globaltimer readings per CTA index (CTAs below the
// trace's row count), written by thread 0.
enum TracePoint : int {
  TR_RT_START = 0, TR_RT_X = 1, TR_RT_DONE = 2, TR_SEL_KEYS = 3, TR_SEL_CANDS = 19, TR_SEL_RANKED = 22,
  TR_GU_START = 4, TR_GU_XQ = 5, TR_GU_WAITED = 6, TR_GU_PICKED = 7, TR_GU_DATA = 8, TR_GU_END = 9,
  TR_DN_START = 12, TR_DN_PICKED = 13, TR_DN_REQUESTED = 14, TR_DN_WAITED = 15, TR_DN_QUANT = 16,
  TR_DN_DATA = 17, TR_DN_END = 18, TR_GU_DOTS = 10, TR_GU_SUMS = 11, TR_DN_LOOP = 20,
  TR_DN_SUMS = 21,
  TR_POINTS = 24
};
__device__ __forceinline__ void tr(const DecodeArgs& a, int point, int rows) {
  if (a.trace && threadIdx.x == 0 && blockIdx.y == 0 && (int)blockIdx.x < rows)
    a.trace[(size_t)blockIdx.x * TR_POINTS + point] = globaltimer();
}

__device__ __forceinline__ void report_timeout(const DecodeArgs& a) {
  atomicOr(a.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
}

// ===========================================================================
// Selection: the picks and their weights from the complete router logits
// ===========================================================================
// (key, expert) order of the selection: the larger key first, the lower expert among
// equal keys (expert indices are unique, so the order is strict).
__device__ __forceinline__ bool before(uint32_t k1, int i1, uint32_t k2, int i2) {
  return k1 > k2 || (k1 == k2 && i1 < i2);
}
// Sorts a lane's N (<= 4) entries into selection order (insertion network).
template <int N>
__device__ __forceinline__ void sort_list(uint32_t (&kv)[N], int (&ki)[N]) {
#pragma unroll
  for (int a = 1; a < N; ++a)
#pragma unroll
    for (int b = a; b > 0; --b)
      if (before(kv[b], ki[b], kv[b - 1], ki[b - 1])) {
        const uint32_t tk = kv[b]; kv[b] = kv[b - 1]; kv[b - 1] = tk;
        const int ti = ki[b]; ki[b] = ki[b - 1]; ki[b - 1] = ti;
      }
}

// Every thread of a 256-thread CTA calls it (it synchronises the CTA). `sel` holds E
// probs, E keys and 256 (key, expert) candidates; rids/rw receive the k picks in
// selection order and their weights.
//   1. each thread: sigmoid and selection key of experts tid, tid + 256, ...
//   2. groups (n_groups > 1): each warp scores groups (the two largest s, summed);
//      warp 0 keeps groups_used of them, the largest score first, the lowest group
//      on ties; the keys of the other groups' experts become 0
//   3. k <= 8: tau = the k-th largest of the 16 keys that are some warp's largest or second
//      largest. At least k keys reach tau, so every pick does: the keys >= tau are gathered
//      (typically little more than k of them) and each takes its rank among them; ranks
//      below k are the picks.
//   4. otherwise (or when more than 256 keys reach tau, i.e. many exact ties): each warp
//      takes its top k in k rounds over the lanes' sorted lists, then warp 0 merges the 8
//      sorted candidate lists in k rounds
//   5. warp 0: the weights from the picked sigmoids
// Key 0 is below every real key (every float's key is at least that of -inf). With
// trows > 0 thread 0 records the timeline points of the selection's phases.
// The routing weights of the ranked picks rids[0..k) from their sigmoids (probs at the
// start of `sel`): w_j = p_j / max(sum p, norm_min) * scale. Warp 0 computes them; the
// whole CTA calls this (it ends with a barrier).
__device__ __forceinline__ void pick_weights(const DecodeArgs& a, const uint8_t* sel, const int* rids, float* rw) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) == 0) {
    const float* probs = reinterpret_cast<const float*>(sel);
    const float pj = lane < a.p.K ? probs[rids[lane]] : 0.f;
    const float wsum = fmaxf(warp_sum(pj), a.norm_min);
    if (lane < a.p.K) rw[lane] = pj / wsum * a.scale;
  }
  __syncthreads();
}

template <int N>
__device__ void select_picks_n(const DecodeArgs& a, const float* lg, uint8_t* sel, float* gscore, int* rids,
                               float* rw, int trows, bool weights) {
  const DecodePlan& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* probs = reinterpret_cast<float*>(sel);
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel + (size_t)p.E * 4);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(sel + (size_t)p.E * 8);
  int* cidx = reinterpret_cast<int*>(sel + (size_t)p.E * 8 + 1024);
  __shared__ unsigned long long kept_groups;
  __shared__ uint32_t wtop[16];
  __shared__ uint32_t tau_s;
  __shared__ int wcnt[8];
  uint32_t kv[N];  // this thread's keys: experts tid + 256 i
  {
    float l[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {  // loads first
      const int e = tid + 256 * i;
      l[i] = e < p.E ? __ldcg(lg + e) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int e = tid + 256 * i;
      kv[i] = 0u;
      if (e < p.E) {
        const float pr = 1.f / (1.f + expf(-l[i]));
        probs[e] = pr;
        kv[i] = order_key(pr + (a.bias ? __ldg(a.bias + e) : 0.f));
        if (p.G > 1) keys[e] = kv[i];
      }
    }
  }
  tr(a, TR_SEL_KEYS, trows);
  if (p.G > 1) {
    if (tid == 0) kept_groups = ~0ull;
    __syncthreads();
    const int per = p.E / p.G;
    #pragma unroll 1
    for (int g = warp; g < p.G; g += 8) {
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
    __syncthreads();
    if (warp == 0) {
      // groups lane and lane + 32, groups_used rounds of the largest score (a score's
      // key is never 0: only a NaN's is)
      uint32_t gk[2];
      int gi[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        gi[i] = lane + 32 * i;
        gk[i] = gi[i] < p.G ? order_key(gscore[gi[i]]) : 0u;
      }
      sort_list(gk, gi);
      unsigned long long kept = 0ull;
#pragma unroll 1
      for (int j = 0; j < p.Gu; ++j) {
        const uint32_t mk = __reduce_max_sync(0xffffffffu, gk[0]);
        const int win = (int)__reduce_min_sync(0xffffffffu, gk[0] == mk && mk != 0u ? (unsigned)gi[0] : 0xffffffffu);
        kept |= 1ull << (win & 63);
        if (gk[0] == mk && gi[0] == win) {
          gk[0] = gk[1]; gi[0] = gi[1]; gk[1] = 0u;
        }
      }
      if (lane == 0) kept_groups = kept;
    }
    __syncthreads();
    // experts of dropped groups take key 0. The group of expert e is floor((e + 1/2) / per)
    // in fp32: exact, since the quotient stays at least 1/(2 per) >= 1/1024 away from an
    // integer and e < 1024.
    const unsigned long long kg = kept_groups;
    const float inv_per = 1.f / (float)per;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int e = tid + 256 * i;
      const int g = (int)(((float)e + 0.5f) * inv_per);
      if (e < p.E && !((kg >> g) & 1ull)) kv[i] = 0u;
    }
  }
  // each warp's two largest keys (as a multiset: the lane holding the largest offers its
  // next one)
  {
    uint32_t m1 = 0u, m2 = 0u;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if (kv[i] > m1) {
        m2 = m1;
        m1 = kv[i];
      } else if (kv[i] > m2) {
        m2 = kv[i];
      }
    }
    const uint32_t w1 = __reduce_max_sync(0xffffffffu, m1);
    const int hl = __ffs(__ballot_sync(0xffffffffu, m1 == w1)) - 1;
    const uint32_t w2 = __reduce_max_sync(0xffffffffu, lane == hl ? m2 : m1);
    if (lane == 0) {
      wtop[2 * warp] = w1;
      wtop[2 * warp + 1] = w2;
    }
  }
  __syncthreads();
  bool pruned = p.K <= 8;
  if (pruned) {
    // tau: the k-th largest of the 16 warp top-two keys (lane l < 16 ranks entry l)
    if (warp == 0) {
      const uint32_t v = lane < 16 ? wtop[lane] : 0u;
      int rank = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t o = __shfl_sync(0xffffffffu, v, i);
        rank += (o > v || (o == v && i < lane)) ? 1 : 0;
      }
      if (lane < 16 && rank == p.K - 1) tau_s = v;
    }
    __syncthreads();
    const uint32_t tau = tau_s;
    unsigned bal[N];
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      bal[i] = __ballot_sync(0xffffffffu, kv[i] != 0u && kv[i] >= tau);
      cnt += __popc(bal[i]);
    }
    if (lane == 0) wcnt[warp] = cnt;
    __syncthreads();
    int off = 0, C = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = wcnt[w];
      off += w < warp ? c : 0;
      C += c;
    }
    if (C <= 256) {
      const unsigned below = (1u << lane) - 1u;
#pragma unroll
      for (int i = 0; i < N; ++i) {
        if ((bal[i] >> lane) & 1u) {
          const int pos = off + __popc(bal[i] & below);
          ckey[pos] = kv[i];
          cidx[pos] = tid + 256 * i;
        }
        off += __popc(bal[i]);
      }
    }
    __syncthreads();
    tr(a, TR_SEL_CANDS, trows);
    if (C <= 256) {
      #pragma unroll 1
      for (int j = tid; j < C; j += 256) {
        const uint32_t kj = ckey[j];
        const int ij = cidx[j];
        int rank = 0;
        #pragma unroll 4
        for (int c = 0; c < C; ++c) rank += before(ckey[c], cidx[c], kj, ij) ? 1 : 0;
        if (rank < p.K) rids[rank] = ij;
      }
    } else {
      pruned = false;
    }
  }
  if (!pruned) {
    // stage 1: each warp's top k, from lane lists sorted into selection order
    int ki[N];
#pragma unroll
    for (int i = 0; i < N; ++i) ki[i] = tid + 256 * i;
    sort_list(kv, ki);
    #pragma unroll 1
    for (int j = 0; j < p.K; ++j) {
      const uint32_t mk = __reduce_max_sync(0xffffffffu, kv[0]);
      const int win = (int)__reduce_min_sync(0xffffffffu, kv[0] == mk && mk != 0u ? (unsigned)ki[0] : 0xffffffffu);
      if (lane == 0) {
        ckey[warp * p.K + j] = mk;
        cidx[warp * p.K + j] = win;
      }
      if (mk != 0u && kv[0] == mk && ki[0] == win) {  // the winner drops its head
#pragma unroll
        for (int i = 0; i + 1 < N; ++i) {
          kv[i] = kv[i + 1];
          ki[i] = ki[i + 1];
        }
        kv[N - 1] = 0u;
      }
    }
    __syncthreads();
    tr(a, TR_SEL_CANDS, trows);
    if (warp == 0) {
      // stage 2: lane l < 8 walks warp l's sorted candidates
      int h = 0;
      uint32_t bk = lane < 8 ? ckey[lane * p.K] : 0u;
      int bi = lane < 8 ? cidx[lane * p.K] : 0x7fffffff;
      #pragma unroll 1
      for (int j = 0; j < p.K; ++j) {
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        int win = (int)__reduce_min_sync(0xffffffffu, bk == mk && mk != 0u ? (unsigned)bi : 0xffffffffu);
        if (win < 0 || win >= p.E) win = j % p.E;  // unreachable for a valid configuration
        if (lane == 0) rids[j] = win;
        if (lane < 8 && bk == mk && bi == win) {
          ++h;
          bk = h < p.K ? ckey[lane * p.K + h] : 0u;
          bi = h < p.K ? cidx[lane * p.K + h] : 0x7fffffff;
        }
      }
    }
  }
  __syncthreads();
  tr(a, TR_SEL_RANKED, trows);
  if (weights) pick_weights(a, sel, rids, rw);
}
// The picks of the token whose logits row is `lg`; with !weights the caller takes the
// weights later (pick_weights), e.g. after it has requested the picked rows.
__device__ __forceinline__ void select_picks(const DecodeArgs& a, const float* lg, uint8_t* sel, float* gscore,
                                             int* rids, float* rw, int trows = 0, bool weights = true) {
  if (a.p.E <= 256) select_picks_n<1>(a, lg, sel, gscore, rids, rw, trows, weights);
  else if (a.p.E <= 512) select_picks_n<2>(a, lg, sel, gscore, rids, rw, trows, weights);
  else select_picks_n<4>(a, lg, sel, gscore, rids, rw, trows, weights);
}

// ===========================================================================
// Router: logits
// ===========================================================================
// The logits go to every copy of the logits array (the consumers read copy blockIdx.x % rep).
__global__ void __launch_bounds__(RT_THREADS) dec_router(const DecodeArgs a, int trows) {
  __shared__ float part[RT_THREADS / 32][DEC_TMAX];
  __shared__ float red[RT_THREADS / 32][DEC_TMAX];  // sums of squares (with a norm vector)
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
  float4 nv[6];  // the norm vector's quarter (with a prologue)
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    const int j = lane + 32 * i;
    nv[i] = (a.norm && has && j < nq4) ? __ldg(reinterpret_cast<const float4*>(a.norm + q * (p.H / 4)) + j)
                                       : make_float4(1.f, 1.f, 1.f, 1.f);
  }
  pdl_wait_prior_grids();  // x may come from the previous kernel
  pdl_launch_dependents();
  tr(a, TR_RT_X, trows);
  // this call's published picks start empty (the previous call's kernels are complete:
  // the wait above covers them, and every reader of this call starts after this grid)
  if (a.T == 1 && blockIdx.x == 0 && tid < p.K) st_relaxed_u64(a.pub + tid, PUB_EMPTY);
  // the prologue (with a norm vector): token t's input is x_t * r_t * norm, r_t =
  // 1/rms(x_t). The dot takes x_t * norm and its sum is scaled by r_t; the sum of squares
  // comes from the same loads (a row's four quarter warps cover x_t once).
#pragma unroll 1
  for (int t = 0; t < a.T; ++t) {
    const float* xt = a.x + (size_t)t * p.H + q * (p.H / 4);
    float acc = 0.f, ss = 0.f;
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      const int j = lane + 32 * i;
      if (has && j < nq4) {
        const float4 xv = __ldcg(reinterpret_cast<const float4*>(xt) + j);
        acc = fmaf(wv[i].x, xv.x * nv[i].x, acc);
        acc = fmaf(wv[i].y, xv.y * nv[i].y, acc);
        acc = fmaf(wv[i].z, xv.z * nv[i].z, acc);
        acc = fmaf(wv[i].w, xv.w * nv[i].w, acc);
        ss = fmaf(xv.x, xv.x, fmaf(xv.y, xv.y, fmaf(xv.z, xv.z, fmaf(xv.w, xv.w, ss))));
      }
    }
    acc = warp_sum(acc);
    if (a.norm) ss = warp_sum(ss);
    if (lane == 0) {
      part[warp][t] = acc;
      red[warp][t] = ss;
    }
  }
  __syncthreads();
  for (int u = tid; u < 2 * a.T; u += RT_THREADS) {
    const int rr = u & 1, t = u >> 1;
    const int row2 = blockIdx.x * 2 + rr;
    if (row2 < p.E) {
      float v = ((part[4 * rr][t] + part[4 * rr + 1][t]) + part[4 * rr + 2][t]) + part[4 * rr + 3][t];
      if (a.norm) {
        const float sq = ((red[4 * rr][t] + red[4 * rr + 1][t]) + red[4 * rr + 2][t]) + red[4 * rr + 3][t];
        v *= 1.f / sqrtf(sq / (float)p.H + a.eps);
      }
      for (int c = 0; c < p.rep; ++c) a.logits[(size_t)c * a.lg_copy + (size_t)t * p.E + row2] = v;
    }
  }
  tr(a, TR_RT_DONE, trows);
}

// ===========================================================================
// Selection of a call of several tokens: one CTA per token
// ===========================================================================
__global__ void __launch_bounds__(256) dec_select(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t ssm[];
  __shared__ float gscore[64];
  __shared__ int rids[32];
  __shared__ float rw[32];
  const int t = blockIdx.x;
  pdl_wait_prior_grids();  // the logits
  pdl_launch_dependents();
  select_picks(a, a.logits + (size_t)(t % a.p.rep) * a.lg_copy + (size_t)t * a.p.E, ssm, gscore, rids, rw);
  if (threadIdx.x < a.p.K) {
    const size_t o = (size_t)t * a.p.K + threadIdx.x;
    a.ids[o] = rids[threadIdx.x];
    a.wts[o] = rw[threadIdx.x];
    if (a.topk_ids) a.topk_ids[o] = rids[threadIdx.x];
    if (a.topk_w) a.topk_w[o] = rw[threadIdx.x];
  }
}

// ===========================================================================
// Gate/up: 16 intermediate values of a slot per CTA
// ===========================================================================
// Dynamic shared memory: 4 windows (chunk c: gate window 2c, up window 2c + 1, each
// 8 rows), then x: f32 chunks [8][nbH] and block sums [nbH], or (fixed point) the planes
// [nbH][64] and info [nbH].
template <int QT, int MAXB, bool FX>
__global__ void __launch_bounds__(GU_THREADS, 3) dec_gate_up(const DecodeArgs a, int trows) {
  extern __shared__ __align__(128) uint8_t gsm[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ float rowdot[GU_THREADS / 32][4];
  __shared__ float actv[GU_VALUES];  // fixed point: the CTA's activations, quantised by warp 0
  __shared__ float gscore[64];
  __shared__ int rids[32];
  __shared__ float rw[32];
  const DecodePlan& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int v0 = blockIdx.x * GU_VALUES;  // first activation index of the CTA
  const int tok = blockIdx.y;             // the call's token
  const int cp = blockIdx.x % p.rep;      // the copy of the logits this CTA reads
  const bool shared = v0 < p.Fs;          // the shared expert's values need no routing
  const int ff = shared ? p.Fs : p.F;
  const int f0 = shared ? v0 : (v0 - p.Fs) % p.F;
  tr(a, TR_GU_START, trows);
  uint8_t* win = gsm;
  uint8_t* xplanes = gsm + (size_t)4 * p.gu_win;  // x: fixed-point planes, or f32 chunks
  float4* xinfo = reinterpret_cast<float4*>(xplanes + (size_t)p.nbH * 64);
  float4* xs = reinterpret_cast<float4*>(xplanes);
  float* xsum = reinterpret_cast<float*>(xplanes + (size_t)p.nbH * 128);
  uint8_t* sel = xplanes + (size_t)p.nbH * (FX ? ACT_BLOCK_SMEM_FX : ACT_BLOCK_SMEM);
  const uint32_t rows8 = 8u * p.rb_h;
  if (tid == 0) {
    mbar_init(&bars[0], 2);
    mbar_init(&bars[1], 2);
    fence_mbar_init();
  }
  __syncthreads();
  // window t (t < 4) of a record: 8 gate (t even) or up (t odd) rows of chunk t / 2,
  // copied by thread t; each chunk's barrier takes its two threads' arrivals
  auto issue = [&](const uint8_t* rec) {
    const int c = tid >> 1;
    const uint8_t* src = rec + (size_t)((tid & 1) * ff + f0 + 8 * c) * p.rb_h;
    mbar_arrive_expect_tx(&bars[c], window_span(src, rows8));
    copy_window(win + (size_t)tid * p.gu_win, src, rows8, &bars[c], policy_evict_first());
  };
  if (shared && tid < 4) issue(a.shared);
  // x -> activation blocks (x is complete: the router kernel waited for it before this
  // launch was triggered); routed CTAs do this while the router kernel runs. With a norm
  // vector the blocks hold x * norm; r = 1/rms(x) comes from the same loads and scales the
  // row dots (every dot is linear in x).
  const float* xt = a.x + (size_t)tok * p.H;
  __shared__ float red[GU_THREADS / 32];
  {
    float ss = 0.f;
    if constexpr (FX) quant_blocks<2>(xt, p.nbH, p.nbH, xplanes, xinfo, tid, GU_THREADS, a.norm, 1.f, a.norm ? &ss : nullptr);
    else store_blocks_f32<4>(xt, p.nbH, p.nbH, xs, xsum, tid, GU_THREADS, a.norm, a.norm ? &ss : nullptr);
    if (a.norm) {
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
    }
  }
  __syncthreads();
  float r = 1.f;
  if (a.norm) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < GU_THREADS / 32; ++w) tot += red[w];
    r = 1.f / sqrtf(tot / (float)p.H + a.eps);
  }
  tr(a, TR_GU_XQ, trows);
  const uint8_t* rec = a.shared;
  if (shared) {
    pdl_launch_dependents();
  } else {
    pdl_wait_prior_grids();  // the logits
    tr(a, TR_GU_WAITED, trows);
    const int slot = (v0 - p.Fs) / p.F;
    if (a.T == 1) {
      // the picks, then (fixed point) this CTA's rows requested before the weights are taken,
      // so the rows' HBM latency starts sooner; the f32 form measured slower that way (15.8
      // against 15.2 us on the Flint layer) and keeps the weights first
      select_picks(a, a.logits + (size_t)cp * a.lg_copy, sel, gscore, rids, rw, trows, !FX);
      rec = a.experts + (size_t)rids[slot] * p.rec_bytes;
      if (FX) {
        if (tid < 4) issue(rec);
        pick_weights(a, sel, rids, rw);
      }
      if (v0 == p.Fs && tid < p.K) {  // one CTA reports the picks
        if (a.topk_ids) a.topk_ids[tid] = rids[tid];
        if (a.topk_w) a.topk_w[tid] = rw[tid];
        // for down CTAs that start after this point: one 64-bit store per pick
        st_relaxed_u64(a.pub + tid, (unsigned long long)(uint32_t)rids[tid] |
                                        ((unsigned long long)__float_as_uint(rw[tid]) << 32));
      }
      if (!FX && tid < 4) issue(rec);
    } else {
      int e = __ldcg(a.ids + (size_t)tok * p.K + slot);  // made by the selection kernel
      if ((unsigned)e >= (unsigned)p.E) {  // only a workspace that was not zeroed before its first use
        if (tid == 0) atomicOr(a.ctrl + CTRL_STATUS, DEV_ERR_BAD_PICK);
        e = 0;
      }
      rec = a.experts + (size_t)e * p.rec_bytes;
      if (tid < 4) issue(rec);
    }
    // the down kernel may start once every CTA is here: by then the picks are published
    // (its CTAs that still find them missing select for themselves)
    pdl_launch_dependents();
  }
  tr(a, TR_GU_PICKED, trows);
  const RowMap mh = row_map(p.nbH, lane);
  ActBlock xc[FX ? MAXB : 1];
  if constexpr (FX) {
#pragma unroll
    for (int i = 0; i < MAXB; ++i) {
      const int b = mh.sub + mh.lpr * i;
      if (b < p.nbH) load_act_block_s(xc[i], smem_addr(xplanes), smem_addr(xinfo), b, p.nbH);
    }
  }
  // warp w: values 2w, 2w + 1 of the CTA (chunk w / 4); its rows r = 0..3 are gate
  // (r even) and up (r odd) of value 2w + r / 2
  const int c = warp >> 2;
  const bool ok = mbar_wait(&bars[c], 0);
  if (!ok && lane == 0) report_timeout(a);
  tr(a, TR_GU_DATA, trows);
  const uint8_t* gsrc = rec + (size_t)(f0 + 8 * c) * p.rb_h;
  const uint8_t* usrc = rec + (size_t)(ff + f0 + 8 * c) * p.rb_h;
  const uint32_t gwin = smem_addr(win) + (uint32_t)(2 * c) * p.gu_win + (uint32_t)(reinterpret_cast<uintptr_t>(gsrc) & 15u);
  const uint32_t uwin = smem_addr(win) + (uint32_t)(2 * c + 1) * p.gu_win + (uint32_t)(reinterpret_cast<uintptr_t>(usrc) & 15u);
  const int vl = 2 * (warp & 3);  // first value of the warp within the chunk
  float dots[4] = {0.f, 0.f, 0.f, 0.f};
  if (ok) {
    if constexpr (FX) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int r = mh.rsub + mh.rps * s;
        if (r < 4) {
          const uint32_t row = ((r & 1) ? uwin : gwin) + (uint32_t)(vl + (r >> 1)) * p.rb_h;
#pragma unroll
          for (int i = 0; i < MAXB; ++i) {
            const int b = mh.sub + mh.lpr * i;
            if (b < p.nbH) {
              dots[s] += row_block_dot<QT>(row, b, xc[i]);
            }
          }
        }
      }
    } else {
      // each x block is loaded once for the warp's rows
#pragma unroll
      for (int i = 0; i < MAXB; ++i) {
        const int b = mh.sub + mh.lpr * i;
        if (b < p.nbH) {
          XBlock xb;
          load_xblock(xb, smem_addr(xs), smem_addr(xsum), b, p.nbH);
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const int r = mh.rsub + mh.rps * s;
            if (r < 4) {
              const uint32_t row = ((r & 1) ? uwin : gwin) + (uint32_t)(vl + (r >> 1)) * p.rb_h;
              dots[s] += row_block_dot_f32<QT>(row, b, xb);
            }
          }
        }
      }
    }
  }
  tr(a, TR_GU_DOTS, trows);
  group_sum_n(dots, mh.lpr);
  tr(a, TR_GU_SUMS, trows);
  if (mh.sub == 0) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int r = mh.rsub + mh.rps * s;
      if (r < 4) rowdot[warp][r] = dots[s];
    }
  }
  __syncwarp();
  if (lane < 2) {
    const float act =
        swiglu_act(rowdot[warp][2 * lane] * r, rowdot[warp][2 * lane + 1] * r, shared ? a.lim_s : a.lim);
    if constexpr (FX) actv[2 * warp + lane] = act;
    else
      for (int c = 0; c < p.rep; ++c) a.act[(size_t)c * a.act_copy + (size_t)tok * p.act_stride + v0 + 2 * warp + lane] = act;
  }
  if constexpr (FX) {
    // The CTA's 16 activations are half h of activation block gb: warp 0 quantises them as
    // quant_task does a half (one power of two from their largest magnitude) and writes the
    // half's two plane chunks and its {scale, sum} into every copy, in the layout the down
    // kernel stages as is: per token, planes [4][nact][16 B] (chunk 2P + h: plane P of half
    // h), then info [nact][16 B] ({s0, X0, s1, X1}).
    static_assert(GU_VALUES == 16, "one CTA makes half an activation block");
    __syncthreads();
    if (warp == 0) {
      const float v = lane < GU_VALUES ? actv[lane] : 0.f;
      float amax = fabsf(v);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFF);
      float inv = 0.f, sc = 0.f;
      if (eb >= 30) {
        inv = __uint_as_float((uint32_t)(140 - eb + 127) << 23);
        sc = __uint_as_float((uint32_t)(eb - 140 + 127) << 23);
      }
      const int q = round_small(v * inv);
      int X = q;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) X += __shfl_xor_sync(0xffffffffu, X, o);
      // word w of plane P: byte P of q of values 4w .. 4w + 3 (lanes 4w .. 4w + 3)
      uint32_t b0 = ((uint32_t)q & 0xFFu) << (8 * (lane & 3));
      uint32_t b1 = (((uint32_t)q >> 8) & 0xFFu) << (8 * (lane & 3));
      b0 |= __shfl_xor_sync(0xffffffffu, b0, 1);
      b1 |= __shfl_xor_sync(0xffffffffu, b1, 1);
      b0 |= __shfl_xor_sync(0xffffffffu, b0, 2);
      b1 |= __shfl_xor_sync(0xffffffffu, b1, 2);
      const uint4 lo = make_uint4(__shfl_sync(0xffffffffu, b0, 0), __shfl_sync(0xffffffffu, b0, 4),
                                  __shfl_sync(0xffffffffu, b0, 8), __shfl_sync(0xffffffffu, b0, 12));
      const uint4 hi = make_uint4(__shfl_sync(0xffffffffu, b1, 0), __shfl_sync(0xffffffffu, b1, 4),
                                  __shfl_sync(0xffffffffu, b1, 8), __shfl_sync(0xffffffffu, b1, 12));
      const int gb = v0 >> 5, h = (v0 >> 4) & 1;
      if (lane < p.rep) {
        uint8_t* rec = reinterpret_cast<uint8_t*>(a.act + (size_t)lane * a.act_copy + (size_t)tok * p.act_stride);
        *reinterpret_cast<uint4*>(rec + ((size_t)h * p.nact + gb) * 16) = lo;
        *reinterpret_cast<uint4*>(rec + ((size_t)(2 + h) * p.nact + gb) * 16) = hi;
        *reinterpret_cast<float2*>(rec + (size_t)64 * p.nact + (size_t)gb * 16 + 8 * h) = make_float2(sc, (float)X);
      }
    }
  }
  tr(a, TR_GU_END, trows);
}

// ===========================================================================
// Down: R output rows per CTA over every slot, weighted, in a fixed order
// ===========================================================================
// Dynamic shared memory: the shared window, then K routed windows, then one piece of
// activation blocks: f32 chunks [8][piece] and block sums [piece], or (fixed point)
// planes [4][piece][16 B] and info [piece]. The threads form RG row groups of 256 / RG threads;
// group g owns rows g R / RG .. (g + 1) R / RG - 1, and its thread t takes blocks t,
// t + 256 / RG, ... of each piece with all of the group's rows: an activation block
// is read once for R / RG block dots.
template <int QT, bool FX>
__global__ void __launch_bounds__(DN_THREADS, 3) dec_down(const DecodeArgs a, int trows) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ float gscore[64];
  __shared__ int rids[32];
  __shared__ float rw[32];
  __shared__ uint32_t woff[33];  // offset of each window's first row in the window
  __shared__ float part[DN_THREADS / 32][8];
  const DecodePlan& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.dn_rows, h0 = blockIdx.x * R;
  const int tok = blockIdx.y;  // the call's token
  const int nwin = p.K + (p.Fs ? 1 : 0);
  tr(a, TR_DN_START, trows);
  const size_t win_r = (size_t)p.dn_win_fs;  // first routed window
  uint8_t* aplanes = dsm + win_r + (size_t)p.K * p.dn_win_f;  // activations: fixed-point planes, or f32 chunks
  float4* ainfo = reinterpret_cast<float4*>(aplanes + (size_t)p.dn_piece * 64);
  float4* axs = reinterpret_cast<float4*>(aplanes);
  float* axsum = reinterpret_cast<float*>(aplanes + (size_t)p.dn_piece * 128);
  uint8_t* sel = aplanes + (size_t)p.dn_piece * (FX ? ACT_BLOCK_SMEM_FX : ACT_BLOCK_SMEM);
  if (tid == 0) {
    mbar_init(&bar, (uint32_t)nwin);
    fence_mbar_init();
  }
  const int cp = blockIdx.x % p.rep;  // the copy of the logits and activations this CTA reads
  // the picks (the router is complete: every routed gate/up CTA waited for it before
  // this launch was triggered)
  if (a.T == 1) {
    // The picks: those the gate/up kernel has published if all k are there (a down CTA
    // that could not start before the gate/up CTAs left finds them), else made here.
    // Nothing waits on them: an entry is either empty or this call's pick.
    bool mine = true;
    if (tid < p.K) {
      const unsigned long long v = ld_relaxed_u64(a.pub + tid);
      mine = v != PUB_EMPTY;
      rids[tid] = (int)(uint32_t)v;
      rw[tid] = __uint_as_float((uint32_t)(v >> 32));
    }
    if (!__syncthreads_and(mine)) select_picks(a, a.logits + (size_t)cp * a.lg_copy, sel, gscore, rids, rw);
  } else {
    // made by the selection kernel, complete once every routed gate/up CTA has waited
    if (tid < p.K) {
      int e = __ldcg(a.ids + (size_t)tok * p.K + tid);
      if ((unsigned)e >= (unsigned)p.E) {  // only a workspace that was not zeroed before its first use
        atomicOr(a.ctrl + CTRL_STATUS, DEV_ERR_BAD_PICK);
        e = 0;
      }
      rids[tid] = e;
      rw[tid] = __ldcg(a.wts + (size_t)tok * p.K + tid);
    }
    __syncthreads();
  }
  tr(a, TR_DN_PICKED, trows);
  if (tid < nwin) {
    // this CTA's rows of slot window tid's down matrix, copied by thread tid
    const bool sh = p.Fs && tid == 0;
    const int j = tid - (p.Fs ? 1 : 0);
    const uint8_t* src = sh ? a.shared + (size_t)2 * p.Fs * p.rb_h + (size_t)h0 * p.rb_fs
                            : a.experts + (size_t)rids[j] * p.rec_bytes + (size_t)2 * p.F * p.rb_h +
                                  (size_t)h0 * p.rb_f;
    const uint32_t bytes = (uint32_t)R * (sh ? p.rb_fs : p.rb_f);
    mbar_arrive_expect_tx(&bar, window_span(src, bytes));
    copy_window(dsm + (sh ? 0 : win_r + (size_t)j * p.dn_win_f), src, bytes, &bar, policy_evict_first());
    woff[sh ? 32 : j] = (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u);
  }
  tr(a, TR_DN_REQUESTED, trows);
  // the residual and accumulate inputs: complete before this call's first kernel started,
  // so they are read ahead of the wait
  float xres = 0.f, oin = 0.f;
  if (tid < R) {
    const size_t h = (size_t)tok * p.H + h0 + tid;
    if (a.flags & FLAG_RESIDUAL) xres = __ldcg(a.x + h);
    if (a.flags & FLAG_ACCUMULATE) oin = __ldcg(a.out + h);
  }
  pdl_wait_prior_grids();  // the activations
  pdl_launch_dependents();
  tr(a, TR_DN_WAITED, trows);
  const int nact = p.nact;
  const int RPG = R / p.dn_rg;                 // rows per group
  const int TPG = DN_THREADS / p.dn_rg;        // threads per group (a multiple of 32)
  const int grp = tid / TPG, tl = tid % TPG;
  float acc[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r] = 0.f;
  bool ok = true;
  #pragma unroll 1
  for (int pb = 0; pb < nact; pb += p.dn_piece) {
    const int np = nact - pb < p.dn_piece ? nact - pb : p.dn_piece;
    if constexpr (FX) {
      // the gate/up kernel wrote the blocks already quantised: planes chunk c of block
      // pb + i and its info, 16 bytes each, go to shared memory as they are (all loads of a
      // thread are issued before its stores)
      const uint8_t* rec = reinterpret_cast<const uint8_t*>(a.act + (size_t)cp * a.act_copy + (size_t)tok * p.act_stride);
      constexpr int U = 4;
      for (int i0 = tid; i0 < 5 * np; i0 += U * DN_THREADS) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * DN_THREADS, c = i / np, bi = i - c * np;
          if (i < 5 * np)
            v[u] = __ldcg(reinterpret_cast<const uint4*>(c < 4 ? rec + ((size_t)c * nact + pb + bi) * 16
                                                               : rec + (size_t)64 * nact + (size_t)(pb + bi) * 16));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * DN_THREADS, c = i / np, bi = i - c * np;
          if (i < 5 * np)
            *reinterpret_cast<uint4*>(c < 4 ? aplanes + ((size_t)c * p.dn_piece + bi) * 16
                                            : reinterpret_cast<uint8_t*>(ainfo) + (size_t)bi * 16) = v[u];
        }
      }
    } else {
      const float* act = a.act + (size_t)cp * a.act_copy + (size_t)tok * p.act_stride + (size_t)pb * 32;
      store_blocks_f32<4>(act, np, p.dn_piece, axs, axsum, tid, DN_THREADS);
    }
    __syncthreads();  // the piece; on the first pass also the window offsets
    if (pb == 0) {
      tr(a, TR_DN_QUANT, trows);
      ok = mbar_wait(&bar, 0);
      if (!ok && lane == 0) report_timeout(a);
      tr(a, TR_DN_DATA, trows);
    }
    if (ok) {
      #pragma unroll 1
      for (int i = tl; i < np; i += TPG) {
        const int cb = pb + i;
        const bool sh = cb < p.nbFs;
        const int j = sh ? 0 : (cb - p.nbFs) / p.nbF;
        const int b = sh ? cb : cb - p.nbFs - j * p.nbF;
        const uint32_t w0 = smem_addr(dsm) + (sh ? woff[32] : (uint32_t)win_r + (uint32_t)j * p.dn_win_f + woff[j]);
        const uint32_t rb = sh ? p.rb_fs : p.rb_f;
        const float wgt = sh ? 1.f : rw[j];
        const uint32_t wr = w0 + (uint32_t)(grp * RPG) * rb;
        if constexpr (FX) {
          ActBlock ab;
          load_act_block_s(ab, smem_addr(aplanes), smem_addr(ainfo), i, p.dn_piece);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            if (r < RPG) {
              acc[r] = fmaf(wgt, row_block_dot<QT>(wr + (uint32_t)r * rb, b, ab), acc[r]);
            }
          }
        } else {
          XBlock xb;
          load_xblock(xb, smem_addr(axs), smem_addr(axsum), i, p.dn_piece);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            if (r < RPG) {
              acc[r] = fmaf(wgt, row_block_dot_f32<QT>(wr + (uint32_t)r * rb, b, xb), acc[r]);
            }
          }
        }
      }
    }
    __syncthreads();  // the next piece reuses the buffer
  }
  tr(a, TR_DN_LOOP, trows);
  // each row: warp sums, then its group's warp sums in warp order
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (r < RPG) {
      const float v = warp_sum(acc[r]);
      if (lane == 0) part[warp][r] = v;
    }
  }
  __syncthreads();
  tr(a, TR_DN_SUMS, trows);
  if (tid < R) {
    const int g = tid / RPG, rl = tid % RPG, w0 = g * (TPG / 32);
    float y = 0.f;
    for (int w = 0; w < TPG / 32; ++w) y += part[w0 + w][rl];
    const size_t h = (size_t)tok * p.H + h0 + tid;
    if (a.flags & FLAG_RESIDUAL) y = xres + y;
    if (a.flags & FLAG_ACCUMULATE) y = oin + y;
    a.out[h] = y;
  }
  tr(a, TR_DN_END, trows);
}

// ===========================================================================
// Host side
// ===========================================================================
template <typename... Args>
static cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, int threads, size_t smem, cudaStream_t st, bool pdl,
                              Args... args) {
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), (int)smem);
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
static cudaError_t launch_gate_up(const DecodeArgs& a, cudaStream_t st, bool pdl, bool fx, int trows) {
  const DecodePlan& p = a.p;
  const dim3 grid((unsigned)((p.K * p.F + p.Fs) / GU_VALUES), (unsigned)a.T);
  if (fx) return launch_pdl(dec_gate_up<QT, MAXB, true>, grid, GU_THREADS, (size_t)p.gu_smem, st, pdl, a, trows);
  return launch_pdl(dec_gate_up<QT, MAXB, false>, grid, GU_THREADS, (size_t)p.gu_smem, st, pdl, a, trows);
}

template <int QT>
static cudaError_t launch_down(const DecodeArgs& a, cudaStream_t st, bool pdl, bool fx, int trows) {
  const DecodePlan& p = a.p;
  const dim3 grid((unsigned)(p.H / p.dn_rows), (unsigned)a.T);
  if (fx) return launch_pdl(dec_down<QT, true>, grid, DN_THREADS, (size_t)p.dn_smem, st, pdl, a, trows);
  return launch_pdl(dec_down<QT, false>, grid, DN_THREADS, (size_t)p.dn_smem, st, pdl, a, trows);
}

// The chain: router, (several tokens) selection, gate/up in the gate/up rows' block type,
// down in the down rows' block type; `fx` selects the 16-bit fixed-point activations.
cudaError_t decode_launch(const DecodeArgs& a, int maxb, cudaStream_t st, bool pdl, bool fx, int trows) {
  const DecodePlan& p = a.p;
  cudaError_t e = launch_pdl(dec_router, dim3((unsigned)ceil_div(p.E, 2)), RT_THREADS, (size_t)0, st, pdl, a, trows);
  if (e != cudaSuccess) return e;
  if (a.T > 1) {  // one selection per token, shared by the gate/up and down CTAs
    e = launch_pdl(dec_select, dim3((unsigned)a.T), 256, (size_t)select_smem(p.E), st, pdl, a);
    if (e != cudaSuccess) return e;
  }
  switch (p.qtype * 8 + maxb) {
    case 2 * 8 + 1: e = launch_gate_up<2, 1>(a, st, pdl, fx, trows); break;
    case 2 * 8 + 2: e = launch_gate_up<2, 2>(a, st, pdl, fx, trows); break;
    case 2 * 8 + 3: e = launch_gate_up<2, 3>(a, st, pdl, fx, trows); break;
    case 3 * 8 + 1: e = launch_gate_up<3, 1>(a, st, pdl, fx, trows); break;
    case 3 * 8 + 2: e = launch_gate_up<3, 2>(a, st, pdl, fx, trows); break;
    case 3 * 8 + 3: e = launch_gate_up<3, 3>(a, st, pdl, fx, trows); break;
    case 12 * 8 + 1: e = launch_gate_up<12, 1>(a, st, pdl, fx, trows); break;
    case 12 * 8 + 2: e = launch_gate_up<12, 2>(a, st, pdl, fx, trows); break;
    case 12 * 8 + 3: e = launch_gate_up<12, 3>(a, st, pdl, fx, trows); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  switch (p.qtype_dn) {
    case 2: return launch_down<2>(a, st, pdl, fx, trows);
    case 3: return launch_down<3>(a, st, pdl, fx, trows);
    case 12: return launch_down<12>(a, st, pdl, fx, trows);
    case 14: return launch_down<14>(a, st, pdl, fx, trows);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
