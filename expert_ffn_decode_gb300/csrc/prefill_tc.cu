// Tile pipeline of the batched MoE-FFN step for sm_103a: the router, gate/up and
// down contractions as warp-specialised persistent kernels on the tensor cores.
//
// One CTA per SM, 640 threads:
//   warp 0       weight producer: 2-D TMA tensor copies of the raw weight rows of each
//                pipeline chunk (one box of 64 or 128 rows) into shared-memory stages (3-D
//                maps for K-quant records; one bulk copy of 128 whole rows for Q6_K down rows)
//   warps 1, 19  MMA issuers: tcgen05.mma with A in tensor memory, B in shared memory,
//                f32 accumulator in tensor memory; commits release the stages. One thread
//                issues a small-N MMA only every ~50-100 cycles (its waits, fence and commits
//                included), so two threads share the A units of a tile: unit n goes to issuer
//                n % 2, which owns its own accumulation chains (the sums stay deterministic)
//   warp 2       token-operand producer: one bulk copy per 128 K values of a pre-tiled
//                image of the chunk's token rows
//   warps 3..14  converters in three groups of four warps (one per TMEM lane quarter;
//                thread = tile row = TMEM lane). Every converter warp waits for every raw
//                chunk and releases it; 128-value A unit n of the tile stream goes to group
//                n % 3, which owns one TMEM A slot: raw 4-bit blocks, Q4_K or Q6_K
//                super-blocks (or f32 router rows) -> f16 rows of A, written with tcgen05.st
//   warps 15..18 the epilogue, one warp per TMEM lane quarter (tcgen05.ld), on one of two
//                accumulators while the MMAs of the next tile run on the other
//
// Work units (one accumulator tile, M = 128 weight rows x N = chunk tokens):
//   router   64 experts (f32 rows split into f16 hi rows 0..63 and lo rows 64..127)
//            x 64 tokens (x hi and lo columns): logit = sum of the four products
//   gate/up  64 gate rows (rows 0..63) and the matching up rows (64..127) of one
//            expert x one chunk of its sorted (token, pick) pairs (x hi and lo columns)
//   down     128 down rows of one expert x the chunk's activations
// Every stage wait is bounded; a timeout anywhere stops every role of the CTA and
// sets the status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "plan.h"
#include "prefill_host.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int TP_CONV_WARPS = 12;                 // three groups of four (one warp per TMEM lane quarter)
constexpr int TP_GROUPS = TP_CONV_WARPS / 4;      // A unit n is converted by group n % TP_GROUPS
constexpr int TP_EPI_WARPS = 4;                   // one per lane quarter
constexpr int TP_EPI_WARP0 = 3 + TP_CONV_WARPS;   // first epilogue warp
constexpr int TP_MMA_WARP2 = TP_EPI_WARP0 + TP_EPI_WARPS;  // the second MMA issuer
// producers, the first MMA issuer, converters, epilogue, the second MMA issuer
constexpr int TP_THREADS = 96 + 32 * (TP_CONV_WARPS + TP_EPI_WARPS) + 32;
constexpr int TP_KB = 128;                        // K values per token-operand stage
constexpr int TP_B_STAGE = 128 * TP_KB * 2;       // up to 128 rows: 32 KB
constexpr int TP_SCRATCH = 64 * 65 * 4;           // gate/up and router epilogue exchange
constexpr int TP_SMEM_MAX = 227 * 1024 - 2048;    // dynamic shared memory (static arrays + alignment aside)
constexpr uint32_t TP_TMEM_COLS = 512;
constexpr uint32_t TP_A_COL = 128;                // A slots follow the first accumulator's columns [0, 128)
constexpr uint32_t TP_ACC1_COL = 384;             // the second accumulator (router, gate/up): [384, 512)
// Every TMEM column a tile kernel touches lies inside its allocation: the converter groups' A
// slots (64 columns each) sit between the two accumulators, and a tile's accumulation chains
// stay inside its accumulator's 128 (down: 64) columns (tile_chains).
static_assert(TP_A_COL >= 128u && TP_A_COL + 64u * (TP_CONV_WARPS / 4) <= TP_ACC1_COL, "TMEM A slots");
static_assert(TP_ACC1_COL + 128u <= TP_TMEM_COLS, "TMEM accumulators");

// Q6_K down rows on the tile pipeline: a raw stage holds 128 whole rows of at most this many
// values (a Q6_K row of 768 values is 630 bytes, so single rows do not start on 16-byte
// bounds, but 128 consecutive rows span a multiple of 16 bytes).
constexpr int TP_Q6_KMAX = 768;

// Stage geometry per contraction. MODE 0 gate/up, 1 down, 2 router.
template <int MODE, int QT>
struct Geo {
  // A raw chunk is ROWS rows x KR K values. Its row segments (SEG bytes) are odd multiples
  // of 16 bytes, stored densely by the TMA: a quarter warp reading one 16-byte word of 8
  // consecutive rows then hits 8 different bank groups. Wide segments keep each TMA row
  // request long (240 and 144 bytes against 80 for a single 128-value unit). A Q4_K chunk
  // is one 144-byte super-block of each row; a Q6_K chunk is whole rows (one bulk copy).
  static constexpr bool Q6 = QT == 14;
  static constexpr int ROWS = MODE == 2 ? 64 : 128;                  // raw rows per stage
  static constexpr int KR = MODE == 2 ? 128 : (QT == 3 ? 384 : (Q6 ? TP_Q6_KMAX : 256));  // K values per raw chunk
  static constexpr int SEG = MODE == 2   ? 512
                             : Q6        ? TP_Q6_KMAX / 256 * 210
                             : QT == 12  ? 144
                                         : KR / 32 * (QT == 3 ? 20 : 18);  // bytes per row (at most, Q6_K)
  static constexpr int STAGE = ROWS * SEG;
  static constexpr int NAU = KR / TP_KB;                             // 128-value A units per chunk
  // token-operand stages: with two MMA issuers each owns every other unit's stage, so gate/up
  // keeps three (a stage refill is an L2 round trip); the down contraction's Q6_K stages leave
  // room for two
  static constexpr int NSB = MODE == 0 ? 3 : 2;
  static constexpr int SCR = MODE == 1 ? 0 : TP_SCRATCH;
  static constexpr int NSA0 = (TP_SMEM_MAX - NSB * TP_B_STAGE - SCR - 1024) / STAGE;
  static constexpr int NSA = NSA0 > 16 ? 16 : NSA0;                  // raw stages (one shared ring)
  static constexpr int NACC = 2;                                     // accumulators (down tiles: N <= 64)
  static constexpr int RAW_BYTES = (NSA * STAGE + 1023) / 1024 * 1024;  // token stages start 1024-aligned
  static constexpr int SMEM = RAW_BYTES + NSB * TP_B_STAGE + SCR;
  static_assert(NSA >= 2 && SMEM + 1024 <= TP_SMEM_MAX, "shared memory");
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_lo(float a, float b, uint32_t hi) {
  __half2 h = *reinterpret_cast<__half2*>(&hi);
  const float2 f = __half22float2(h);
  return pack_h2(a - f.x, b - f.y);
}

// ---- bounded waits shared by the roles -----------------------------------------------
__device__ __forceinline__ bool tp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > MBAR_TIMEOUT_NS) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// The whole warp waits; the answer is the same on every lane.
__device__ __forceinline__ bool tp_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = tp_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ---- tensor memory stores / loads ------------------------------------------------------
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T over K = 16.
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// ---- dequantisation of one nibble word into 4 packed f16 pairs (slots 8w .. 8w + 7) ------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Value of nibble q is d*q + m (Q4_1) or d*(q - 8) (Q4_0): the nibble enters the
// mantissa of an f16 whose exponent makes it an exact integer offset (1024 + q for a
// low nibble, 64 + q for a high nibble), the offset is subtracted exactly, and one
// fused multiply-add (or multiply) applies the scale and offset with a single rounding.
template <int QT>
__device__ __forceinline__ void dequant4(uint32_t qw, __half2 d2, __half2 m2, uint32_t* o) {
  const uint32_t sh = qw >> 8;
  __half2 lo02 = u2h(lop3_and_or(qw, 0x000F000Fu, 0x64006400u));
  __half2 lo13 = u2h(lop3_and_or(sh, 0x000F000Fu, 0x64006400u));
  __half2 hi02 = u2h(lop3_and_or(qw, 0x00F000F0u, 0x54005400u));
  __half2 hi13 = u2h(lop3_and_or(sh, 0x00F000F0u, 0x54005400u));
  if constexpr (QT == 3) {
    const __half2 b1024 = u2h(0x64006400u), b64 = u2h(0x54005400u);
    o[0] = h2u(__hfma2(__hsub2(lo02, b1024), d2, m2));
    o[1] = h2u(__hfma2(__hsub2(lo13, b1024), d2, m2));
    o[2] = h2u(__hfma2(__hsub2(hi02, b64), d2, m2));
    o[3] = h2u(__hfma2(__hsub2(hi13, b64), d2, m2));
  } else {
    const __half2 b1032 = __float2half2_rn(1032.f), b72 = __float2half2_rn(72.f);
    o[0] = h2u(__hmul2(__hsub2(lo02, b1032), d2));
    o[1] = h2u(__hmul2(__hsub2(lo13, b1032), d2));
    o[2] = h2u(__hmul2(__hsub2(hi02, b72), d2));
    o[3] = h2u(__hmul2(__hsub2(hi13, b72), d2));
  }
}

// Q4_1: the thread's block H (20 bytes at byte 20H of the 80-byte row segment), read as
// the two 16-byte words that cover it.
template <int H>
__device__ __forceinline__ void convert_q41(const uint8_t* row, uint32_t (&o)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(row) + H;
  const uint4 a = p[0], b = p[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const __half2 dmh = u2h(w[H]);  // block H starts at word 5H = 4H + H
  const __half2 d2 = __low2half2(dmh), m2 = __high2half2(dmh);
  dequant4<3>(w[H + 1], d2, m2, o + 0);
  dequant4<3>(w[H + 2], d2, m2, o + 4);
  dequant4<3>(w[H + 3], d2, m2, o + 8);
  dequant4<3>(w[H + 4], d2, m2, o + 12);
}

// Q4_0: the thread's blocks 2P and 2P + 1 (18 bytes each) of the 144-byte row segment.
template <int P>
__device__ __forceinline__ void convert_q40(const uint8_t* row, uint32_t (&o)[32]) {
  constexpr int byte0 = 36 * P;
  constexpr int u0 = byte0 >> 4;
  const uint4* q = reinterpret_cast<const uint4*>(row) + u0;
  const uint4 a = q[0], b = q[1], c = q[2];
  const uint32_t w[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const int off = byte0 + 18 * blk - 16 * u0;  // byte offset of the block in w (even)
    const int wi = off >> 2;
    uint32_t dw, q0, q1, q2, q3;
    if (off & 2) {  // d in the high half of w[wi]; nibble words aligned from w[wi + 1]
      dw = w[wi] >> 16;
      q0 = w[wi + 1];
      q1 = w[wi + 2];
      q2 = w[wi + 3];
      q3 = w[wi + 4];
    } else {  // d in the low half; each nibble word straddles two words
      dw = w[wi] & 0xFFFFu;
      q0 = __byte_perm(w[wi], w[wi + 1], 0x5432);
      q1 = __byte_perm(w[wi + 1], w[wi + 2], 0x5432);
      q2 = __byte_perm(w[wi + 2], w[wi + 3], 0x5432);
      q3 = __byte_perm(w[wi + 3], w[wi + 4], 0x5432);
    }
    const __half2 d2 = u2h(dw | (dw << 16));
    dequant4<2>(q0, d2, d2, o + 16 * blk + 0);
    dequant4<2>(q1, d2, d2, o + 16 * blk + 4);
    dequant4<2>(q2, d2, d2, o + 16 * blk + 8);
    dequant4<2>(q3, d2, d2, o + 16 * blk + 12);
  }
}

// Q4_K super-block (144 bytes: f16 d and dmin, 12 packed 6-bit scale and min bytes, then
// four runs of 32 bytes; run c holds sub-block 2c in its low nibbles and 2c + 1 in its high
// nibbles, value i of each in byte i). Sub-block s takes scale sc and min mn (s < 4: the low
// six bits of bytes s and s + 4; s >= 4: the nibbles of byte s + 4 with the top two bits of
// bytes s - 4 and s); value = d sc q - dmin mn. Here d sc and -dmin mn are rounded to f16 and
// the value is one f16 fused multiply-add of the exact nibble, as for a Q4_1 block.
__device__ __forceinline__ void q4k_scale(const uint4& hd, int s, __half2& d2, __half2& m2) {
  const int i0 = s < 4 ? s : s + 4, i1 = s < 4 ? s + 4 : s - 4, i2 = s;  // bytes read
  auto byte = [&](int i) -> uint32_t {
    const uint32_t w = i < 4 ? hd.y : (i < 8 ? hd.z : hd.w);
    return (w >> (8 * (i & 3))) & 0xFFu;
  };
  uint32_t sc, mn;
  if (s < 4) {
    sc = byte(i0) & 63u;
    mn = byte(i1) & 63u;
  } else {
    sc = (byte(i0) & 15u) | ((byte(i1) >> 6) << 4);
    mn = (byte(i0) >> 4) | ((byte(i2) >> 6) << 4);
  }
  const float2 f = __half22float2(u2h(hd.x));
  d2 = __float2half2_rn(f.x * (float)sc);
  m2 = __float2half2_rn(-(f.y * (float)mn));
}

// A unit J (sub-blocks 4J .. 4J + 3, 128 values) of the thread's Q4_K row segment -> TMEM
// columns col .. col + 63. Each sub-block's nibbles are regrouped into the Q4_1 block order
// (values 4w .. 4w + 3 in the low and 16 + 4w .. in the high nibbles of word w) first.
__device__ __forceinline__ void convert_q4k(const uint8_t* row, int J, uint32_t col) {
  const uint4 hd = *reinterpret_cast<const uint4*>(row);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4* run = reinterpret_cast<const uint4*>(row + 16 + 32 * (2 * J + h));
    const uint4 ra = run[0], rb = run[1];
    const uint32_t R[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      __half2 d2, m2;
      q4k_scale(hd, 4 * J + 2 * h + hi, d2, m2);
      uint32_t o[16];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t qw = ((R[w] >> (4 * hi)) & 0x0F0F0F0Fu) | (((R[w + 4] >> (4 * hi)) & 0x0F0F0F0Fu) << 4);
        dequant4<3>(qw, d2, m2, o + 4 * w);
      }
      tmem_st16(col + 16u * (2 * h + hi), o);
    }
  }
}

// N words of shared memory from an address on a 2-byte bound: aligned words, funnel-shifted.
// Reads one word past the N (the callers' stages are followed by more shared memory).
template <int N>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t (&o)[N]) {
  const uintptr_t u = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(u & ~uintptr_t(3));
  const uint32_t sh = (uint32_t)(u & 3u) * 8u;
  uint32_t t[N + 1];
#pragma unroll
  for (int i = 0; i <= N; ++i) t[i] = w[i];
#pragma unroll
  for (int i = 0; i < N; ++i) o[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

// Q6_K super-block (210 bytes: ql[128], qh[64], 16 int8 scales, f16 d) in two halves of 128
// values; sub-block r of half n, value i: the nibble (low for r < 2) of ql[64n + 32 (r % 2) + i]
// with bits 2r, 2r + 1 of qh[32n + i] above it, scale[8n + 2r + i / 16]; value = d scale (q - 32).
// A unit J is half J % 2 of super-block J / 2 -> TMEM columns col .. col + 63. The 6-bit q
// enters an f16 mantissa (1024 + q), 1056 is subtracted exactly, one f16 multiply by the
// f16-rounded d scale follows.
__device__ __forceinline__ void convert_q6k(const uint8_t* row, int J, uint32_t col) {
  const uint8_t* sb = row + 210 * (J >> 1);
  const int n = J & 1;
  uint32_t ql[16], qh[8], sc[2], dw[1];
  lds_words(sb + 64 * n, ql);
  lds_words(sb + 128 + 32 * n, qh);
  lds_words(sb + 192 + 8 * n, sc);
  lds_words(sb + 208, dw);
  const float d = __half2float(__ushort_as_half((unsigned short)(dw[0] & 0xFFFFu)));
  const __half2 b1056 = __float2half2_rn(1056.f);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t scw = sc[r >> 1] >> (16 * (r & 1));
    const __half2 d0 = __float2half2_rn(d * (float)(int)(int8_t)(scw & 0xFFu));
    const __half2 d1 = __float2half2_rn(d * (float)(int)(int8_t)((scw >> 8) & 0xFFu));
    const int ls = 4 * (r >> 1), hs = 2 * r, qo = 8 * (r & 1);
    uint32_t o[16];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t ulo = ((ql[qo + w] >> ls) & 0x0F0F0F0Fu) | (((qh[w] >> hs) & 0x03030303u) << 4);
      const uint32_t uhi = ((ql[qo + 4 + w] >> ls) & 0x0F0F0F0Fu) | (((qh[4 + w] >> hs) & 0x03030303u) << 4);
      o[4 * w + 0] = h2u(__hmul2(__hsub2(u2h((ulo & 0x00FF00FFu) | 0x64006400u), b1056), d0));
      o[4 * w + 1] = h2u(__hmul2(__hsub2(u2h(((ulo >> 8) & 0x00FF00FFu) | 0x64006400u), b1056), d0));
      o[4 * w + 2] = h2u(__hmul2(__hsub2(u2h((uhi & 0x00FF00FFu) | 0x64006400u), b1056), d1));
      o[4 * w + 3] = h2u(__hmul2(__hsub2(u2h(((uhi >> 8) & 0x00FF00FFu) | 0x64006400u), b1056), d1));
    }
    tmem_st16(col + 16u * r, o);
  }
}

// Router rows: the 32 f32 values of sub-box H of a row (values 32H .. 32H + 31 of the
// 128-value chunk; the sub-box is stored with the 128-byte swizzle: 16-byte chunk j of
// row r sits at chunk j ^ (r & 7)) -> f16 hi or lo parts in the permuted slot order.
__device__ __forceinline__ void convert_f32(const uint8_t* sub, int r, bool lo, uint32_t (&o)[16]) {
  const uint8_t* rowp = sub + r * 128;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 x0 = *reinterpret_cast<const float4*>(rowp + ((w ^ (r & 7)) << 4));
    const float4 x1 = *reinterpret_cast<const float4*>(rowp + (((4 + w) ^ (r & 7)) << 4));
    uint32_t* d = o + 4 * w;
    const uint32_t h0 = pack_h2(x0.x, x0.z), h1 = pack_h2(x0.y, x0.w);
    const uint32_t h2 = pack_h2(x1.x, x1.z), h3 = pack_h2(x1.y, x1.w);
    if (lo) {
      d[0] = pack_lo(x0.x, x0.z, h0);
      d[1] = pack_lo(x0.y, x0.w, h1);
      d[2] = pack_lo(x1.x, x1.z, h2);
      d[3] = pack_lo(x1.y, x1.w, h3);
    } else {
      d[0] = h0;
      d[1] = h1;
      d[2] = h2;
      d[3] = h3;
    }
  }
}

// ---- tensor maps of the weight matrices ------------------------------------------------------
// The expert records are viewed as 2-D byte arrays: with rows of a gate/up row's bytes
// (each record is 3F such rows: gate, up, then the down matrix) and with rows of a down
// row's bytes (each record is 3H such rows, the down matrix from row 2H). The router is
// an E x H f32 array read in 32-value sub-boxes with the 128-byte swizzle.
struct TileMaps {
  CUtensorMap gu, gu_s, dn, dn_s, rt;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The same from a 3-D map (K-quant records: x = byte of the row, y = row of the record's
// gate/up or down rows, z = expert).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ---- work units ----------------------------------------------------------------------------
struct TileUnit {
  const CUtensorMap* map;  // weight rows
  int y0, y1;              // first map row of the tile (gate/up: gate rows, up rows)
  int z;                   // K-quant maps: the expert (0 for the shared expert)
  const uint8_t* src;      // Q6_K down: the tile's first row (128 whole rows, one bulk copy)
  int rbs;                 // Q6_K down: bytes per row
  const uint8_t* b;        // token-operand image of the chunk (first 128-value block)
  int nk;                  // raw chunks (the last one may hold fewer than NAU A units)
  int kdim;                // reduction length
  int n, npad, nb;         // chunk tokens, rounded to 16, operand rows (hi + lo: 2 npad)
  int row0, prow, mt;      // chunk's first row, padded-row offset, M tile
  bool shared;             // shared expert (token chunk)
  int e0;                  // router: first expert of the tile
  int k0, ks;              // router: the K slice's first 128-value unit, the slice
};

template <int MODE, int QT>
__device__ __forceinline__ int tile_units(const PrefillArgs& a) {
  const int ntok = (a.T + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX;
  if (MODE == 2) return ntok * ((a.E + 63) / 64) * a.rt_slices;
  const int nr = (int)a.nchunks[0];
  const int nsh = a.Fs ? ntok : 0;
  const int mt_r = MODE == 0 ? a.F / 64 : a.H / 128;
  const int mt_s = MODE == 0 ? a.Fs / 64 : a.H / 128;
  return nr * mt_r + nsh * mt_s;
}

template <int MODE, int QT>
__device__ __forceinline__ TileUnit tile_unit(const PrefillArgs& a, const TileMaps& maps, int u) {
  using G = Geo<MODE, QT>;
  TileUnit t;
  const int nkh = a.H / TP_KB;
  if (MODE == 2) {
    // unit u: K slice u % slices of tile u / slices (token chunk j, experts 64 e ...)
    const int et = (a.E + 63) / 64;
    t.ks = u % a.rt_slices;
    u /= a.rt_slices;
    const int j = u / et, e = u % et;
    t.e0 = 64 * e;
    t.k0 = t.ks * a.rt_ups;
    t.map = &maps.rt;
    t.y0 = t.y1 = t.e0;
    t.row0 = j * PREFILL_TILE_NMAX;
    t.n = min(PREFILL_TILE_NMAX, a.T - t.row0);
    t.npad = (t.n + 15) & ~15;
    t.nb = 2 * t.npad;
    t.prow = t.row0;
    t.nk = min(a.rt_ups, nkh - t.k0);  // KR = 128: one raw chunk per A unit
    t.kdim = t.nk * TP_KB;
    t.b = a.ximg + (size_t)2 * t.prow * nkh * 256 + (size_t)t.k0 * t.nb * 256;
    t.mt = 0;
    t.shared = false;
    return t;
  }
  const int nr = (int)a.nchunks[0];
  const int mt_r = MODE == 0 ? a.F / 64 : a.H / 128;
  const int mt_s = MODE == 0 ? a.Fs / 64 : a.H / 128;
  int slot, mt;
  if (u < nr * mt_r) {
    const GemmChunk ch = a.chunks[u / mt_r];
    mt = u % mt_r;
    slot = ch.slot;
    t.row0 = ch.row0;
    t.n = ch.n;
    t.prow = ch.prow;
    t.shared = false;
  } else {
    const int v = u - nr * mt_r;
    const int j = v / mt_s;
    mt = v % mt_s;
    slot = 0;
    t.row0 = j * PREFILL_TILE_NMAX;
    t.n = min(PREFILL_TILE_NMAX, a.T - t.row0);
    t.prow = t.row0;
    t.shared = true;
  }
  t.mt = mt;
  t.e0 = 0;
  t.npad = (t.n + 15) & ~15;
  const int ff = t.shared ? a.Fs : a.F;
  constexpr bool KQ = QT == 12 || QT == 14;
  t.z = t.shared ? 0 : slot;
  t.src = nullptr;
  t.rbs = 0;
  if (MODE == 0) {
    t.map = t.shared ? &maps.gu_s : &maps.gu;
    t.y0 = KQ ? 64 * mt : slot * 3 * ff + 64 * mt;  // gate rows
    t.y1 = t.y0 + ff;                                // up rows
    t.nb = 2 * t.npad;
    t.nk = (a.H + G::KR - 1) / G::KR;
    t.kdim = a.H;
    const uint8_t* img = t.shared ? a.ximg : a.ximg_routed;
    t.b = img + (size_t)2 * t.prow * nkh * 256;
  } else {
    t.map = t.shared ? &maps.dn_s : &maps.dn;
    t.y0 = t.y1 = KQ ? 128 * mt : slot * 3 * a.H + 2 * a.H + 128 * mt;
    if (QT == 14) {  // the expert's down matrix follows its 2 ff gate/up rows
      t.rbs = (int)(t.shared ? a.rb_fs : a.rb_f);
      const uint8_t* rec = t.shared ? a.shared : a.experts + (size_t)slot * a.rec_bytes;
      t.src = rec + (size_t)2 * ff * a.rb_h + (size_t)128 * mt * t.rbs;
    }
    t.nb = t.npad;
    t.nk = (ff + G::KR - 1) / G::KR;
    t.kdim = ff;
    const uint8_t* img = t.shared ? a.aimg_s : a.aimg;
    t.b = img + (size_t)t.prow * (ff / TP_KB) * 256;
  }
  return t;
}

// First TMEM column of accumulator ab: the down tiles' two 64-column accumulators share
// [0, 128); the router and gate/up tiles take [0, 128) and [384, 512).
template <int MODE>
__device__ __forceinline__ uint32_t acc_col(int ab) {
  return MODE == 1 ? 64u * (uint32_t)ab : (ab ? TP_ACC1_COL : 0u);
}

// Independent accumulators of a tile: as many nb-column chains as fit in the tile's
// accumulator columns (128; down tiles: 64 each of two), at most 4.
template <int MODE>
__device__ __forceinline__ int tile_chains(int nb) {
  const int cols = MODE == 1 ? 64 : 128;
  return nb * 4 <= cols ? 4 : (nb * 2 <= cols ? 2 : 1);
}

// A tile whose A units the two MMA issuers share (unit n to issuer n % 2): it has at least two
// accumulation chains and two A units. Every role derives the owner of a unit from this.
template <int MODE>
__device__ __forceinline__ bool tile_split(const TileUnit& t) {
  return tile_chains<MODE>(t.nb) >= 2 && t.kdim / TP_KB >= 2;
}

// Sum over the tile's chains of 8 accumulator columns starting at column c.
template <int MODE>
__device__ __forceinline__ void acc_ld8(uint32_t acc, int nb, int c, float (&v)[8]) {
  const int nch = tile_chains<MODE>(nb);
  uint32_t r[8];
  tmem_ld8(acc + (uint32_t)c, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
  for (int ch = 1; ch < nch; ++ch) {
    tmem_ld8(acc + (uint32_t)(ch * nb + c), r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] += __uint_as_float(r[i]);
  }
}

// ---- the persistent tile kernel -----------------------------------------------------------
template <int MODE, int QT>
__global__ void __launch_bounds__(TP_THREADS, 1) tile_gemm(const PrefillArgs a, const __grid_constant__ TileMaps maps) {
  using G = Geo<MODE, QT>;
  extern __shared__ __align__(1024) uint8_t tsm_dyn[];
  // stages start on a 1024-byte boundary (the router's swizzled boxes need it)
  uint8_t* raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tsm_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* bring = raw + G::RAW_BYTES;                                      // [NSB][B_STAGE]
  float* scratch = reinterpret_cast<float*>(bring + G::NSB * TP_B_STAGE);  // gate/up and router epilogues
  __shared__ __align__(8) uint64_t raw_full[G::NSA], raw_empty[G::NSA];
  // a_full and b_full have one barrier per owning MMA issuer: an issuer skips the other's
  // units, and a parity wait must never fall two phases behind the barrier it waits on
  __shared__ __align__(8) uint64_t a_full[TP_GROUPS][2], a_empty[TP_GROUPS], b_full[G::NSB][2], b_empty[G::NSB];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin, scr_full, scr_empty;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  volatile int* abrt = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < G::NSA; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], TP_CONV_WARPS);  // every converter warp releases every chunk
    }
    for (int i = 0; i < TP_GROUPS; ++i) {
      mbar_init(&a_full[i][0], 4);  // the group's four warps
      mbar_init(&a_full[i][1], 4);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < G::NSB; ++i) {
      mbar_init(&b_full[i][0], 1);
      mbar_init(&b_full[i][1], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 2);  // both issuers commit every tile
      mbar_init(&acc_empty[i], TP_EPI_WARPS);
    }
    mbar_init(&fin, 2);
    mbar_init(&scr_full, TP_EPI_WARPS / 2);   // epilogue warps of lanes 64..127
    mbar_init(&scr_empty, TP_EPI_WARPS / 2);  // epilogue warps of lanes 0..63
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base, TP_TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int units = tile_units<MODE, QT>(a);

  if (warp == 0) {
    // ------------------------------ weight producer ------------------------------
    // weight rows stream through L2 once; router rows are read by every token chunk
    const uint64_t pol_w = MODE == 2 ? policy_evict_last() : policy_evict_first();
    uint32_t ka = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const TileUnit t = tile_unit<MODE, QT>(a, maps, u);
      for (int kc = 0; kc < t.nk && ok; ++kc, ++ka) {
        const int sa = (int)(ka % G::NSA);
        if (ka >= (uint32_t)G::NSA && !tp_wait_warp(&raw_empty[sa], ((ka / G::NSA) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* dst = raw + sa * G::STAGE;
          mbar_arrive_expect_tx(&raw_full[sa], QT == 14 ? (uint32_t)(128 * t.rbs) : (uint32_t)G::STAGE);
          if (MODE == 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(dst + j * 8192, t.map, (t.k0 + kc) * 128 + 32 * j, t.y0, &raw_full[sa], pol_w);
          } else if (QT == 14) {  // 128 whole down rows: one contiguous span of 128 rbs bytes
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
                    smem_addr(dst)),
                "l"(t.src), "r"((uint32_t)(128 * t.rbs)), "r"(smem_addr(&raw_full[sa])), "l"(pol_w)
                : "memory");
          } else if (QT == 12) {  // K-quant records through 3-D maps (x byte, y row, z expert)
            tma_load_3d(dst, t.map, kc * G::SEG, t.y0, t.z, &raw_full[sa], pol_w);
            if (MODE == 0) tma_load_3d(dst + 64 * G::SEG, t.map, kc * G::SEG, t.y1, t.z, &raw_full[sa], pol_w);
          } else if (MODE == 0) {
            tma_load_2d(dst, t.map, kc * G::SEG, t.y0, &raw_full[sa], pol_w);
            tma_load_2d(dst + 64 * G::SEG, t.map, kc * G::SEG, t.y1, &raw_full[sa], pol_w);
          } else {
            tma_load_2d(dst, t.map, kc * G::SEG, t.y0, &raw_full[sa], pol_w);
          }
        }
        __syncwarp();
      }
    }
    // every copy this warp issued has landed before the CTA may exit (this matters only
    // when a timed-out wait stopped the consumers early)
    if (lane == 0) {
      for (int sa = 0; sa < G::NSA; ++sa) {
        const uint32_t f = ka > (uint32_t)sa ? (ka - sa - 1) / G::NSA + 1 : 0u;  // fills of this stage
        if (f) mbar_wait(&raw_full[sa], (f - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------ token-operand producer ------------------------------
    uint32_t rb = 0;
    // bit 2 sb + o: (stage sb, issuer o) filled at least once / its fill count is odd
    uint32_t filled = 0, fodd = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const TileUnit t = tile_unit<MODE, QT>(a, maps, u);
      const uint32_t bbytes = (uint32_t)t.nb * 256u;
      const bool split = tile_split<MODE>(t);
      for (int kk = 0; kk < t.kdim / TP_KB; ++kk) {  // one stage per 128-value A unit
        const int sb = (int)(rb % G::NSB);
        const int own = split ? (int)(rb & 1u) : 0;
        // with as many token stages as A slots, unit n's stage and slot have the same index and
        // one commit (on a_empty) releases both
        constexpr bool kOneRelease = G::NSB == TP_GROUPS;
        if (rb >= (uint32_t)G::NSB &&
            !tp_wait_warp(kOneRelease ? &a_empty[sb] : &b_empty[sb], ((rb / G::NSB) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&b_full[sb][own], bbytes);
          const uint8_t* src = t.b + (size_t)kk * bbytes;
          asm volatile(
              "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  smem_addr(bring + sb * TP_B_STAGE)),
              "l"(src), "r"(bbytes), "r"(smem_addr(&b_full[sb][own]))
              : "memory");
        }
        __syncwarp();
        filled |= 1u << (2 * sb + own);
        fodd ^= 1u << (2 * sb + own);
        ++rb;
      }
    }
    if (lane == 0) {
      for (int sb = 0; sb < G::NSB; ++sb)
        for (int o = 0; o < 2; ++o)  // the last fill's phase parity is (count - 1) & 1
          if ((filled >> (2 * sb + o)) & 1u) mbar_wait(&b_full[sb][o], ((fodd >> (2 * sb + o)) & 1u) ^ 1u);
    }
    __syncwarp();
  } else if (warp == 1 || warp == TP_MMA_WARP2) {
    // ------------------------------ MMA issuers ------------------------------
    // Both issuers walk every tile and A unit in order (so their unit, stage and parity
    // counts agree) and issue the units they own. A tile with at least two chains and two
    // A units is split: unit n goes to issuer n % 2, and each issuer accumulates into its
    // own chains only (four chains: chains iss and 2 + iss; two: chain iss), so every chain
    // receives its MMAs from one thread in a fixed order. Other tiles go to issuer 0 alone.
    const int iss = warp == 1 ? 0 : 1;
    if (lane == 0) {
      uint32_t n = 0, rb = 0, uc = 0;
      // bit g / sb: parity of this issuer's next wait on a_full[g][iss] / b_full[sb][iss]
      uint32_t pa = 0, pb = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
        const TileUnit t = tile_unit<MODE, QT>(a, maps, u);
        const uint32_t idesc = idesc_f16_f32(128, t.nb);
        const int nch = tile_chains<MODE>(t.nb);
        const int nku = t.kdim / TP_KB;  // A units of the tile
        const bool split = tile_split<MODE>(t);
        const int ab = (int)(uc % G::NACC);
        const uint32_t acc = tmem + acc_col<MODE>(ab);  // accumulator columns
        if (uc >= (uint32_t)G::NACC && !tp_wait(&acc_empty[ab], ((uc / G::NACC) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        bool fresh = true;  // no MMA of this issuer in this tile yet
        for (int kk = 0; kk < nku && ok; ++kk, ++n, ++rb) {  // A units in order
          if ((split ? (int)(n & 1u) : 0) != iss) continue;
          const int g = (int)(n % TP_GROUPS);  // A unit n was converted by group n % 3
          if (!tp_wait(&a_full[g][iss], (pa >> g) & 1u, abrt)) {
            ok = false;
            break;
          }
          pa ^= 1u << g;
          const int sb = (int)(rb % G::NSB);
          if (!tp_wait(&b_full[sb][iss], (pb >> sb) & 1u, abrt)) {
            ok = false;
            break;
          }
          pb ^= 1u << sb;
          tc_fence_after_sync();
          const uint8_t* B = bring + sb * TP_B_STAGE;
          const uint32_t ta0 = tmem + TP_A_COL + 64u * g;  // the group's A slot
          // B descriptor of K step j: the stage's, its start address (in 16-byte units, bits
          // 0-13; a stage ends below 228 KB, so the field does not carry) advanced 2 j nb units
          const uint64_t bd0 = smem_desc(B, 16u * t.nb, 128);
#pragma unroll
          for (int j = 0; j < TP_KB / 16; ++j) {
            // narrow tiles keep several independent accumulation chains in flight instead of
            // one latency-bound chain; the first MMA into a chain in the tile overwrites it
            int ch;
            bool accum;
            if (!split) {
              ch = j & (nch - 1);
              accum = kk > 0 || j >= nch;
            } else if (nch == 4) {
              ch = 2 * (j & 1) + iss;
              accum = !fresh || j >= 2;
            } else {
              ch = iss;
              accum = !fresh || j >= 1;
            }
            mma_f16_ta(acc + (uint32_t)(ch * t.nb), ta0 + 8u * j, bd0 + (uint64_t)(2 * j * t.nb), idesc, accum);
          }
          fresh = false;
          if constexpr (G::NSB != TP_GROUPS) mma_commit(&b_empty[sb]);  // else sb == g: a_empty releases both
          mma_commit(&a_empty[g]);
        }
        if (ok) mma_commit(&acc_full[ab]);  // arrives once this issuer's MMAs are done
      }
      // every MMA issued has completed before the columns are freed: this wait ignores the
      // abort flag (MMAs in flight complete by themselves; freeing TMEM under them would not)
      mma_commit(&fin);
      mbar_wait(&fin, 0);
    }
    __syncwarp();
  } else if (warp < TP_EPI_WARP0) {
    // ------------------------------ converters ------------------------------
    const int q = warp & 3, grp = (warp - 3) >> 2;  // lane quarter, converter group
    const int m = 32 * q + lane;                     // TMEM lane = tile row
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t ka = 0, n = 0, uc = 0;  // raw chunks, A units and tiles so far
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const TileUnit t = tile_unit<MODE, QT>(a, maps, u);
      const bool split = tile_split<MODE>(t);  // unit nj then goes to MMA issuer nj % 2
      for (int kc = 0; kc < t.nk; ++kc, ++ka) {
        // every warp waits for every chunk and releases it: a warp can then never release
        // a stage's next use before its current one has landed
        const int sa = (int)(ka % G::NSA);
        if (!tp_wait_warp(&raw_full[sa], (ka / G::NSA) & 1u, abrt)) {
          ok = false;
          break;
        }
        const uint8_t* stage = raw + sa * G::STAGE;
        const int nau = min(G::NAU, (t.kdim - kc * G::KR) / TP_KB);
        const uint32_t col = tmem + lane_addr + TP_A_COL + 64u * grp;  // the group's A slot
        for (int j = 0; j < nau; ++j) {
          const uint32_t nj = n + j;  // A unit nj goes to group nj % 4
          if ((int)(nj % TP_GROUPS) != grp) continue;
          const uint32_t i = nj / TP_GROUPS;  // the group's own A unit count
          if (i >= 1 && !tp_wait_warp(&a_empty[grp], (i - 1) & 1u, abrt)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (MODE == 2) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              uint32_t o[16];
              convert_f32(stage + jj * 8192, m & 63, m >= 64, o);
              tmem_st16(col + 16u * jj, o);
            }
          } else if (QT == 12) {
            convert_q4k(stage + m * G::SEG, j, col);
          } else if (QT == 14) {
            convert_q6k(stage + m * t.rbs, j, col);
          } else if (QT == 3) {
            const uint8_t* row = stage + m * G::SEG + 80 * j;  // blocks 4j .. 4j + 3
            uint32_t o[16];
            convert_q41<0>(row, o);
            tmem_st16(col + 0u, o);
            convert_q41<1>(row, o);
            tmem_st16(col + 16u, o);
            convert_q41<2>(row, o);
            tmem_st16(col + 32u, o);
            convert_q41<3>(row, o);
            tmem_st16(col + 48u, o);
          } else {
            const uint8_t* row = stage + m * G::SEG;
            uint32_t o[32];
            if (j == 0) {
              convert_q40<0>(row, o);
              tmem_st32(col + 0u, o);
              convert_q40<1>(row, o);
              tmem_st32(col + 32u, o);
            } else {
              convert_q40<2>(row, o);
              tmem_st32(col + 0u, o);
              convert_q40<3>(row, o);
              tmem_st32(col + 32u, o);
            }
          }
          tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[grp][split ? (int)(nj & 1u) : 0]);
        }
        if (!ok) break;
        n += nau;
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[sa]);
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    // one warp per lane quarter, every column of the tile; the MMAs of the next tile run
    // on the other accumulator meanwhile
    const int q = warp & 3;
    const int m = 32 * q + lane;  // TMEM lane = tile row
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const TileUnit t = tile_unit<MODE, QT>(a, maps, u);
      // ---- the tile on accumulator ab ----
      const int ab = (int)(uc % G::NACC);
      const uint32_t acc = tmem + lane_addr + acc_col<MODE>(ab);
      if (!tp_wait_warp(&acc_full[ab], (uc / G::NACC) & 1u, abrt)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int half = t.npad;  // every column
      const int c_lo = 0;
      if (MODE == 2 || MODE == 0) {
        // lanes 64..127 (router: lo rows; gate/up: up rows) hand their column sums over
        if (m >= 64) {
          if (uc > 0 && !tp_wait_warp(&scr_empty, (uc - 1) & 1u, abrt)) {
            ok = false;
            break;
          }
          for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
            float v0[8], v1[8];
            acc_ld8<MODE>(acc, t.nb, c0, v0);
            acc_ld8<MODE>(acc, t.nb, t.npad + c0, v1);
#pragma unroll
            for (int i = 0; i < 8; ++i) scratch[(m - 64) * 65 + c0 + i] = v0[i] + v1[i];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&scr_full);
        } else {
          if (!tp_wait_warp(&scr_full, uc & 1u, abrt)) {
            ok = false;
            break;
          }
          const int ff = t.shared ? a.Fs : a.F;
          const int nkf = ff / TP_KB;
          const int f0 = 64 * t.mt + 32 * q;  // the warp's 32 gate rows: one 32-value block
          uint8_t* img = MODE == 0 ? (t.shared ? a.aimg_s : a.aimg) : nullptr;
          uint8_t* ibase =
              MODE == 0 ? img + ((size_t)t.prow * nkf + (size_t)(f0 / TP_KB) * t.npad) * 256 : nullptr;
          const int kcore = ((f0 & (TP_KB - 1)) >> 3) + (lane & 3);  // piece written by lanes 0..3
          for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
            float v0[8], v1[8];
            acc_ld8<MODE>(acc, t.nb, c0, v0);
            acc_ld8<MODE>(acc, t.nb, t.npad + c0, v1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c = c0 + i;
              const float v = v0[i] + v1[i];
              const float other = scratch[m * 65 + c];
              if (MODE == 2) {
                if (c < t.n && t.e0 + m < a.E)
                  a.logits[((size_t)t.ks * a.T + t.row0 + c) * a.E + t.e0 + m] = v + other;
              } else {
                // act = silu(gate) * up (clamped) for f = f0 + lane, gathered into the four 16-byte
                // pieces of the block (slot 8w + k holds value 4w + {0,2,1,3}[k], +16 for k >= 4)
                const float act = swiglu_act(v, other, t.shared ? a.lim_s : a.lim);
                const uint32_t hv = (uint32_t)__half_as_ushort(__float2half_rn(act));
                const int w = lane & 3;
                uint32_t pk[4];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                  const int ka2 = 2 * k2, kb2 = 2 * k2 + 1;
                  const int ea = (ka2 < 4 ? 0 : 16) + 4 * w + ((ka2 & 3) == 1 ? 2 : ((ka2 & 3) == 2 ? 1 : (ka2 & 3)));
                  const int eb = (kb2 < 4 ? 0 : 16) + 4 * w + ((kb2 & 3) == 1 ? 2 : ((kb2 & 3) == 2 ? 1 : (kb2 & 3)));
                  const uint32_t va = __shfl_sync(0xffffffffu, hv, ea);
                  const uint32_t vb = __shfl_sync(0xffffffffu, hv, eb);
                  pk[k2] = va | (vb << 16);
                }
                if (lane < 4 && c < t.n)
                  *reinterpret_cast<uint4*>(ibase + (kcore * (t.npad >> 3) + (c >> 3)) * 128 + (c & 7) * 16) =
                      make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&scr_empty);
        }
      } else {
        const int hrow = 128 * t.mt + m;
        for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
          float v0[8];
          acc_ld8<MODE>(acc, t.nb, c0, v0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + i;
            if (c < t.n) {
              const float y = v0[i];
              if (t.shared) a.sbuf[(size_t)(t.row0 + c) * a.H + hrow] = y;
              else a.ybuf[(size_t)(t.row0 + c) * a.H + hrow] = a.wsorted[t.row0 + c] * y;
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  __syncthreads();
  if (tid == 0 && *abrt) atomicOr(a.status, DEV_ERR_MBAR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TP_TMEM_COLS);
  }
}

// ---- token-operand images ------------------------------------------------------------------
// x rows of each chunk as f16 hi and lo parts, tiled as the MMA's B operand. Grid (chunk, row
// group slice, K slice): CTA (c, y, z) takes the chunk's 8-row groups y, y + gridDim.y, ...
// (token chunks, or routed chunks when `routed`), warp w the 128-value K blocks w + 8 m with
// m = z modulo gridDim.z of each, two blocks a round with all their loads issued before the
// first store. Lane (q = lane / 8, r = lane % 8) takes row r of the group and pieces q, q + 4,
// q + 8, q + 12 of the block (a piece: 8 values, one 16-byte core-matrix row), so the eight
// lanes of a piece write one whole 128-byte core matrix with each store.
__global__ void __launch_bounds__(256) tile_images(const PrefillArgs a, int routed) {
  const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane & 7, q = lane >> 3;
  int n, row0, prow;
  uint8_t* base;
  const int nkh = a.H / TP_KB;
  if (routed) {
    if (c >= (int)a.nchunks[0]) return;
    const GemmChunk ch = a.chunks[c];
    n = ch.n;
    row0 = ch.row0;
    prow = ch.prow;
    base = a.ximg_routed;
  } else {
    row0 = c * PREFILL_TILE_NMAX;
    if (row0 >= a.T) return;
    n = min(PREFILL_TILE_NMAX, a.T - row0);
    prow = row0;
    base = a.ximg;
  }
  const int npad = (n + 15) & ~15, nb = 2 * npad;
  base += (size_t)2 * prow * nkh * 256;
  for (int g = blockIdx.y; 8 * g < n; g += gridDim.y) {
    const int row = 8 * g + r;
    const bool valid = row < n;
    const int tok = !valid ? 0 : routed ? (int)(a.perm[row0 + row] / (uint32_t)a.K) : row0 + row;
    const float* xrow = a.x + (size_t)tok * a.H;
    const int rl = npad + row;  // the lo part's row
    const uint32_t hi_off = (uint32_t)((row >> 3) * 128 + (row & 7) * 16), lo_off = (uint32_t)((rl >> 3) * 128 + (rl & 7) * 16);
    // K blocks warp + 8 m with m = z (mod Z), Z = gridDim.z; two (m0, m0 + Z) a round, all
    // their loads issued before any store
    const int Z = (int)gridDim.z;
    for (int m0 = (int)blockIdx.z; warp + 8 * m0 < nkh; m0 += 2 * Z) {
      float4 x0[2][4], x1[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = warp + 8 * (m0 + h * Z);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int gs = kk * TP_KB + 8 * (q + 4 * u);  // first slot of the piece
          const float4* xr = reinterpret_cast<const float4*>(xrow + 32 * (gs >> 5));
          if (valid && kk < nkh) {
            x0[h][u] = __ldg(xr + ((gs & 31) >> 3));
            x1[h][u] = __ldg(xr + 4 + ((gs & 31) >> 3));
          }
        }
      }
      if (valid) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kk = warp + 8 * (m0 + h * Z);
          if (kk >= nkh) break;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int kc8 = q + 4 * u;
            uint4 hi, lo;
            hi.x = pack_h2(x0[h][u].x, x0[h][u].z);
            hi.y = pack_h2(x0[h][u].y, x0[h][u].w);
            hi.z = pack_h2(x1[h][u].x, x1[h][u].z);
            hi.w = pack_h2(x1[h][u].y, x1[h][u].w);
            lo.x = pack_lo(x0[h][u].x, x0[h][u].z, hi.x);
            lo.y = pack_lo(x0[h][u].y, x0[h][u].w, hi.y);
            lo.z = pack_lo(x1[h][u].x, x1[h][u].z, hi.z);
            lo.w = pack_lo(x1[h][u].y, x1[h][u].w, hi.w);
            uint8_t* blk = base + (size_t)kk * nb * 256 + (size_t)kc8 * (nb >> 3) * 128;
            *reinterpret_cast<uint4*>(blk + hi_off) = hi;
            *reinterpret_cast<uint4*>(blk + lo_off) = lo;
          }
        }
      }
    }
  }
}

// ---- host side -----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over `rows` rows of `row_bytes` bytes (u8 elements) or f32 elements.
cudaError_t encode_2d(CUtensorMap* m, const void* base, bool f32, uint64_t inner, uint64_t rows, uint32_t box_x,
                      uint32_t box_y, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (f32 ? 4 : 1)};
  const cuuint32_t box[2] = {box_x, box_y};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE, int QT>
cudaError_t launch_tile(const PrefillArgs& a, const TileMaps& maps, cudaStream_t st) {
  using G = Geo<MODE, QT>;
  auto kern = tile_gemm<MODE, QT>;
  const int smem = G::SMEM + 1024;  // + alignment slack
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<a.nc, TP_THREADS, smem, st>>>(a, maps);
  return cudaGetLastError();
}

// 3-D map over `n` blocks of `rows` rows of `row_bytes` bytes, block i at base + i * stride2
// (the K-quant expert records: rows of a record are whole super-blocks, but a record need
// not be a whole number of them); boxes of box_x bytes x box_y rows x 1 block.
cudaError_t encode_3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t n,
                      uint64_t stride2, uint32_t box_x, uint32_t box_y) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {row_bytes, rows, n};
  const cuuint64_t strides[2] = {row_bytes, stride2};
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_maps(const PrefillArgs& a, TileMaps* m) {
  std::memset(m, 0, sizeof *m);
  cudaError_t e;
  if (a.qtype == 12) {
    // K-quant records: gate and up rows (2F of rb_h bytes), then H down rows of rb_f bytes;
    // Q4_K down rows through a map as well, Q6_K down rows by bulk copies of whole rows
    const uint32_t seg = Geo<0, 12>::SEG;
    if ((e = encode_3d(&m->gu, a.experts, a.rb_h, (uint64_t)2 * a.F, (uint64_t)a.E, a.rec_bytes, seg, 64)) !=
        cudaSuccess)
      return e;
    if (a.qtype_dn == 12 &&
        (e = encode_3d(&m->dn, a.experts + (size_t)2 * a.F * a.rb_h, a.rb_f, (uint64_t)a.H, (uint64_t)a.E,
                       a.rec_bytes, seg, 128)) != cudaSuccess)
      return e;
    if (a.Fs) {
      const uint64_t srec = (uint64_t)2 * a.Fs * a.rb_h + (uint64_t)a.H * a.rb_fs;
      if ((e = encode_3d(&m->gu_s, a.shared, a.rb_h, (uint64_t)2 * a.Fs, 1, srec, seg, 64)) != cudaSuccess) return e;
      if (a.qtype_dn == 12 && (e = encode_3d(&m->dn_s, a.shared + (size_t)2 * a.Fs * a.rb_h, a.rb_fs, (uint64_t)a.H,
                                             1, srec, seg, 128)) != cudaSuccess)
        return e;
    }
    return encode_2d(&m->rt, a.router_w, true, (uint64_t)a.H, (uint64_t)a.E, 32, 64, true);
  }
  const uint32_t seg = a.qtype == 3 ? Geo<0, 3>::SEG : Geo<0, 2>::SEG;
  if ((e = encode_2d(&m->gu, a.experts, false, a.rb_h, (uint64_t)a.E * 3 * a.F, seg, 64, false)) != cudaSuccess)
    return e;
  if ((e = encode_2d(&m->dn, a.experts, false, a.rb_f, (uint64_t)a.E * 3 * a.H, seg, 128, false)) != cudaSuccess)
    return e;
  if (a.Fs) {
    if ((e = encode_2d(&m->gu_s, a.shared, false, a.rb_h, (uint64_t)3 * a.Fs, seg, 64, false)) != cudaSuccess)
      return e;
    if ((e = encode_2d(&m->dn_s, a.shared, false, a.rb_fs, (uint64_t)3 * a.H, seg, 128, false)) != cudaSuccess)
      return e;
  }
  return encode_2d(&m->rt, a.router_w, true, (uint64_t)a.H, (uint64_t)a.E, 32, 64, true);
}

// =============================================================================================
// Swapped down contraction: tokens as A (M = 128 operand rows), weights as B (N = 256 rows)
// =============================================================================================
// One MMA then covers 256 down rows x 16 K values, twice what the weights-as-A layout covers,
// so the contraction issues half the MMAs. A tile is 256 down rows of one expert (or of the
// shared expert) x one chunk of <= 64 token rows; the activation image holds plain token rows.
//
// One CTA per SM, 480 threads:
//   warp 0       weight producer: 2-D TMA boxes of 128 raw rows x KR K values into raw stages
//   warp 1       MMA issuer: A (token image) and B (converted weights) from shared memory,
//                accumulators in TMEM (two of 256 columns); commits release the stages
//   warp 2       token-operand producer: one bulk copy per 64 K values of the chunk's image
//                (half of a 128-value image block: its pieces are contiguous)
//   warps 3..10  converters, thread = weight row: each 32-value block of the raw stage ->
//                one B unit (256 rows x 32 K, f16, K-major core matrices) in shared memory
//   warps 11..14 the epilogue, one warp per TMEM lane quarter (lane = token row): weighted
//                rows into the routed or shared output buffer
// The same layout for gate/up (each 128-row image holding 64 tokens' hi and lo parts) measured
// slower than the weights-as-A kernel: its converters and epilogue, not the MMAs, set the pace.
constexpr int SW_CONV_WARPS = 8;
constexpr int SW_EPI_WARPS = 4;
constexpr int SW_EPI_WARP0 = 3 + SW_CONV_WARPS;
constexpr int SW_THREADS = 32 * (3 + SW_CONV_WARPS + SW_EPI_WARPS);
constexpr int SW_N = 256;                       // weight rows per tile (MMA N)
constexpr int SW_KU = 32;                       // K values per B unit (one 4-bit block per row)
constexpr int SW_BU = SW_N * SW_KU * 2;         // 16 KB
constexpr int SW_NBU = 4;                       // B unit slots: converters run up to four units ahead
constexpr int SW_KA = 64;                       // K values per token-operand stage (half an image block)
constexpr int SW_A_STAGE = 128 * SW_KA * 2;     // 16 KB (up to 128 image rows)
constexpr int SW_NA = 2;                        // token-operand stages
constexpr uint32_t SW_TMEM_COLS = 512;          // two 256-column accumulators

template <int QT>
struct SwGeo {
  static constexpr int BLK = QT == 3 ? 20 : 18;
  static constexpr int KR = 256;                       // K values per raw stage
  static constexpr int SEG = KR / 32 * BLK;            // 160 / 144 bytes
  static constexpr int STAGE = SW_N * SEG;
  static constexpr int NBR = KR / SW_KU;               // B units per raw stage
  static constexpr int NSA = 3;                        // raw stages
  static constexpr int SMEM = NSA * STAGE + SW_NBU * SW_BU + SW_NA * SW_A_STAGE;
  static_assert(SMEM + 1024 <= TP_SMEM_MAX, "shared memory");
};

struct SwMaps {
  CUtensorMap dn, dn_s;  // boxes of 128 rows x SEG bytes
};

struct SwUnit {
  const CUtensorMap* map;
  int y0, y1;        // map rows of B rows 0..127 and 128..255
  const uint8_t* a;  // the chunk's activation image (first 128-value block)
  int kdim;          // reduction length (F or Fs)
  int n, npad;       // chunk tokens, rounded to 16 (= image rows)
  int row0, prow, mt;
  bool shared;
};

// Tiles: routed chunks x H/256 row tiles, then token chunks x H/256 for the shared expert.
__device__ __forceinline__ int sw_units(const PrefillArgs& a) {
  const int ntok = (a.T + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX;
  const int nr = (int)a.nchunks[0];
  const int nsh = a.Fs ? ntok : 0;
  return (nr + nsh) * (a.H / SW_N);
}

__device__ __forceinline__ SwUnit sw_unit(const PrefillArgs& a, const SwMaps& maps, int u) {
  SwUnit t;
  const int nr = (int)a.nchunks[0];
  const int mt_r = a.H / SW_N, mt_s = a.H / SW_N;
  int slot, mt;
  if (u < nr * mt_r) {
    const GemmChunk ch = a.chunks[u / mt_r];
    mt = u % mt_r;
    slot = ch.slot;
    t.row0 = ch.row0;
    t.n = ch.n;
    t.prow = ch.prow;
    t.shared = false;
  } else {
    const int v = u - nr * mt_r;
    mt = v % mt_s;
    slot = 0;
    t.row0 = (v / mt_s) * PREFILL_TILE_NMAX;
    t.n = min(PREFILL_TILE_NMAX, a.T - t.row0);
    t.prow = t.row0;
    t.shared = true;
  }
  t.mt = mt;
  t.npad = (t.n + 15) & ~15;
  const int ff = t.shared ? a.Fs : a.F;
  t.map = t.shared ? &maps.dn_s : &maps.dn;
  t.y0 = slot * 3 * a.H + 2 * a.H + SW_N * mt;  // down rows of the expert's packed matrix
  t.y1 = t.y0 + 128;
  t.kdim = ff;
  const uint8_t* img = t.shared ? a.aimg_s : a.aimg;
  t.a = img + (size_t)t.prow * (ff / TP_KB) * 256;
  return t;
}

// Block J (compile-time) of a raw row segment -> its 32 values as f16 in the permuted slot
// order: o[4 p + i] is piece p (slots 8p .. 8p + 7) word i. The block is read as the two
// 16-byte words that cover it.
template <int QT, int J>
__device__ __forceinline__ void sw_convert(const uint8_t* row, uint32_t (&o)[16]) {
  constexpr int BLK = QT == 3 ? 20 : 18;
  constexpr int off = J * BLK;
  constexpr int q0 = off >> 4, rel = off - 16 * q0;  // byte offset in the two words
  const uint4* p = reinterpret_cast<const uint4*>(row) + q0;
  const uint4 x = p[0], y = p[1];
  const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
  if constexpr (QT == 3) {
    constexpr int wi = rel >> 2;
    const __half2 dmh = u2h(w[wi]);
    const __half2 d2 = __low2half2(dmh), m2 = __high2half2(dmh);
#pragma unroll
    for (int k = 0; k < 4; ++k) dequant4<3>(w[wi + 1 + k], d2, m2, o + 4 * k);
  } else {
    constexpr int wi = rel >> 2;
    uint32_t dw, q[4];
    if constexpr ((rel & 2) != 0) {  // d in the high half of w[wi]; nibble words aligned
      dw = w[wi] >> 16;
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = w[wi + 1 + k];
    } else {  // d in the low half; each nibble word straddles two words
      dw = w[wi] & 0xFFFFu;
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = __byte_perm(w[wi + k], w[wi + 1 + k], 0x5432);
    }
    const __half2 d2 = u2h(dw | (dw << 16));
#pragma unroll
    for (int k = 0; k < 4; ++k) dequant4<2>(q[k], d2, d2, o + 4 * k);
  }
}

// Block j (0 .. 11, a compile-time value once the caller's loop is unrolled) of a raw row.
template <int QT>
__device__ __forceinline__ void sw_convert_j(const uint8_t* row, int j, uint32_t (&o)[16]) {
  switch (j) {
    case 0: sw_convert<QT, 0>(row, o); break;
    case 1: sw_convert<QT, 1>(row, o); break;
    case 2: sw_convert<QT, 2>(row, o); break;
    case 3: sw_convert<QT, 3>(row, o); break;
    case 4: sw_convert<QT, 4>(row, o); break;
    case 5: sw_convert<QT, 5>(row, o); break;
    case 6: sw_convert<QT, 6>(row, o); break;
    case 7: sw_convert<QT, 7>(row, o); break;
    case 8: sw_convert<QT, 8>(row, o); break;
    case 9: sw_convert<QT, 9>(row, o); break;
    case 10: sw_convert<QT, 10>(row, o); break;
    default: sw_convert<QT, 11>(row, o); break;
  }
}

template <int QT>
__global__ void __launch_bounds__(SW_THREADS, 1) swap_down(const PrefillArgs a, const __grid_constant__ SwMaps maps) {
  using G = SwGeo<QT>;
  extern __shared__ __align__(1024) uint8_t ssm_dyn[];
  uint8_t* raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ssm_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* bunits = raw + G::NSA * G::STAGE;       // [SW_NBU][SW_BU]
  uint8_t* astage = bunits + SW_NBU * SW_BU;       // [SW_NA][SW_A_STAGE]
  __shared__ __align__(8) uint64_t raw_full[G::NSA], raw_empty[G::NSA];
  __shared__ __align__(8) uint64_t bu_full[SW_NBU], bu_empty[SW_NBU], a_full[SW_NA], a_empty[SW_NA];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  volatile int* abrt = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < G::NSA; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], SW_CONV_WARPS);
    }
    for (int i = 0; i < SW_NBU; ++i) {
      mbar_init(&bu_full[i], SW_CONV_WARPS);
      mbar_init(&bu_empty[i], 1);
    }
    for (int i = 0; i < SW_NA; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], SW_EPI_WARPS);
    }
    mbar_init(&fin, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base, SW_TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int units = sw_units(a);

  if (warp == 0) {
    // ------------------------------ weight producer ------------------------------
    const uint64_t pol = policy_evict_first();
    uint32_t ka = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const SwUnit t = sw_unit(a, maps, u);
      const int nk = (t.kdim + G::KR - 1) / G::KR;
      for (int kc = 0; kc < nk; ++kc, ++ka) {
        const int sa = (int)(ka % G::NSA);
        if (ka >= (uint32_t)G::NSA && !tp_wait_warp(&raw_empty[sa], ((ka / G::NSA) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* dst = raw + sa * G::STAGE;
          mbar_arrive_expect_tx(&raw_full[sa], (uint32_t)G::STAGE);
          tma_load_2d(dst, t.map, kc * G::SEG, t.y0, &raw_full[sa], pol);
          tma_load_2d(dst + 128 * G::SEG, t.map, kc * G::SEG, t.y1, &raw_full[sa], pol);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {  // every copy issued has landed before the CTA may exit
      for (int sa = 0; sa < G::NSA; ++sa) {
        const uint32_t f = ka > (uint32_t)sa ? (ka - sa - 1) / G::NSA + 1 : 0u;
        if (f) mbar_wait(&raw_full[sa], (f - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------ token-operand producer ------------------------------
    uint32_t rb = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const SwUnit t = sw_unit(a, maps, u);
      const uint32_t bytes = (uint32_t)t.npad * 16u * (SW_KA / 8);  // 8 pieces of npad rows
      for (int kk = 0; kk < t.kdim / SW_KA; ++kk, ++rb) {
        const int s2 = (int)(rb % SW_NA);
        if (rb >= (uint32_t)SW_NA && !tp_wait_warp(&a_empty[s2], ((rb / SW_NA) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&a_full[s2], bytes);
          asm volatile(
              "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  smem_addr(astage + s2 * SW_A_STAGE)),
              "l"(t.a + (size_t)kk * bytes), "r"(bytes), "r"(smem_addr(&a_full[s2]))
              : "memory");
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      for (int s2 = 0; s2 < SW_NA; ++s2) {
        const uint32_t f = rb > (uint32_t)s2 ? (rb - s2 - 1) / SW_NA + 1 : 0u;
        if (f) mbar_wait(&a_full[s2], (f - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(128, SW_N);
      uint32_t nbu = 0, rb = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
        const SwUnit t = sw_unit(a, maps, u);
        const int ab = (int)(uc & 1u);
        const uint32_t acc = tmem + 256u * ab;
        if (uc >= 2u && !tp_wait(&acc_empty[ab], ((uc >> 1) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        for (int kk = 0; kk < t.kdim / SW_KA && ok; ++kk, ++rb) {
          const int s2 = (int)(rb % SW_NA);
          if (!tp_wait(&a_full[s2], (rb / SW_NA) & 1u, abrt)) {
            ok = false;
            break;
          }
          const uint8_t* A = astage + s2 * SW_A_STAGE;
          for (int q = 0; q < SW_KA / SW_KU; ++q, ++nbu) {  // the stage's two B units
            const int sb = (int)(nbu % SW_NBU);
            if (!tp_wait(&bu_full[sb], (nbu / SW_NBU) & 1u, abrt)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint8_t* B = bunits + sb * SW_BU;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              // K values 32 q + 16 j .. + 15: token-image pieces 4 q + 2 j, + 1; B unit pieces 2 j, 2 j + 1
              const uint64_t ad = smem_desc(A + (size_t)(4 * q + 2 * j) * 16 * t.npad, 16u * t.npad, 128);
              const uint64_t bd = smem_desc(B + 2 * j * 4096, 4096, 128);
              mma_f16(acc, ad, bd, idesc, kk > 0 || q > 0 || j > 0);
            }
            mma_commit(&bu_empty[sb]);
          }
          if (!ok) break;
          mma_commit(&a_empty[s2]);
        }
        if (ok) mma_commit(&acc_full[ab]);
      }
      mma_commit(&fin);
      mbar_wait(&fin, 0);  // not cut short by an abort: the MMAs in flight end before TMEM is freed
    }
    __syncwarp();
  } else if (warp < SW_EPI_WARP0) {
    // ------------------------------ converters ------------------------------
    const int r = tid - 96;  // weight row of the tile (0..255)
    uint32_t ka = 0, nbu = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const SwUnit t = sw_unit(a, maps, u);
      const int nk = (t.kdim + G::KR - 1) / G::KR;
      for (int kc = 0; kc < nk && ok; ++kc, ++ka) {
        const int sa = (int)(ka % G::NSA);
        if (!tp_wait_warp(&raw_full[sa], (ka / G::NSA) & 1u, abrt)) {
          ok = false;
          break;
        }
        const uint8_t* row = raw + sa * G::STAGE + r * G::SEG;
        const int nvalid = min(G::NBR, (t.kdim - kc * G::KR) / SW_KU);
#pragma unroll
        for (int j = 0; j < G::NBR; ++j) {
          if (j < nvalid && ok) {
            const int sb = (int)(nbu % SW_NBU);
            if (nbu >= (uint32_t)SW_NBU && !tp_wait_warp(&bu_empty[sb], ((nbu / SW_NBU) - 1) & 1u, abrt)) {
              ok = false;
            } else {
              uint32_t o[16];
              sw_convert_j<QT>(row, j, o);
              uint8_t* dst = bunits + sb * SW_BU + r * 16;
#pragma unroll
              for (int pc = 0; pc < 4; ++pc)
                *reinterpret_cast<uint4*>(dst + pc * 4096) = make_uint4(o[4 * pc], o[4 * pc + 1], o[4 * pc + 2], o[4 * pc + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bu_full[sb]);
              ++nbu;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[sa]);
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const SwUnit t = sw_unit(a, maps, u);
      const int ab = (int)(uc & 1u);
      const uint32_t acc = tmem + lane_addr + 256u * ab;
      if (!tp_wait_warp(&acc_full[ab], (uc >> 1) & 1u, abrt)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int tr = 32 * q + lane;  // token row of the chunk
      if (32 * q < t.npad) {
        const int h0 = SW_N * t.mt;
        float* dst = nullptr;
        float wgt = 1.f;
        if (tr < t.n) {
          if (t.shared) dst = a.sbuf + (size_t)(t.row0 + tr) * a.H + h0;
          else {
            dst = a.ybuf + (size_t)(t.row0 + tr) * a.H + h0;
            wgt = a.wsorted[t.row0 + tr];
          }
        }
        for (int c0 = 0; c0 < SW_N; c0 += 8) {
          uint32_t v[8];
          tmem_ld8(acc + (uint32_t)c0, v);
          tmem_ld_wait();
          if (dst) {
            float4* d4 = reinterpret_cast<float4*>(dst + c0);
            d4[0] = make_float4(wgt * __uint_as_float(v[0]), wgt * __uint_as_float(v[1]), wgt * __uint_as_float(v[2]),
                                wgt * __uint_as_float(v[3]));
            d4[1] = make_float4(wgt * __uint_as_float(v[4]), wgt * __uint_as_float(v[5]), wgt * __uint_as_float(v[6]),
                                wgt * __uint_as_float(v[7]));
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  __syncthreads();
  if (tid == 0 && *abrt) atomicOr(a.status, DEV_ERR_MBAR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, SW_TMEM_COLS);
  }
}

template <int QT>
cudaError_t launch_swap(const PrefillArgs& a, const SwMaps& maps, cudaStream_t st) {
  using G = SwGeo<QT>;
  auto kern = swap_down<QT>;
  const int smem = G::SMEM + 1024;  // + alignment slack
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<a.nc, SW_THREADS, smem, st>>>(a, maps);
  return cudaGetLastError();
}

cudaError_t make_sw_maps(const PrefillArgs& a, SwMaps* m) {
  std::memset(m, 0, sizeof *m);
  const uint32_t seg = a.qtype == 3 ? SwGeo<3>::SEG : SwGeo<2>::SEG;
  cudaError_t e;
  if ((e = encode_2d(&m->dn, a.experts, false, a.rb_f, (uint64_t)a.E * 3 * a.H, seg, 128, false)) != cudaSuccess)
    return e;
  if (a.Fs && (e = encode_2d(&m->dn_s, a.shared, false, a.rb_fs, (uint64_t)3 * a.H, seg, 128, false)) != cudaSuccess)
    return e;
  return cudaSuccess;
}

}  // namespace

cudaError_t tile_router_launch(const PrefillArgs& a, cudaStream_t st) {
  TileMaps maps;
  cudaError_t e = make_maps(a, &maps);
  if (e != cudaSuccess) return e;
  return launch_tile<2, 3>(a, maps, st);
}

cudaError_t tile_images_launch(const PrefillArgs& a, bool routed, cudaStream_t st) {
  int grid;
  if (routed) {
    const int P = a.T * a.K;
    grid = (P + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX + a.E;  // routed chunks at most
  } else {
    grid = (a.T + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX;
  }
  // one CTA per 8-row group of a chunk: the CTAs past a routed chunk's rows exit at once, and
  // a full chunk's eight groups run side by side (two groups a CTA, looping, measured 12 us
  // slower on the Ling K-quant batch, whose most-picked experts fill several chunks). The few
  // token chunks also split their K blocks over two CTAs.
  tile_images<<<dim3(grid, PREFILL_TILE_NMAX / 8, routed ? 1 : 2), 256, 0, st>>>(a, routed ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t swap_down_launch(const PrefillArgs& a, cudaStream_t st) {
  SwMaps maps;
  cudaError_t e = make_sw_maps(a, &maps);
  if (e != cudaSuccess) return e;
  return a.qtype == 3 ? launch_swap<3>(a, maps, st) : launch_swap<2>(a, maps, st);
}

cudaError_t tile_gemm_launch(const PrefillArgs& a, int mode, cudaStream_t st) {
  TileMaps maps;
  cudaError_t e = make_maps(a, &maps);
  if (e != cudaSuccess) return e;
  const int qt = mode == 0 ? a.qtype : a.qtype_dn;
  switch (qt) {
    case 2: return mode == 0 ? launch_tile<0, 2>(a, maps, st) : launch_tile<1, 2>(a, maps, st);
    case 3: return mode == 0 ? launch_tile<0, 3>(a, maps, st) : launch_tile<1, 3>(a, maps, st);
    case 12: return mode == 0 ? launch_tile<0, 12>(a, maps, st) : launch_tile<1, 12>(a, maps, st);
    case 14: return mode == 0 ? cudaErrorInvalidValue : launch_tile<1, 14>(a, maps, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
