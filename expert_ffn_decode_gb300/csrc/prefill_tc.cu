// Tile pipeline of the batched MoE-FFN step for sm_103a: the router, gate/up and
// down contractions as warp-specialised persistent kernels on the tensor cores.
//
// One CTA per SM, 320 threads:
//   warp 0      producer: cp.async.bulk copies of the raw weight rows of each
//               pipeline chunk into a ring of shared-memory stages, and of the
//               token operand (a pre-tiled image, one copy per 128 K values)
//   warp 1      MMA issuer: tcgen05.mma with A in tensor memory, B in shared memory,
//               f32 accumulator in tensor memory; commits release the stages
//   warps 2..9  converters: raw 4-bit blocks (or f32 router rows) -> f16 rows of A,
//               written to tensor memory with tcgen05.st (thread = row = TMEM lane);
//               then the epilogue of each tile (tcgen05.ld)
//
// Work units (one accumulator tile, M = 128 weight rows x N = chunk tokens):
//   router   64 experts (f32 rows split into f16 hi rows 0..63 and lo rows 64..127)
//            x 64 tokens (x hi and lo columns): logit = sum of the four products
//   gate/up  64 gate/up row pairs (interleaved: even rows gate, odd rows up) of one
//            expert x one chunk of its sorted (token, pick) pairs (x hi and lo columns)
//   down     128 down rows of one expert x the chunk's activations
// Every stage wait is bounded; a timeout anywhere stops every role of the CTA and
// sets the status word.
#include <cuda_fp16.h>

#include <cstdint>

#include "common.cuh"
#include "plan.h"
#include "prefill_host.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int TP_THREADS = 320;
constexpr int TP_CONV_WARPS = 8;
constexpr int TP_KB = 128;                        // K values per token-operand stage
constexpr int TP_B_STAGE = 128 * TP_KB * 2;       // up to 128 rows: 32 KB
constexpr int TP_NSB = 3;
constexpr int TP_RAW_BUDGET = 104 * 1024;
constexpr int TP_SCRATCH = 64 * 65 * 4;           // router epilogue exchange
constexpr int TP_MAX_NSA = 16;
constexpr uint32_t TP_TMEM_COLS = 512;
constexpr uint32_t TP_A_COL = 128;                // A stages follow the accumulator (128 columns)

// Stage geometry per contraction. MODE 0 gate/up, 1 down, 2 router.
template <int MODE, int QT>
struct Geo {
  static constexpr int ROWS = MODE == 2 ? 64 : 128;             // raw rows per stage
  static constexpr int SEG = MODE == 2 ? 512 : (QT == 3 ? 80 : 144);  // bytes per row per chunk
  static constexpr int PITCH = MODE == 2 ? 528 : SEG;           // odd multiple of 16: conflict-free LDS.128
  static constexpr int KC = MODE == 2 ? 128 : (QT == 3 ? 128 : 256);  // K values per chunk
  static constexpr int STAGE = ROWS * PITCH;
  static constexpr int NSA = (TP_RAW_BUDGET / STAGE) < TP_MAX_NSA ? (TP_RAW_BUDGET / STAGE) : TP_MAX_NSA;
  static constexpr uint32_t ACOLS = KC / 2;                     // TMEM columns per A stage
  static constexpr int NSUB = KC / TP_KB;                       // token stages per chunk
  static constexpr int SMEM = NSA * STAGE + TP_NSB * TP_B_STAGE + (MODE == 2 ? TP_SCRATCH : 0);
};

__device__ __forceinline__ int kslot_dev(int e) {
  const int hi = e >> 4, r = e & 15, w = r >> 2, j = r & 3;
  return 8 * w + 4 * hi + ((j == 1) ? 2 : (j == 2 ? 1 : j));
}

// Byte offset of (row r, slot s) inside one 128-value block of an operand image with nb rows.
__device__ __forceinline__ uint32_t img_off(int r, int s, int nb) {
  return (uint32_t)(((s >> 3) * (nb >> 3) + (r >> 3)) * 128 + (r & 7) * 16 + (s & 7) * 2);
}

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

// Q4_1: the thread's two blocks (40 bytes at byte 40h of the 80-byte row segment).
__device__ __forceinline__ void convert_q41(const uint8_t* row, int h, uint32_t (&o)[32]) {
  const uint4* p = reinterpret_cast<const uint4*>(row) + (h ? 2 : 0);
  const uint4 a = p[0], b = p[1], c = p[2];
  const uint32_t w[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
  // h = 0: blocks at words 0 and 5; h = 1 (window starts at word 8): words 2 and 7
  const int w0 = h ? 2 : 0;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const int base = w0 + 5 * blk;
    uint32_t dm, q0, q1, q2, q3;
    if (h) {
      dm = blk ? w[7] : w[2];
      q0 = blk ? w[8] : w[3];
      q1 = blk ? w[9] : w[4];
      q2 = blk ? w[10] : w[5];
      q3 = blk ? w[11] : w[6];
    } else {
      dm = blk ? w[5] : w[0];
      q0 = blk ? w[6] : w[1];
      q1 = blk ? w[7] : w[2];
      q2 = blk ? w[8] : w[3];
      q3 = blk ? w[9] : w[4];
    }
    (void)base;
    const __half2 dmh = u2h(dm);
    const __half2 d2 = __low2half2(dmh), m2 = __high2half2(dmh);
    dequant4<3>(q0, d2, m2, o + 16 * blk + 0);
    dequant4<3>(q1, d2, m2, o + 16 * blk + 4);
    dequant4<3>(q2, d2, m2, o + 16 * blk + 8);
    dequant4<3>(q3, d2, m2, o + 16 * blk + 12);
  }
}

// Q4_0: two of the thread's four blocks (pair p of 2), 18 bytes each, from the 144-byte
// row segment; the thread's blocks are 4h .. 4h + 3.
template <int H>
__device__ __forceinline__ void convert_q40_pair(const uint8_t* row, int p, uint32_t (&o)[32]) {
  // blocks b0 = 4H + 2p and b0 + 1 span bytes [18 b0, 18 b0 + 36): load the covering uint4s
  const int byte0 = 18 * (4 * H + 2 * p);
  const int u0 = byte0 >> 4;
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

// Router rows: 64 f32 values (values 64h .. 64h + 63 of the 128-value chunk) -> f16 hi
// or lo parts in the permuted slot order.
__device__ __forceinline__ void convert_f32(const uint8_t* row, int h, bool lo, uint32_t (&o)[32]) {
  const float4* p = reinterpret_cast<const float4*>(row) + 16 * h;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 x0 = p[8 * blk + w], x1 = p[8 * blk + 4 + w];
      uint32_t* d = o + 16 * blk + 4 * w;
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
}

// ---- work units ----------------------------------------------------------------------------
struct TileUnit {
  const uint8_t* a0;   // raw row 0 of the tile (chunk 0)
  uint32_t a_rs;       // bytes between consecutive rows (row pairs for gate/up)
  uint32_t a_odd;      // gate/up: byte distance from a gate row to its up row
  int mrows;           // valid raw rows
  const uint8_t* b;    // token-operand image of the chunk (first 128-value block)
  int nk;              // pipeline chunks
  int n, npad, nb;     // chunk tokens, rounded to 16, operand rows (hi + lo: 2 npad)
  int row0, prow, mt;  // chunk's first row, padded-row offset, M tile
  bool shared;         // shared expert (token chunk)
  int e0;              // router: first expert of the tile
};

template <int MODE, int QT>
__device__ __forceinline__ int tile_units(const PrefillArgs& a) {
  const int ntok = (a.T + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX;
  if (MODE == 2) return ntok * ((a.E + 63) / 64);
  const int nr = (int)a.nchunks[0];
  const int nsh = a.Fs ? ntok : 0;
  const int mt_r = MODE == 0 ? a.F / 64 : a.H / 128;
  const int mt_s = MODE == 0 ? a.Fs / 64 : a.H / 128;
  return nr * mt_r + nsh * mt_s;
}

template <int MODE, int QT>
__device__ __forceinline__ TileUnit tile_unit(const PrefillArgs& a, int u) {
  using G = Geo<MODE, QT>;
  TileUnit t;
  const int nkh = a.H / TP_KB;
  if (MODE == 2) {
    const int et = (a.E + 63) / 64;
    const int j = u / et, e = u % et;
    t.e0 = 64 * e;
    t.a0 = reinterpret_cast<const uint8_t*>(a.router_w) + (size_t)t.e0 * a.H * 4;
    t.a_rs = (uint32_t)a.H * 4;
    t.a_odd = 0;
    t.mrows = min(64, a.E - t.e0);
    t.row0 = j * PREFILL_TILE_NMAX;
    t.n = min(PREFILL_TILE_NMAX, a.T - t.row0);
    t.npad = (t.n + 15) & ~15;
    t.nb = 2 * t.npad;
    t.prow = t.row0;
    t.b = a.ximg + (size_t)2 * t.prow * nkh * 256;
    t.nk = a.H / G::KC;
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
    slot = a.E;
    t.row0 = j * PREFILL_TILE_NMAX;
    t.n = min(PREFILL_TILE_NMAX, a.T - t.row0);
    t.prow = t.row0;
    t.shared = true;
  }
  t.mt = mt;
  t.e0 = 0;
  t.npad = (t.n + 15) & ~15;
  const int ff = t.shared ? a.Fs : a.F;
  const uint8_t* rec = t.shared ? a.shared : a.experts + (size_t)slot * a.rec_bytes;
  if (MODE == 0) {
    t.nb = 2 * t.npad;
    t.a0 = rec + (size_t)(64 * mt) * a.rb_h;
    t.a_rs = a.rb_h;
    t.a_odd = (uint32_t)ff * a.rb_h;
    t.mrows = 128;
    t.nk = a.H / G::KC;
    const uint8_t* img = t.shared ? a.ximg : a.ximg_routed;
    t.b = img + (size_t)2 * t.prow * nkh * 256;
  } else {
    const uint32_t rb = t.shared ? a.rb_fs : a.rb_f;
    t.nb = t.npad;
    t.a0 = rec + (size_t)2 * ff * a.rb_h + (size_t)(128 * mt) * rb;
    t.a_rs = rb;
    t.a_odd = 0;
    t.mrows = 128;
    t.nk = ff / G::KC;
    const uint8_t* img = t.shared ? a.aimg_s : a.aimg;
    t.b = img + (size_t)t.prow * (ff / TP_KB) * 256;
  }
  return t;
}

// Byte address of raw row m (stage chunk kc) of a tile.
template <int MODE>
__device__ __forceinline__ const uint8_t* raw_src(const TileUnit& t, int m, int kc, int seg) {
  if (MODE == 0) return t.a0 + (size_t)(m >> 1) * t.a_rs + ((m & 1) ? t.a_odd : 0u) + (size_t)kc * seg;
  return t.a0 + (size_t)m * t.a_rs + (size_t)kc * seg;
}

// ---- the persistent tile kernel -----------------------------------------------------------
template <int MODE, int QT>
__global__ void __launch_bounds__(TP_THREADS, 1) tile_gemm(const PrefillArgs a) {
  using G = Geo<MODE, QT>;
  extern __shared__ __align__(1024) uint8_t tsm_dyn[];
  uint8_t* raw = tsm_dyn;                                   // [NSA][STAGE]
  uint8_t* bring = tsm_dyn + G::NSA * G::STAGE;             // [NSB][B_STAGE]
  float* scratch = reinterpret_cast<float*>(bring + TP_NSB * TP_B_STAGE);  // router only
  __shared__ __align__(8) uint64_t raw_full[G::NSA], raw_empty[G::NSA];
  __shared__ __align__(8) uint64_t a_full[2], a_empty[2], b_full[TP_NSB], b_empty[TP_NSB];
  __shared__ __align__(8) uint64_t acc_full, acc_empty, fin, scr_full, scr_empty;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  volatile int* abrt = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < G::NSA; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], TP_CONV_WARPS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], TP_CONV_WARPS);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < TP_NSB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, TP_CONV_WARPS);
    mbar_init(&fin, 1);
    mbar_init(&scr_full, 4);   // router epilogue: the four warps of lanes 64..127
    mbar_init(&scr_empty, 4);  // ... and the four warps of lanes 0..63
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
    // ------------------------------ producer ------------------------------
    // weight rows stream through L2 once; router rows are read by every token chunk
    const uint64_t pol_w = MODE == 2 ? policy_evict_last() : policy_evict_first();
    uint32_t ra = 0, rb = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const TileUnit t = tile_unit<MODE, QT>(a, u);
      const uint32_t bbytes = (uint32_t)t.nb * 256u;
      for (int kc = 0; kc < t.nk && ok; ++kc) {
        const int sa = (int)(ra % G::NSA);
        if (ra >= (uint32_t)G::NSA && !tp_wait_warp(&raw_empty[sa], ((ra / G::NSA) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&raw_full[sa], (uint32_t)t.mrows * G::SEG);
        __syncwarp();
        for (int m = lane; m < t.mrows; m += 32)
          bulk_g2s(raw + sa * G::STAGE + m * G::PITCH, raw_src<MODE>(t, m, kc, G::SEG), G::SEG, &raw_full[sa],
                   pol_w);
        ++ra;
        for (int sub = 0; sub < G::NSUB; ++sub) {
          const int sb = (int)(rb % TP_NSB);
          if (rb >= (uint32_t)TP_NSB && !tp_wait_warp(&b_empty[sb], ((rb / TP_NSB) - 1) & 1u, abrt)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&b_full[sb], bbytes);
            const uint8_t* src = t.b + (size_t)(kc * G::NSUB + sub) * bbytes;
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(bring + sb * TP_B_STAGE)),
                "l"(src), "r"(bbytes), "r"(smem_addr(&b_full[sb]))
                : "memory");
          }
          __syncwarp();
          ++rb;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      uint32_t ka = 0, rb = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
        const TileUnit t = tile_unit<MODE, QT>(a, u);
        const uint32_t idesc = idesc_f16_f32(128, t.nb);
        if (uc > 0 && !tp_wait(&acc_empty, (uc - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        for (int kc = 0; kc < t.nk && ok; ++kc) {
          const int st = (int)(ka & 1u);
          if (!tp_wait(&a_full[st], (ka >> 1) & 1u, abrt)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          for (int sub = 0; sub < G::NSUB; ++sub) {
            const int sb = (int)(rb % TP_NSB);
            if (!tp_wait(&b_full[sb], (rb / TP_NSB) & 1u, abrt)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint8_t* B = bring + sb * TP_B_STAGE;
#pragma unroll
            for (int j = 0; j < TP_KB / 16; ++j) {
              const uint64_t bd = smem_desc(B + 2 * j * 16 * t.nb, 16u * t.nb, 128);
              const uint32_t ta = tmem + TP_A_COL + (uint32_t)st * G::ACOLS + (uint32_t)(sub * 64 + 8 * j);
              mma_f16_ta(tmem, ta, bd, idesc, (kc | sub | j) != 0);
            }
            mma_commit(&b_empty[sb]);
            ++rb;
          }
          mma_commit(&a_empty[st]);
          ++ka;
        }
        if (ok) mma_commit(&acc_full);
      }
      // every MMA issued has completed before the columns are freed
      mma_commit(&fin);
      tp_wait(&fin, 0, abrt);
    }
    __syncwarp();
  } else {
    // ------------------------------ converters + epilogue ------------------------------
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int m = 32 * q + lane;  // TMEM lane = tile row
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t ra = 0, ka = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const TileUnit t = tile_unit<MODE, QT>(a, u);
      for (int kc = 0; kc < t.nk; ++kc) {
        const int sa = (int)(ra % G::NSA);
        if (!tp_wait_warp(&raw_full[sa], (ra / G::NSA) & 1u, abrt)) {
          ok = false;
          break;
        }
        const int st = (int)(ka & 1u);
        if (ka >= 2 && !tp_wait_warp(&a_empty[st], ((ka >> 1) - 1) & 1u, abrt)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t col = TP_A_COL + (uint32_t)st * G::ACOLS;
        if (MODE == 2) {
          uint32_t o[32];
          convert_f32(raw + sa * G::STAGE + (m & 63) * G::PITCH, h, m >= 64, o);
          tmem_st32(tmem + lane_addr + col + 32u * h, o);
        } else if (QT == 3) {
          uint32_t o[32];
          convert_q41(raw + sa * G::STAGE + m * G::PITCH, h, o);
          tmem_st32(tmem + lane_addr + col + 32u * h, o);
        } else {
          uint32_t o[32];
          const uint8_t* row = raw + sa * G::STAGE + m * G::PITCH;
          if (h == 0) convert_q40_pair<0>(row, 0, o); else convert_q40_pair<1>(row, 0, o);
          tmem_st32(tmem + lane_addr + col + 64u * h, o);
          if (h == 0) convert_q40_pair<0>(row, 1, o); else convert_q40_pair<1>(row, 1, o);
          tmem_st32(tmem + lane_addr + col + 64u * h + 32u, o);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        fence_proxy_async_smem();  // raw stage reads done before the next bulk copy into it
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&raw_empty[sa]);
          mbar_arrive(&a_full[st]);
        }
        ++ra;
        ++ka;
      }
      if (!ok) break;
      // ---- epilogue ----
      if (!tp_wait_warp(&acc_full, uc & 1u, abrt)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int half = t.npad >> 1;  // columns per warp of a lane quarter (a multiple of 8)
      const int c_lo = h * half;
      if (MODE == 2) {
        // logit = (hi.x_hi + hi.x_lo) + (lo.x_hi + lo.x_lo): lanes 64..127 hand their sums
        // over through shared memory
        if (m >= 64) {
          if (uc > 0 && !tp_wait_warp(&scr_empty, (uc - 1) & 1u, abrt)) {
            ok = false;
            break;
          }
          for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
            uint32_t r0[8], r1[8];
            tmem_ld8(tmem + lane_addr + (uint32_t)c0, r0);
            tmem_ld8(tmem + lane_addr + (uint32_t)(t.npad + c0), r1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              scratch[(m - 64) * 65 + c0 + i] = __uint_as_float(r0[i]) + __uint_as_float(r1[i]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&scr_full);
        } else {
          if (!tp_wait_warp(&scr_full, uc & 1u, abrt)) {
            ok = false;
            break;
          }
          for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
            uint32_t r0[8], r1[8];
            tmem_ld8(tmem + lane_addr + (uint32_t)c0, r0);
            tmem_ld8(tmem + lane_addr + (uint32_t)(t.npad + c0), r1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c = c0 + i;
              const float v = (__uint_as_float(r0[i]) + __uint_as_float(r1[i])) + scratch[m * 65 + c];
              if (c < t.n && t.e0 + m < a.E) a.logits[(size_t)(t.row0 + c) * a.E + t.e0 + m] = v;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&scr_empty);
        }
      } else if (MODE == 0) {
        const int ff = t.shared ? a.Fs : a.F;
        const int f = 64 * t.mt + (m >> 1);
        const int nkf = ff / TP_KB;
        uint8_t* img = t.shared ? a.aimg_s : a.aimg;
        uint8_t* base = img + ((size_t)t.prow * nkf + (size_t)(f / TP_KB) * t.npad) * 256;
        const int s = kslot_dev(f & 31) + (f & (TP_KB - 1) & ~31);
        for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
          uint32_t r0[8], r1[8];
          tmem_ld8(tmem + lane_addr + (uint32_t)c0, r0);
          tmem_ld8(tmem + lane_addr + (uint32_t)(t.npad + c0), r1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float v = __uint_as_float(r0[i]) + __uint_as_float(r1[i]);  // x_hi + x_lo parts
            const float other = __shfl_xor_sync(0xffffffffu, v, 1);
            const int c = c0 + i;
            if (!(m & 1) && c < t.n) {
              const float act = v / (1.f + expf(-v)) * other;  // silu(gate) * up
              *reinterpret_cast<__half*>(base + img_off(c, s, t.npad)) = __float2half_rn(act);
            }
          }
        }
      } else {
        const int hrow = 128 * t.mt + m;
        for (int c0 = c_lo; c0 < c_lo + half; c0 += 8) {
          uint32_t r0[8];
          tmem_ld8(tmem + lane_addr + (uint32_t)c0, r0);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + i;
            if (c < t.n) {
              const float y = __uint_as_float(r0[i]);
              if (t.shared) a.sbuf[(size_t)(t.row0 + c) * a.H + hrow] = y;
              else a.ybuf[(size_t)(t.row0 + c) * a.H + hrow] = a.wsorted[t.row0 + c] * y;
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
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
// x rows of each chunk as f16 hi and lo parts, tiled as the MMA's B operand. Block c of the
// grid takes chunk c (token chunks, or routed chunks when `routed`).
__global__ void __launch_bounds__(256) tile_images(const PrefillArgs a, int routed) {
  const int c = blockIdx.x;
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
  const int pieces = a.H / 8;
  for (int i = threadIdx.x; i < n * pieces; i += blockDim.x) {
    const int r = i / pieces, p = i % pieces;
    const int tok = routed ? (int)(a.perm[row0 + r] / (uint32_t)a.K) : row0 + r;
    const int kk = p >> 4, kc8 = p & 15;
    const int g = kk * TP_KB + 8 * kc8;  // first slot of the piece
    const int b = g >> 5, w = (g & 31) >> 3;
    const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)tok * a.H + 32 * b);
    const float4 x0 = __ldg(xr + w), x1 = __ldg(xr + 4 + w);
    uint4 hi, lo;
    hi.x = pack_h2(x0.x, x0.z);
    hi.y = pack_h2(x0.y, x0.w);
    hi.z = pack_h2(x1.x, x1.z);
    hi.w = pack_h2(x1.y, x1.w);
    lo.x = pack_lo(x0.x, x0.z, hi.x);
    lo.y = pack_lo(x0.y, x0.w, hi.y);
    lo.z = pack_lo(x1.x, x1.z, hi.z);
    lo.w = pack_lo(x1.y, x1.w, hi.w);
    uint8_t* blk = base + (size_t)kk * nb * 256;
    *reinterpret_cast<uint4*>(blk + ((kc8 * (nb >> 3) + (r >> 3)) * 128 + (r & 7) * 16)) = hi;
    const int rl = npad + r;
    *reinterpret_cast<uint4*>(blk + ((kc8 * (nb >> 3) + (rl >> 3)) * 128 + (rl & 7) * 16)) = lo;
  }
}

template <int MODE, int QT>
cudaError_t launch_tile(const PrefillArgs& a, cudaStream_t st) {
  using G = Geo<MODE, QT>;
  auto kern = tile_gemm<MODE, QT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<a.nc, TP_THREADS, G::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tile_router_launch(const PrefillArgs& a, cudaStream_t st) { return launch_tile<2, 3>(a, st); }

cudaError_t tile_images_launch(const PrefillArgs& a, bool routed, cudaStream_t st) {
  int grid;
  if (routed) {
    const int P = a.T * a.K;
    grid = (P + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX + a.E;  // routed chunks at most
  } else {
    grid = (a.T + PREFILL_TILE_NMAX - 1) / PREFILL_TILE_NMAX;
  }
  tile_images<<<grid, 256, 0, st>>>(a, routed ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t tile_gemm_launch(const PrefillArgs& a, int mode, cudaStream_t st) {
  if (mode == 0) return a.qtype == 3 ? launch_tile<0, 3>(a, st) : launch_tile<0, 2>(a, st);
  return a.qtype == 3 ? launch_tile<1, 3>(a, st) : launch_tile<1, 2>(a, st);
}

}  // namespace moe
