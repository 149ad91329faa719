// Fused single-token MoE-FFN step (decode, T = 1) for sm_103a.
//
// One persistent CTA per SM runs the whole step. A slot is a pick of the token or
// the shared expert; a slot with ff intermediate values has ff / 32 columns, dealt to
// the CTAs in turn. Phases of a CTA:
//   router rows (F32, one row per ring item)                    -> published logits
//   x -> activation blocks
//   its shared-expert columns (they need no routing): 32 gate and 32 up rows ->
//   SwiGLU values, published; then its share of the shared expert's down rows over
//   the whole published activation vector -> published output rows
//   every CTA's logits seen; sigmoid, selection bias, (group) top-k and weight
//   normalisation, computed by every CTA
//   its routed columns, the same way, each down row weighted by its pick's weight
//   every slot's output rows seen; out = their sum in a fixed slot order
// Weights stream through a ring of shared-memory slots filled by 1-D bulk async
// copies (cp.async.bulk, completion counted on mbarriers) issued by the lanes of one
// producer warp; eleven consumer warps compute. Gate/up rows and down rows are both
// contiguous runs of a record, so every byte arrives in whole-row copies.
// Routing-independent rows (router, shared expert) are requested before the kernel
// waits on the previous grid (programmatic dependent launch).
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
#include "plan.h"
#include "select.cuh"

namespace moe {

constexpr int NCW = 11;              // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int NCT = NCW * 32;        // consumer threads
constexpr int BAR_CONS = 1;          // named barrier: consumer warps only
constexpr int MAX_SLOTS = 16;        // ring slots (one issuing producer lane each)

// Shared-memory carve-up (byte offsets, computed identically on host and device).
struct SmemLayout {
  uint32_t ring, xplanes, xinfo, aplanes, ainfo, probs, keys, gscore, rids, rw, items, bars, misc, total;
};

MOE_HD uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

MOE_HD SmemLayout smem_layout(const DecodePlan& p) {
  SmemLayout L;
  uint32_t o = 0;
  L.ring = o;
  o += (uint32_t)p.nslots * p.slot_bytes;
  const int nbx = p.H / 32;
  const int nba = (p.F > p.Fs ? p.F : p.Fs) / 32;  // a slot's activation blocks
  L.xplanes = o = align_up(o, 16);
  o += (uint32_t)nbx * 96u;
  L.xinfo = o = align_up(o, 16);
  o += (uint32_t)nbx * 8u;
  L.aplanes = o = align_up(o, 16);
  o += (uint32_t)nba * 96u;
  L.ainfo = o = align_up(o, 16);
  o += (uint32_t)nba * 8u;
  L.probs = o = align_up(o, 16);
  o += (uint32_t)p.E * 4u;
  L.keys = o = align_up(o, 16);
  o += (uint32_t)p.E * 4u;
  L.gscore = o = align_up(o, 16);
  o += 64u * 4u;
  L.rids = o = align_up(o, 16);
  o += 32u * 4u;
  L.rw = o;
  o += 33u * 4u;
  L.items = o = align_up(o, 16);
  o += (uint32_t)p.max_items * (uint32_t)sizeof(Item);
  L.bars = o = align_up(o, 8);
  o += (uint32_t)p.nslots * 16u + 8u;
  L.misc = o = align_up(o, 16);
  o += 16u;
  L.total = align_up(o, 128);
  return L;
}

// ---------------------------------------------------------------------------
// Activation blocks
// ---------------------------------------------------------------------------

// Quantise blocks [0, nb) of a global f32 vector into the shared planes. Four
// consecutive threads share a block (8 values each); the block's 32 values v_i
// become integers q_i = v_i * 2^k, |q_i| <= 2^22, the power of two chosen from the
// block's largest magnitude; plane P holds byte P of every q_i (value i at byte
// P*32 + i) and info[b] = {2^-k, sum q_i}. A block whose values are all below
// 2^-97 in magnitude is taken as zero. When `copy` is not null the f32 values are
// stored there too. Every thread of a group runs the same number of rounds.
// The source is an f32 vector in global memory, an f32 vector in shared memory
// (kShared), or published words of generation `gen` (then every value is awaited;
// `ok` is cleared on a timeout). Whole warps call it (the groups use shuffles).
template <typename Src, bool kShared = false>
__device__ __forceinline__ void quant_blocks(const Src* src, int nb, uint8_t* planes, float2* info,
                                             float* copy, int t, int nthreads, uint32_t gen, bool& ok) {
  for (int base = 0; base < 4 * nb; base += nthreads) {
    const int idx = base + t, b = idx >> 2, qq = idx & 3;
    const bool active = idx < 4 * nb;
    float v[8];
    if (active) {
      if constexpr (sizeof(Src) == 4) {
        const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)b * 32 + qq * 8);
        const float4 a = kShared ? s4[0] : __ldcg(s4), c = kShared ? s4[1] : __ldcg(s4 + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
      } else {
        const uint64_t* w = src + (size_t)b * 32 + qq * 8;
        uint64_t u[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const ulonglong2 pr = __ldcg(reinterpret_cast<const ulonglong2*>(w) + i);
          u[2 * i] = pr.x;
          u[2 * i + 1] = pr.y;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = await_tagged(w + i, u[i], gen, ok);
      }
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
      if (copy) {
        float4* c4 = reinterpret_cast<float4*>(copy + (size_t)b * 32 + qq * 8);
        c4[0] = make_float4(v[0], v[1], v[2], v[3]);
        c4[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
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

// Block b of a row starting at shared-memory address `row` times activation block a.
template <int QT>
__device__ __forceinline__ float block_dot(const uint8_t* row, int b, const ActBlock& a) {
  if constexpr (QT == 3) {  // Q4_1: word 0 = f16 d | f16 m << 16, words 1..4 the nibbles
    const uint32_t* w = reinterpret_cast<const uint32_t*>(row + 20 * b);
    uint32_t dm = w[0];
    uint32_t qw[4] = {w[1], w[2], w[3], w[4]};
    float S = nibble_dot(qw, a);
    __half2 h = *reinterpret_cast<__half2*>(&dm);
    float2 f = __half22float2(h);
    return a.s * fmaf(f.x, S, f.y * a.X);
  } else {  // Q4_0: f16 d, then 16 nibble bytes; the block sits on a 2-byte boundary
    uintptr_t addr = reinterpret_cast<uintptr_t>(row) + 18u * (uint32_t)b;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(addr & ~uintptr_t(3));
    uint32_t sh = (uint32_t)(addr & 3u) * 8u;  // 0 or 16
    uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
    uint32_t dbits = __funnelshift_rc(w0, w1, sh) & 0xFFFFu;
    uint32_t qw[4] = {__funnelshift_rc(w0, w1, 16 + sh), __funnelshift_rc(w1, w2, 16 + sh),
                      __funnelshift_rc(w2, w3, 16 + sh), __funnelshift_rc(w3, w4, 16 + sh)};
    float S = nibble_dot(qw, a);
    float d = __half2float(__ushort_as_half((unsigned short)dbits));
    return a.s * d * fmaf(-8.f, a.X, S);
  }
}

// Block b of a row in global memory (read-only during the kernel) times block a.
template <int QT>
__device__ __forceinline__ float block_dot_g(const uint8_t* row, int b, const ActBlock& a) {
  if constexpr (QT == 3) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(row + 20 * b);  // 4-byte aligned
    uint32_t dm = __ldg(w);
    const uint32_t qw[4] = {__ldg(w + 1), __ldg(w + 2), __ldg(w + 3), __ldg(w + 4)};
    const float S = nibble_dot(qw, a);
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&dm));
    return a.s * fmaf(f.x, S, f.y * a.X);
  } else {  // 2-byte aligned blocks: nine 16-bit loads, all inside the block
    const unsigned short* h = reinterpret_cast<const unsigned short*>(row + 18 * b);
    unsigned short u[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) u[i] = __ldg(h + i);
    const uint32_t qw[4] = {(uint32_t)u[1] | ((uint32_t)u[2] << 16), (uint32_t)u[3] | ((uint32_t)u[4] << 16),
                            (uint32_t)u[5] | ((uint32_t)u[6] << 16), (uint32_t)u[7] | ((uint32_t)u[8] << 16)};
    const float S = nibble_dot(qw, a);
    const float d = __half2float(__ushort_as_half(u[0]));
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
__device__ __forceinline__ float group_sum(float v, int lpr) {
  for (int o = lpr / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// group_sum of N independent values at once (their shuffles interleave)
template <int N>
__device__ __forceinline__ void group_sum_n(float (&v)[N], int lpr) {
  for (int o = lpr / 2; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Timeline points (MOE_TRACE): one u64 %globaltimer value each, per CTA.
enum TracePoint : int {
  TR_START = 0, TR_PDL_DONE, TR_ROUTER_DONE, TR_X_READY, TR_SHARED_DONE, TR_LOGITS, TR_KEYS, TR_TOPK,
  TR_ROUTED, TR_GU_DONE, TR_COLS_DONE, TR_PARTIALS, TR_END, TR_PRODUCER_READY, TR_PRODUCER_ROUTED,
  TR_PRODUCER_DONE, TR_ROUTER_DATA, TR_GU_DATA, TR_ACT_READY, TR_GU_LAST, TR_DN_DATA, TR_POINTS = 24
};

// MAXB: activation blocks per lane of a row (every row has at most 1024 * MAXB values).
template <int QT, int MAXB>
__global__ void __launch_bounds__(NTHREADS, 1) moe_decode_kernel(const DecodeArgs args) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DecodePlan& p = args.p;
  const SmemLayout L = smem_layout(p);
  uint8_t* ring = smem + L.ring;
  uint8_t* xplanes = smem + L.xplanes;
  float2* xinfo = reinterpret_cast<float2*>(smem + L.xinfo);
  uint8_t* aplanes = smem + L.aplanes;
  float2* ainfo = reinterpret_cast<float2*>(smem + L.ainfo);
  float* probs = reinterpret_cast<float*>(smem + L.probs);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L.keys);
  float* gscore = reinterpret_cast<float*>(smem + L.gscore);
  int* rids = reinterpret_cast<int*>(smem + L.rids);
  float* rw = reinterpret_cast<float*>(smem + L.rw);  // [K] picks' weights, [K] = 1 (shared)
  Item* items = reinterpret_cast<Item*>(smem + L.items);  // the CTA's ring items, in order
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + p.nslots;
  uint64_t* routed_bar = empty + p.nslots;  // one arrival: the picks are in shared memory
  // [0] error seen, [1] generation
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);
  __shared__ uint32_t s_armed[MAX_SLOTS];  // uses of each ring slot armed so far
  volatile uint32_t* armed = s_armed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  // optional timeline: %globaltimer at fixed points, written by one thread
  auto trace = [&](int point) {
    if (args.trace && lane == 0 && (warp == 0 || warp == NCW))
      args.trace[(size_t)c * TR_POINTS + point] = globaltimer();
  };
  trace(TR_START);
  const CtaShare cs = cta_share(p, c);

  if (tid == 0) {
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);  // every consumer warp releases every item
    }
    mbar_init(routed_bar, 1);
    fence_mbar_init();
    misc[0] = 0;
    rw[p.K] = 1.f;  // the shared expert's weight
    for (int s = 0; s < MAX_SLOTS; ++s) s_armed[s] = 0;
  }
  // the item list, computed once (the producer and every consumer warp read it)
  for (int n = tid; n < cs.n_items; n += NTHREADS) items[n] = item_at(p, cs, c, n);
  __syncthreads();
  pdl_launch_dependents();

  // ======================= producer warp =======================
  // Lane s < nslots owns ring slot s and issues its items n = s, s + nslots, ...
  // in order (one issuing thread per slot: issue cost is per thread, so the
  // slots fill in parallel).
  if (warp == NCW) {
    const uint64_t pol = policy_evict_first();
    trace(TR_PRODUCER_READY);
    auto issue = [&](int n) -> bool {
      const Item it = items[n];
      const int s = n % p.nslots, use = n / p.nslots;
      if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1))) return false;
      uint8_t* dst = ring + (size_t)s * p.slot_bytes;
      mbar_arrive_expect_tx(&full[s], it.bytes);
      if (it.kind == ITEM_ROUTER) {
        bulk_g2s(dst, args.router_w + (size_t)it.row0 * p.H, it.bytes, &full[s], pol);
      } else {
        const uint8_t* base = it.slot < p.K ? args.experts + (size_t)rids[it.slot] * p.rec_bytes : args.shared;
        const int ff = slot_ff(p, it.slot);
        if (it.kind == ITEM_GU) {
          const uint32_t half = it.bytes / 2;
          bulk_g2s(dst, base + (size_t)it.row0 * p.rb_h, half, &full[s], pol);
          bulk_g2s(dst + half, base + (size_t)(ff + it.row0) * p.rb_h, half, &full[s], pol);
        } else {
          const uint8_t* dn = base + (size_t)2 * ff * p.rb_h;
          bulk_g2s(dst, dn + (size_t)it.row0 * dn_row_bytes(p, it.slot), it.bytes, &full[s], pol);
        }
      }
      // Consumers wait for a use only once it is armed. Arming use u follows the
      // producer's wait for the release of use u - 1, which every consumer warp gave
      // after seeing use u - 1 land: a consumer that sees the count has seen the
      // barrier pass the phase before u, so its parity wait for u cannot alias.
      armed[s] = (uint32_t)(use + 1);
      return true;
    };
    bool ok = true;
    if (lane < p.nslots) {
      bool routed = false;
      for (int n = lane; n < cs.n_items && ok; n += p.nslots) {
        if (n >= cs.n_pre && !routed) {
          // the picks (valid ids even when routing failed) are in shared memory after this wait
          ok = mbar_wait(routed_bar, 0);
          routed = true;
          if (args.trace && n == cs.n_pre) args.trace[(size_t)c * TR_POINTS + 16] = globaltimer();
          if (!ok) break;
        }
        ok = issue(n);
      }
    } else if (args.trace && lane >= 16 && lane < 21) {
      // timeline only: when the first routed items land (observing a phase is harmless)
      const int j = lane - 16, n = cs.n_pre + j;
      const int pts[5] = {18, 21, 22, 23, 20};
      if (n < cs.n_items) {
        const int s = n % p.nslots, use = n / p.nslots;
        const unsigned long long t0 = globaltimer();
        while (armed[s] <= (uint32_t)use && globaltimer() - t0 < MBAR_TIMEOUT_NS) __nanosleep(32);
        if (armed[s] > (uint32_t)use && mbar_wait(&full[s], use & 1u))
          args.trace[(size_t)c * TR_POINTS + pts[j]] = globaltimer();
      }
    }
    if (!ok) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
    trace(TR_PRODUCER_DONE);
    return;
  }

  // ======================= consumer warps =======================
  // Every item the producer issues is waited for and released below on every
  // path, so no copy is in flight when the CTA exits. Errors only skip results.
  const int H = p.H, K = p.K;
  const int nbH = H / 32;

  pdl_wait_prior_grids();  // x (and out, when accumulating) may come from the previous kernel
  trace(TR_PDL_DONE);
  if (tid == 0) misc[1] = ld_relaxed(args.ctrl + CTRL_GEN) + 1u;
  named_bar_sync(BAR_CONS, NCT);
  const uint32_t gen = misc[1];
  uint32_t* ctr_logits = args.ctrl + CTRL_LOGITS + (gen & 1u);
  uint32_t* ctr_part = args.ctrl + CTRL_ACT + (gen & 1u);
  uint32_t* ctr_slot = args.ctrl + CTRL_SLOT + (gen & 1u) * CTRL_SLOTS;  // columns published, per slot
  bool err = false;  // this thread saw a timeout

  // Item n's copy is awaited only once its slot's use has been armed: then the
  // slot's full barrier is in the phase of this use (a parity wait cannot alias an
  // older phase of the slot).
  auto wait_full = [&](int n) -> bool {
    const int s = n % p.nslots;
    const uint32_t use = (uint32_t)(n / p.nslots);
    // One lane per warp waits, sleeping briefly between reads (spinning warps would
    // crowd the shared-memory pipe the producer's barrier and copy instructions use);
    // then every lane takes the completed phase itself (an immediate try_wait).
    bool ok = true;
    if (lane == 0) {
      const unsigned long long t0 = globaltimer();
      uint32_t it = 0;
      while (armed[s] <= use) {
        __nanosleep(64);
        if ((++it & 15u) == 0 && globaltimer() - t0 > MBAR_TIMEOUT_NS) { ok = false; break; }
      }
      if (ok) ok = mbar_wait(&full[s], use & 1u);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) ok = mbar_wait(&full[s], use & 1u);
    if (!ok && lane == 0) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
    return ok;
  };
  auto release = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[n % p.nslots]);
  };
  auto slot_buf = [&](int n) -> const uint8_t* { return ring + (size_t)(n % p.nslots) * p.slot_bytes; };

  // Every warp walks the ring items [n0, n1) in order and releases each; an item's
  // work units are dealt to the warps in turn across the walk, so every warp has
  // work while the copies land. unit(it, buf, u) does unit u of item it.
  int ucount = 0;
  auto walk = [&](int n0, int n1, int per_unit, auto&& unit) {
    for (int n = n0; n < n1; ++n) {
      const Item it = items[n];
      const int units = ceil_div((int)it.nrows, per_unit);
      const int first = ucount + (warp - ucount % NCW + NCW) % NCW;
      // a warp with no unit in the item releases it at once: a warp with units
      // releases only after the copy landed, so the slot is not refilled early
      if (first >= ucount + units) {
        release(n);
        ucount += units;
        continue;
      }
      if (wait_full(n)) {
        if (args.trace && lane == 0 && n == cs.n_pre) args.trace[(size_t)c * TR_POINTS + TR_GU_DATA] = globaltimer();
        if (args.trace && lane == 0 && n == cs.n_pre + GU_ITEMS * cs.n_rc - 1)
          args.trace[(size_t)c * TR_POINTS + TR_GU_LAST] = globaltimer();
        if (args.trace && lane == 0 && n == cs.n_pre + GU_ITEMS * cs.n_rc)
          args.trace[(size_t)c * TR_POINTS + TR_DN_DATA] = globaltimer();
        const uint8_t* buf = slot_buf(n);
        for (int u = first; u < ucount + units; u += NCW) unit(it, buf, u - ucount);
      } else {
        err = true;
      }
      release(n);
      ucount += units;
    }
  };

  // ---- router rows: x (f32, from global) . router row -> published logits ----
  {
    walk(0, cs.n_r, 1, [&](const Item& it, const uint8_t* buf, int) {
      const float* row = reinterpret_cast<const float*>(buf);
      float acc = 0.f;
      for (int h = lane * 4; h < H; h += 128) {
        const float4 wv = *reinterpret_cast<const float4*>(row + h);
        const float4 xv = __ldcg(reinterpret_cast<const float4*>(args.x + h));
        acc = fmaf(wv.x, xv.x, acc);
        acc = fmaf(wv.y, xv.y, acc);
        acc = fmaf(wv.z, xv.z, acc);
        acc = fmaf(wv.w, xv.w, acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) st_relaxed_u64(args.logits + it.row0, tagged(gen, acc));
    });
    named_bar_sync(BAR_CONS, NCT);
    trace(TR_ROUTER_DONE);
    if (tid == 0) red_relaxed_add(ctr_logits, 1u);  // a hint: readers check each logit's generation
  }

  // ---- x -> activation blocks ----
  {
    bool ok = true;
    quant_blocks(args.x, nbH, xplanes, xinfo, nullptr, tid, NCT, 0u, ok);
  }
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_X_READY);

  // gate/up items [n0, n1): SwiGLU values of their pairs, published; then each of the
  // ncols columns (columns col(i)) counts itself in its slot (a hint: readers still
  // check every value's generation)
  auto gate_up = [&](int n0, int n1, bool shared, int ncols) {
    const RowMap mh = row_map(nbH, lane);
    ActBlock xc[MAXB];
#pragma unroll
    for (int i = 0; i < MAXB; ++i) {
      const int b = mh.sub + mh.lpr * i;
      if (b < nbH) load_act_block(xc[i], xplanes, xinfo, b);
    }
    walk(n0, n1, mh.rps, [&](const Item& it, const uint8_t* buf, int u) {
      const int r = u * mh.rps + mh.rsub;
      float gu[2] = {0.f, 0.f};
      if (r < ITEM_PAIRS) {
        const uint8_t* grow = buf + (size_t)r * p.rb_h;
        const uint8_t* urow = buf + (size_t)(ITEM_PAIRS + r) * p.rb_h;
#pragma unroll
        for (int i = 0; i < MAXB; ++i) {
          const int b = mh.sub + mh.lpr * i;
          if (b < nbH) {
            gu[0] += block_dot<QT>(grow, b, xc[i]);
            gu[1] += block_dot<QT>(urow, b, xc[i]);
          }
        }
      }
      group_sum_n(gu, mh.lpr);
      uint64_t* dst = args.act + (it.slot < K ? it.slot * p.F : K * p.F);
      if (r < ITEM_PAIRS && mh.sub == 0) st_relaxed_u64(dst + it.row0 + r, tagged(gen, silu_mul(gu[0], gu[1])));
    });
    named_bar_sync(BAR_CONS, NCT);
    if (tid < ncols) {
      int slot, bc;
      column_at(p, shared ? shared_column(p, cs, c, tid) : routed_column(p, c, tid), slot, bc);
      red_relaxed_add(ctr_slot + slot, 1u);
    }
  };

  // down items [n0, n1) of the CTA's columns (shared or routed): per column, the
  // slot's whole activation vector (every CTA of the slot has published its part)
  // -> activation blocks, then its down rows -> weighted, published output rows
  auto down = [&](bool shared, int ncols, int n0) {
    int n = n0;
    for (int i = 0; i < ncols; ++i) {
      const int g = shared ? shared_column(p, cs, c, i) : routed_column(p, c, i);
      int slot, bc;
      column_at(p, g, slot, bc);
      const int m = column_dn_items(p, slot, bc);
      if (m == 0) continue;
      const int ff = slot_ff(p, slot), nbF = ff / 32;
      // every column of the slot has published its values
      if (tid == 0 && !await_count(ctr_slot + slot, (uint32_t)slot_cols(p, slot))) misc[0] = 1;
      named_bar_sync(BAR_CONS, NCT);
      {
        bool ok = true;
        quant_blocks(args.act + (slot < K ? slot * p.F : K * p.F), nbF, aplanes, ainfo, nullptr, tid, NCT, gen, ok);
        if (!ok) err = true;
      }
      named_bar_sync(BAR_CONS, NCT);
      const RowMap mf = row_map(nbF, lane);
      ActBlock ac[MAXB];
#pragma unroll
      for (int j = 0; j < MAXB; ++j) {
        const int b = mf.sub + mf.lpr * j;
        if (b < nbF) load_act_block(ac[j], aplanes, ainfo, b);
      }
      const float w = rw[slot];
      const uint32_t rb = dn_row_bytes(p, slot);
      uint64_t* ys = args.ys + (size_t)slot * H;
      walk(n, n + m, mf.rps, [&](const Item& it, const uint8_t* buf, int u) {
        const int r = u * mf.rps + mf.rsub;
        float y = 0.f;
        if (r < (int)it.nrows) {
          const uint8_t* row = buf + (size_t)r * rb;
#pragma unroll
          for (int j = 0; j < MAXB; ++j) {
            const int b = mf.sub + mf.lpr * j;
            if (b < nbF) y += block_dot<QT>(row, b, ac[j]);
          }
        }
        y = group_sum(y, mf.lpr);
        if (r < (int)it.nrows && mf.sub == 0) st_relaxed_u64(ys + it.row0 + r, tagged(gen, w * y));
      });
      n += m;
      named_bar_sync(BAR_CONS, NCT);  // the activation blocks are reused by the next column
    }
  };

  // ---- two rounds of columns: the shared expert's (no routing needed), then, once the
  // picks are made, the routed ones; one copy of the code serves both rounds ----
  for (int round = 0; round < 2; ++round) {
    const bool shared = round == 0;
    const int ncols = shared ? cs.n_sc : cs.n_rc;
    const int n_gu = shared ? cs.n_r : cs.n_pre;  // first gate/up item of the round
    if (!shared) {
      // ---- routing: every CTA's logits are written; select ----
      if (tid == 0 && !await_count(ctr_logits, (uint32_t)p.nc)) misc[0] = 1;
      named_bar_sync(BAR_CONS, NCT);
      trace(TR_LOGITS);
      for (int e = tid; e < p.E; e += NCT) {
        bool ok = true;
        const float l = await_tagged(args.logits + e, ld_relaxed_u64(args.logits + e), gen, ok);
        if (!ok) err = true;
        const float pr = 1.f / (1.f + expf(-l));
        probs[e] = pr;
        keys[e] = order_key(pr + (args.bias ? __ldg(args.bias + e) : 0.f));
      }
      named_bar_sync(BAR_CONS, NCT);
      trace(TR_KEYS);
      if (p.G > 1) {
        // group score: the two largest s of the group, summed (multiset top-2)
        const int per = p.E / p.G;
        for (int g = warp; g < p.G; g += NCW) {
          float a = -INFINITY, bsec = -INFINITY;
          for (int e = g * per + lane; e < (g + 1) * per; e += 32) {
            uint32_t k = keys[e];
            float v = __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
            if (v > a) { bsec = a; a = v; } else if (v > bsec) { bsec = v; }
          }
    #pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            float oa = __shfl_xor_sync(0xffffffffu, a, o);
            float ob = __shfl_xor_sync(0xffffffffu, bsec, o);
            float hi = fmaxf(a, oa), lo = fminf(a, oa);
            bsec = fmaxf(lo, fmaxf(bsec, ob));
            a = hi;
          }
          if (lane == 0) gscore[g] = a + bsec;
        }
        named_bar_sync(BAR_CONS, NCT);
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
              bool kept = g < 32 ? ((keep_lo >> g) & 1u) : ((keep_hi >> (g - 32)) & 1u);
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
        if (p.E <= 256) topk_rounds<8>(keys, p.E, K, rids, lane);
        else if (p.E <= 512) topk_rounds<16>(keys, p.E, K, rids, lane);
        else topk_rounds<32>(keys, p.E, K, rids, lane);
        trace(TR_TOPK);
        // weights from the picked sigmoids
        const float pj = lane < K ? probs[rids[lane]] : 0.f;
        const float wsum = fmaxf(warp_sum(pj), args.norm_min);
        if (lane < K) {
          const float wj = pj / wsum * args.scale;
          rw[lane] = wj;
          if (c == 0) {
            if (args.topk_ids) args.topk_ids[lane] = rids[lane];
            if (args.topk_w) args.topk_w[lane] = wj;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(routed_bar);  // the producer may now fetch the picked experts
      }
      named_bar_sync(BAR_CONS, NCT);  // the picks and weights are visible to every consumer
      trace(TR_ROUTED);
    }
    gate_up(n_gu, n_gu + GU_ITEMS * ncols, shared, ncols);
    trace(shared ? TR_SHARED_DONE : TR_GU_DONE);
    down(shared, ncols, n_gu + GU_ITEMS * ncols);
  }
  trace(TR_COLS_DONE);
  if (tid == 0) red_relaxed_add(ctr_part, 1u);  // a hint: readers check each value's generation

  // ---- out[h] = sum over the slots of their weighted down rows, in slot order ----
  if (tid == 0 && !await_count(ctr_part, (uint32_t)p.nc)) misc[0] = 1;
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_PARTIALS);
  const int nslot = K + (p.Fs ? 1 : 0);
  for (int r = tid; r < cs.d_len; r += NCT) {
    const int h = cs.d_lo + r;
    constexpr int BATCH = 8;
    float acc = 0.f;
    for (int s0 = 0; s0 < nslot; s0 += BATCH) {
      uint64_t v[BATCH];
#pragma unroll
      for (int j = 0; j < BATCH; ++j)
        v[j] = s0 + j < nslot ? __ldcg(reinterpret_cast<const unsigned long long*>(args.ys + (size_t)(s0 + j) * H + h))
                              : 0ull;
#pragma unroll
      for (int j = 0; j < BATCH; ++j) {
        if (s0 + j < nslot) {
          bool ok = true;
          // slot order: the picks, then the shared expert (slot K)
          acc += await_tagged(args.ys + (size_t)(s0 + j) * H + h, v[j], gen, ok);
          if (!ok) err = true;
        }
      }
    }
    if (args.flags & FLAG_RESIDUAL) acc = __ldcg(args.x + h) + acc;
    if (args.flags & FLAG_ACCUMULATE) acc = __ldcg(args.out + h) + acc;
    if (!err) args.out[h] = acc;
  }
  if (err) misc[0] = 1;
  named_bar_sync(BAR_CONS, NCT);
  if (misc[0] != 0 && tid == 0) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_POLL_TIMEOUT);

  // ---- exit: the last CTA out prepares the next call's counters ----
  trace(TR_END);
  if (tid == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(args.ctrl + CTRL_EXIT, 1u) + 1u;
    if (done == (uint32_t)p.nc) {
      args.ctrl[CTRL_EXIT] = 0;
      args.ctrl[CTRL_LOGITS + ((gen + 1u) & 1u)] = 0;
      args.ctrl[CTRL_ACT + ((gen + 1u) & 1u)] = 0;
      for (int j = 0; j < CTRL_SLOTS; ++j) args.ctrl[CTRL_SLOT + ((gen + 1u) & 1u) * CTRL_SLOTS + j] = 0;
      args.ctrl[CTRL_GEN] = gen;
      __threadfence();
    }
  }
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
#include "decode_host.h"

namespace moe {

template <int QT, int MAXB>
static cudaError_t launch_one(const DecodeArgs& a, uint32_t smem, cudaStream_t st, bool pdl) {
  auto kern = moe_decode_kernel<QT, MAXB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.p.nc);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int QT, int MAXB>
static cudaError_t occupancy_one(uint32_t smem, int* blocks) {
  auto kern = moe_decode_kernel<QT, MAXB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, NTHREADS, smem);
}

#define MOE_DISPATCH(FN, ...)                                        \
  switch (qtype * 8 + maxb) {                                        \
    case 2 * 8 + 1: return FN<2, 1>(__VA_ARGS__);                    \
    case 2 * 8 + 2: return FN<2, 2>(__VA_ARGS__);                    \
    case 2 * 8 + 3: return FN<2, 3>(__VA_ARGS__);                    \
    case 3 * 8 + 1: return FN<3, 1>(__VA_ARGS__);                    \
    case 3 * 8 + 2: return FN<3, 2>(__VA_ARGS__);                    \
    case 3 * 8 + 3: return FN<3, 3>(__VA_ARGS__);                    \
    default: return cudaErrorInvalidValue;                           \
  }

cudaError_t decode_launch(const DecodeArgs& a, int qtype, int maxb, uint32_t smem, cudaStream_t st,
                          bool pdl) {
  MOE_DISPATCH(launch_one, a, smem, st, pdl)
}

cudaError_t decode_occupancy(int qtype, int maxb, uint32_t smem, int* blocks) {
  MOE_DISPATCH(occupancy_one, smem, blocks)
}

uint32_t decode_smem_bytes(const DecodePlan& p) { return smem_layout(p).total; }

}  // namespace moe
