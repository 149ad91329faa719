// Fused single-token MoE-FFN step (decode, T = 1) for sm_103a.
//
// One persistent CTA per SM runs the whole step:
//   router GEMV (F32 router rows, one row per item)          -> logits
//   all CTAs' logits written (arrival counter); sigmoid, selection bias,
//   (group) top-k and weight normalisation, computed by every CTA
//   gate/up GEMV of every pick and of the shared expert, SwiGLU -> act
//   all CTAs' act written (arrival counter); down GEMV of the output rows the
//   CTA owns, for every slot; weighted combine                     -> out
// Weights stream through a ring of shared-memory slots filled by 1-D bulk async
// copies (cp.async.bulk, completion counted on mbarriers) issued by the lanes
// of one producer warp; eleven consumer warps compute. Down rows bypass the ring: the
// producer prefetches the CTA's down rows into L2 (the shared expert's at once,
// the picks' as soon as they are known) and the consumers read them with plain
// loads once the activations are complete. Routing-independent rows (router,
// shared expert) are requested before the kernel waits on the previous grid
// (programmatic dependent launch).
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
constexpr int BAR_CONS = 1;          // named barrier: consumer warps only
constexpr int MAX_SLOTS = 16;        // ring slots (one issuing producer lane each)

// Shared-memory carve-up (byte offsets, computed identically on host and device).
struct SmemLayout {
  uint32_t ring, qplanes, qinfo, xf, probs, partial, keys, gscore, rids, rw, bars, misc, total;
};

MOE_HD uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

MOE_HD SmemLayout smem_layout(const DecodePlan& p) {
  SmemLayout L;
  uint32_t o = 0;
  L.ring = o;
  o += (uint32_t)p.nslots * p.slot_bytes;
  int nb_act = (p.K * p.F + p.Fs) / 32;
  int nbq = nb_act > p.H / 32 ? nb_act : p.H / 32;
  L.qplanes = o = align_up(o, 16);
  o += (uint32_t)nbq * 96u;
  L.qinfo = o = align_up(o, 16);
  o += (uint32_t)nbq * 8u;
  L.xf = o = align_up(o, 16);
  o += (uint32_t)p.H * 4u;
  L.probs = o = align_up(o, 16);
  o += (uint32_t)p.E * 4u;
  L.partial = o = align_up(o, 16);
  o += (uint32_t)(p.K + 1) * (uint32_t)p.max_dn_rows * 4u;
  L.keys = o = align_up(o, 16);
  o += (uint32_t)p.E * 4u;
  L.gscore = o = align_up(o, 16);
  o += 64u * 4u;
  L.rids = o = align_up(o, 16);
  o += 32u * 4u;
  L.rw = o;
  o += 32u * 4u;
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
// The source is either an f32 vector or published words of generation `gen`
// (then every value is awaited; `ok` is cleared on a timeout).
template <typename Src>
__device__ __forceinline__ void quant_blocks(const Src* src, int nb, uint8_t* planes, float2* info,
                                             float* copy, int t, int nthreads, uint32_t gen, bool& ok) {
  for (int base = 0; base < 4 * nb; base += nthreads) {
    const int idx = base + t, b = idx >> 2, qq = idx & 3;
    const bool active = idx < 4 * nb;
    float v[8];
    if (active) {
      if constexpr (sizeof(Src) == 4) {
        const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)b * 32 + qq * 8);
        const float4 a = __ldcg(s4), c = __ldcg(s4 + 1);
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
constexpr int ROWS_PER_STEP = 4;  // row steps a warp keeps in flight together

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }


// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Timeline points (MOE_TRACE): one u64 %globaltimer value each, per CTA.
enum TracePoint : int {
  TR_START = 0, TR_PDL_DONE, TR_X_READY, TR_PRE_DONE, TR_LOGITS, TR_ROUTED, TR_GU_DONE,
  TR_ACT_READY, TR_DN_DONE, TR_END, TR_PRODUCER_READY, TR_PRODUCER_ROUTED, TR_PRODUCER_DONE,
  TR_ROUTER_DATA, TR_ROUTER_DONE, TR_ACT_COUNTED, TR_POINTS = 24
};

template <int QT, int MAXB>
__global__ void __launch_bounds__(NTHREADS, 1) moe_decode_kernel(const DecodeArgs args) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DecodePlan& p = args.p;
  const SmemLayout L = smem_layout(p);
  uint8_t* ring = smem + L.ring;
  uint8_t* qplanes = smem + L.qplanes;
  float2* qinfo = reinterpret_cast<float2*>(smem + L.qinfo);
  float* xf = reinterpret_cast<float*>(smem + L.xf);
  float* probs = reinterpret_cast<float*>(smem + L.probs);
  float* partial = reinterpret_cast<float*>(smem + L.partial);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L.keys);
  float* gscore = reinterpret_cast<float*>(smem + L.gscore);
  int* rids = reinterpret_cast<int*>(smem + L.rids);
  float* rw = reinterpret_cast<float*>(smem + L.rw);
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
    for (int s = 0; s < MAX_SLOTS; ++s) s_armed[s] = 0;
  }
  __syncthreads();
  pdl_launch_dependents();

  // ======================= producer warp =======================
  // Lane s < nslots owns ring slot s and issues its items n = s, s + nslots, ...
  // in order (one issuing thread per slot: issue cost is per thread, so the
  // slots fill in parallel). Lanes 16..31 prefetch the CTA's down rows into L2.
  if (warp == NCW) {
    const uint64_t pol = policy_evict_first();
    trace(TR_PRODUCER_READY);
    auto issue = [&](int n) -> bool {
      const Item it = item_at(p, cs, n);
      const int s = n % p.nslots, use = n / p.nslots;
      if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1))) return false;
      uint8_t* dst = ring + (size_t)s * p.slot_bytes;
      mbar_arrive_expect_tx(&full[s], it.bytes);
      if (it.kind == ITEM_ROUTER) {
        bulk_g2s(dst, args.router_w + (size_t)it.row0 * p.H, it.bytes, &full[s], pol);
      } else {
        const uint8_t* base = it.slot < p.K ? args.experts + (size_t)rids[it.slot] * p.rec_bytes : args.shared;
        const int ff = slot_ff(p, it.slot);
        const uint32_t half = it.bytes / 2;
        bulk_g2s(dst, base + (size_t)it.row0 * p.rb_h, half, &full[s], pol);
        bulk_g2s(dst + half, base + (size_t)(ff + it.row0) * p.rb_h, half, &full[s], pol);
      }
      __threadfence_block();                   // the arrive above is visible before the count
      armed[s] = (uint32_t)(use + 1);          // this slot's uses are armed in order
      return true;
    };
    // down rows [d_lo, d_lo + d_len) of slot s go to L2 ahead of their use
    auto prefetch_down = [&](int s) {
      const uint8_t* base = s < p.K ? args.experts + (size_t)rids[s] * p.rec_bytes : args.shared;
      const uint32_t rb = dn_row_bytes(p, s);
      if (cs.d_len > 0)
        bulk_prefetch_l2(base + (size_t)2 * slot_ff(p, s) * p.rb_h + (size_t)cs.d_lo * rb,
                         (uint32_t)cs.d_len * rb);
    };
    bool ok = true;
    if (lane < p.nslots) {
      bool routed = false;
      for (int n = lane; n < cs.n_items && ok; n += p.nslots) {
        if (n >= cs.n_pre && !routed) {
          // the picks (valid ids even when routing failed) are in shared memory after this wait
          ok = mbar_wait(routed_bar, 0);
          routed = true;
          trace(TR_PRODUCER_ROUTED);
          if (!ok) break;
        }
        ok = issue(n);
      }
    } else if (lane >= 16) {
      if (lane == 31 && p.Fs) prefetch_down(p.K);
      if (lane - 16 < p.K) {
        ok = mbar_wait(routed_bar, 0);
        if (ok)
          for (int j = lane - 16; j < p.K; j += 16) prefetch_down(j);
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
  const int NCT = NCW * 32;

  pdl_wait_prior_grids();  // x (and out, when accumulating) may come from the previous kernel
  trace(TR_PDL_DONE);
  if (tid == 0) misc[1] = ld_relaxed(args.ctrl + CTRL_GEN) + 1u;

  // activation blocks of x -> shared planes, and an f32 copy for the router
  bool err = false;  // this thread saw a timeout
  {
    bool ok = true;
    quant_blocks(args.x, nbH, qplanes, qinfo, xf, tid, NCT, 0u, ok);
  }
  named_bar_sync(BAR_CONS, NCT);
  const uint32_t gen = misc[1];
  uint32_t* ctr_logits = args.ctrl + CTRL_LOGITS + (gen & 1u);
  uint32_t* ctr_act = args.ctrl + CTRL_ACT + (gen & 1u);
  trace(TR_X_READY);

  // this lane's x blocks for gate/up rows, kept in registers
  const RowMap mh = row_map(nbH, lane);
  ActBlock xc[MAXB];
#pragma unroll
  for (int i = 0; i < MAXB; ++i) {
    int b = mh.sub + mh.lpr * i;
    if (b < nbH) load_act_block(xc[i], qplanes, qinfo, b);
  }

  // Item n's copy is awaited only once its slot's use has been armed: then the
  // slot's full barrier is in the phase of this use (a parity wait cannot alias an
  // older phase of the slot).
  auto wait_full = [&](int n) -> bool {
    const int s = n % p.nslots;
    const uint32_t use = (uint32_t)(n / p.nslots);
    bool ok = true;
    if (armed[s] <= use) {
      const unsigned long long t0 = globaltimer();
      uint32_t it = 0;
      while (armed[s] <= use)
        if ((++it & 63u) == 0 && globaltimer() - t0 > MBAR_TIMEOUT_NS) { ok = false; break; }
    }
    if (ok) ok = mbar_wait(&full[s], use & 1u);
    if (!ok && lane == 0) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
    return ok;
  };
  auto release = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[n % p.nslots]);
  };
  auto slot_buf = [&](int n) -> const uint8_t* { return ring + (size_t)(n % p.nslots) * p.slot_bytes; };

  // gate/up unit: pairs unit*rps + [0, rps) of an item of slot `slot` (its pairs
  // [row0, row0 + m), gate rows then up rows in buf), one pair per lane group
  auto do_gu_unit = [&](const Item& it, const uint8_t* buf, int unit) {
    const int m = (int)it.nrows;
    const int r = unit * mh.rps + mh.rsub;
    float gu[2] = {0.f, 0.f};
    if (r < m) {
      const uint8_t* grow = buf + (size_t)r * p.rb_h;
      const uint8_t* urow = buf + (size_t)(m + r) * p.rb_h;
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
    if (r < m && mh.sub == 0) st_relaxed_u64(dst + it.row0 + r, tagged(gen, silu_mul(gu[0], gu[1])));
  };

  // router item: one row of H f32 values in buf, dot with the f32 copy of x
  auto do_router = [&](const Item& it, const float* buf) {
    float acc = 0.f;
    for (int h = lane * 4; h < H; h += 128) {
      float4 wv = *reinterpret_cast<const float4*>(buf + h);
      float4 xv = *reinterpret_cast<const float4*>(xf + h);
      acc = fmaf(wv.x, xv.x, acc);
      acc = fmaf(wv.y, xv.y, acc);
      acc = fmaf(wv.z, xv.z, acc);
      acc = fmaf(wv.w, xv.w, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) st_relaxed_u64(args.logits + it.row0, tagged(gen, acc));
  };

  // Every warp walks the ring items [n0, n1) in order and releases each; the
  // items' work units (a router row, or rps gate/up pairs) are dealt to the warps
  // in turn across the walk, so every warp has work while the copies land.
  auto walk_items = [&](int n0, int n1) {
    int ucount = 0;
    for (int n = n0; n < n1; ++n) {
      const Item it = item_at(p, cs, n);
      const int units = it.kind == ITEM_ROUTER ? 1 : ceil_div((int)it.nrows, mh.rps);
      const int first = ucount + (warp - ucount % NCW + NCW) % NCW;
      if (wait_full(n)) {
        if (n == 0) trace(TR_ROUTER_DATA);
        const uint8_t* buf = slot_buf(n);
        for (int u = first; u < ucount + units; u += NCW) {
          if (it.kind == ITEM_ROUTER) do_router(it, reinterpret_cast<const float*>(buf));
          else do_gu_unit(it, buf, u - ucount);
        }
      } else {
        err = true;
      }
      release(n);
      ucount += units;
    }
  };

  // ---- router rows: write the logits, then count this CTA in ----
  walk_items(0, cs.n_r);
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_ROUTER_DONE);
  if (tid == 0) red_relaxed_add(ctr_logits, 1u);  // a hint: readers check each logit's generation
  trace(TR_PRE_DONE);

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
  trace(TR_ROUTED);

  // ---- gate/up items: the shared expert's (already in the ring), then the picks' ----
  walk_items(cs.n_r, cs.n_items);
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_GU_DONE);
  if (tid == 0) {
    red_relaxed_add(ctr_act, 1u);  // a hint: readers check each activation's generation
    if (!await_count(ctr_act, (uint32_t)p.nc)) misc[0] = 1;
  }
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_ACT_COUNTED);

  // ---- activations of every slot -> shared planes ----
  {
    bool ok = true;
    quant_blocks(args.act, (K * p.F + p.Fs) / 32, qplanes, qinfo, nullptr, tid, NCT, gen, ok);
    if (!ok) err = true;
  }
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_ACT_READY);

  // ---- down rows, read through L2: partial[slot][row] = W_down[row] . act[slot] ----
  // Tasks: for every slot (shared first), the CTA's output rows in runs of
  // rps * ROWS_PER_STEP rows (one warp step each), dealt to the warps in turn.
  {
    const int nslot = K + (p.Fs ? 1 : 0);
    int t_first = 0;  // index of the slot's first task in the deal
    for (int si = 0; si < nslot; ++si) {
      const int slot = p.Fs ? (si == 0 ? K : si - 1) : si;
      const int nb = slot_ff(p, slot) / 32;
      const RowMap mf = row_map(nb, lane);
      const int run = mf.rps * ROWS_PER_STEP;
      const int ntask = ceil_div(cs.d_len, run);
      // this warp's tasks of the slot: t with (t_first + t) % NCW == warp
      const int t0 = (warp - t_first % NCW + NCW) % NCW;
      if (t0 < ntask) {
        const int b0 = (slot < K ? slot * p.F : K * p.F) / 32;  // first act block of the slot
        const uint32_t rb = dn_row_bytes(p, slot);
        const uint8_t* base = slot < K ? args.experts + (size_t)rids[slot] * p.rec_bytes : args.shared;
        const uint8_t* dn = base + (size_t)2 * slot_ff(p, slot) * p.rb_h;
        ActBlock ac[MAXB];
#pragma unroll
        for (int i = 0; i < MAXB; ++i) {
          const int b = mf.sub + mf.lpr * i;
          if (b < nb) load_act_block(ac[i], qplanes, qinfo, b0 + b);
        }
        float* part = partial + slot * p.max_dn_rows;
        for (int t = t0; t < ntask; t += NCW) {
          float y[ROWS_PER_STEP];
#pragma unroll
          for (int k = 0; k < ROWS_PER_STEP; ++k) {
            const int r = t * run + k * mf.rps + mf.rsub;
            y[k] = 0.f;
            if (r < cs.d_len) {
              const uint8_t* row = dn + (size_t)(cs.d_lo + r) * rb;
#pragma unroll
              for (int i = 0; i < MAXB; ++i) {
                const int b = mf.sub + mf.lpr * i;
                if (b < nb) y[k] += block_dot_g<QT>(row, b, ac[i]);
              }
            }
          }
          group_sum_n(y, mf.lpr);
#pragma unroll
          for (int k = 0; k < ROWS_PER_STEP; ++k) {
            const int r = t * run + k * mf.rps + mf.rsub;
            if (r < cs.d_len && mf.sub == 0) part[r] = y[k];
          }
        }
      }
      t_first += ntask;
    }
  }
  if (err) misc[0] = 1;
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_DN_DONE);

  // ---- combine: out[h] = sum_j w_j y_j[h] + shared[h] (+ x[h] | + out[h]) ----
  if (misc[0] == 0) {
    for (int r = tid; r < cs.d_len; r += NCT) {
      float acc = 0.f;
      for (int j = 0; j < K; ++j) acc = fmaf(rw[j], partial[j * p.max_dn_rows + r], acc);
      if (p.Fs) acc += partial[K * p.max_dn_rows + r];
      const int h = cs.d_lo + r;
      if (args.flags & FLAG_RESIDUAL) acc = __ldcg(args.x + h) + acc;
      if (args.flags & FLAG_ACCUMULATE) acc = __ldcg(args.out + h) + acc;
      args.out[h] = acc;
    }
  } else if (tid == 0) {
    atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_POLL_TIMEOUT);
  }

  // ---- exit: the last CTA out prepares the next call's counters ----
  named_bar_sync(BAR_CONS, NCT);
  trace(TR_END);
  if (tid == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(args.ctrl + CTRL_EXIT, 1u) + 1u;
    if (done == (uint32_t)p.nc) {
      args.ctrl[CTRL_EXIT] = 0;
      args.ctrl[CTRL_LOGITS + ((gen + 1u) & 1u)] = 0;
      args.ctrl[CTRL_ACT + ((gen + 1u) & 1u)] = 0;
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
