// Fused single-token MoE-FFN step (decode, T = 1) for sm_103a.
//
// One persistent CTA per SM runs the whole step:
//   router GEMV (F32 router rows, one row per item)         -> logits
//   grid barrier A; sigmoid, selection bias, (group) top-k, weight normalisation
//   gate/up GEMV of every picked expert and of the shared expert, SwiGLU -> act
//   grid barrier B; down GEMV of every slot, weighted combine         -> out
// Weights stream through a ring of shared-memory slots filled by 1-D bulk async
// copies (cp.async.bulk, completion counted on mbarriers) issued by one
// producer warp; seven consumer warps compute. Routing-independent rows
// (router, shared expert) are requested before the kernel waits on the
// previous grid (programmatic dependent launch), so their latency overlaps the
// previous kernel.
//
// Dequant-dot: a 4-bit block (ggml Q4_0/Q4_1, 32 values) times 32 activations.
// Activations are held per 32-block as integers v = x * 2^k with |v| < 2^22
// (power-of-two block scale; error at most 2^-22 of the block's largest
// magnitude), split into byte planes; dp4a forms sum(q * v) exactly in int32,
// the block result d * s * sum(q v) (+ m * s * sum(v) for Q4_1, - 8 d s sum(v)
// for Q4_0) is accumulated in fp32. The block formats and the per-block dot
// identity follow flint_moe_ssd.js (WGSL section, Q41DOT and its comment).
#include <cstdint>
#include <cuda_fp16.h>

#include "common.cuh"
#include "plan.h"

namespace moe {

constexpr int NCW = 7;               // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int BAR_CONS = 1;          // named barrier: consumer warps only
constexpr int BAR_ROUTED = 2;        // named barrier: consumers arrive, producer waits

// Shared-memory carve-up (byte offsets, computed identically on host and device).
struct SmemLayout {
  uint32_t ring, qplanes, qinfo, items, partial, keys, gscore, rids, rw, bars, misc, total;
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
  L.items = o = align_up(o, 16);
  o += (uint32_t)p.max_items * (uint32_t)sizeof(Item);
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
  o += (uint32_t)p.nslots * 16u;
  L.misc = o = align_up(o, 16);
  o += 16u;
  L.total = align_up(o, 128);
  return L;
}

// ---------------------------------------------------------------------------
// Activation blocks
// ---------------------------------------------------------------------------

// Quantise one 32-value block held one value per lane; writes the three byte
// planes (plane P, value i at byte P*32 + i) and {scale, sum(v)}.
__device__ __forceinline__ void quant_block(float xv, uint8_t* planes, float2* info, int lane) {
  float amax = warp_max(fabsf(xv));
  int eb = (int)((__float_as_uint(amax) >> 23) & 0xFF);  // amax < 2^(eb - 126)
  float inv = 0.f, s = 0.f;
  if (eb >= 30) {  // |x| < 2^-97 everywhere: the block is taken as zero
    inv = __uint_as_float((uint32_t)(148 - eb + 127) << 23);   // 2^(148 - eb)
    s = __uint_as_float((uint32_t)(eb - 148 + 127) << 23);     // 2^(eb - 148)
  }
  int v = (inv != 0.f) ? round_small(xv * inv) : 0;  // |v| <= 2^22
  planes[lane] = (uint8_t)(v & 0xFF);
  planes[32 + lane] = (uint8_t)((v >> 8) & 0xFF);
  planes[64 + lane] = (uint8_t)((v >> 16) & 0xFF);
  int X = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) *info = make_float2(s, (float)X);
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

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// ---------------------------------------------------------------------------
// Grid barrier on a monotonic counter (one thread per CTA). Returns false on
// timeout and records it in the status word.
// ---------------------------------------------------------------------------
__device__ bool grid_barrier(uint32_t* ctrl, int word, uint32_t target, uint32_t where) {
  __threadfence();
  red_release_add(ctrl + word, 1u);
  unsigned long long t0 = globaltimer();
  uint32_t it = 0;
  while (ld_acquire(ctrl + word) < target) {
    if ((++it & 255u) == 0 && globaltimer() - t0 > BARRIER_TIMEOUT_NS) {
      atomicOr(ctrl + CTRL_STATUS, DEV_ERR_BARRIER_TIMEOUT);
      atomicCAS(ctrl + CTRL_WHERE, 0u, where);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int QT, int MAXB>
__global__ void __launch_bounds__(NTHREADS, 2) moe_decode_kernel(const DecodeArgs args) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DecodePlan& p = args.p;
  const SmemLayout L = smem_layout(p);
  uint8_t* ring = smem + L.ring;
  uint8_t* qplanes = smem + L.qplanes;
  float2* qinfo = reinterpret_cast<float2*>(smem + L.qinfo);
  Item* items = reinterpret_cast<Item*>(smem + L.items);
  float* partial = reinterpret_cast<float*>(smem + L.partial);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L.keys);
  float* gscore = reinterpret_cast<float*>(smem + L.gscore);
  int* rids = reinterpret_cast<int*>(smem + L.rids);
  float* rw = reinterpret_cast<float*>(smem + L.rw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + p.nslots;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);  // [0] abort, [1] router rows done

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  __shared__ int s_n_items, s_n_pre, s_n_gu_end, s_dn_lo, s_dn_hi;

  if (tid == 0) {
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
    int n_pre, n_gu_end, dn_lo, dn_hi;
    s_n_items = build_items(p, c, items, &n_pre, &n_gu_end, &dn_lo, &dn_hi);
    s_n_pre = n_pre;
    s_n_gu_end = n_gu_end;
    s_dn_lo = dn_lo;
    s_dn_hi = dn_hi;
    misc[0] = 0;
    misc[1] = 0;
  }
  __syncthreads();
  pdl_launch_dependents();
  const int n_items = s_n_items, n_pre = s_n_pre, n_gu_end = s_n_gu_end;
  const int dn_lo = s_dn_lo, dn_hi = s_dn_hi;
  int n_router = 0;
  {
    int lo, hi;
    share(p.E, c, p.nc, lo, hi);
    n_router = hi - lo;
  }

  // ======================= producer warp =======================
  if (warp == NCW) {
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int n) -> bool {
      const Item it = items[n];
      const int s = n % p.nslots, use = n / p.nslots;
      if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1))) return false;
      uint8_t* dst = ring + (size_t)s * p.slot_bytes;
      mbar_arrive_expect_tx(&full[s], it.bytes);
      if (it.kind == ITEM_ROUTER) {
        bulk_g2s(dst, args.router_w + (size_t)it.row0 * p.H, it.bytes, &full[s], pol);
      } else {
        const uint8_t* base;
        if (it.slot < p.K) base = args.experts + (size_t)rids[it.slot] * p.rec_bytes;
        else base = args.shared;
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
      return true;
    };
    bool ok = true;
    if (lane == 0) {
      for (int n = 0; n < n_pre && ok; ++n) ok = issue(n);
      if (!ok) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
    }
    __syncwarp();
    named_bar_sync(BAR_ROUTED, NTHREADS);  // the routing is in shared memory now
    if (lane == 0 && ok && misc[0] == 0) {
      for (int n = n_pre; n < n_items && ok; ++n) ok = issue(n);
      if (!ok) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
    }
    return;
  }

  // ======================= consumer warps =======================
  const int H = p.H, K = p.K;
  const int nbH = H / 32;
  bool abort = false;

  pdl_wait_prior_grids();  // x (and out, when accumulating) may come from the previous kernel

  // activation blocks of x -> shared planes
  for (int b = warp; b < nbH; b += NCW) {
    float xv = __ldcg(args.x + b * 32 + lane);
    quant_block(xv, qplanes + (size_t)b * 96, qinfo + b, lane);
  }
  named_bar_sync(BAR_CONS, NCW * 32);

  // this lane's x blocks for gate/up rows, kept in registers
  const RowMap mh = row_map(nbH, lane);
  ActBlock xc[MAXB];
#pragma unroll
  for (int i = 0; i < MAXB; ++i) {
    int b = mh.sub + mh.lpr * i;
    if (b < nbH) load_act_block(xc[i], qplanes, qinfo, b);
  }

  auto wait_full = [&](int n) -> bool {
    const int s = n % p.nslots;
    bool ok = mbar_wait(&full[s], (uint32_t)((n / p.nslots) & 1));
    if (!ok && lane == 0) atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_MBAR_TIMEOUT);
    return ok;
  };
  auto release = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[n % p.nslots]);
  };

  // gate/up item: pairs [row0, row0 + m) of slot `slot`; gate rows then up rows in buf
  auto do_gu = [&](const Item& it, const uint8_t* buf) {
    const int m = (int)it.nrows;
    const int ff = slot_ff(p, it.slot);
    float* dst = args.act + (it.slot < K ? it.slot * p.F : K * p.F);
    for (int r0 = 0; r0 < m; r0 += mh.rps) {
      const int r = r0 + mh.rsub;
      float g = 0.f, u = 0.f;
      if (r < m) {
        const uint8_t* grow = buf + (size_t)r * p.rb_h;
        const uint8_t* urow = buf + (size_t)(m + r) * p.rb_h;
#pragma unroll
        for (int i = 0; i < MAXB; ++i) {
          int b = mh.sub + mh.lpr * i;
          if (b < nbH) {
            g += block_dot<QT>(grow, b, xc[i]);
            u += block_dot<QT>(urow, b, xc[i]);
          }
        }
      }
      g = group_sum(g, mh.lpr);
      u = group_sum(u, mh.lpr);
      if (r < m && mh.sub == 0) dst[it.row0 + r] = silu_mul(g, u);
    }
    (void)ff;
  };

  // router item: one row of H f32 values in buf, dot with x (global, fp32)
  auto do_router = [&](const Item& it, const float* buf) {
    float acc = 0.f;
    for (int h = lane * 4; h < H; h += 128) {
      float4 wv = *reinterpret_cast<const float4*>(buf + h);
      float4 xv = __ldcg(reinterpret_cast<const float4*>(args.x + h));
      acc = fmaf(wv.x, xv.x, acc);
      acc = fmaf(wv.y, xv.y, acc);
      acc = fmaf(wv.z, xv.z, acc);
      acc = fmaf(wv.w, xv.w, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      args.logits[it.row0] = acc;
      __threadfence();
      uint32_t done = atomicAdd(&misc[1], 1u) + 1;
      if ((int)done == n_router) {
        // every router row of this CTA is written: arrive at barrier A
        __threadfence();
        red_release_add(args.ctrl + CTRL_BAR_A, 1u);
      }
    }
  };

  // ---- routing-independent items: router rows, shared gate/up ----
  for (int n = warp; n < n_pre; n += NCW) {
    const Item it = items[n];
    if (!wait_full(n)) { abort = true; release(n); continue; }
    const uint8_t* buf = ring + (size_t)(n % p.nslots) * p.slot_bytes;
    if (it.kind == ITEM_ROUTER) do_router(it, reinterpret_cast<const float*>(buf));
    else do_gu(it, buf);
    release(n);
  }
  if (n_router == 0 && tid == 0) red_release_add(args.ctrl + CTRL_BAR_A, 1u);

  // ---- barrier A: every logit of the token is written ----
  if (tid == 0) {
    unsigned long long t0 = globaltimer();
    uint32_t itc = 0;
    while (ld_acquire(args.ctrl + CTRL_BAR_A) < (uint32_t)p.nc) {
      if ((++itc & 255u) == 0 && globaltimer() - t0 > BARRIER_TIMEOUT_NS) {
        atomicOr(args.ctrl + CTRL_STATUS, DEV_ERR_BARRIER_TIMEOUT);
        atomicCAS(args.ctrl + CTRL_WHERE, 0u, 1u);
        misc[0] = 1;
        break;
      }
    }
  }
  if (abort && lane == 0) misc[0] = 1;
  named_bar_sync(BAR_CONS, NCW * 32);
  abort = misc[0] != 0;

  // ---- routing ----
  if (!abort) {
    // selection keys s = sigmoid(logit) + bias
    for (int e = tid; e < p.E; e += NCW * 32) {
      float l = __ldcg(args.logits + e);
      float pr = 1.f / (1.f + expf(-l));
      float sv = pr + (args.bias ? args.bias[e] : 0.f);
      keys[e] = order_key(sv);
    }
    named_bar_sync(BAR_CONS, NCW * 32);
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
      named_bar_sync(BAR_CONS, NCW * 32);
    }
    if (warp == 0) {
      // kept groups: groups_used rounds of the largest group score, lowest group on ties
      uint32_t keep_mask_lo = 0xffffffffu, keep_mask_hi = 0xffffffffu;  // groups 0..63
      if (p.G > 1) {
        keep_mask_lo = keep_mask_hi = 0;
        for (int j = 0; j < p.Gu; ++j) {
          int best = -1;
          float bv = 0.f;
          for (int g = 0; g < p.G; ++g) {
            bool kept = g < 32 ? ((keep_mask_lo >> g) & 1u) : ((keep_mask_hi >> (g - 32)) & 1u);
            if (!kept && (best < 0 || gscore[g] > bv)) { best = g; bv = gscore[g]; }
          }
          if (best < 32) keep_mask_lo |= 1u << best; else keep_mask_hi |= 1u << (best - 32);
        }
      }
      const int per = p.E / p.G;
      auto allowed = [&](int e) -> bool {
        if (p.G <= 1) return true;
        int g = e / per;
        return g < 32 ? ((keep_mask_lo >> g) & 1u) : ((keep_mask_hi >> (g - 32)) & 1u);
      };
      // lane-local best (largest key, lowest index) over e = lane + 32 i, skipping taken ones
      uint32_t taken = 0u;  // bit i: expert lane + 32 i already picked
      uint32_t bk = 0u;
      int bi = 0x7fffffff;
      auto local_best = [&]() {
        bk = 0u;
        bi = 0x7fffffff;
        for (int i = 0, e = lane; e < p.E; ++i, e += 32) {
          if (!allowed(e) || ((taken >> i) & 1u)) continue;
          uint32_t k = keys[e];
          if (bi == 0x7fffffff || k > bk) { bk = k; bi = e; }
        }
      };
      local_best();
      for (int j = 0; j < K; ++j) {
        uint32_t mk = __reduce_max_sync(0xffffffffu, bi != 0x7fffffff ? bk : 0u);
        unsigned cand = (bi != 0x7fffffff && bk == mk) ? (unsigned)bi : 0xffffffffu;
        int win = (int)__reduce_min_sync(0xffffffffu, cand);
        if (win < 0 || win >= p.E) win = 0;  // unreachable for a valid configuration
        if (lane == 0) rids[j] = win;
        if ((win & 31) == lane) {
          taken |= 1u << (win >> 5);
          local_best();
        }
      }
      __syncwarp();
      // weights from the picked sigmoids
      float pj = 0.f;
      if (lane < K) {
        float l = __ldcg(args.logits + rids[lane]);
        pj = 1.f / (1.f + expf(-l));
      }
      float wsum = fmaxf(warp_sum(pj), args.norm_min);
      if (lane < K) {
        float wj = pj / wsum * args.scale;
        rw[lane] = wj;
        if (c == 0) {
          if (args.topk_ids) args.topk_ids[lane] = rids[lane];
          if (args.topk_w) args.topk_w[lane] = wj;
        }
      }
    }
    named_bar_sync(BAR_CONS, NCW * 32);
  }
  const bool routed_ok = !abort;          // otherwise the producer issues nothing more
  named_bar_arrive(BAR_ROUTED, NTHREADS);  // the producer may now fetch the picked experts

  // ---- routed gate/up items ----
  for (int n = n_pre + warp; n < n_gu_end; n += NCW) {
    if (abort) break;
    const Item it = items[n];
    if (!wait_full(n)) { abort = true; release(n); continue; }
    do_gu(it, ring + (size_t)(n % p.nslots) * p.slot_bytes);
    release(n);
  }

  // ---- barrier B: every activation of every slot is written ----
  named_bar_sync(BAR_CONS, NCW * 32);
  if (tid == 0) {
    if (abort || misc[0]) {
      misc[0] = 1;
      red_release_add(args.ctrl + CTRL_BAR_B, 1u);
    } else if (!grid_barrier(args.ctrl, CTRL_BAR_B, (uint32_t)p.nc, 2u)) {
      misc[0] = 1;
    }
  }
  named_bar_sync(BAR_CONS, NCW * 32);
  abort = misc[0] != 0;

  if (!abort) {
    // activation blocks of every slot -> shared planes (x planes are no longer needed)
    const int nb_act = (K * p.F + p.Fs) / 32;
    for (int b = warp; b < nb_act; b += NCW) {
      float av = __ldcg(args.act + b * 32 + lane);
      quant_block(av, qplanes + (size_t)b * 96, qinfo + b, lane);
    }
    named_bar_sync(BAR_CONS, NCW * 32);
  }

  // ---- down items: partial[slot][row] = W_down[row] . act[slot] ----
  const int dn_rows = dn_hi - dn_lo;
  if (!abort) {
    for (int n = n_gu_end + warp; n < n_items; n += NCW) {
      const Item it = items[n];
      if (!wait_full(n)) { abort = true; release(n); continue; }
      const uint8_t* buf = ring + (size_t)(n % p.nslots) * p.slot_bytes;
      const int ff = slot_ff(p, it.slot);
      const int nb = ff / 32;
      const uint32_t rb = dn_row_bytes(p, it.slot);
      const int b0 = (it.slot < K ? it.slot * p.F : K * p.F) / 32;  // first act block of the slot
      const RowMap mf = row_map(nb, lane);
      ActBlock ac[MAXB];
#pragma unroll
      for (int i = 0; i < MAXB; ++i) {
        int b = mf.sub + mf.lpr * i;
        if (b < nb) load_act_block(ac[i], qplanes, qinfo, b0 + b);
      }
      const int m = (int)it.nrows;
      for (int r0 = 0; r0 < m; r0 += mf.rps) {
        const int r = r0 + mf.rsub;
        float y = 0.f;
        if (r < m) {
          const uint8_t* row = buf + (size_t)r * rb;
#pragma unroll
          for (int i = 0; i < MAXB; ++i) {
            int b = mf.sub + mf.lpr * i;
            if (b < nb) y += block_dot<QT>(row, b, ac[i]);
          }
        }
        y = group_sum(y, mf.lpr);
        if (r < m && mf.sub == 0) partial[it.slot * p.max_dn_rows + (it.row0 - dn_lo) + r] = y;
      }
      release(n);
    }
  } else if (routed_ok) {
    // drain: wait for every down copy issued into this CTA's ring before exiting
    for (int n = n_gu_end + warp; n < n_items; n += NCW) {
      if (!wait_full(n)) break;
      release(n);
    }
  }
  named_bar_sync(BAR_CONS, NCW * 32);

  // ---- combine: out[h] = sum_j w_j y_j[h] + shared[h] (+ x[h] | + out[h]) ----
  if (!misc[0] && !abort) {
    for (int r = tid; r < dn_rows; r += NCW * 32) {
      float acc = 0.f;
      for (int j = 0; j < K; ++j) acc = fmaf(rw[j], partial[j * p.max_dn_rows + r], acc);
      if (p.Fs) acc += partial[K * p.max_dn_rows + r];
      const int h = dn_lo + r;
      if (args.flags & FLAG_RESIDUAL) acc = __ldcg(args.x + h) + acc;
      if (args.flags & FLAG_ACCUMULATE) acc = __ldcg(args.out + h) + acc;
      args.out[h] = acc;
    }
  }

  // ---- exit: the last CTA out resets the counters for the next call ----
  named_bar_sync(BAR_CONS, NCW * 32);
  if (tid == 0) {
    __threadfence();
    uint32_t done = atomicAdd(args.ctrl + CTRL_EXIT, 1u) + 1;
    if (done == (uint32_t)p.nc) {
      args.ctrl[CTRL_BAR_A] = 0;
      args.ctrl[CTRL_BAR_B] = 0;
      args.ctrl[CTRL_EXIT] = 0;
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
