// Work plan of the fused decode kernel: how one token's MoE-FFN step is cut
// into byte-balanced copy items per CTA. Shared by the host (sizing, launch
// configuration) and the device (each CTA enumerates its own items).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

enum ItemKind : uint16_t { ITEM_ROUTER = 0, ITEM_GU = 1 };

// One copy item: a contiguous run of rows that one consumer warp processes out
// of the shared-memory ring.
//  ROUTER: router row `row0` (H f32 values).
//  GU:     pair rows [row0, row0 + nrows) of expert slot `slot`: the gate rows
//          then the up rows, landed back to back in the slot buffer.
// Slot k (k < top_k) is the k-th pick of the token; slot top_k is the shared expert.
// Down rows do not go through the ring: they are prefetched into L2 and read
// directly by the warps that own them.
struct Item {
  uint16_t kind;
  uint16_t slot;
  uint32_t row0;
  uint32_t nrows;
  uint32_t bytes;
};

struct DecodePlan {
  // layer shape
  int H, E, K, F, Fs, G, Gu, qtype;
  // bytes
  uint32_t blk;         // bytes per 32-value block (18 or 20)
  uint32_t rb_h;        // bytes per gate/up row (H values)
  uint32_t rb_f;        // bytes per routed down row (F values)
  uint32_t rb_fs;       // bytes per shared down row (Fs values)
  uint64_t rec_bytes;   // bytes per routed expert record
  // schedule
  int nc;               // CTAs (one per SM)
  uint32_t slot_bytes;  // ring slot size
  int nslots;           // ring slots
  int gu_align;         // GU partition unit (pairs) keeping copies 16-byte aligned
  int gu_r;             // max pairs per GU item
  int dn_align;         // output-row partition unit keeping down-row runs 16-byte aligned
  int max_dn_rows;      // output rows of the busiest CTA
};

MOE_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows per 16-byte-aligned run: the smallest r with r * row_bytes % 16 == 0.
MOE_HD int align_rows(uint32_t row_bytes) {
  int r = 1;
  while ((row_bytes * r) % 16u) r *= 2;
  return r;
}

// Contiguous share [lo, hi) of `units` for CTA c of nc (units * nc stays far
// below 2^31 for every accepted configuration).
MOE_HD void share(int units, int c, int nc, int& lo, int& hi) {
  lo = units * c / nc;
  hi = units * (c + 1) / nc;
}

MOE_HD uint32_t dn_row_bytes(const DecodePlan& p, int slot) { return slot < p.K ? p.rb_f : p.rb_fs; }
MOE_HD int slot_ff(const DecodePlan& p, int slot) { return slot < p.K ? p.F : p.Fs; }

// CTA c's share of the step, in closed form. Ring items, in processing order:
//   router rows [r_lo, r_lo + n_r)                         (routing-independent)
//   shared gate/up pairs [s_lo, s_lo + s_len), gu_r a piece (routing-independent)
//   for each pick j: its gate/up pairs [g_lo, g_lo + g_len), gu_r a piece
// The CTA also owns output rows [d_lo, d_lo + d_len): it computes the down rows
// of every slot for them and writes their combined result.
struct CtaShare {
  int r_lo, n_r;
  int s_lo, s_len, n_s;
  int g_lo, g_len, n_g;
  int d_lo, d_len;
  int n_pre, n_items;
};

MOE_HD CtaShare cta_share(const DecodePlan& p, int c) {
  CtaShare s;
  int lo, hi;
  share(p.E, c, p.nc, lo, hi);
  s.r_lo = lo;
  s.n_r = hi - lo;
  s.s_lo = s.s_len = s.n_s = 0;
  if (p.Fs) {
    share(p.Fs / p.gu_align, c, p.nc, lo, hi);
    s.s_lo = lo * p.gu_align;
    s.s_len = (hi - lo) * p.gu_align;
    s.n_s = ceil_div(s.s_len, p.gu_r);
  }
  share(p.F / p.gu_align, c, p.nc, lo, hi);
  s.g_lo = lo * p.gu_align;
  s.g_len = (hi - lo) * p.gu_align;
  s.n_g = ceil_div(s.g_len, p.gu_r);
  share(p.H / p.dn_align, c, p.nc, lo, hi);
  s.d_lo = lo * p.dn_align;
  s.d_len = (hi - lo) * p.dn_align;
  s.n_pre = s.n_r + s.n_s;
  s.n_items = s.n_pre + p.K * s.n_g;
  return s;
}

// Item n (0 <= n < n_items) of the CTA with share s.
MOE_HD Item item_at(const DecodePlan& p, const CtaShare& s, int n) {
  auto piece = [](int lo, int len, int step, int i, uint32_t& row0, uint32_t& m) {
    row0 = (uint32_t)(lo + i * step);
    int left = len - i * step;
    m = (uint32_t)(left < step ? left : step);
  };
  Item it;
  if (n < s.n_r) {
    it.kind = ITEM_ROUTER;
    it.slot = 0;
    it.row0 = (uint32_t)(s.r_lo + n);
    it.nrows = 1;
    it.bytes = (uint32_t)p.H * 4u;
    return it;
  }
  n -= s.n_r;
  if (n < s.n_s) {
    it.kind = ITEM_GU;
    it.slot = (uint16_t)p.K;
    piece(s.s_lo, s.s_len, p.gu_r, n, it.row0, it.nrows);
    it.bytes = 2u * it.nrows * p.rb_h;
    return it;
  }
  n -= s.n_s;
  it.kind = ITEM_GU;
  it.slot = (uint16_t)(n / s.n_g);
  piece(s.g_lo, s.g_len, p.gu_r, n % s.n_g, it.row0, it.nrows);
  it.bytes = 2u * it.nrows * p.rb_h;
  return it;
}

constexpr uint32_t FLAG_ACCUMULATE = 1u;  // out = out + contribution
constexpr uint32_t FLAG_RESIDUAL = 2u;    // out = x + contribution

// Arguments of the fused decode kernel (one token).
struct DecodeArgs {
  const float* x;             // [H]
  const float* router_w;      // [E][H]
  const float* bias;          // [E] or null
  const uint8_t* experts;     // E packed records
  const uint8_t* shared;      // shared record or null
  float* out;                 // [H]
  int32_t* topk_ids;          // [K] or null
  float* topk_w;              // [K] or null
  uint32_t* ctrl;             // control block
  unsigned long long* trace;  // [nc][16] timeline, or null
  uint64_t* logits;           // [E] published words {generation, f32}
  uint64_t* act;              // [K*F + Fs] published words (shared expert at K*F)
  float scale, norm_min;
  uint32_t flags;
  DecodePlan p;
};

}  // namespace moe
