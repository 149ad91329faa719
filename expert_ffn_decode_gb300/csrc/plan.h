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

enum ItemKind : uint16_t { ITEM_ROUTER = 0, ITEM_GU = 1, ITEM_DN = 2 };

// One copy item: a contiguous run of rows that one consumer warp processes.
//  ROUTER: router row `row0` (H f32 values).
//  GU:     pair rows [row0, row0 + nrows) of expert slot `slot`: the gate rows
//          then the up rows, landed back to back in the slot buffer.
//  DN:     down rows [row0, row0 + nrows) of expert slot `slot`.
// Slot k (k < top_k) is the k-th pick of the token; slot top_k is the shared expert.
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
  int dn_align;         // DN partition unit (rows)
  int dn_r, dn_r_s;     // max rows per DN item (routed, shared)
  int max_items;        // items of the busiest CTA
  int max_dn_rows;      // DN rows of the busiest CTA
};

MOE_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows per 16-byte-aligned run: the smallest r with r * row_bytes % 16 == 0.
MOE_HD int align_rows(uint32_t row_bytes) {
  int r = 1;
  while ((row_bytes * r) % 16u) r *= 2;
  return r;
}

// Contiguous share [lo, hi) of `units` for CTA c of nc.
MOE_HD void share(int units, int c, int nc, int& lo, int& hi) {
  lo = (int)((int64_t)units * c / nc);
  hi = (int)((int64_t)units * (c + 1) / nc);
}

MOE_HD uint32_t dn_row_bytes(const DecodePlan& p, int slot) { return slot < p.K ? p.rb_f : p.rb_fs; }
MOE_HD int slot_ff(const DecodePlan& p, int slot) { return slot < p.K ? p.F : p.Fs; }

// Enumerate CTA c's items in processing order; writes them to `out` when it is
// not null and returns the count. Order: router rows, shared gate/up pairs
// (both independent of the routing), routed gate/up pairs, then down rows of
// every slot (routed picks first, shared last). `n_pre` receives the number of
// routing-independent items, `n_gu_end` the index one past the last GU item.
MOE_HD int build_items(const DecodePlan& p, int c, Item* out, int* n_pre, int* n_gu_end,
                       int* dn_lo, int* dn_hi) {
  int n = 0;
  auto put = [&](uint16_t kind, uint16_t slot, uint32_t row0, uint32_t nrows, uint32_t bytes) {
    if (out) out[n] = Item{kind, slot, row0, nrows, bytes};
    ++n;
  };
  int lo, hi;
  // router rows
  share(p.E, c, p.nc, lo, hi);
  for (int e = lo; e < hi; ++e) put(ITEM_ROUTER, 0, (uint32_t)e, 1, (uint32_t)p.H * 4u);
  // shared gate/up pairs
  if (p.Fs) {
    share(p.Fs / p.gu_align, c, p.nc, lo, hi);
    for (int r = lo * p.gu_align; r < hi * p.gu_align; r += p.gu_r) {
      int m = hi * p.gu_align - r < p.gu_r ? hi * p.gu_align - r : p.gu_r;
      put(ITEM_GU, (uint16_t)p.K, (uint32_t)r, (uint32_t)m, 2u * (uint32_t)m * p.rb_h);
    }
  }
  if (n_pre) *n_pre = n;
  // routed gate/up pairs: one linear space of K*F pairs, expert-major
  share(p.K * p.F / p.gu_align, c, p.nc, lo, hi);
  {
    int a = lo * p.gu_align, b = hi * p.gu_align;
    while (a < b) {
      int j = a / p.F, r = a - j * p.F;
      int seg_end = (j + 1) * p.F < b ? (j + 1) * p.F : b;
      int m = seg_end - a < p.gu_r ? seg_end - a : p.gu_r;
      put(ITEM_GU, (uint16_t)j, (uint32_t)r, (uint32_t)m, 2u * (uint32_t)m * p.rb_h);
      a += m;
    }
  }
  if (n_gu_end) *n_gu_end = n;
  // down rows: this CTA owns rows [lo, hi) of the output for every slot
  share(p.H / p.dn_align, c, p.nc, lo, hi);
  lo *= p.dn_align;
  hi *= p.dn_align;
  if (dn_lo) *dn_lo = lo;
  if (dn_hi) *dn_hi = hi;
  int nslot = p.K + (p.Fs ? 1 : 0);
  for (int s = 0; s < nslot; ++s) {
    int rmax = s < p.K ? p.dn_r : p.dn_r_s;
    uint32_t rb = dn_row_bytes(p, s);
    for (int r = lo; r < hi; r += rmax) {
      int m = hi - r < rmax ? hi - r : rmax;
      put(ITEM_DN, (uint16_t)s, (uint32_t)r, (uint32_t)m, (uint32_t)m * rb);
    }
  }
  return n;
}

constexpr uint32_t FLAG_ACCUMULATE = 1u;
constexpr uint32_t FLAG_RESIDUAL = 2u;

// Arguments of the fused decode kernel (one token).
struct DecodeArgs {
  const float* x;           // [H]
  const float* router_w;    // [E][H]
  const float* bias;        // [E] or null
  const uint8_t* experts;   // E packed records
  const uint8_t* shared;    // shared record or null
  float* out;               // [H]
  int32_t* topk_ids;        // [K] or null
  float* topk_w;            // [K] or null
  uint32_t* ctrl;           // control block
  float* logits;            // [E]
  float* act;               // [K*F + Fs]
  float scale, norm_min;
  uint32_t flags;
  DecodePlan p;
};

}  // namespace moe
