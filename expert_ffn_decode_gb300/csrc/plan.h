// Work plan of the fused decode kernel: how one token's MoE-FFN step is cut into
// per-CTA work. Shared by the host (sizing, launch configuration) and the device
// (each CTA enumerates its own work in closed form).
//
// A slot is a pick of the token (k of them) or the shared expert. A slot with ff
// intermediate values has P = ff / 32 *columns*; column bc of the slot owns
//   gate/up: the slot's 32 gate rows and 32 up rows [32 bc, 32 bc + 32) (all of x),
//            whose SwiGLU values it publishes;
//   down:    the slot's down rows [lo, hi), a contiguous 1/P share of the H rows,
//            which it applies to the slot's whole published activation vector.
// Columns are dealt to the CTAs in turn (routed columns first, pick-major, then the
// shared expert's). Every down row of every slot is computed once, weighted by the
// slot's routing weight and published; a fixed-order sum over the slots gives out.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

enum ItemKind : uint16_t { ITEM_ROUTER = 0, ITEM_GU = 1, ITEM_DN = 2 };

constexpr int COL_VALUES = 32;  // intermediate values per column
constexpr int ITEM_PAIRS = 8;   // gate/up row pairs per ring item (copies stay 16-byte aligned)
constexpr int GU_ITEMS = COL_VALUES / ITEM_PAIRS;

// One copy item: what one ring slot receives.
//  ROUTER: router row `row0` (H f32 values).
//  GU:     gate rows [row0, row0 + ITEM_PAIRS) of slot `slot`, then the same up rows,
//          landed back to back (2 * ITEM_PAIRS rows of rb_h bytes).
//  DN:     down rows [row0, row0 + nrows) of slot `slot` (rows of the slot's down bytes).
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
  int ncol_r;           // routed columns: K * F / 32
  int ncol;             // all columns: ncol_r + Fs / 32
  int dn_align;         // down-row shares are multiples of this (16-byte aligned copies)
  int dn_r, dn_rs;      // max down rows per item (routed, shared)
  uint32_t slot_bytes;  // ring slot size
  int nslots;           // ring slots
  int max_items;        // ring items of the busiest CTA
};

MOE_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows per 16-byte-aligned run: the smallest r with r * row_bytes % 16 == 0.
MOE_HD int align_rows(uint32_t row_bytes) {
  int r = 1;
  while ((row_bytes * r) % 16u) r *= 2;
  return r;
}

// Contiguous share [lo, hi) of `units` for part c of n (units * n stays far below
// 2^31 for every accepted configuration).
MOE_HD void share(int units, int c, int n, int& lo, int& hi) {
  lo = units * c / n;
  hi = units * (c + 1) / n;
}

MOE_HD uint32_t dn_row_bytes(const DecodePlan& p, int slot) { return slot < p.K ? p.rb_f : p.rb_fs; }
MOE_HD int slot_ff(const DecodePlan& p, int slot) { return slot < p.K ? p.F : p.Fs; }
MOE_HD int slot_cols(const DecodePlan& p, int slot) { return slot_ff(p, slot) / COL_VALUES; }

// Column g of the step: routed columns first (pick-major), then the shared expert's.
MOE_HD void column_at(const DecodePlan& p, int g, int& slot, int& bc) {
  if (g < p.ncol_r) {
    slot = g / (p.F / COL_VALUES);
    bc = g % (p.F / COL_VALUES);
  } else {
    slot = p.K;
    bc = g - p.ncol_r;
  }
}

// Down rows [lo, hi) of column bc of a slot.
MOE_HD void column_rows(const DecodePlan& p, int slot, int bc, int& lo, int& hi) {
  share(p.H / p.dn_align, bc, slot_cols(p, slot), lo, hi);
  lo *= p.dn_align;
  hi *= p.dn_align;
}
MOE_HD int column_dn_items(const DecodePlan& p, int slot, int bc) {
  int lo, hi;
  column_rows(p, slot, bc, lo, hi);
  return ceil_div(hi - lo, slot < p.K ? p.dn_r : p.dn_rs);
}

// CTA c's share of the step, in closed form.
//   router rows [r_lo, r_lo + n_r)
//   columns g = c + i * nc (i < n_rc: routed; then n_sc shared ones)
//   output rows [d_lo, d_lo + d_len) of the final sum over the slots
// Ring items in processing order (phases):
//   0 router rows | 1 gate/up of the shared columns | 2 down of the shared columns |
//   3 gate/up of the routed columns | 4 down of the routed columns
// Phases 0-2 need no routing (n_pre items).
struct CtaShare {
  int r_lo, n_r;
  int n_rc, n_sc;
  int d_lo, d_len;
  int n_sdn, n_rdn;  // down items of the shared / routed columns
  int n_pre, n_items;
};

// Global column index of CTA c's i-th shared (routed) column.
MOE_HD int shared_column(const DecodePlan& p, const CtaShare& s, int c, int i) { return c + (s.n_rc + i) * p.nc; }
MOE_HD int routed_column(const DecodePlan& p, int c, int i) { return c + i * p.nc; }

MOE_HD CtaShare cta_share(const DecodePlan& p, int c) {
  CtaShare s;
  int lo, hi;
  share(p.E, c, p.nc, lo, hi);
  s.r_lo = lo;
  s.n_r = hi - lo;
  const int nmine = c < p.ncol ? (p.ncol - 1 - c) / p.nc + 1 : 0;
  s.n_rc = c < p.ncol_r ? (p.ncol_r - 1 - c) / p.nc + 1 : 0;
  s.n_sc = nmine - s.n_rc;
  share(p.H, c, p.nc, lo, hi);
  s.d_lo = lo;
  s.d_len = hi - lo;
  s.n_sdn = 0;
  for (int i = 0; i < s.n_sc; ++i) {
    int slot, bc;
    column_at(p, shared_column(p, s, c, i), slot, bc);
    s.n_sdn += column_dn_items(p, slot, bc);
  }
  s.n_rdn = 0;
  for (int i = 0; i < s.n_rc; ++i) {
    int slot, bc;
    column_at(p, routed_column(p, c, i), slot, bc);
    s.n_rdn += column_dn_items(p, slot, bc);
  }
  s.n_pre = s.n_r + GU_ITEMS * s.n_sc + s.n_sdn;
  s.n_items = s.n_pre + GU_ITEMS * s.n_rc + s.n_rdn;
  return s;
}

// Item n (0 <= n < n_items) of CTA c with share s.
MOE_HD Item item_at(const DecodePlan& p, const CtaShare& s, int c, int n) {
  Item it;
  it.nrows = 0;
  if (n < s.n_r) {
    it.kind = ITEM_ROUTER;
    it.slot = 0;
    it.row0 = (uint32_t)(s.r_lo + n);
    it.nrows = 1;
    it.bytes = (uint32_t)p.H * 4u;
    return it;
  }
  n -= s.n_r;
  // gate/up items of column g
  auto gu_item = [&](int g, int j) {
    int slot, bc;
    column_at(p, g, slot, bc);
    it.kind = ITEM_GU;
    it.slot = (uint16_t)slot;
    it.row0 = (uint32_t)(bc * COL_VALUES + j * ITEM_PAIRS);
    it.nrows = ITEM_PAIRS;
    it.bytes = 2u * ITEM_PAIRS * p.rb_h;
  };
  // down item j of the columns listed by col(i), i < ncols
  auto dn_item = [&](bool shared, int ncols, int j) {
    for (int i = 0; i < ncols; ++i) {
      const int g = shared ? shared_column(p, s, c, i) : routed_column(p, c, i);
      int slot, bc;
      column_at(p, g, slot, bc);
      const int m = column_dn_items(p, slot, bc);
      if (j < m) {
        int lo, hi;
        column_rows(p, slot, bc, lo, hi);
        const int step = slot < p.K ? p.dn_r : p.dn_rs;
        const int r0 = lo + j * step;
        it.kind = ITEM_DN;
        it.slot = (uint16_t)slot;
        it.row0 = (uint32_t)r0;
        it.nrows = (uint32_t)(hi - r0 < step ? hi - r0 : step);
        it.bytes = it.nrows * dn_row_bytes(p, slot);
        return;
      }
      j -= m;
    }
  };
  if (n < GU_ITEMS * s.n_sc) {
    gu_item(shared_column(p, s, c, n / GU_ITEMS), n % GU_ITEMS);
    return it;
  }
  n -= GU_ITEMS * s.n_sc;
  if (n < s.n_sdn) {
    dn_item(true, s.n_sc, n);
    return it;
  }
  n -= s.n_sdn;
  if (n < GU_ITEMS * s.n_rc) {
    gu_item(routed_column(p, c, n / GU_ITEMS), n % GU_ITEMS);
    return it;
  }
  n -= GU_ITEMS * s.n_rc;
  dn_item(false, s.n_rc, n);
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
  unsigned long long* trace;  // [nc][24] timeline, or null
  uint64_t* logits;           // [E] published words {generation, f32}
  uint64_t* act;              // [K * F + Fs] published SwiGLU values (shared expert at K * F)
  uint64_t* ys;               // [K + 1][H] published weighted down rows (shared expert last)
  float scale, norm_min;
  uint32_t flags;
  DecodePlan p;
};

}  // namespace moe
