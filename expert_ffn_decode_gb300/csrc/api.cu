// C ABI of the routed MoE-FFN step: validation, workspace, planning, launches.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moeffn.h"
#include "common.cuh"
#include "decode_host.h"
#include "plan.h"
#include "prefill_host.h"

namespace {

// The calling thread's last error text, formatted in place (no allocation).
thread_local char g_err[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // clear the sticky launch error, if any
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The device address of page-locked host memory mapped into the current device's address
// space, or null for any other pointer (pageable host memory, device memory).
void* mapped_host(const void* p) {
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
}

// Bytes of a weight row of n values: 32-value blocks of 18 (Q4_0) or 20 (Q4_1) bytes, or
// 256-value super-blocks of 144 (Q4_K) or 210 (Q6_K) bytes.
uint32_t row_bytes(int n, int qtype) {
  switch (qtype) {
    case MOE_Q4_0: return (uint32_t)(n / 32) * 18u;
    case MOE_Q4_1: return (uint32_t)(n / 32) * 20u;
    case MOE_Q4_K: return (uint32_t)(n / 256) * 144u;
    default: return (uint32_t)(n / 256) * 210u;
  }
}
bool kquant(int qtype) { return qtype == MOE_Q4_K || qtype == MOE_Q6_K; }
// The down rows' block type.
int down_type(const moe_cfg* c) { return c->qtype_down ? c->qtype_down : c->qtype; }

// ---- configuration checks ------------------------------------------------------
int check_cfg(const moe_cfg* c) {
  if (!c) return fail(MOE_ERR_NULL_PTR, "cfg is NULL");
  if (c->qtype != MOE_Q4_0 && c->qtype != MOE_Q4_1 && c->qtype != MOE_Q4_K)
    return fail(MOE_ERR_INVALID_CFG, "qtype %d: expected MOE_Q4_0 (2), MOE_Q4_1 (3) or MOE_Q4_K (12)", c->qtype);
  if (c->qtype_down != 0 && c->qtype_down != MOE_Q4_0 && c->qtype_down != MOE_Q4_1 && c->qtype_down != MOE_Q4_K &&
      c->qtype_down != MOE_Q6_K)
    return fail(MOE_ERR_INVALID_CFG, "qtype_down %d: expected 0, MOE_Q4_0, MOE_Q4_1, MOE_Q4_K or MOE_Q6_K",
                c->qtype_down);
  if (c->hidden <= 0 || c->hidden % 32 || c->hidden > 3072)
    return fail(MOE_ERR_INVALID_CFG, "hidden %d: must be a positive multiple of 32, at most 3072", c->hidden);
  if (c->expert_ff <= 0 || c->expert_ff % 32 || c->expert_ff > 3072)
    return fail(MOE_ERR_INVALID_CFG, "expert_ff %d: must be a positive multiple of 32, at most 3072",
                c->expert_ff);
  if (c->shared_ff < 0 || c->shared_ff % 32 || c->shared_ff > 3072)
    return fail(MOE_ERR_INVALID_CFG, "shared_ff %d: must be 0 or a multiple of 32, at most 3072",
                c->shared_ff);
  if (kquant(c->qtype) && c->hidden % 256)
    return fail(MOE_ERR_INVALID_CFG, "hidden %d: K-quant gate/up rows need a multiple of 256", c->hidden);
  if (kquant(down_type(c)) && (c->expert_ff % 256 || c->shared_ff % 256))
    return fail(MOE_ERR_INVALID_CFG, "expert_ff %d, shared_ff %d: K-quant down rows need multiples of 256",
                c->expert_ff, c->shared_ff);
  if (c->n_experts < 1 || c->n_experts > 1024)
    return fail(MOE_ERR_INVALID_CFG, "n_experts %d: must be in [1, 1024]", c->n_experts);
  if (c->top_k < 1 || c->top_k > 32 || c->top_k > c->n_experts)
    return fail(MOE_ERR_INVALID_CFG, "top_k %d: must be in [1, min(n_experts, 32)]", c->top_k);
  if (c->n_groups < 1 || c->n_experts % c->n_groups)
    return fail(MOE_ERR_INVALID_CFG, "n_groups %d must divide n_experts %d", c->n_groups, c->n_experts);
  if (c->n_groups > 1) {
    const int per = c->n_experts / c->n_groups;
    if (per < 2) return fail(MOE_ERR_INVALID_CFG, "groups of %d expert: need at least 2 per group", per);
    if (c->n_groups > 64) return fail(MOE_ERR_INVALID_CFG, "n_groups %d > 64", c->n_groups);
    if (c->groups_used < 1 || c->groups_used > c->n_groups)
      return fail(MOE_ERR_INVALID_CFG, "groups_used %d: must be in [1, n_groups]", c->groups_used);
    if (c->top_k > c->groups_used * per)
      return fail(MOE_ERR_INVALID_CFG, "top_k %d exceeds the %d experts of the kept groups", c->top_k,
                  c->groups_used * per);
  }
  if (c->n_tokens < 0) return fail(MOE_ERR_INVALID_CFG, "n_tokens %d < 0", c->n_tokens);
  if (!std::isfinite(c->weights_scale))
    return fail(MOE_ERR_INVALID_CFG, "weights_scale is not finite");
  if (!(c->norm_min >= 0.f) || !std::isfinite(c->norm_min))
    return fail(MOE_ERR_INVALID_CFG, "norm_min must be finite and >= 0");
  if (!(c->swiglu_limit >= 0.f) || !std::isfinite(c->swiglu_limit) || !(c->swiglu_limit_shared >= 0.f) ||
      !std::isfinite(c->swiglu_limit_shared))
    return fail(MOE_ERR_INVALID_CFG, "swiglu limits must be finite and >= 0");
  if (!(c->rms_eps >= 0.f) || !std::isfinite(c->rms_eps))
    return fail(MOE_ERR_INVALID_CFG, "rms_eps must be finite and >= 0");
  if (c->flags & ~(MOE_ACCUMULATE | MOE_RESIDUAL | MOE_HOST_IO | MOE_NO_PDL | MOE_TRACE | MOE_BATCHED |
                   MOE_F32_ACT | MOE_GRAPH))
    return fail(MOE_ERR_INVALID_CFG, "unknown flag bits 0x%x", c->flags);
  return MOE_OK;
}

// ---- workspace layout -----------------------------------------------------------
struct WsLayout {
  size_t ctrl, logits, act, ids, wts, pub, x_stage, out_stage, ids_stage, w_stage, trace, xn, prefill, total;
  int rep;                    // copies of the decode chain's broadcast arrays
  size_t lg_copy, act_copy;   // floats from one copy to the next
};

// SMs of the current device (the timeline keeps one row per SM); without a
// device, an upper bound for sizing.
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    sms = 256;
  }
  return sms;
}

// Tokens of one batched pass for a call (0: the call takes the decode path). Calls of
// at least PREFILL_MIN_T tokens, or any call with MOE_BATCHED, take the batched path.
int prefill_pass_tokens(const moe_cfg* c) {
  const int T = c->n_tokens;
  if (T < 1 || (T < moe::PREFILL_MIN_T && !(c->flags & MOE_BATCHED))) return 0;
  return T < moe::PREFILL_CHUNK_T ? T : moe::PREFILL_CHUNK_T;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Tokens per decode call for a call on the decode path (1 otherwise).
int decode_call_tokens(const moe_cfg* c) {
  const int T = c->n_tokens;
  if (prefill_pass_tokens(c) || T < 1) return 1;
  return T < moe::DEC_TMAX ? T : moe::DEC_TMAX;
}

// decode_only: the layout of calls that always decode (moe_ffn_forward_noalloc), up
// to DEC_TMAX tokens at a time and without the batched path's regions. `rep`: copies of
// the decode chain's broadcast arrays.
WsLayout ws_layout(const moe_cfg* c, bool decode_only = false, int rep = moe::DEC_REP) {
  WsLayout L;
  size_t o = 0;
  L.ctrl = o;
  o += moe::CTRL_BYTES;
  const size_t td = decode_only ? (size_t)(c->n_tokens < moe::DEC_TMAX ? c->n_tokens : moe::DEC_TMAX)
                                : (size_t)decode_call_tokens(c);  // tokens of one decode call
  // decode: `rep` copies of the arrays every CTA reads, each copy 256-byte aligned
  L.rep = rep;
  L.lg_copy = up256(td * c->n_experts * 4) / 4;
  L.act_copy = up256(td * ((size_t)c->top_k * c->expert_ff + c->shared_ff) * 4) / 4;
  L.logits = o;  // router logits [rep][td][E] f32
  o += (size_t)rep * L.lg_copy * 4;
  L.act = o;     // SwiGLU activations of every slot [rep][td][K * F + Fs] f32
  o += (size_t)rep * L.act_copy * 4;
  L.ids = o;     // decode: picks and weights [td][K] (calls of several tokens)
  o = up256(o + td * c->top_k * 4);
  L.wts = o;
  o = up256(o + td * c->top_k * 4);
  L.pub = o;     // decode: the picks a single-token call publishes for its down kernel [K] u64
  o = up256(o + (size_t)c->top_k * 8);
  const size_t T = (size_t)c->n_tokens;
  L.x_stage = L.out_stage = L.ids_stage = L.w_stage = 0;
  if (c->flags & MOE_HOST_IO) {
    L.x_stage = o;
    o = up256(o + T * c->hidden * 4);
    L.out_stage = o;
    o = up256(o + T * c->hidden * 4);
    L.ids_stage = o;
    o = up256(o + T * c->top_k * 4);
    L.w_stage = o;
    o = up256(o + T * c->top_k * 4);
  }
  L.trace = 0;
  if (c->flags & MOE_TRACE) {
    L.trace = o;
    o = up256(o + (size_t)device_sms() * 24 * 8);
  }
  L.prefill = 0;
  L.xn = 0;
  if (const int tp = decode_only ? 0 : prefill_pass_tokens(c)) {
    if (c->ffn_norm) {
      L.xn = o;  // batched passes: the normalised tokens [pass][H] f32
      o = up256(o + (size_t)tp * c->hidden * 4);
    }
    L.prefill = o;
    const bool tile = moe::prefill_tile_ok(c->hidden, c->expert_ff, c->shared_ff, c->qtype, down_type(c));
    o = up256(o + moe::prefill_ws_layout(tp, c->hidden, c->n_experts, c->top_k, c->expert_ff, c->shared_ff, tile)
                      .total);
  }
  L.total = o;
  return L;
}

// ---- decode plans (cached per device and layer shape) ------------------------------
struct PlanEntry {
  int device;
  moe_cfg key;
  moe::DecodePlan plan;
  int maxb;  // blocks per lane of a gate/up row
  int sms;   // SMs of the device
};
std::mutex g_mu;
std::vector<PlanEntry> g_plans;

bool same_shape(const moe_cfg& a, const moe_cfg& b) {
  return a.hidden == b.hidden && a.n_experts == b.n_experts && a.top_k == b.top_k &&
         a.expert_ff == b.expert_ff && a.shared_ff == b.shared_ff && a.n_groups == b.n_groups &&
         (a.n_groups == 1 || a.groups_used == b.groups_used) && a.qtype == b.qtype &&
         down_type(&a) == down_type(&b) && (a.flags & MOE_F32_ACT) == (b.flags & MOE_F32_ACT);
}

int make_plan(const moe_cfg* c, int device, PlanEntry* out) {
  moe::DecodePlan p{};
  p.H = c->hidden;
  p.E = c->n_experts;
  p.K = c->top_k;
  p.F = c->expert_ff;
  p.Fs = c->shared_ff;
  p.G = c->n_groups;
  p.Gu = c->n_groups > 1 ? c->groups_used : 1;
  p.qtype = c->qtype;
  p.qtype_dn = down_type(c);
  p.rb_h = row_bytes(p.H, p.qtype);
  p.rb_f = row_bytes(p.F, p.qtype_dn);
  p.rb_fs = p.Fs ? row_bytes(p.Fs, p.qtype_dn) : p.rb_f;
  p.rec_bytes = (uint64_t)2 * p.F * p.rb_h + (uint64_t)p.H * p.rb_f;
  p.nbH = p.H / 32;
  p.nbF = p.F / 32;
  p.nbFs = p.Fs / 32;
  p.nact = p.nbFs + p.K * p.nbF;
  p.act_stride = p.K * p.F + p.Fs;
  p.rep = moe::DEC_REP;
  const uint32_t budget = 200u * 1024u;  // dynamic shared memory of one CTA
  // shared bytes per 32-value activation block: f32 chunks and sum, or fixed-point planes and info
  const uint32_t blk = (c->flags & MOE_F32_ACT) ? moe::ACT_BLOCK_SMEM : moe::ACT_BLOCK_SMEM_FX;
  // gate/up: 4 windows of 8 rows, the x blocks and the selection
  p.gu_win = moe::window_bytes(8u * p.rb_h);
  p.gu_smem = 4u * p.gu_win + (uint32_t)p.nbH * blk + moe::select_smem(p.E);
  if (p.gu_smem > budget) return fail(MOE_ERR_UNSUPPORTED, "gate/up rows too long for shared memory");
  // down: the activation blocks in one piece when they fit in 40 KiB, else pieces of
  // 256; then as many rows per CTA (8, 4, 2, 1) as the windows allow
  p.dn_piece = (size_t)p.nact * blk <= 40 * 1024 ? p.nact : 256;
  for (p.dn_rows = 8; p.dn_rows >= 1; p.dn_rows /= 2) {
    p.dn_win_f = moe::window_bytes((uint32_t)p.dn_rows * p.rb_f);
    p.dn_win_fs = p.Fs ? moe::window_bytes((uint32_t)p.dn_rows * p.rb_fs) : 0u;
    p.dn_smem = p.dn_win_fs + (uint32_t)p.K * p.dn_win_f + (uint32_t)p.dn_piece * blk + moe::select_smem(p.E);
    if (p.dn_smem <= budget) break;
  }
  if (p.dn_rows < 1) return fail(MOE_ERR_UNSUPPORTED, "down rows too long for shared memory");
  // row groups: split the threads over the rows while a group still has a thread for
  // each block of a piece
  p.dn_rg = 1;
  while (p.dn_rg < p.dn_rows && 256 / (2 * p.dn_rg) >= p.dn_piece) p.dn_rg *= 2;
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  out->device = device;
  out->key = *c;
  out->plan = p;
  out->maxb = (p.nbH + 31) / 32;
  out->sms = sms;
  return MOE_OK;
}

int get_plan(const moe_cfg* c, PlanEntry* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  for (const auto& pe : g_plans)
    if (pe.device == dev && same_shape(pe.key, *c)) {
      *out = pe;
      return MOE_OK;
    }
  PlanEntry pe;
  int rc = make_plan(c, dev, &pe);
  if (rc != MOE_OK) return rc;
  g_plans.push_back(pe);
  *out = pe;
  return MOE_OK;
}

// ---- library-owned workspaces -----------------------------------------------------
struct OwnedWs {
  int device;
  void* ptr;
  size_t bytes;
};
std::vector<OwnedWs> g_ws;

int owned_workspace(size_t bytes, void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& w : g_ws)
    if (w.device == dev) {
      if (w.bytes >= bytes) {
        *ptr = w.ptr;
        return MOE_OK;
      }
      e = cudaFree(w.ptr);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFree");
      w.ptr = nullptr;
      w.bytes = 0;
      e = cudaMalloc(&w.ptr, bytes);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
      e = cudaMemset(w.ptr, 0, bytes);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
      w.bytes = bytes;
      *ptr = w.ptr;
      return MOE_OK;
    }
  OwnedWs w{dev, nullptr, bytes};
  e = cudaMalloc(&w.ptr, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  e = cudaMemset(w.ptr, 0, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  g_ws.push_back(w);
  *ptr = w.ptr;
  return MOE_OK;
}

// Checks the call and enqueues all of its work (copies and kernels) on `st`.
int enqueue(const float* x, const float* router_w, const float* bias, const void* experts,
            const void* shared, const moe_cfg* c, float* out, void* ws, size_t ws_bytes, cudaStream_t st,
            int32_t* ids, float* wts) {
  int rc = check_cfg(c);
  if (rc != MOE_OK) return rc;
  const int T = c->n_tokens;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !experts || !out) return fail(MOE_ERR_NULL_PTR, "x, router_w, expert_blocks and out must not be NULL");
  if (c->shared_ff > 0 && !shared) return fail(MOE_ERR_NULL_PTR, "shared_ff > 0 needs shared_blocks");
  if (!ws) return fail(MOE_ERR_NULL_PTR, "workspace is NULL");
  if (!aligned(router_w, 16) || !aligned(experts, 16) || (shared && !aligned(shared, 16)))
    return fail(MOE_ERR_ALIGNMENT, "router_w, expert_blocks and shared_blocks must be 16-byte aligned");
  if (!(c->flags & MOE_HOST_IO) && (!aligned(x, 16) || !aligned(out, 16)))
    return fail(MOE_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
  if (bias && !aligned(bias, 4)) return fail(MOE_ERR_ALIGNMENT, "router_bias must be 4-byte aligned");
  if (c->ffn_norm && !aligned(c->ffn_norm, 16)) return fail(MOE_ERR_ALIGNMENT, "ffn_norm must be 16-byte aligned");
  if (!aligned(ws, 256)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const size_t xbytes = (size_t)T * c->hidden * 4;
  {
    const char* xa = reinterpret_cast<const char*>(x);
    const char* oa = reinterpret_cast<const char*>(out);
    if (xa < oa + xbytes && oa < xa + xbytes) return fail(MOE_ERR_INVALID_CFG, "x and out overlap");
  }
  const WsLayout W = ws_layout(c);
  if (ws_bytes < W.total)
    return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes, this call needs %zu", ws_bytes, W.total);

  PlanEntry pe;
  rc = get_plan(c, &pe);
  if (rc != MOE_OK) return rc;

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const bool host = (c->flags & MOE_HOST_IO) != 0;
  const float* dx = x;
  float* dout = out;
  int32_t* dids = ids;
  float* dw = wts;
  cudaError_t e;
  // Host outputs in page-locked memory mapped into the device's address space are written
  // in place by the kernels (one pass of stores, no copy back); other host outputs are staged.
  bool out_direct = false, ids_direct = false, w_direct = false;
  if (host) {
    dx = reinterpret_cast<const float*>(wsb + W.x_stage);
    dout = reinterpret_cast<float*>(wsb + W.out_stage);
    dids = ids ? reinterpret_cast<int32_t*>(wsb + W.ids_stage) : nullptr;
    dw = wts ? reinterpret_cast<float*>(wsb + W.w_stage) : nullptr;
    if (void* m = mapped_host(out)) {
      dout = static_cast<float*>(m);
      out_direct = true;
    }
    if (void* m = ids ? mapped_host(ids) : nullptr) {
      dids = static_cast<int32_t*>(m);
      ids_direct = true;
    }
    if (void* m = wts ? mapped_host(wts) : nullptr) {
      dw = static_cast<float*>(m);
      w_direct = true;
    }
    e = cudaMemcpyAsync(const_cast<float*>(dx), x, xbytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "copy of x to the device");
    if ((c->flags & MOE_ACCUMULATE) && !out_direct) {
      e = cudaMemcpyAsync(dout, out, xbytes, cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) return cuda_fail(e, "copy of out to the device");
    }
  }

  if (const int tp = prefill_pass_tokens(c)) {
    // batched path: router, top-k, expert sort and grouped tensor-core GEMMs
    const bool tile = moe::prefill_tile_ok(c->hidden, c->expert_ff, c->shared_ff, c->qtype, down_type(c));
    const moe::PrefillWs P = moe::prefill_ws_layout(tp, c->hidden, c->n_experts, c->top_k, c->expert_ff,
                                                    c->shared_ff, tile);
    uint8_t* pb = wsb + W.prefill;
    moe::PrefillArgs pa{};
    pa.router_w = router_w;
    pa.bias = bias;
    pa.experts = static_cast<const uint8_t*>(experts);
    pa.shared = static_cast<const uint8_t*>(shared);
    pa.logits = reinterpret_cast<float*>(pb + P.logits);
    pa.ids = reinterpret_cast<int32_t*>(pb + P.ids);
    pa.wts = reinterpret_cast<float*>(pb + P.wts);
    pa.offsets = reinterpret_cast<uint32_t*>(pb + P.offsets);
    pa.perm = reinterpret_cast<uint32_t*>(pb + P.perm);
    pa.wsorted = reinterpret_cast<float*>(pb + P.wsorted);
    pa.pos_of = reinterpret_cast<uint32_t*>(pb + P.pos_of);
    pa.chunks = reinterpret_cast<moe::GemmChunk*>(pb + P.chunks);
    pa.nchunks = reinterpret_cast<uint32_t*>(pb + P.nchunks);
    if (tile) {
      pa.ximg = pb + P.ximg;
      pa.ximg_routed = pb + P.ximg_routed;
      pa.aimg = pb + P.aimg;
      pa.aimg_s = pb + P.aimg_s;
    } else {
      pa.x16 = reinterpret_cast<__half*>(pb + P.x16);
      pa.act16 = reinterpret_cast<__half*>(pb + P.act16);
      pa.act16s = reinterpret_cast<__half*>(pb + P.act16s);
    }
    pa.tile = tile ? 1 : 0;
    pa.nmax = tile ? moe::PREFILL_TILE_NMAX : moe::PREFILL_NMAX;
    pa.ybuf = reinterpret_cast<float*>(pb + P.ybuf);
    pa.sbuf = reinterpret_cast<float*>(pb + P.sbuf);
    pa.status = reinterpret_cast<uint32_t*>(wsb + W.ctrl) + moe::CTRL_STATUS;
    pa.H = c->hidden;
    pa.E = c->n_experts;
    pa.K = c->top_k;
    pa.F = c->expert_ff;
    pa.Fs = c->shared_ff;
    pa.G = c->n_groups;
    pa.Gu = c->n_groups > 1 ? c->groups_used : 1;
    pa.qtype = c->qtype;
    pa.qtype_dn = down_type(c);
    pa.scale = c->weights_scale;
    pa.norm_min = c->norm_min;
    pa.lim = c->swiglu_limit;
    pa.lim_s = c->swiglu_limit_shared;
    pa.norm = c->ffn_norm;
    pa.eps = c->rms_eps;
    pa.xn = c->ffn_norm ? reinterpret_cast<float*>(wsb + W.xn) : nullptr;
    pa.flags = c->flags & (MOE_ACCUMULATE | MOE_RESIDUAL);
    pa.rb_h = pe.plan.rb_h;
    pa.rb_f = pe.plan.rb_f;
    pa.rb_fs = pe.plan.rb_fs;
    pa.rec_bytes = pe.plan.rec_bytes;
    pa.nc = pe.sms;
    for (int t0 = 0; t0 < T; t0 += tp) {
      pa.T = T - t0 < tp ? T - t0 : tp;
      pa.x = dx + (size_t)t0 * c->hidden;
      pa.xres = pa.x;
      pa.out = dout + (size_t)t0 * c->hidden;
      pa.topk_ids = dids ? dids + (size_t)t0 * c->top_k : nullptr;
      pa.topk_w = dw ? dw + (size_t)t0 * c->top_k : nullptr;
      e = moe::prefill_launch(pa, st);
      if (e != cudaSuccess) return cuda_fail(e, "prefill kernel launch");
    }
  }

  moe::DecodeArgs a{};
  a.router_w = router_w;
  a.bias = bias;
  a.experts = static_cast<const uint8_t*>(experts);
  a.shared = static_cast<const uint8_t*>(shared);
  a.ctrl = reinterpret_cast<uint32_t*>(wsb + W.ctrl);
  a.logits = reinterpret_cast<float*>(wsb + W.logits);
  a.act = reinterpret_cast<float*>(wsb + W.act);
  a.lg_copy = W.lg_copy;
  a.act_copy = W.act_copy;
  a.ids = reinterpret_cast<int32_t*>(wsb + W.ids);
  a.wts = reinterpret_cast<float*>(wsb + W.wts);
  a.pub = reinterpret_cast<unsigned long long*>(wsb + W.pub);
  a.trace = (c->flags & MOE_TRACE) ? reinterpret_cast<unsigned long long*>(wsb + W.trace) : nullptr;
  a.scale = c->weights_scale;
  a.norm_min = c->norm_min;
  a.lim = c->swiglu_limit;
  a.lim_s = c->swiglu_limit_shared;
  a.norm = c->ffn_norm;
  a.eps = c->rms_eps;
  a.flags = c->flags & (MOE_ACCUMULATE | MOE_RESIDUAL);
  a.p = pe.plan;
  a.p.rep = W.rep;
  const bool pdl = (c->flags & MOE_NO_PDL) == 0;
  const int td = decode_call_tokens(c);
  for (int t = 0; t < T && !prefill_pass_tokens(c); t += td) {
    a.T = T - t < td ? T - t : td;
    a.x = dx + (size_t)t * c->hidden;
    a.out = dout + (size_t)t * c->hidden;
    a.topk_ids = dids ? dids + (size_t)t * c->top_k : nullptr;
    a.topk_w = dw ? dw + (size_t)t * c->top_k : nullptr;
    e = moe::decode_launch(a, pe.maxb, st, pdl, (c->flags & MOE_F32_ACT) == 0, pe.sms);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  }
  if (host) {
    if (!out_direct) {
      e = cudaMemcpyAsync(out, dout, xbytes, cudaMemcpyDeviceToHost, st);
      if (e != cudaSuccess) return cuda_fail(e, "copy of out to the host");
    }
    if (ids && !ids_direct) {
      e = cudaMemcpyAsync(ids, dids, (size_t)T * c->top_k * 4, cudaMemcpyDeviceToHost, st);
      if (e != cudaSuccess) return cuda_fail(e, "copy of topk_ids to the host");
    }
    if (wts && !w_direct) {
      e = cudaMemcpyAsync(wts, dw, (size_t)T * c->top_k * 4, cudaMemcpyDeviceToHost, st);
      if (e != cudaSuccess) return cuda_fail(e, "copy of topk_w to the host");
    }
  }
  return MOE_OK;
}

// ---- replayed graphs (MOE_GRAPH) ---------------------------------------------------
// With MOE_GRAPH, an argument set seen before runs as one launch of a CUDA graph of its whole
// enqueued work, captured the second time the set is seen (the first time it runs as it is,
// which also sets every kernel's shared-memory limit outside any capture). The cache holds
// the last GRAPH_SLOTS sets per process. A call made while its stream is being captured, a
// traced call, and a call whose capture fails run directly.
constexpr int GRAPH_SLOTS = 64;

struct GraphKey {
  int device;
  const void* p[10];  // x, router_w, bias, experts, shared, out, ws, ids, wts, ffn_norm
  size_t ws_bytes;
  int32_t i[12];      // the cfg's integer fields (flags included)
  float f[6];         // the cfg's float fields
};

bool same_key(const GraphKey& a, const GraphKey& b) {
  if (a.device != b.device || a.ws_bytes != b.ws_bytes) return false;
  for (int k = 0; k < 10; ++k)
    if (a.p[k] != b.p[k]) return false;
  for (int k = 0; k < 12; ++k)
    if (a.i[k] != b.i[k]) return false;
  for (int k = 0; k < 6; ++k)
    if (std::memcmp(&a.f[k], &b.f[k], sizeof(float)) != 0) return false;
  return true;
}

struct GraphSlot {
  bool used;
  bool no_graph;       // its capture failed: always run directly
  GraphKey key;
  cudaGraphExec_t exec;
  unsigned long long last;
};
GraphSlot g_graphs[GRAPH_SLOTS];
unsigned long long g_graph_tick = 0;
std::mutex g_graph_mu;
cudaStream_t g_capture_stream[64];

int run(const float* x, const float* router_w, const float* bias, const void* experts, const void* shared,
        const moe_cfg* c, float* out, void* ws, size_t ws_bytes, cudaStream_t st, int32_t* ids, float* wts) {
  if (!c || !(c->flags & MOE_GRAPH) || (c->flags & MOE_TRACE) || c->n_tokens <= 0)
    return enqueue(x, router_w, bias, experts, shared, c, out, ws, ws_bytes, st, ids, wts);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    cs = cudaStreamCaptureStatusActive;
  }
  int dev = 0;
  if (cs != cudaStreamCaptureStatusNone || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return enqueue(x, router_w, bias, experts, shared, c, out, ws, ws_bytes, st, ids, wts);
  }
  GraphKey k{};
  k.device = dev;
  const void* ps[10] = {x, router_w, bias, experts, shared, out, ws, ids, wts, c->ffn_norm};
  for (int j = 0; j < 10; ++j) k.p[j] = ps[j];
  k.ws_bytes = ws_bytes;
  const int32_t is[12] = {c->hidden, c->n_experts, c->top_k, c->expert_ff, c->shared_ff, c->n_groups,
                          c->groups_used, c->n_tokens, c->qtype, (int32_t)c->flags, c->qtype_down, 0};
  for (int j = 0; j < 12; ++j) k.i[j] = is[j];
  const float fs[6] = {c->weights_scale, c->norm_min, c->swiglu_limit, c->swiglu_limit_shared, c->rms_eps, 0.f};
  for (int j = 0; j < 6; ++j) k.f[j] = fs[j];

  std::unique_lock<std::mutex> lk(g_graph_mu);
  GraphSlot* hit = nullptr;
  for (auto& g : g_graphs)
    if (g.used && same_key(g.key, k)) {
      hit = &g;
      break;
    }
  if (hit && hit->exec) {
    hit->last = ++g_graph_tick;
    const cudaGraphExec_t ex = hit->exec;
    const cudaError_t e = cudaGraphLaunch(ex, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "graph launch");
  }
  if (!hit || hit->no_graph) {
    if (!hit) {  // first sight: remember the set (evicting the least recently used slot)
      GraphSlot* v = &g_graphs[0];
      for (auto& g : g_graphs) {
        if (!g.used) {
          v = &g;
          break;
        }
        if (g.last < v->last) v = &g;
      }
      if (v->used && v->exec) cudaGraphExecDestroy(v->exec);
      *v = GraphSlot{true, false, k, nullptr, ++g_graph_tick};
    }
    lk.unlock();
    return enqueue(x, router_w, bias, experts, shared, c, out, ws, ws_bytes, st, ids, wts);
  }
  // second sight: capture the call's work on the library's capture stream
  if (!g_capture_stream[dev]) {
    cudaError_t e = cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      g_capture_stream[dev] = nullptr;
      hit->no_graph = true;
      lk.unlock();
      cudaGetLastError();
      return enqueue(x, router_w, bias, experts, shared, c, out, ws, ws_bytes, st, ids, wts);
    }
  }
  const cudaStream_t cap = g_capture_stream[dev];
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int rc = MOE_ERR_CUDA;
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
    rc = enqueue(x, router_w, bias, experts, shared, c, out, ws, ws_bytes, cap, ids, wts);
    const cudaError_t e = cudaStreamEndCapture(cap, &graph);
    if (rc == MOE_OK && (e != cudaSuccess || cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)) {
      exec = nullptr;
      rc = MOE_ERR_CUDA;
    }
    if (graph) cudaGraphDestroy(graph);
  }
  cudaGetLastError();
  if (!exec) {
    hit->no_graph = true;
    lk.unlock();
    g_err[0] = 0;
    return enqueue(x, router_w, bias, experts, shared, c, out, ws, ws_bytes, st, ids, wts);
  }
  hit->exec = exec;
  hit->last = ++g_graph_tick;
  const cudaError_t e = cudaGraphLaunch(exec, st);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "graph launch");
}

void clear_graphs() {
  std::lock_guard<std::mutex> lk(g_graph_mu);
  for (auto& g : g_graphs) {
    if (g.used && g.exec) cudaGraphExecDestroy(g.exec);
    g = GraphSlot{};
  }
  for (auto& s : g_capture_stream) {
    if (s) cudaStreamDestroy(s);
    s = nullptr;
  }
}

// The error a nonzero status word reports.
int status_error(uint32_t bits) {
  if (bits & moe::DEV_ERR_MBAR_TIMEOUT)
    return fail(MOE_ERR_TIMEOUT, "a device-side wait timed out (status bits 0x%x); control block reset", bits);
  return fail(MOE_ERR_WORKSPACE,
              "a decode pick in the workspace was out of range (status bits 0x%x): the workspace was not "
              "zero-filled before its first use; control block reset", bits);
}

int read_status(void* ws, cudaStream_t st) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t ctrl[16];
  e = cudaMemcpy(ctrl, ws, sizeof ctrl, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (ctrl[moe::CTRL_STATUS] != 0) {
    // the counters of an interrupted call are not trustworthy: restart the control block
    const uint32_t bits = ctrl[moe::CTRL_STATUS];
    e = cudaMemset(ws, 0, moe::CTRL_BYTES);
    if (e != cudaSuccess) return cuda_fail(e, "control block reset");
    return status_error(bits);
  }
  return MOE_OK;
}

}  // namespace

// One thread waits on a fresh mbarrier (one arrival expected, none made) through the
// bounded wait; when it gives up it sets the timeout bit, as a stalled copy's wait would.
__global__ void selftest_timeout_kernel(uint32_t* ctrl) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bar, 1);
    moe::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !moe::mbar_wait(&bar, 0)) atomicOr(ctrl + moe::CTRL_STATUS, moe::DEV_ERR_MBAR_TIMEOUT);
}

extern "C" {

int moe_ffn_forward(const float* x, const float* router_w, const float* router_bias,
                    const void* expert_blocks, const void* shared_blocks, const moe_cfg* cfg, float* out) {
  g_err[0] = 0;
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (cfg->n_tokens == 0) return MOE_OK;
  const size_t need = ws_layout(cfg).total;
  void* ws = nullptr;
  rc = owned_workspace(need, &ws);
  if (rc != MOE_OK) return rc;
  rc = run(x, router_w, router_bias, expert_blocks, shared_blocks, cfg, out, ws, need, nullptr, nullptr,
           nullptr);
  if (rc != MOE_OK) return rc;
  return read_status(ws, nullptr);
}

int moe_ffn_forward_ex(const float* x, const float* router_w, const float* router_bias,
                       const void* expert_blocks, const void* shared_blocks, const moe_cfg* cfg, float* out,
                       void* workspace, size_t workspace_bytes, void* stream, int32_t* topk_ids,
                       float* topk_w) {
  g_err[0] = 0;
  return run(x, router_w, router_bias, expert_blocks, shared_blocks, cfg, out, workspace, workspace_bytes,
             static_cast<cudaStream_t>(stream), topk_ids, topk_w);
}

size_t moe_workspace_size(const moe_cfg* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return ws_layout(cfg).total;
}

size_t moe_trace_offset(const moe_cfg* cfg) {
  if (check_cfg(cfg) != MOE_OK || !(cfg->flags & MOE_TRACE)) return 0;
  return ws_layout(cfg).trace;
}

int moe_workspace_status(void* workspace, void* stream) {
  g_err[0] = 0;
  if (!workspace) return fail(MOE_ERR_NULL_PTR, "workspace is NULL");
  return read_status(workspace, static_cast<cudaStream_t>(stream));
}

int moe_selftest_timeout(void* workspace, void* stream) {
  g_err[0] = 0;
  if (!workspace) return fail(MOE_ERR_NULL_PTR, "workspace is NULL");
  selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(workspace));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "self-test launch");
}

const char* moe_last_error(void) { return g_err; }

int moe_shutdown(void) {
  clear_graphs();
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = MOE_OK;
  for (auto& w : g_ws) {
    if (w.ptr) {
      int prev = 0;
      cudaGetDevice(&prev);
      cudaSetDevice(w.device);
      if (cudaFree(w.ptr) != cudaSuccess) rc = MOE_ERR_CUDA;
      cudaSetDevice(prev);
    }
  }
  g_ws.clear();
  g_plans.clear();
  return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The step without any allocation, for callers that cannot allocate memory.
// ---------------------------------------------------------------------------
namespace {

// Fixed scratch for moe_ffn_forward_noalloc: the control block, the logits and the
// SwiGLU activations of the tokens of one launch (one token of the largest layer the
// checks admit, 32 picks of 3072 values plus a shared expert of 3072, needs about 401 KiB).
// It is device memory that exists from the moment the library's code is loaded on a
// device until the process exits; every call on that device shares it.
constexpr size_t NOALLOC_SCRATCH_BYTES = 512 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// The scratch's device address on the current device. In host code the array's name only
// stands in for the symbol; the address a kernel needs comes from cudaGetSymbolAddress with
// that device current. It is looked up on every call (cheap once the library's module is
// loaded on the device), so no address outlives the context it came from.
int noalloc_scratch(void** ptr) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the fixed scratch");
  *ptr = p;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_ffn_forward_noalloc(const float* x, const float* router_w, const float* router_bias,
                                       const void* expert_blocks, const void* shared_blocks,
                                       const moe_cfg* c, float* out, void* stream) {
  g_err[0] = 0;
  int rc = check_cfg(c);
  if (rc != MOE_OK) return rc;
  if (c->flags & (MOE_HOST_IO | MOE_TRACE))
    return fail(MOE_ERR_UNSUPPORTED, "moe_ffn_forward_noalloc takes device buffers only, without MOE_TRACE");
  const int T = c->n_tokens;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !expert_blocks || !out)
    return fail(MOE_ERR_NULL_PTR, "x, router_w, expert_blocks and out must not be NULL");
  if (c->shared_ff > 0 && !shared_blocks) return fail(MOE_ERR_NULL_PTR, "shared_ff > 0 needs shared_blocks");
  if (!aligned(router_w, 16) || !aligned(expert_blocks, 16) || (shared_blocks && !aligned(shared_blocks, 16)) ||
      !aligned(x, 16) || !aligned(out, 16) || (router_bias && !aligned(router_bias, 4)) ||
      (c->ffn_norm && !aligned(c->ffn_norm, 16)))
    return fail(MOE_ERR_ALIGNMENT, "x, out, router_w and the blocks must be 16-byte aligned, the bias 4-byte");
  const size_t xbytes = (size_t)T * c->hidden * 4;
  {
    const char* xa = reinterpret_cast<const char*>(x);
    const char* oa = reinterpret_cast<const char*>(out);
    if (xa < oa + xbytes && oa < xa + xbytes) return fail(MOE_ERR_INVALID_CFG, "x and out overlap");
  }
  // the calls decode up to td tokens at a time with `rep` copies of the broadcast arrays:
  // the most copies for which one token's scratch fits, then as many tokens as fit
  moe_cfg c1 = *c;
  int td = 1, rep = moe::DEC_REP;
  c1.n_tokens = 1;
  while (rep > 1 && ws_layout(&c1, true, rep).total > NOALLOC_SCRATCH_BYTES) --rep;
  for (td = T < moe::DEC_TMAX ? T : moe::DEC_TMAX; td > 1; --td) {
    c1.n_tokens = td;
    if (ws_layout(&c1, true, rep).total <= NOALLOC_SCRATCH_BYTES) break;
  }
  c1.n_tokens = td;
  const WsLayout W = ws_layout(&c1, true, rep);
  if (W.total > NOALLOC_SCRATCH_BYTES)
    return fail(MOE_ERR_UNSUPPORTED,
                "this layer needs %zu bytes of scratch; the fixed scratch of moe_ffn_forward_noalloc holds %zu",
                W.total, NOALLOC_SCRATCH_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != MOE_OK) return rc;
  PlanEntry pe;  // planned on every call: the plan cache of the other entry points would grow
  rc = make_plan(c, dev, &pe);
  if (rc != MOE_OK) return rc;

  uint8_t* wsb = static_cast<uint8_t*>(scratch);
  moe::DecodeArgs a{};
  a.router_w = router_w;
  a.bias = router_bias;
  a.experts = static_cast<const uint8_t*>(expert_blocks);
  a.shared = static_cast<const uint8_t*>(shared_blocks);
  a.ctrl = reinterpret_cast<uint32_t*>(wsb + W.ctrl);
  a.logits = reinterpret_cast<float*>(wsb + W.logits);
  a.act = reinterpret_cast<float*>(wsb + W.act);
  a.lg_copy = W.lg_copy;
  a.act_copy = W.act_copy;
  a.ids = reinterpret_cast<int32_t*>(wsb + W.ids);
  a.wts = reinterpret_cast<float*>(wsb + W.wts);
  a.pub = reinterpret_cast<unsigned long long*>(wsb + W.pub);
  a.trace = nullptr;
  a.scale = c->weights_scale;
  a.norm_min = c->norm_min;
  a.lim = c->swiglu_limit;
  a.lim_s = c->swiglu_limit_shared;
  a.norm = c->ffn_norm;
  a.eps = c->rms_eps;
  a.flags = c->flags & (MOE_ACCUMULATE | MOE_RESIDUAL);
  a.p = pe.plan;
  a.p.rep = W.rep;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool pdl = (c->flags & MOE_NO_PDL) == 0;
  for (int t = 0; t < T; t += td) {
    a.T = T - t < td ? T - t : td;
    a.x = x + (size_t)t * c->hidden;
    a.out = out + (size_t)t * c->hidden;
    a.topk_ids = nullptr;
    a.topk_w = nullptr;
    e = moe::decode_launch(a, pe.maxb, st, pdl, (c->flags & MOE_F32_ACT) == 0, 0);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  }
  // wait, then read the status word; after a device-side timeout the control block
  // is zeroed so the next call starts clean
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t status = 0;
  e = cudaMemcpy(&status, wsb + moe::CTRL_STATUS * 4, sizeof status, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (status != 0) {
    e = cudaMemset(wsb + W.ctrl, 0, moe::CTRL_BYTES);
    if (e != cudaSuccess) return cuda_fail(e, "control block reset");
    return status_error(status);
  }
  return MOE_OK;
}
