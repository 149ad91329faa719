// Small device helpers for sm_103a: mbarriers, 1-D bulk async copies,
// programmatic-dependent-launch control, timers and the integer dot products used
// by the 4-bit kernels. Every wait here is bounded.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

namespace moe {

// ---- control block (first 512 bytes of every workspace) ---------------------
// A workspace starts zeroed. The status word is sticky until the host clears it.
enum CtrlWord : int {
  CTRL_STATUS = 8,   // device error bits (see DEV_ERR_*)
};
constexpr int CTRL_BYTES = 512;

enum DevErr : uint32_t {
  DEV_ERR_MBAR_TIMEOUT = 2u,   // a copy or a slot release never arrived
  DEV_ERR_BAD_PICK = 4u,       // a decode pick read from the workspace was out of range
};

// Raises a kernel's dynamic shared memory limit on the current device when a launch needs
// more than any earlier one did. The attribute persists, so later launches skip the
// driver call (it is on every call's host path). The table of raised limits is a fixed
// array (no allocation); once it is full, launches of further kernels set the attribute
// every time.
inline cudaError_t ensure_smem(const void* kern, int bytes) {
  struct Entry {
    int dev;
    const void* kern;
    int bytes;
  };
  constexpr int kMax = 512;
  static std::mutex mu;
  static Entry done[kMax];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n; ++i) {
    Entry& d = done[i];
    if (d.dev == dev && d.kern == kern) {
      if (d.bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) d.bytes = bytes;
      return e;
    }
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < kMax) done[n++] = Entry{dev, kern, bytes};
  return e;
}

// Spin limit, measured on %globaltimer: an mbarrier wait gives up after this many
// nanoseconds.
constexpr unsigned long long MBAR_TIMEOUT_NS = 500ull * 1000 * 1000;  // 0.5 s

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// The expected-bytes arrival orders nothing of the issuing thread: the copy's own
// completion is what signals the waiters, so the arrival is relaxed (a release would
// first wait for the thread's earlier stores).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && globaltimer() - t0 > MBAR_TIMEOUT_NS) return false;
  }
}

// ---- bulk async copy global -> shared (no tensor map) -------------------------
// Both addresses 16-byte aligned, size a multiple of 16; completion is counted
// in bytes on the mbarrier. `policy` is an L2 cache-policy descriptor.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- programmatic dependent launch --------------------------------------------
__device__ __forceinline__ void pdl_wait_prior_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- integer dot products ---------------------------------------------------------
// dp4a with unsigned bytes in a and unsigned (uu) or signed (us) bytes in b.
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// 64-bit relaxed (single-copy atomic) global store and load at GPU scope.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// dp4a with signed bytes in a and unsigned (su) or signed (ss) bytes in b.
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ---- f32 block dots ------------------------------------------------------------
// A small unsigned integer q (a byte holding 0..63) becomes the f32 number 2^23 + q when it
// is placed in the low mantissa byte of 2^23 (bit pattern 0x4B000000); subtracting 2^23 (or
// 2^23 + c) then leaves q (or q - c) exactly. Byte j (0..3) of w:
__device__ __forceinline__ float magic_byte(uint32_t w, int j) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | (uint32_t)j));
}
constexpr float MAGIC_2P23 = 8388608.0f;  // 2^23

// Packed pairs of f32 (two lanes of one 64-bit register pair): a - c on both lanes, and
// a + q * x on both lanes, each rounded as the scalar f32 operation is.
__device__ __forceinline__ void sub2_f32(float& q0, float& q1, float c) {
  asm("{.reg .b64 q, c;\n mov.b64 q, {%0, %1};\n mov.b64 c, {%2, %2};\n sub.rn.f32x2 q, q, c;\n"
      " mov.b64 {%0, %1}, q;}" : "+f"(q0), "+f"(q1) : "f"(c));
}
__device__ __forceinline__ void fma2_f32(float& a0, float& a1, float q0, float q1, float x0, float x1) {
  asm("{.reg .b64 q, x, a;\n mov.b64 q, {%2, %3};\n mov.b64 x, {%4, %5};\n mov.b64 a, {%0, %1};\n"
      " fma.rn.f32x2 a, q, x, a;\n mov.b64 {%0, %1}, a;}"
      : "+f"(a0), "+f"(a1) : "f"(q0), "f"(q1), "f"(x0), "f"(x1));
}
// a0/a1 += (q_j - off) * x_j for the four byte values q_j of w and the four floats of x.
__device__ __forceinline__ void word_dot_f32(uint32_t w, const float4& x, float off, float& a0, float& a1) {
  float q0 = magic_byte(w, 0), q1 = magic_byte(w, 1), q2 = magic_byte(w, 2), q3 = magic_byte(w, 3);
  sub2_f32(q0, q1, off);
  sub2_f32(q2, q3, off);
  fma2_f32(a0, a1, q0, q1, x.x, x.y);
  fma2_f32(a0, a1, q2, q3, x.z, x.w);
}

// Round-to-nearest-even of |y| <= 2^22 to an integer by the add-and-subtract of
// 1.5 * 2^23 (the float then holds the integer in its low mantissa bits).
__device__ __forceinline__ int round_small(float y) {
  return __float_as_int(y + 12582912.0f) - 0x4B400000;
}

// Float -> 32-bit key whose unsigned order is the float order (-0 taken as +0).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// SwiGLU of one intermediate value: silu(g) * u, or with a clamp limit L > 0,
// min(silu(g), L) * clamp(u, -L, L) (ling_moe_ssd.js, the swiglu kernel).
__device__ __forceinline__ float swiglu_act(float g, float u, float L) {
  float sg = g / (1.f + expf(-g));
  if (L > 0.f) {
    u = fminf(fmaxf(u, -L), L);
    sg = fminf(sg, L);
  }
  return sg * u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 1 / sqrt(mean(x^2) + eps) over a row of H floats (H a multiple of 4, x 16-byte
// aligned), by a whole CTA of blockDim.x threads (a multiple of 32, at most 1024);
// `red` is 32 floats of shared memory. Every thread gets the result; the summation
// order is fixed. Synchronises the CTA.
__device__ __forceinline__ float block_rms_scale(const float* x, int H, float eps, float* red) {
  float ss = 0.f;
  for (int h = 4 * (int)threadIdx.x; h < H; h += 4 * (int)blockDim.x) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(x + h));
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  __syncthreads();  // red may be reused
  return 1.f / sqrtf(tot / (float)H + eps);
}

}  // namespace moe
