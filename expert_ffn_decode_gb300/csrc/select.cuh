// Expert selection shared by the decode and prefill kernels.
#pragma once

#include <cstdint>

namespace moe {

// Top-k by one warp: k rounds, each taking the largest key, the lowest expert
// index among equal keys. Lane l holds the keys of experts l + 32 i (i < EPL) in
// registers; key 0 marks an expert that cannot be picked (every real key is at
// least 0x007FFFFF, the key of -inf). Writes the picks in order to ids[0, k).
template <int EPL>
__device__ __forceinline__ void lane_best(const uint32_t (&kv)[EPL], int lane, uint32_t& bk, int& bi) {
  // a max tree over the lane's keys that keeps the lower index on ties
  uint32_t tk[EPL];
  int ti[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    tk[i] = kv[i];
    ti[i] = i;
  }
#pragma unroll
  for (int w = 1; w < EPL; w *= 2)
#pragma unroll
    for (int i = 0; i + w < EPL; i += 2 * w) {
      const bool right = tk[i + w] > tk[i];
      tk[i] = right ? tk[i + w] : tk[i];
      ti[i] = right ? ti[i + w] : ti[i];
    }
  bk = tk[0];
  bi = lane + 32 * ti[0];
}

// k rounds over the lane keys kv (kv[i]: expert lane + 32 i); kv is consumed.
template <int EPL>
__device__ __forceinline__ void topk_rounds_kv(uint32_t (&kv)[EPL], int E, int k, int* ids, int lane) {
  uint32_t bk;
  int bi;
  lane_best(kv, lane, bk, bi);
  for (int j = 0; j < k; ++j) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const unsigned cand = (bk == mk && mk != 0u) ? (unsigned)bi : 0xffffffffu;
    int win = (int)__reduce_min_sync(0xffffffffu, cand);
    if (win < 0 || win >= E) win = j % E;  // unreachable for a valid configuration
    if (lane == 0) ids[j] = win;
#pragma unroll
    for (int i = 0; i < EPL; ++i) kv[i] = (lane + 32 * i == win) ? 0u : kv[i];
    if ((win & 31) == lane) lane_best(kv, lane, bk, bi);
  }
}

}  // namespace moe
