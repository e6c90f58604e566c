// Warp-wide top-k with renormalised softmax weights (page "Perplexity's Lily beats MLX-LM on
// MacBook M5 because it only runs one model", section "Why Qwen3.6-35B-A3B is a weird
// workload": the router scores the experts and picks the top k).
//
// Each (logit, expert) pair becomes a 64-bit key: an order-preserving image of the fp32 logit
// in the high word (-0.0 folded onto +0.0) and (0xFFFFFFFF - expert) in the low word, so the
// largest key is the largest logit and, among equal logits, the lowest expert index. k rounds
// of a shuffle max-reduction pick the experts in descending order.
#pragma once

#include <stdint.h>

#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ uint32_t orderable_f32(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_orderable_f32(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Whole warp: selects the top k (k <= 16 <= 32) of row[0..E) (E <= 1024). Lane j < k returns
// its slot's expert in *e_out and weight in *w_out. Returns true (on every lane) if any logit
// of the row was NaN or infinite; the selection then stays within [0, E) but is meaningless.
__device__ __forceinline__ bool warp_topk_softmax(const float* row, int E, int k, int* e_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  const int per_lane = (E + 31) >> 5;
  unsigned long long key[32];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    key[i] = 0ull;
    const int e = lane + 32 * i;
    if (i < per_lane && e < E) {
      const float v = __ldcg(row + e);
      bad |= !isfinite(v);
      key[i] = ((unsigned long long)orderable_f32(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
    }
  }
  int my_e = 0;
  float my_v = 0.f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < 32; ++i) best = key[i] > best ? key[i] : best;
    best = warp_max_u64(best);
    const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    if ((e & 31) == lane) {
      const int slot = e >> 5;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i == slot) key[i] = 0ull;
    }
    if (lane == j) {
      my_e = e;
      my_v = from_orderable_f32((uint32_t)(best >> 32));
    }
  }
  // Softmax restricted to the selected experts; slot 0 holds the largest logit.
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const float ex = lane < k ? expf(my_v - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  *e_out = min(max(my_e, 0), E - 1);
  *w_out = ex / sum;
  return __any_sync(0xFFFFFFFFu, bad);
}

}  // namespace moe
