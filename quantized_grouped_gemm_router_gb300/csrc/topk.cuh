// Warp-wide top-k with renormalised softmax weights (page "Perplexity's Lily beats MLX-LM on
// MacBook M5 because it only runs one model", section "Why Qwen3.6-35B-A3B is a weird
// workload": the router scores the experts and picks the top k).
//
// Logits become order-preserving unsigned keys (-0.0 folded onto +0.0); the largest key is the
// largest logit, and equal logits are split by the lower expert index.
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

// Whole warp: selects the top k (k <= 16 <= 32) of row[0..E) (E <= 32 * SLOTS). Lane j < k
// returns its slot's expert in *e_out and weight in *w_out. Returns true (on every lane) if any
// logit of the row was NaN or infinite; the selection then stays within [0, E) but is
// meaningless.
//
// Lane l holds experts l, l+32, ... as order-preserving 32-bit keys and keeps its best untaken
// one (largest key, lowest index among equal keys). Each round takes the warp maximum of the
// lanes' bests with one redux.sync, then the lowest expert index among the lanes holding that
// maximum with a second one; only the winning lane rescans its own keys.
template <int SLOTS>
__device__ __forceinline__ bool warp_topk_softmax(const float* row, int E, int k, int* e_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t key[SLOTS];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;  // below every finite logit's key
    if (e < E) {
      const float v = __ldcg(row + e);
      bad |= !isfinite(v);
      key[i] = max(orderable_f32(v), 1u);
    }
  }
  uint32_t taken = 0u, bv = 0u;
  int bi = 0;
  auto local_best = [&]() {
    bv = 0u;
    bi = 0;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (!((taken >> i) & 1u) && key[i] > bv) {
        bv = key[i];
        bi = i;
      }
  };
  local_best();
  int my_e = 0;
  float my_v = 0.f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const uint32_t vmax = __reduce_max_sync(0xFFFFFFFFu, bv);
    const uint32_t cand = (bv == vmax && bv != 0u) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
    const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (lane == j) {
      my_e = (int)emin;
      my_v = from_orderable_f32(vmax);
    }
    if ((int)(emin & 31u) == lane) {
      taken |= 1u << (emin >> 5);
      local_best();
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

// Compare-exchange keeping a >= b (descending order).
__device__ __forceinline__ void cx_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}
// Sorts 8 keys descending (Batcher's odd-even merge network, 19 compare-exchanges).
__device__ __forceinline__ void sort8_desc(uint64_t (&v)[8]) {
  cx_desc(v[0], v[1]); cx_desc(v[2], v[3]); cx_desc(v[4], v[5]); cx_desc(v[6], v[7]);
  cx_desc(v[0], v[2]); cx_desc(v[1], v[3]); cx_desc(v[4], v[6]); cx_desc(v[5], v[7]);
  cx_desc(v[1], v[2]); cx_desc(v[5], v[6]);
  cx_desc(v[0], v[4]); cx_desc(v[1], v[5]); cx_desc(v[2], v[6]); cx_desc(v[3], v[7]);
  cx_desc(v[2], v[4]); cx_desc(v[3], v[5]);
  cx_desc(v[1], v[2]); cx_desc(v[3], v[4]); cx_desc(v[5], v[6]);
}

// Whole warp, E <= 256, k <= 8: the same selection and weights as warp_topk_softmax<8>, with no
// serial rounds. Every expert gets the unique key (orderable logit << 32) | ~index, so a larger
// key is a larger logit, or an equal logit with a lower index. Each lane sorts its 8 keys; five
// butterfly steps then merge the lane's sorted top 8 with its partner's (a bitonic merge keeps
// the larger half), after which every lane holds the warp's top 8 in order.
__device__ __forceinline__ bool warp_top8_softmax(const float* row, int E, int k, int* e_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  uint64_t v[8];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = 0ull;  // below every real key
    if (e < E) {
      const float x = __ldcg(row + e);
      bad |= !isfinite(x);
      v[i] = ((uint64_t)max(orderable_f32(x), 1u) << 32) | (uint32_t)~(uint32_t)e;
    }
  }
  sort8_desc(v);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    uint64_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __shfl_xor_sync(0xFFFFFFFFu, v[i], off);
    // v descending, o descending: max(v[i], o[7-i]) is a bitonic sequence holding the top 8
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = v[i] > o[7 - i] ? v[i] : o[7 - i];
    cx_desc(v[0], v[4]); cx_desc(v[1], v[5]); cx_desc(v[2], v[6]); cx_desc(v[3], v[7]);
    cx_desc(v[0], v[2]); cx_desc(v[1], v[3]); cx_desc(v[4], v[6]); cx_desc(v[5], v[7]);
    cx_desc(v[0], v[1]); cx_desc(v[2], v[3]); cx_desc(v[4], v[5]); cx_desc(v[6], v[7]);
  }
  uint64_t mine = v[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if (lane == i) mine = v[i];
  const int my_e = (int)~(uint32_t)mine;
  const float my_v = from_orderable_f32((uint32_t)(mine >> 32));
  // Softmax restricted to the selected experts; slot 0 holds the largest logit.
  const float vmax = from_orderable_f32((uint32_t)(v[0] >> 32));
  const float ex = lane < k ? expf(my_v - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  *e_out = min(max(my_e, 0), E - 1);
  *w_out = ex / sum;
  return __any_sync(0xFFFFFFFFu, bad);
}

// Dispatch on the number of experts per lane and on k.
__device__ __forceinline__ bool warp_topk_softmax(const float* row, int E, int k, int* e_out, float* w_out) {
  if (E <= 256 && k <= 8) return warp_top8_softmax(row, E, k, e_out, w_out);
  if (E <= 256) return warp_topk_softmax<8>(row, E, k, e_out, w_out);
  return warp_topk_softmax<32>(row, E, k, e_out, w_out);
}

}  // namespace moe
