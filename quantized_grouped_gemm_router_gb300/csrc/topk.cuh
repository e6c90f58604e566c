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

// Whole warp, E <= 32 * SLOTS, k <= 16: the same selection and weights as warp_topk_softmax,
// computed by a threshold and exact ranks instead of k serial rounds. Every expert has the unique
// key (orderable logit << 32) | ~index. Each lane's largest key belongs to a different expert, so
// the k-th largest key overall is at least tau, the k-th largest of the 32 lane maxima; only the
// experts with a key >= tau (about k + 1 for Gaussian logits) are candidates. They are gathered
// one per lane and ranked by counting the larger candidate keys. If more than 32 experts pass the
// threshold (ties of the logits), the serial selection runs instead.
// Returns true (on every lane) if a logit of the row was NaN or infinite. Lane l gets *rank_out =
// the slot (0..k-1) of the expert it holds, with its expert and weight, or -1.
template <int SLOTS>
__device__ __forceinline__ bool warp_select_topk(const float* row, int E, int k, int* rank_out, int* e_out,
                                                 float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t key[SLOTS];
  bool bad = false;
  uint32_t bk = 0u;
  int bi = 0;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;  // below every real key
    if (e < E) {
      const float v = __ldcg(row + e);
      bad |= !isfinite(v);
      key[i] = max(orderable_f32(v), 1u);
    }
    if (key[i] > bk) {  // strict: the lowest index wins among equal keys
      bk = key[i];
      bi = i;
    }
  }
  const unsigned long long lu = bk ? ((unsigned long long)bk << 32) | (uint32_t)~(uint32_t)(lane + 32 * bi) : 0ull;
  int lr = 0;  // rank of this lane's maximum among the 32
#pragma unroll 8
  for (int j = 0; j < 32; ++j) lr += __shfl_sync(0xFFFFFFFFu, lu, j) > lu ? 1 : 0;
  const int n_valid = __popc(__ballot_sync(0xFFFFFFFFu, bk != 0u));
  unsigned long long tau = 0ull;
  if (k <= n_valid) {
    const unsigned src = __ballot_sync(0xFFFFFFFFu, lu != 0ull && lr == k - 1);
    tau = __shfl_sync(0xFFFFFFFFu, lu, __ffs(src) - 1);
  }
  // gather the candidates (keys >= tau) one per lane, in (slot i, lane) order
  unsigned long long cand = 0ull;
  int n = 0;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = lane + 32 * i;
    const unsigned long long u = ((unsigned long long)key[i] << 32) | (uint32_t)~(uint32_t)e;
    const unsigned b = __ballot_sync(0xFFFFFFFFu, e < E && u >= tau);
    const int c = lane - n;  // this lane's candidate slot, if it falls in this row
    const int src = (c >= 0 && c < __popc(b)) ? __fns(b, 0, c + 1) : 0;
    const unsigned long long got = __shfl_sync(0xFFFFFFFFu, u, src);
    if (c >= 0 && c < __popc(b)) cand = got;
    n += __popc(b);
  }
  if (n > 32) {  // ties at the threshold: serial selection (lane j holds slot j)
    const bool b2 = warp_topk_softmax<SLOTS>(row, E, k, e_out, w_out);
    *rank_out = lane < k ? lane : -1;
    return b2;
  }
  int rank = 0;
  for (int j = 0; j < n; ++j) rank += __shfl_sync(0xFFFFFFFFu, cand, j) > cand ? 1 : 0;
  const bool mine = lane < n && rank < k;
  const float my_v = from_orderable_f32((uint32_t)(cand >> 32));
  // Softmax restricted to the selected experts, relative to the largest logit (rank 0).
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, __ffs(__ballot_sync(0xFFFFFFFFu, mine && rank == 0)) - 1);
  const float ex = mine ? expf(my_v - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  *rank_out = mine ? rank : -1;
  *e_out = min(max((int)~(uint32_t)cand, 0), E - 1);
  *w_out = ex / sum;
  return __any_sync(0xFFFFFFFFu, bad);
}

// Dispatch on the number of experts per lane.
__device__ __forceinline__ bool warp_select_topk(const float* row, int E, int k, int* rank_out, int* e_out,
                                                 float* w_out) {
  if (E <= 256) return warp_select_topk<8>(row, E, k, rank_out, e_out, w_out);
  return warp_select_topk<32>(row, E, k, rank_out, e_out, w_out);
}

}  // namespace moe
