// GPU-resident routing (page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs
// one model", section "Prefill: keep routing on the GPU, dequantize in flight": after the top-8
// selection, histogram, prefix scan, scatter and block map run on the GPU with no host round
// trip). Three launches (four in prefill):
//   route_topk_kernel    8 tokens per CTA, one per warp: top-k on order-preserving logit keys
//                        (ties to the lower index), renormalised softmax weights (after summing
//                        the router GEMM's K slices when it was split)
//   route_hist_kernel    one CTA per chunk (64 tokens, more above 4096 tokens): histogram in shared
//                        memory, added into the per-expert totals; the last CTA to finish (ticket)
//                        scans the totals into counts, offsets and the tile block map. In prefill
//                        its extra CTAs make the fp16 copy of x meanwhile.
//   route_scatter_kernel one CTA per chunk: the chunk's base inside each expert (the earlier chunks'
//                        counts summed), then stable placement of its assignments (per-warp
//                        histograms and a prefix in warp order, then in-warp ranks by
//                        __match_any_sync; no global atomics). In prefill its extra CTAs zero the
//                        combine accumulator rows meanwhile.
//   route_rows_kernel    (prefill) copies each assignment's fp16 token row to its sorted
//                        position, so the grouped GEMM reads every tile as contiguous rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kTopkThreads = 256;
constexpr int kTopkTokens = 8;    // tokens per CTA of the top-k kernel: one per warp

// Exclusive scan of up to 4*blockDim values held 4 per thread (v[0..3] are items 4t..4t+3).
// Returns the exclusive prefix of item 4t; *total receives the sum of all items.
__device__ int block_exclusive_scan4(const int (&v)[4], int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int mine = v[0] + v[1] + v[2] + v[3];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < nwarps) s_warp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int before_warp = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[nwarps - 1];
  __syncthreads();
  return before_warp + incl - mine;
}

// Share `part` of `parts` of the fp16 copy of x (token order, the expert GEMMs' operand; exact
// inside the fp16 range, anything beyond it is reported): 8 loads in flight per thread.
__device__ void copy_x16_share(const RouteParams& p, int part, int parts) {
  constexpr int kU = 8;
  const int lane = threadIdx.x & 31;
  const size_t n8 = (size_t)p.T * p.d / 8, step = (size_t)parts * blockDim.x;
  const uint4* xs = reinterpret_cast<const uint4*>(p.x);
  uint4* xd = reinterpret_cast<uint4*>(p.x16 + (size_t)p.T * p.k * p.d);
  bool over = false;
  for (size_t i0 = (size_t)part * blockDim.x + threadIdx.x; i0 < n8; i0 += kU * step) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const size_t i = i0 + u * step;
      v[u] = i < n8 ? xs[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const size_t i = i0 + u * step;
      const uint32_t in[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(in[j] << 16), hi = __uint_as_float(in[j] & 0xFFFF0000u);
        over |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
        const __half2 h = __floats2half2_rn(lo, hi);
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      if (i < n8) xd[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (__any_sync(0xFFFFFFFFu, over) && lane == 0) set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
}

// Share `part` of `parts` of the zeroing of the combine accumulator rows [T, d].
__device__ void zero_yacc_share(const RouteParams& p, int part, int parts) {
  const size_t n4 = (size_t)p.T * p.d / 4, step = (size_t)parts * blockDim.x;
  float4* y = reinterpret_cast<float4*>(p.yacc);
  for (size_t i = (size_t)part * blockDim.x + threadIdx.x; i < n4; i += step) y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Extra CTAs the histogram (fp16 copy of x) and scatter (accumulator zeroing) launches carry: the
// two byte streams run beside those latency-bound kernels instead of in front of the selections.
// One CTA per 64 KB written, two per SM at most.
constexpr int kStreamCtas = 304;
inline int stream_ctas(size_t bytes) {
  const size_t n = (bytes + 65535) / 65536;
  return (int)(n < 8 ? 8 : n > (size_t)kStreamCtas ? kStreamCtas : n);
}

// The top-k of the CTA's kTopkTokens tokens, one per warp: a selection is a latency-bound chain,
// so every token gets its own warp and they all run at once.
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(const RouteParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k;
  const int t_begin = blockIdx.x * kTopkTokens;
  const int t_end = min(p.T, t_begin + kTopkTokens);
  if (blockIdx.x == 0)  // the histogram kernel adds every chunk into these
    for (int e = tid; e < E; e += kTopkThreads) p.totals[e] = 0;
  for (int t = t_begin + warp; t < t_end; t += kTopkThreads / 32) {
    if (p.ksplit > 1) {  // the router GEMM's K slices: their partial logits summed in slice order
      float* row = const_cast<float*>(p.logits) + (size_t)t * E;
      const size_t slice = (size_t)p.T * E;
      for (int e0 = 0; e0 < E; e0 += 8 * 32) {  // 8 experts per lane, every slice's loads in flight
        float v[kMaxRouterSplit][8];
#pragma unroll
        for (int s = 0; s < kMaxRouterSplit; ++s)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = e0 + lane + 32 * i;
            v[s][i] = s < p.ksplit && e < E ? __ldcg(row + s * slice + e) : 0.f;
          }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float a = v[0][i];
#pragma unroll
          for (int s = 1; s < kMaxRouterSplit; ++s) a += v[s][i];  // zero beyond ksplit: exact
          if (e0 + lane + 32 * i < E) row[e0 + lane + 32 * i] = a;
        }
      }
      __syncwarp();
    }
    int my_e;
    float my_w;
    const bool bad = warp_topk_softmax(p.logits + (size_t)t * E, E, k, &my_e, &my_w);
    if (bad && lane == 0) set_device_status(p.hdr, MOE_ERR_NONFINITE);
    if (lane < k) {
      p.topk_idx[(size_t)t * k + lane] = my_e;
      p.topk_w[(size_t)t * k + lane] = my_w;
    }
  }
}

// Histogram of one p.chunk-token chunk in shared memory, kept per chunk (the scatter's bases) and
// added into the per-expert totals. The last CTA to finish (ticket) turns the totals into counts,
// offsets and the tile block map.
__global__ void __launch_bounds__(kTopkThreads) route_hist_kernel(const RouteParams p) {
  __shared__ int s_counts[kMaxExperts];
  __shared__ int s_warp[32];
  __shared__ int s_last;
  pdl_wait();
  pdl_launch_dependents();
  if ((int)blockIdx.x >= p.n_chunks) {  // a stream CTA: its share of the fp16 copy of x
    copy_x16_share(p, blockIdx.x - p.n_chunks, gridDim.x - p.n_chunks);
    return;
  }
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const int E = p.E, k = p.k;
  for (int e = tid; e < E; e += blockDim.x) s_counts[e] = 0;
  __syncthreads();
  const int a_begin = c * p.chunk * k, a_end = min(p.T, (c + 1) * p.chunk) * k;
  for (int a = a_begin + tid; a < a_end; a += blockDim.x) atomicAdd(&s_counts[p.topk_idx[a]], 1);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    const int n = s_counts[e];
    p.chunk_counts[(size_t)c * E + e] = n;
    if (n) atomicAdd(p.totals + e, n);  // integer adds: the totals do not depend on their order
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&p.hdr->ticket, 1u) == (unsigned)p.n_chunks - 1u);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  for (int e = tid; e < E; e += blockDim.x) s_counts[e] = __ldcg(p.totals + e);  // own histogram done
  __syncthreads();
  int cnt[4], tiles[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * tid + i;
    cnt[i] = e < E ? s_counts[e] : 0;
    tiles[i] = (cnt[i] + p.tile_rows - 1) / p.tile_rows;
  }
  int total_rows, total_tiles;
  const int off0 = block_exclusive_scan4(cnt, s_warp, &total_rows);
  const int tile0 = block_exclusive_scan4(tiles, s_warp, &total_tiles);
  int off = off0, tl = tile0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * tid + i;
    if (e < E) {
      p.counts[e] = cnt[i];
      p.offsets[e] = off;
      for (int r = 0; r < tiles[i]; ++r) {
        int32_t* tm = p.tile_map + 3 * (size_t)(tl + r);
        tm[0] = e;
        tm[1] = r * p.tile_rows;
        tm[2] = min(p.tile_rows, cnt[i] - r * p.tile_rows);
        p.tile_row0[tl + r] = off + r * p.tile_rows;
      }
    }
    off += cnt[i];
    tl += tiles[i];
  }
  if (tid == 0) {
    p.offsets[E] = total_rows;
    *p.n_tiles = total_tiles;
    p.hdr->ticket = 0u;  // ready for the next call
  }
}

// One CTA of kScatterWarps warps per chunk. Warp w takes the chunk's w-th run of consecutive
// assignments (a = t*k + j ascending); a per-warp histogram and a prefix over the warps (in
// warp order) give each warp its experts' first free positions, then each warp places its run
// 32 assignments at a time (in-warp ranks by __match_any_sync): the result is the stable order.
// No atomics: every counter has a single writer (the lowest lane of an expert's peer group).
constexpr int kScatterWarps = 8;
__global__ void __launch_bounds__(kScatterWarps * 32) route_scatter_kernel(const RouteParams p) {
  __shared__ int s_run[kScatterWarps][kMaxExperts];  // counts, then first free positions
  pdl_wait();
  pdl_launch_dependents();
  if ((int)blockIdx.x >= p.n_chunks) {  // a stream CTA: its share of the accumulator zeroing
    zero_yacc_share(p, blockIdx.x - p.n_chunks, gridDim.x - p.n_chunks);
    return;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int E = p.E;
  for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) s_run[i / E][i % E] = 0;
  __syncthreads();
  const int a_begin = c * p.chunk * p.k;
  const int a_end = min(p.T, (c + 1) * p.chunk) * p.k;
  const int per = (a_end - a_begin + kScatterWarps - 1) / kScatterWarps;
  const int w_begin = min(a_end, a_begin + w * per), w_end = min(a_end, w_begin + per);
  const unsigned lt_mask = (1u << lane) - 1u;
  // This warp's histogram, 32 assignments at a time: the lowest lane of each expert's peer group
  // adds the group's size (one writer per counter, no atomics).
  for (int base = w_begin; base < w_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < w_end;
    const int e = valid ? p.topk_idx[a] : -1 - lane;  // invalid lanes get unique keys
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (valid && (peers & lt_mask) == 0u) s_run[w][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    // the chunk's first position inside expert e: the earlier chunks' counts, 16 loads in flight
    int base = 0;
    for (int c0 = 0; c0 < c; c0 += 16) {
      int v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = c0 + j < c ? __ldcg(p.chunk_counts + (size_t)(c0 + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) base += v[j];
    }
    int pos = p.offsets[e] + base;
#pragma unroll
    for (int v = 0; v < kScatterWarps; ++v) {
      const int n = s_run[v][e];
      s_run[v][e] = pos;
      pos += n;
    }
  }
  __syncthreads();
  int* run = s_run[w];
  for (int base = w_begin; base < w_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < w_end;
    const int e = valid ? p.topk_idx[a] : -1 - lane;  // invalid lanes get unique keys
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (valid) {
      const int pos = run[e] + __popc(peers & lt_mask);
      p.perm[pos] = a;
      p.inv_perm[a] = pos;
      p.row_tw[pos] = make_int2(a / p.k, __float_as_int(p.topk_w[a]));
    }
    __syncwarp();
    if (valid && (peers & lt_mask) == 0u) run[e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per sorted row: x16[pos] = x16[A + perm[pos] / k] (16-byte copies, d/8 per row; every
// lane's loads of a row, up to 8, are in flight at once).
__global__ void __launch_bounds__(256) route_rows_kernel(const RouteParams p) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int kU = 8;
  const int A = p.T * p.k, n16 = p.d / 8;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (int pos = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pos < A; pos += warps) {
    const int t = p.row_tw[pos].x;
    const uint4* src = reinterpret_cast<const uint4*>(p.x16 + ((size_t)A + t) * p.d);
    uint4* dst = reinterpret_cast<uint4*>(p.x16 + (size_t)pos * p.d);
    for (int i0 = lane; i0 < n16; i0 += kU * 32) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) v[u] = i0 + 32 * u < n16 ? src[i0 + 32 * u] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (i0 + 32 * u < n16) dst[i0 + 32 * u] = v[u];
    }
  }
}

__global__ void __launch_bounds__(256) cast_kernel(const float* __restrict__ yacc, uint16_t* __restrict__ y, size_t n8) {
  pdl_wait();
  pdl_launch_dependents();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(yacc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(yacc)[2 * i + 1];
    __nv_bfloat162 o0 = __floats2bfloat162_rn(a.x, a.y), o1 = __floats2bfloat162_rn(a.z, a.w);
    __nv_bfloat162 o2 = __floats2bfloat162_rn(b.x, b.y), o3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t*>(&o0);
    o.y = *reinterpret_cast<uint32_t*>(&o1);
    o.z = *reinterpret_cast<uint32_t*>(&o2);
    o.w = *reinterpret_cast<uint32_t*>(&o3);
    reinterpret_cast<uint4*>(y)[i] = o;
  }
}

}  // namespace

// Every launch is chained to its predecessor with programmatic dependent launch: it starts while
// the predecessor finishes and waits for it (pdl_wait) before touching any data.
cudaError_t launch_route_topk(const RouteParams& p, cudaStream_t s) {
  return launch_pdl(route_topk_kernel, (p.T + kTopkTokens - 1) / kTopkTokens, kTopkThreads, 0, 1, s, p);
}

cudaError_t launch_route_group(const RouteParams& p, cudaStream_t s) {
  const size_t rows_bytes = (size_t)p.T * p.d * 2;  // fp16 copy; the accumulator takes twice that
  cudaError_t err = launch_pdl(route_hist_kernel, p.n_chunks + (p.x ? stream_ctas(rows_bytes) : 0), kTopkThreads, 0, 1,
                               s, p);
  if (err != cudaSuccess) return err;
  return launch_pdl(route_scatter_kernel, p.n_chunks + (p.yacc ? stream_ctas(2 * rows_bytes) : 0),
                    kScatterWarps * 32, 0, 1, s, p);
}

// The fp16 copy of x and the accumulator zeroing on their own (the host-routing ablation, whose
// histogram and scatter run on the host).
__global__ void __launch_bounds__(256) route_streams_kernel(const RouteParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int half = gridDim.x / 2;
  if ((int)blockIdx.x < half) {
    if (p.x) copy_x16_share(p, blockIdx.x, half);
  } else if (p.yacc) {
    zero_yacc_share(p, blockIdx.x - half, gridDim.x - half);
  }
}

cudaError_t launch_route_streams(const RouteParams& p, cudaStream_t s) {
  return launch_pdl(route_streams_kernel, 2 * kStreamCtas, 256, 0, 1, s, p);
}

cudaError_t launch_route_rows(const RouteParams& p, cudaStream_t s) {
  const int rows = p.T * p.k, per_cta = 8;  // 8 warps of 256 threads
  const int blocks = (rows + per_cta - 1) / per_cta < 152 * 8 ? (rows + per_cta - 1) / per_cta : 152 * 8;
  return launch_pdl(route_rows_kernel, blocks, 256, 0, 1, s, p);
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t s) {
  cudaError_t err = launch_route_topk(p, s);
  if (err != cudaSuccess) return err;
  if ((err = launch_route_group(p, s)) != cudaSuccess || !p.x) return err;
  return launch_route_rows(p, s);
}

cudaError_t launch_cast(const float* yacc, uint16_t* y, size_t n, cudaStream_t s) {
  const size_t n8 = n / 8;
  const int blocks = (int)((n8 + 255) / 256 < 1216 ? (n8 + 255) / 256 : 1216);
  return launch_pdl(cast_kernel, blocks > 0 ? blocks : 1, 256, 0, 1, s, yacc, y, n8);
}

}  // namespace moe
