// Batch-1 decode path: Q4 GEMVs that stream only the selected experts' packed weights.
//
// Page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model":
// section "Prefill and decode are different problems" (decode at batch 1 is a matrix-vector
// product bound by memory bandwidth; "minimize bytes moved per token"), section "Decode:
// minimize bytes per token" (fusion of the input projections with the gate activation and of
// the output projection with the routing scores and the shared expert), section "What didn't
// work" (the GEMV runs near the weight-read rate and its arithmetic barely matters).
//
// Three launches on one stream:
//   decode_router_kernel  one warp per expert: logit = W_r[e] . x (+ b_e); the last CTA to
//                         finish selects the top k and their renormalised weights
//   decode_gateup_kernel  one CTA per (selected or shared expert, 32 intermediate rows):
//                         gate and up GEMV rows over the packed blocks, SwiGLU in registers
//   decode_down_kernel    one CTA per 16 output rows: the down GEMV of all k+1 experts, scaled
//                         by the routing weights (shared expert weight 1) and summed in a fixed
//                         order (deterministic, no atomics), written as bf16
// Weights stream with 128-bit non-allocating loads; per group of 64 inputs the dot product is
// scale * sum(q*x) + bias * sum(x), with sum(x) computed once per input vector.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kDecThreads = 256;
constexpr int kGateUpRows = 32;   // intermediate rows per gate/up CTA
constexpr int kDownRows = 16;     // output rows per down CTA

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_stream32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// One row of one 64-column block: sum_c (scale*q_c + bias) * x_c, with x (64 fp32 values,
// shared memory) and gsum = sum_c x_c. Codes are read as (128 + q) bf16 pairs, so the
// accumulated value is sum (128 + q) x; scale*acc + (bias - 128*scale)*gsum removes the offset.
__device__ __forceinline__ float dot_block(const uint4 c0, const uint4 c1, uint32_t sb, const float* xs, float gsum) {
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t = ((words[c] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
      acc0 = fmaf(bf16lo(t), xs[8 * c + 2 * i], acc0);
      acc1 = fmaf(bf16hi(t), xs[8 * c + 2 * i + 1], acc1);
    }
  }
  const float s = bf16lo(sb), b = bf16hi(sb);
  return s * (acc0 + acc1) + (b - 128.f * s) * gsum;
}

__global__ void __launch_bounds__(kDecThreads) decode_router_kernel(const DecodeParams p) {
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * (kDecThreads / 32) + warp;
  if (e < p.E) {
    const uint16_t* w = p.router_w + (size_t)e * p.d;
    float acc = 0.f;
    for (int i = lane * 8; i < p.d; i += 256) {
      const uint4 xv = *reinterpret_cast<const uint4*>(p.x + i);
      const uint4 wv = ld_stream(w + i);
      const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = fmaf(bf16lo(xa[j]), bf16lo(wa[j]), acc);
        acc = fmaf(bf16hi(xa[j]), bf16hi(wa[j]), acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) p.logits[e] = acc + (p.router_bias ? p.router_bias[e] : 0.f);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&p.hdr->dticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  int my_e;
  float my_w;
  const bool bad = warp_topk_softmax(p.logits, p.E, p.k, &my_e, &my_w);
  if (lane < p.k) {
    p.topk_idx[lane] = my_e;
    p.topk_w[lane] = my_w;
  }
  if (lane == 0) {
    if (bad) set_device_status(p.hdr, MOE_ERR_NONFINITE);
    p.hdr->dticket = 0u;
  }
}

// Dynamic shared memory: x as fp32 [d], group sums [d/64], partials [8 warps][2][32].
__global__ void __launch_bounds__(kDecThreads) decode_gateup_kernel(const DecodeParams p) {
  extern __shared__ float dsm[];
  float* s_x = dsm;
  float* s_gs = s_x + p.d;
  float* s_part = s_gs + p.d / kGroup;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_slot = p.inter / kGateUpRows;
  const int slot = blockIdx.x / per_slot;
  const int f0 = (blockIdx.x % per_slot) * kGateUpRows;
  const int expert = slot < p.k ? p.topk_idx[slot] : p.E;
  for (int i = tid; i < p.d; i += kDecThreads) s_x[i] = __uint_as_float((uint32_t)p.x[i] << 16);
  __syncthreads();
  const int KB = p.d / kGroup;
  for (int g = tid; g < KB; g += kDecThreads) {
    float s = 0.f;
    for (int c = 0; c < kGroup; ++c) s += s_x[g * kGroup + c];
    s_gs[g] = s;
  }
  __syncthreads();
  const int m = f0 / kBlockRows, r = f0 % kBlockRows + lane;
  const uint8_t* gu = p.packed + (size_t)expert * p.expert_stride + (size_t)m * KB * 2 * kBlockBytes;
  float g_acc = 0.f, u_acc = 0.f;
  for (int kb0 = warp; kb0 < KB; kb0 += 4 * (kDecThreads / 32)) {
    uint4 gc[4][2], uc[4][2];
    uint32_t gsb[4], usb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // issue every load of up to four blocks before any math
      const int kb = kb0 + i * (kDecThreads / 32);
      if (kb < KB) {
        const uint8_t* blk = gu + (size_t)kb * 2 * kBlockBytes;
        gc[i][0] = ld_stream(blk + r * 32);
        gc[i][1] = ld_stream(blk + r * 32 + 16);
        gsb[i] = ld_stream32(blk + kCodeBytes + r * 4);
        uc[i][0] = ld_stream(blk + kBlockBytes + r * 32);
        uc[i][1] = ld_stream(blk + kBlockBytes + r * 32 + 16);
        usb[i] = ld_stream32(blk + kBlockBytes + kCodeBytes + r * 4);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int kb = kb0 + i * (kDecThreads / 32);
      if (kb < KB) {
        g_acc += dot_block(gc[i][0], gc[i][1], gsb[i], s_x + kb * kGroup, s_gs[kb]);
        u_acc += dot_block(uc[i][0], uc[i][1], usb[i], s_x + kb * kGroup, s_gs[kb]);
      }
    }
  }
  s_part[(warp * 2 + 0) * 32 + lane] = g_acc;
  s_part[(warp * 2 + 1) * 32 + lane] = u_acc;
  __syncthreads();
  if (warp == 0) {
    float g = 0.f, u = 0.f;
    for (int w = 0; w < kDecThreads / 32; ++w) {
      g += s_part[(w * 2 + 0) * 32 + lane];
      u += s_part[(w * 2 + 1) * 32 + lane];
    }
    p.hbuf[(size_t)slot * p.inter + f0 + lane] = g / (1.f + expf(-g)) * u;
  }
}

// Dynamic shared memory: h [(k+1) * I], group sums [(k+1) * I/64], partials [(k+1)*I/64][16].
__global__ void __launch_bounds__(kDecThreads) decode_down_kernel(const DecodeParams p) {
  extern __shared__ float dsm[];
  const int KBI = p.inter / kGroup;
  const int slots = p.k + 1, items = slots * KBI;
  float* s_h = dsm;
  float* s_hs = s_h + slots * p.inter;
  float* s_part = s_hs + items;
  const int tid = threadIdx.x;
  for (int i = tid; i < slots * p.inter; i += kDecThreads) s_h[i] = __ldcg(p.hbuf + i);
  __syncthreads();
  for (int it = tid; it < items; it += kDecThreads) {
    float s = 0.f;
    for (int c = 0; c < kGroup; ++c) s += s_h[it * kGroup + c];
    s_hs[it] = s;
  }
  __syncthreads();
  const int i0 = blockIdx.x * kDownRows;
  const int m = i0 / kBlockRows, rin = i0 % kBlockRows;
  const int row = tid % kDownRows, lane_item = tid / kDownRows;
  const int n_il = kDecThreads / kDownRows;
  for (int it0 = lane_item; it0 < items; it0 += 4 * n_il) {
    uint4 c[4][2];
    uint32_t sb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int it = it0 + i * n_il;
      if (it < items) {
        const int slot = it / KBI, kb = it % KBI;
        const int expert = slot < p.k ? __ldcg(p.topk_idx + slot) : p.E;
        const uint8_t* blk = p.packed + (size_t)expert * p.expert_stride + p.gu_bytes +
                             ((size_t)m * KBI + kb) * kBlockBytes;
        c[i][0] = ld_stream(blk + (rin + row) * 32);
        c[i][1] = ld_stream(blk + (rin + row) * 32 + 16);
        sb[i] = ld_stream32(blk + kCodeBytes + (rin + row) * 4);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int it = it0 + i * n_il;
      if (it < items) s_part[it * kDownRows + row] = dot_block(c[i][0], c[i][1], sb[i], s_h + it * kGroup, s_hs[it]);
    }
  }
  __syncthreads();
  if (tid < kDownRows) {
    float y = 0.f;
    for (int slot = 0; slot < slots; ++slot) {
      float ys = 0.f;
      for (int kb = 0; kb < KBI; ++kb) ys += s_part[(slot * KBI + kb) * kDownRows + tid];
      const float w = slot < p.k ? __ldcg(p.topk_w + slot) : 1.f;
      y += w * ys;
    }
    p.y[i0 + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

}  // namespace

size_t decode_smem_gateup(int d) { return ((size_t)d + d / kGroup + 2 * kDecThreads) * sizeof(float); }
size_t decode_smem_down(int k, int inter) {
  const size_t items = (size_t)(k + 1) * (inter / kGroup);
  return ((size_t)(k + 1) * inter + items + items * kDownRows) * sizeof(float);
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s, void* const* events) {
  const size_t sm_gu = decode_smem_gateup(p.d), sm_dn = decode_smem_down(p.k, p.inter);
  static cudaError_t a1 = cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  static cudaError_t a2 = cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (a1 != cudaSuccess) return a1;
  if (a2 != cudaSuccess) return a2;
  cudaError_t err = record_event(events, 0, s);
  if (err != cudaSuccess) return err;
  decode_router_kernel<<<(p.E + 7) / 8, kDecThreads, 0, s>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess || (err = record_event(events, 1, s)) != cudaSuccess) return err;
  decode_gateup_kernel<<<(p.k + 1) * (p.inter / kGateUpRows), kDecThreads, sm_gu, s>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess || (err = record_event(events, 2, s)) != cudaSuccess) return err;
  decode_down_kernel<<<p.d / kDownRows, kDecThreads, sm_dn, s>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return record_event(events, 3, s);
}

}  // namespace moe
