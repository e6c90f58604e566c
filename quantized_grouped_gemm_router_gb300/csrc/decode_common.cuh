// Device building blocks shared by the batch-1 decode (decode.cu) and the small-batch decode
// (decode_batch.cu): launch shapes, shared-memory layout constants, the mma.sync wrappers, the
// nibble-pair conversion, bounded barrier drains and the router GEMV kernel (both paths start with
// it). Included by one translation unit each; everything here has internal linkage.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRThreads = 256;         // router: two experts per CTA, 128 threads each
constexpr int kRMaxChunks = kDecodeMaxD / 8 / 128;
constexpr int kXThreads = 512;         // expert kernel: 16 warps to hide MMA and smem latency
constexpr int kXWarps = kXThreads / 32;
constexpr int kDThreads = 512;         // down kernel: 16 warps, one 32-column part each
constexpr int kDWarps = kDThreads / 32;
constexpr int kDRows = 16;             // output rows per down-kernel CTA (the MMA's M)
constexpr int kDPieceBytes = kDRows * 16;             // codes of one (part, 16 rows) piece
constexpr int kDSBBytes = kDRows * 4;                 // scale/bias of 16 rows for one K block
constexpr int kDCodeSlot = kDWarps * kDPieceBytes;    // one slot's codes for 16 parts
constexpr int kDSBSlot = kDWarps / 2 * kDSBBytes;     // one slot's scale/bias for 8 K blocks
constexpr int kDSlotBytes = kDCodeSlot + kDSBSlot + kDWarps * kHRecBytes;
constexpr int kXMaxGUChunks = 4;       // gate/up run split into up to 4 copies (own barriers, own lanes)
constexpr int kGUStage = 2 * (2 * kDecPartRows * 16 + kDecPartRows * 4);  // gate + up slice of one kb
constexpr int kDnStage = kHalfBytes + kBlockRows * 4;                     // down half-block + sb

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
// 16-byte asynchronous copy global -> shared through L2 only (data an earlier kernel of the chain
// wrote), completed by cp_async_wait_all.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// D = A(16x16, fp16, row-major) * B(16x8, fp16, column-major) + 0, fp32 result.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(d[0]), "f"(d[1]), "f"(d[2]), "f"(d[3]));
}

// The same product accumulated into d, without volatile: the compiler may schedule it freely.
__device__ __forceinline__ void mma16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kRThreads) decode_router_kernel(const DecodeParams p) {
  __shared__ float s_part[kMaxDecodeBatch][kRThreads / 32];
  const int half = threadIdx.x >> 7, t = threadIdx.x & 127, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 2 + half;
  const int nch = p.d >> 3;  // 8-element chunks per row
  uint4 w[kRMaxChunks];
#pragma unroll
  for (int i = 0; i < kRMaxChunks; ++i) {  // static weights: load before waiting on the predecessor
    const int c = t + 128 * i;
    w[i] = (e < p.E && c < nch) ? ld_stream(p.router_w + (size_t)e * p.d + 8 * c) : make_uint4(0, 0, 0, 0);
  }
  pdl_launch_dependents();
  pdl_wait();
  for (int tok = 0; tok < p.T; ++tok) {  // the same weights against every token of the call
    const uint4* xt = reinterpret_cast<const uint4*>(p.x + (size_t)tok * p.d);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kRMaxChunks; ++i) {
      const int c = t + 128 * i;
      if (e < p.E && c < nch) {
        const uint4 xv = __ldcg(xt + c);
        const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc = fmaf(bf16lo(xa[j]), bf16lo(wa[j]), acc);
          acc = fmaf(bf16hi(xa[j]), bf16hi(wa[j]), acc);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) s_part[tok][warp] = acc;
  }
  __syncthreads();
  if (t < p.T && e < p.E) {  // thread t of each half writes token t's logit of its expert
    const float* sp = s_part[t] + 4 * half;
    p.logits[(size_t)t * p.E + e] = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + (p.router_bias ? p.router_bias[e] : 0.f);
  }
}

__host__ __device__ inline int up16(int v) { return (v + 15) & ~15; }

// The four nibble pairs of a packed word (columns 2i, 2i+1 of its eight are nibbles i and i+4) as
// fp16 pairs (base + q0, base + q1), with one byte permute and four LOP3s: nibbles 0/4 sit in
// mantissa bits [3:0] of 1024.0 (ulp 1), nibbles 1/5 in bits [7:4] of 64.0 (ulp 1/16), and the
// byte swap brings nibbles 2/6 and 3/7 to the same places. Columns 0,1 and 4,5 of the word get
// base 1024, columns 2,3 and 6,7 base 64; the caller removes the bases with the matching sums of
// the vector after the product.
__device__ __forceinline__ void q_pairs(uint32_t w, uint32_t (&t)[4]) {
  const uint32_t sw = __byte_perm(w, 0, 0x2301);
  t[0] = (w & 0x000F000Fu) | 0x64006400u;
  t[1] = (w & 0x00F000F0u) | 0x54005400u;
  t[2] = (sw & 0x000F000Fu) | 0x64006400u;
  t[3] = (sw & 0x00F000F0u) | 0x54005400u;
}

// Bounded wait that ignores the abort flag: used after an abort, so that no bulk copy of this CTA
// is still landing in its shared memory when the CTA exits.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitCycles) {
  }
}

}  // namespace
}  // namespace moe
