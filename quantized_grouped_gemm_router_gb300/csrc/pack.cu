// Canonical MLX-style Q4 matrices -> the library's packed expert layout (a pure re-layout:
// codes are permuted inside each 32-bit word and scales/biases are interleaved; no value
// changes). Layout: see PackedLayout in moe_internal.h.
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {
namespace {

struct PackArgs {
  moe_q4_view gate, up, down, sh_gate, sh_up, sh_down;
  uint8_t* packed;
  size_t expert_stride, gu_bytes;
  int d, inter, n_experts;
};

// Canonical word: column j (0..7) in bits 4j. Packed word: column j in nibble slot j/2 + 4*(j%2).
__device__ __forceinline__ uint32_t permute_nibbles(uint32_t w) {
  uint32_t out = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t code = (w >> (4 * j)) & 0xFu;
    out |= code << (4 * ((j >> 1) + 4 * (j & 1)));
  }
  return out;
}

// One CTA of 128 threads packs one 128 x 64 block; thread r packs row r of the block.
__global__ void __launch_bounds__(128) pack_kernel(const PackArgs a) {
  const int e = blockIdx.y;                    // 0..E-1 routed, E shared
  const int kb_d = a.d / kGroup, kb_i = a.inter / kGroup;
  const int n_gu = (a.inter / kBlockRows) * kb_d;  // (m, kb) pairs of the gate|up region
  int blk = blockIdx.x;
  const bool shared = (e == a.n_experts);
  const size_t lead = shared ? 0 : (size_t)e;
  const int r = threadIdx.x;
  uint8_t* eb = a.packed + (size_t)e * a.expert_stride;
  uint32_t words[8];
  uint32_t sb;
  if (blk < 2 * n_gu) {  // gate or up block (m, kb)
    const int pair = blk >> 1, which = blk & 1;      // 0 gate, 1 up
    const int m = pair / kb_d, kb = pair % kb_d;
    const moe_q4_view src = which ? (shared ? a.sh_up : a.up) : (shared ? a.sh_gate : a.gate);
    const size_t row = (size_t)m * kBlockRows + r;
    const uint32_t* q = src.q + (lead * a.inter + row) * (a.d / 8) + (size_t)kb * 8;
    const size_t g = (lead * a.inter + row) * kb_d + kb;
    for (int w = 0; w < 8; ++w) words[w] = permute_nibbles(q[w]);
    sb = (uint32_t)src.scale[g] | ((uint32_t)src.bias[g] << 16);
    const int qtr = r / kQuarterRows, rr = r % kQuarterRows;
    uint8_t* dst = eb + gu_offset(m, qtr, kb, kb_d) + which * kGUMat;
    for (int w = 0; w < 8; ++w)
      reinterpret_cast<uint32_t*>(dst + (w >> 2) * kQuarterRows * 16 + rr * 16)[w & 3] = words[w];
    *reinterpret_cast<uint32_t*>(dst + 2 * kQuarterRows * 16 + rr * 4) = sb;
  } else {               // down block (mm, kbd)
    blk -= 2 * n_gu;
    const int DM = a.d / kBlockRows;
    const int mm = blk / kb_i, kbd = blk % kb_i;
    const moe_q4_view src = shared ? a.sh_down : a.down;
    const size_t row = (size_t)mm * kBlockRows + r;
    const uint32_t* q = src.q + (lead * a.d + row) * (a.inter / 8) + (size_t)kbd * 8;
    const size_t g = (lead * a.d + row) * kb_i + kbd;
    for (int w = 0; w < 8; ++w) words[w] = permute_nibbles(q[w]);
    sb = (uint32_t)src.scale[g] | ((uint32_t)src.bias[g] << 16);
    uint8_t* dn = eb + a.gu_bytes;
    for (int w = 0; w < 8; ++w)
      reinterpret_cast<uint32_t*>(dn + dn_code_offset(kbd, w >> 2, mm, DM) + r * 16)[w & 3] = words[w];
    *reinterpret_cast<uint32_t*>(dn + dn_sb_offset(kbd, mm, DM, kb_i) + r * 4) = sb;
  }
}

}  // namespace

cudaError_t launch_pack(const moe_dims& d, const moe_q4_view* v, uint8_t* packed, cudaStream_t s) {
  const PackedLayout L = packed_layout(d);
  PackArgs a;
  a.gate = v[0];
  a.up = v[1];
  a.down = v[2];
  a.sh_gate = v[3];
  a.sh_up = v[4];
  a.sh_down = v[5];
  a.packed = packed;
  a.expert_stride = L.expert_stride;
  a.gu_bytes = L.gu_bytes;
  a.d = d.d;
  a.inter = d.inter;
  a.n_experts = d.n_experts;
  const int blocks = 2 * (d.inter / kBlockRows) * (d.d / kGroup) + (d.d / kBlockRows) * (d.inter / kGroup);
  pack_kernel<<<dim3(blocks, d.n_experts + 1), 128, 0, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Materialised dequantization (ablation): each thread expands one packed word (8 codes) of one
// expert into 8 fp16 weights, scale * q + bias rounded once to fp16 exactly as the in-tile path
// does; experts no token selected are skipped.
// ------------------------------------------------------------------------------------------
size_t dense_gu_bytes(const moe_dims& d) { return (size_t)(d.n_experts + 1) * 2 * d.inter * d.d * 2; }
size_t dense_dn_bytes(const moe_dims& d) { return (size_t)(d.n_experts + 1) * d.d * d.inter * 2; }

namespace {

__device__ __forceinline__ uint4 expand8(uint32_t w, uint32_t sbw) {
  const __half s = __float2half_rn(__uint_as_float(sbw << 16));
  const __half b = __float2half_rn(__uint_as_float(sbw & 0xFFFF0000u));
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // columns 2j, 2j+1 sit in nibble slots j and j + 4
    const __half lo = __hfma(__ushort2half_rn((w >> (4 * j)) & 0xF), s, b);
    const __half hi = __hfma(__ushort2half_rn((w >> (4 * j + 16)) & 0xF), s, b);
    o[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256) dense_dequant_kernel(const uint8_t* __restrict__ packed, const int32_t* counts,
                                                            uint16_t* dense_gu, uint16_t* dense_dn, int d, int E,
                                                            int inter, size_t expert_stride, size_t gu_bytes) {
  const int e = blockIdx.y;
  if (e < E && __ldcg(counts + e) == 0) return;  // unselected expert (the shared expert, e == E, always runs)
  const int KB = d / kGroup, DM = d / kBlockRows, KBI = inter / kGroup;
  const uint8_t* eb = packed + (size_t)e * expert_stride;
  const size_t gu_words = (size_t)2 * inter * d / 8, dn_words = (size_t)d * inter / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < gu_words + dn_words;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < gu_words) {  // dense gate/up row r of item h, columns 8 cw .. 8 cw + 7
      const int cw = (int)(i % (d / 8));
      const size_t rowi = i / (d / 8);
      const int r = (int)(rowi % 128), h = (int)(rowi / 128);
      const int f = 64 * h + (r & 63), mat = r >> 6;
      const int m = f / kBlockRows, q = (f % kBlockRows) / kQuarterRows, rr = f % kQuarterRows;
      const int c = 8 * cw, kb = c / kGroup, half = (c % kGroup) / 32, w = (c % 32) / 8;
      const uint8_t* blk = eb + gu_offset(m, q, kb, KB) + mat * kGUMat;
      const uint32_t word = *reinterpret_cast<const uint32_t*>(blk + half * kQuarterRows * 16 + rr * 16 + 4 * w);
      const uint32_t sbw = *reinterpret_cast<const uint32_t*>(blk + 2 * kQuarterRows * 16 + rr * 4);
      reinterpret_cast<uint4*>(dense_gu + (size_t)e * 2 * inter * d)[i] = expand8(word, sbw);
    } else {  // dense down row o, columns 8 cw .. 8 cw + 7 of I
      const size_t j = i - gu_words;
      const int cw = (int)(j % (inter / 8)), o = (int)(j / (inter / 8));
      const int mm = o / kBlockRows, r = o % kBlockRows;
      const int c = 8 * cw, kbd = c / kGroup, hd = (c % kGroup) / 32, w = (c % 32) / 8;
      const uint8_t* dn = eb + gu_bytes;
      const uint32_t word = *reinterpret_cast<const uint32_t*>(dn + dn_code_offset(kbd, hd, mm, DM) + r * 16 + 4 * w);
      const uint32_t sbw = *reinterpret_cast<const uint32_t*>(dn + dn_sb_offset(kbd, mm, DM, KBI) + r * 4);
      reinterpret_cast<uint4*>(dense_dn + (size_t)e * d * inter)[j] = expand8(word, sbw);
    }
  }
}

}  // namespace

cudaError_t launch_dense_dequant(const moe_dims& d, const uint8_t* packed, const int32_t* counts, uint16_t* dense_gu,
                                 uint16_t* dense_dn, cudaStream_t s) {
  const PackedLayout P = packed_layout(d);
  const size_t words = (size_t)3 * d.inter * d.d / 8;
  const int blocks = (int)std::min<size_t>((words + 255) / 256, 4096);
  dense_dequant_kernel<<<dim3(blocks, d.n_experts + 1), 256, 0, s>>>(packed, counts, dense_gu, dense_dn, d.d,
                                                                      d.n_experts, d.inter, P.expert_stride, P.gu_bytes);
  return cudaGetLastError();
}

}  // namespace moe
