// Canonical MLX-style Q4 matrices -> the library's packed expert layout (a pure re-layout:
// codes are permuted inside each 32-bit word and scales/biases are interleaved; no value
// changes). Layout: see PackedLayout in moe_internal.h.
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

}  // namespace moe
