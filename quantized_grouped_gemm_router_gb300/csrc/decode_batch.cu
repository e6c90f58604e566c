// Small-batch decode (2..8 tokens at once, e.g. checking a few draft tokens): page "Perplexity's
// Lily beats MLX-LM on MacBook M5 because it only runs one model", section "What didn't work" (2 to
// 5 draft rows route to different experts). The union of the tokens' selected experts is streamed
// once, each distinct expert's blocks serving every token that chose it, the tokens filling the
// columns of the MMAs' B operand:
//   decode_router_kernel        logits of the T tokens (decode_common.cuh)
//   decode_batch_select_kernel  top-k of every token, the distinct experts in ascending order
//   decode_batch_expert_kernel  one block per (distinct or shared expert, 32 intermediate rows):
//                               gate/up GEMV + SwiGLU for every token, then the block's 32 columns
//                               of the down projection -> a partial output row per token that
//                               chose the expert
//   decode_reduce_kernel        y of every token = the sum of its partial rows in a fixed order
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kYThreads = 512;  // reduce: 16 output rows x 32 groups of partial rows
constexpr int kYRows = 16;

// ------------------------------------------------------------------------------------------
// Small-batch decode (2..8 tokens, e.g. checking a few draft tokens at once): the tokens route
// to different experts (page, section "What didn't work": 2 to 5 draft rows touch different
// experts), so the union of their selected experts is streamed once, each distinct expert's
// CTAs serving every token that chose it; the tokens fill the columns of the MMAs' B operand.
// ------------------------------------------------------------------------------------------

// Selection of every token (warp t = token t), then the distinct selected experts in ascending
// order: dexp[0..n_distinct).
__global__ void __launch_bounds__(kMaxDecodeBatch * 32) decode_batch_select_kernel(const DecodeParams p,
                                                                                    int32_t* dexp,
                                                                                    int32_t* n_distinct) {
  __shared__ uint32_t bitmap[kMaxExperts / 32];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kMaxExperts / 32) bitmap[threadIdx.x] = 0u;
  __syncthreads();
  if (warp < p.T) {
    int e;
    float w;
    const bool bad = warp_topk_softmax(p.logits + (size_t)warp * p.E, p.E, p.k, &e, &w);
    if (lane < p.k) {
      p.topk_idx[warp * p.k + lane] = e;
      p.topk_w[warp * p.k + lane] = w;
      atomicOr(&bitmap[e >> 5], 1u << (e & 31));
    }
    if (bad && lane == 0) set_device_status(p.hdr, MOE_ERR_NONFINITE);
  }
  __syncthreads();
  if (warp == 0) {  // lane l owns experts 32 l .. 32 l + 31
    uint32_t bits = bitmap[lane];
    int before = __popc(bits);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, before, o);
      if (lane >= o) before += v;
    }
    const int total = __shfl_sync(0xFFFFFFFFu, before, 31);
    before -= __popc(bits);
    while (bits) {
      const int b = __ffs(bits) - 1;
      dexp[before++] = 32 * lane + b;
      bits &= bits - 1;
    }
    if (lane == 0) *n_distinct = total;
  }
}

// Shared memory of the batch expert kernel.
// Shared memory of the batch expert kernel, under half an SM's so that two blocks fit: the
// gate/up stage area is reused, once the gate/up loop has consumed it, for the cross-warp
// reduction of the gate/up dots and for the down slice (copied in only then).
struct BSmem {
  int gu, red, dn, x16, xsum, h, hsum, tok, misc, bars, total;
};
__host__ __device__ inline BSmem b_smem(int d) {
  const int KB = d / kGroup, DM = d / kBlockRows;
  const int red_bytes = kXWarps * 2 * kDecPartRows * kMaxDecodeBatch * 4;          // [warp][mat][row][token]
  const int area = max(KB * kGUStage, red_bytes + DM * kDnStage);
  BSmem L;
  L.gu = 0;
  L.red = 0;                                                                  // after the gate/up loop
  L.dn = red_bytes;                                                           // after the gate/up loop
  L.x16 = up16(area);                                                         // [token][d] fp16
  L.xsum = up16(L.x16 + kMaxDecodeBatch * d * 2);                             // [token][KB][2]
  L.h = up16(L.xsum + kMaxDecodeBatch * KB * 8);                              // [plane][token][32] fp16
  L.hsum = up16(L.h + 2 * kMaxDecodeBatch * kDecPartRows * 2);                // [token][2]
  L.tok = up16(L.hsum + kMaxDecodeBatch * 8);                                 // weight[8], slot[8]
  L.misc = up16(L.tok + kMaxDecodeBatch * 8);                                 // abort flag, expert
  L.bars = up16(L.misc + 16);
  L.total = L.bars + (kXMaxGUChunks + 1) * 8;
  return L;
}

// One CTA per (distinct selected expert, or the shared expert) x 32 intermediate rows, for every
// token of the call at once. Slots beyond the call's distinct experts exit at once. Token t's
// contribution from its slot j goes to partial row [t][j][part] (the shared expert to [t][k]).
__global__ void __launch_bounds__(kXThreads, 2) decode_batch_expert_kernel(const DecodeParams p,
                                                                           const int32_t* dexp,
                                                                           const int32_t* n_distinct) {
  extern __shared__ __align__(128) uint8_t xs[];
  const BSmem L = b_smem(p.d);
  const int KB = p.d / kGroup, DM = p.d / kBlockRows, KBI = p.inter / kGroup;
  const int parts = p.inter / kDecPartRows, T = p.T, k = p.k;
  const int slot = blockIdx.x / parts, part = blockIdx.x % parts;
  const bool shared = slot == T * k;
  const int m = part / (kBlockRows / kDecPartRows);
  const int kbd = part / 2, hd = part % 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bars = smem_u32(xs + L.bars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(xs + L.misc);
  int* s_expert = reinterpret_cast<int*>(xs + L.misc + 4);
  float* s_w = reinterpret_cast<float*>(xs + L.tok);
  int* s_slot = reinterpret_cast<int*>(xs + L.tok + kMaxDecodeBatch * 4);
  const int NGU = min(kXMaxGUChunks, KB);
  if (tid == 0) {
    for (int i = 0; i <= NGU; ++i) mbar_init(bars + 8u * i, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int expert) {  // the gate/up pieces of the batch-1 expert kernel
    const uint8_t* eb = p.packed + (size_t)expert * p.expert_stride;
    if (lane < NGU) {
      const uint8_t* gu = eb + gu_offset(m, part % (kBlockRows / kDecPartRows), 0, KB);
      const int c = lane, kb0 = c * KB / NGU, kb1 = (c + 1) * KB / NGU;
      const uint32_t bytes = (uint32_t)(kb1 - kb0) * kGUStage;
      mbar_arrive_expect_tx(bars + 8u * c, bytes);
      tma_bulk_g2s(smem_u32(xs + L.gu + kb0 * kGUStage), gu + (size_t)kb0 * kGUStage, bytes, bars + 8u * c);
    }
  };
  auto issue_down = [&](int expert) {  // lane 0 of warp 0: the down slice, into the consumed gate/up area
    const uint8_t* dn = p.packed + (size_t)expert * p.expert_stride + p.gu_bytes;
    mbar_arrive_expect_tx(bars + 8u * NGU, (uint32_t)(DM * (kHalfBytes + kSBBytes)));
    tma_bulk_g2s(smem_u32(xs + L.dn), dn + dn_code_offset(kbd, hd, 0, DM), DM * kHalfBytes, bars + 8u * NGU);
    tma_bulk_g2s(smem_u32(xs + L.dn + DM * kHalfBytes), dn + dn_sb_offset(kbd, 0, DM, KBI), DM * kSBBytes,
                 bars + 8u * NGU);
  };
  if (shared && warp == 0) issue(p.E);  // static weights: before waiting on the selection
  pdl_launch_dependents();
  pdl_wait();
  // Warp 0 finds this block's expert and issues its copies at once, while warps 1..15 stage x (the
  // copies' issue holds warp 0 up for a while).
  if (warp == 0) {
    int e = p.E;
    if (lane == 0 && !shared) {  // both loads in flight at once (dexp holds T*k entries: in bounds)
      const int nd = __ldcg(n_distinct), ex = __ldcg(dexp + slot);
      e = slot < nd ? ex : -1;
    }
    e = __shfl_sync(0xFFFFFFFFu, e, 0);
    if (lane == 0) *s_expert = e;
    if (lane < kMaxDecodeBatch) {  // not chosen: weight 0, slot -1; the shared expert: every token
      s_w[lane] = shared && lane < T ? 1.f : 0.f;
      s_slot[lane] = shared && lane < T ? k : -1;
    }
    if (!shared && e >= 0) issue(e);
  } else {
    // x of every token as fp16 pairs, and per token and 64-column group the sums of x over the
    // base-1024 columns (0,1,4,5 of every 8) and the base-64 columns (2,3,6,7); chunk i of the
    // T x d/8 chunks goes to thread 32 + (i mod 480), every thread's loads first so they overlap
    constexpr int kStagers = kXThreads - 32;
    constexpr int kXIter = (kMaxDecodeBatch * (kBatchMaxD / 8) + kStagers - 1) / kStagers;
    uint32_t* x2w = reinterpret_cast<uint32_t*>(xs + L.x16);
    float* xsw = reinterpret_cast<float*>(xs + L.xsum);
    const int nch = p.d / 8, st = tid - 32;
    bool over = false;
    uint4 xv[kXIter];
#pragma unroll
    for (int it = 0; it < kXIter; ++it) {
      const int i = it * kStagers + st, t = i / nch, c = i % nch;
      xv[it] = t < T ? __ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.d) + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < kXIter; ++it) {
      const int i = it * kStagers + st, t = i / nch, c = i % nch;
      float sa = 0.f, sb = 0.f;
      uint32_t o[4] = {0u, 0u, 0u, 0u};
      if (t < T) {
        const uint32_t in[4] = {xv[it].x, xv[it].y, xv[it].z, xv[it].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = bf16lo(in[j]), hi = bf16hi(in[j]);
          over |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
          if (j == 0 || j == 2) sa += lo + hi; else sb += lo + hi;
          const __half2 h2 = __floats2half2_rn(lo, hi);
          o[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      if (t < kMaxDecodeBatch) *reinterpret_cast<uint4*>(x2w + (size_t)t * (p.d / 2) + 4 * c) = make_uint4(o[0], o[1], o[2], o[3]);
#pragma unroll
      for (int q = 1; q < 8; q <<= 1) {  // 8 consecutive chunks (one 64-column group) per 8 lanes
        sa += __shfl_xor_sync(0xFFFFFFFFu, sa, q);
        sb += __shfl_xor_sync(0xFFFFFFFFu, sb, q);
      }
      if (t < kMaxDecodeBatch && (c & 7) == 0) {
        xsw[(t * KB + (c >> 3)) * 2] = sa;
        xsw[(t * KB + (c >> 3)) * 2 + 1] = sb;
      }
    }
    if (slot == 0 && part == 0 && __any_sync(0xFFFFFFFFu, over) && lane == 0)
      set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }
  __syncthreads();
  const int expert = *s_expert;
  if (expert < 0) return;  // fewer distinct experts than slots (uniform; nothing was issued)
  if (!shared && tid < T * k) {  // the T*k selections, one per thread (each token picks an expert once)
    const int e = __ldcg(p.topk_idx + tid);
    const float w = __ldcg(p.topk_w + tid);
    if (e == expert) {  // read after the barrier that follows the gate/up loop
      s_w[tid / k] = w;
      s_slot[tid / k] = tid % k;
    }
  }
  const uint32_t* x2 = reinterpret_cast<const uint32_t*>(xs + L.x16);
  const float* xsum = reinterpret_cast<const float*>(xs + L.xsum);

  // ---- gate/up: warp w takes K blocks w, w+16, ...; the tokens are the 8 columns of B
  const int g = lane >> 2, tig = lane & 3;
  float acc[2][2][4] = {};  // [gate/up][row tile][(row g, tokens 2tig, 2tig+1), (row g+8, ...)]
  bool gu_ok = true;
  for (int kb = warp; kb < KB; kb += kXWarps) {
    int chunk = 0;
    while (kb >= (chunk + 1) * KB / NGU) ++chunk;
    if (!(gu_ok = mbar_wait(bars + 8u * chunk, 0, s_abort))) break;
    const uint8_t* st = xs + L.gu + kb * kGUStage;
    // B: token g's x for the columns of this lane's two code words (tig and tig + 4)
    const uint4 xa = *reinterpret_cast<const uint4*>(x2 + (size_t)g * (p.d / 2) + kb * (kGroup / 2) + 4 * tig);
    const uint4 xb = *reinterpret_cast<const uint4*>(x2 + (size_t)g * (p.d / 2) + kb * (kGroup / 2) + 16 + 4 * tig);
    const float sa0 = xsum[((2 * tig) * KB + kb) * 2], sb0 = xsum[((2 * tig) * KB + kb) * 2 + 1];
    const float sa1 = xsum[((2 * tig + 1) * KB + kb) * 2], sb1 = xsum[((2 * tig + 1) * KB + kb) * 2 + 1];
#pragma unroll
    for (int mat = 0; mat < 2; ++mat) {
      const uint8_t* ms = st + mat * (kGUStage / 2);
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        const int R0 = rt * 16 + g, R1 = R0 + 8;
        uint32_t a0[4], a1[4], b0[4], b1[4];
        q_pairs(*reinterpret_cast<const uint32_t*>(ms + R0 * 16 + 4 * tig), a0);
        q_pairs(*reinterpret_cast<const uint32_t*>(ms + R1 * 16 + 4 * tig), a1);
        q_pairs(*reinterpret_cast<const uint32_t*>(ms + kDecPartRows * 16 + R0 * 16 + 4 * tig), b0);
        q_pairs(*reinterpret_cast<const uint32_t*>(ms + kDecPartRows * 16 + R1 * 16 + 4 * tig), b1);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(d, a0[0], a1[0], a0[1], a1[1], xa.x, xa.y);
        mma16816(d, a0[2], a1[2], a0[3], a1[3], xa.z, xa.w);
        mma16816(d, b0[0], b1[0], b0[1], b1[1], xb.x, xb.y);
        mma16816(d, b0[2], b1[2], b0[3], b1[3], xb.z, xb.w);
        const uint32_t sbw0 = *reinterpret_cast<const uint32_t*>(ms + 2 * kDecPartRows * 16 + R0 * 4);
        const uint32_t sbw1 = *reinterpret_cast<const uint32_t*>(ms + 2 * kDecPartRows * 16 + R1 * 4);
        const float s0 = bf16lo(sbw0), c0a = bf16hi(sbw0) - 1024.f * s0, c0b = bf16hi(sbw0) - 64.f * s0;
        const float s1 = bf16lo(sbw1), c1a = bf16hi(sbw1) - 1024.f * s1, c1b = bf16hi(sbw1) - 64.f * s1;
        acc[mat][rt][0] += s0 * d[0] + c0a * sa0 + c0b * sb0;
        acc[mat][rt][1] += s0 * d[1] + c0a * sa1 + c0b * sb1;
        acc[mat][rt][2] += s1 * d[2] + c1a * sa0 + c1b * sb0;
        acc[mat][rt][3] += s1 * d[3] + c1a * sa1 + c1b * sb1;
      }
    }
  }
  gu_ok = __all_sync(0xFFFFFFFFu, gu_ok);
  // every warp is done with the gate/up stages: the area now takes the reduction and the down slice
  __syncthreads();
  const bool down_issued = tid == 0 && !*s_abort;  // (meaningful on thread 0, which drains)
  if (down_issued) issue_down(expert);
  float* red = reinterpret_cast<float*>(xs + L.red);  // [warp][mat][row][token]
#pragma unroll
  for (int mat = 0; mat < 2; ++mat)
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = rt * 16 + g + 8 * (q >> 1), tok = 2 * tig + (q & 1);
        red[((warp * 2 + mat) * kDecPartRows + row) * kMaxDecodeBatch + tok] = acc[mat][rt][q];
      }
  __syncthreads();
  __half* hh = reinterpret_cast<__half*>(xs + L.h);            // [token][32] leading part
  __half* hl = hh + kMaxDecodeBatch * kDecPartRows;            // [token][32] remainder
  float* hsum = reinterpret_cast<float*>(xs + L.hsum);         // [token][2]
  if (warp < kMaxDecodeBatch) {  // warp t: SwiGLU of token t's 32 rows, scaled by its routing weight
    const int t = warp;
    float gs = 0.f, us = 0.f;
    for (int w = 0; w < kXWarps; ++w) {
      gs += red[((w * 2 + 0) * kDecPartRows + lane) * kMaxDecodeBatch + t];
      us += red[((w * 2 + 1) * kDecPartRows + lane) * kMaxDecodeBatch + t];
    }
    const float wt = s_w[t];
    const float h = wt != 0.f ? gs / (1.f + expf(-gs)) * us * wt : 0.f;
    const __half hi = __float2half_rn(h);
    hh[t * kDecPartRows + lane] = hi;
    hl[t * kDecPartRows + lane] = __float2half_rn(h - __half2float(hi));
    const bool base1024 = (lane & 2) == 0;
    float ta = base1024 ? h : 0.f, tb = base1024 ? 0.f : h;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ta += __shfl_xor_sync(0xFFFFFFFFu, ta, o);
      tb += __shfl_xor_sync(0xFFFFFFFFu, tb, o);
    }
    if (lane == 0) {
      hsum[2 * t] = ta;
      hsum[2 * t + 1] = tb;
    }
    if (__any_sync(0xFFFFFFFFu, !(fabsf(h) <= 65504.f)) && lane == 0) set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }
  __syncthreads();

  // ---- down: this CTA's 32 columns of W_down against every output row, 4 tokens per MMA (the
  // leading part and remainder of token t's h in columns 2t, 2t + 1 of B)
  const bool down_ok = mbar_wait(bars + 8u * NGU, 0, s_abort);
  const bool ok = !*s_abort && down_ok && gu_ok;
  const int nsets = (T + 3) / 4;
  uint4 hbv[2];
#pragma unroll
  for (int set = 0; set < 2; ++set) {
    const int tok = 4 * set + (g >> 1);
    const __half* src = (g & 1) ? hl : hh;
    hbv[set] = *reinterpret_cast<const uint4*>(src + tok * kDecPartRows + 8 * tig);
  }
  constexpr int kMaxTilesPerWarp = kBatchMaxD / 16 / kXWarps;
  const int ntiles = DM * 8;  // 16-row tiles of the d output rows (warp w: tiles w, w + 16, ...)
  uint32_t c0[kMaxTilesPerWarp], c1[kMaxTilesPerWarp];
#pragma unroll
  for (int i = 0; i < kMaxTilesPerWarp; ++i) {
    if (ok && warp + i * kXWarps < ntiles) {
      const int tile = warp + i * kXWarps, mm = tile >> 3, R0 = (tile & 7) * 16 + g;
      const uint8_t* ds = xs + L.dn + mm * kHalfBytes;
      c0[i] = *reinterpret_cast<const uint32_t*>(ds + R0 * 16 + 4 * tig);
      c1[i] = *reinterpret_cast<const uint32_t*>(ds + (R0 + 8) * 16 + 4 * tig);
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxTilesPerWarp; ++i) {
    if (ok && warp + i * kXWarps < ntiles) {
      const int tile = warp + i * kXWarps, mm = tile >> 3, R0 = (tile & 7) * 16 + g, R1 = R0 + 8;
      uint32_t q0[4], q1[4];
      q_pairs(c0[i], q0);
      q_pairs(c1[i], q1);
      const uint8_t* dsb = xs + L.dn + DM * kHalfBytes + mm * kSBBytes;
      const uint32_t sbw0 = *reinterpret_cast<const uint32_t*>(dsb + R0 * 4);
      const uint32_t sbw1 = *reinterpret_cast<const uint32_t*>(dsb + R1 * 4);
      const float s0 = bf16lo(sbw0), s1 = bf16lo(sbw1);
#pragma unroll
      for (int set = 0; set < 2; ++set) {
        if (set < nsets) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816(d, q0[0], q1[0], q0[1], q1[1], hbv[set].x, hbv[set].y);
          mma16816(d, q0[2], q1[2], q0[3], q1[3], hbv[set].z, hbv[set].w);
          const int tok = 4 * set + tig;  // columns 2 tig, 2 tig + 1: this token's two planes
          const int j = tok < T ? s_slot[tok] : -1;
          if (j >= 0) {
            const float ha = hsum[2 * tok], hb = hsum[2 * tok + 1];
            float* gout = p.partials + (((size_t)tok * (k + 1) + j) * parts + part) * p.d;
            gout[mm * kBlockRows + R0] = s0 * (d[0] + d[1]) + (bf16hi(sbw0) - 1024.f * s0) * ha + (bf16hi(sbw0) - 64.f * s0) * hb;
            gout[mm * kBlockRows + R1] = s1 * (d[2] + d[3]) + (bf16hi(sbw1) - 1024.f * s1) * ha + (bf16hi(sbw1) - 64.f * s1) * hb;
          }
        }
      }
    }
  }
  if (!down_ok && tid == 0) *s_abort = 1;
  __syncthreads();
  if (tid == 0 && *s_abort) {
    for (int i = 0; i < NGU; ++i) mbar_drain(bars + 8u * i, 0);
    if (down_issued) mbar_drain(bars + 8u * NGU, 0);
    set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
  }
}

// y[t][i] = the sum of partials[t][c][i] over c, rounded to bf16, for token t = blockIdx.y (c runs
// over the n_parts partial rows of one token: every (expert slot, 32-row part)). Thread (row r,
// group q) sums the rows c = q, q + 32, ... (loads of 16 consecutive floats per group); warp r
// then adds the 32 group sums of row r by a butterfly. The order is fixed, so the result does
// not depend on timing.
__global__ void __launch_bounds__(kYThreads) decode_reduce_kernel(const DecodeParams p, int n_parts) {
  constexpr int kGroups = kYThreads / kYRows;
  static_assert(kGroups == 32 && kYRows == kYThreads / 32, "one warp per output row for the butterfly");
  __shared__ float s[kYRows][kGroups + 1];
  pdl_launch_dependents();
  pdl_wait();
  const int r = threadIdx.x % kYRows, q = threadIdx.x / kYRows;
  const int row = blockIdx.x * kYRows + r;
  const float* part = p.partials + (size_t)blockIdx.y * n_parts * p.d;
  float acc = 0.f;
  for (int c0 = q; c0 < n_parts; c0 += 8 * kGroups) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + j * kGroups;
      v[j] = c < n_parts ? __ldcg(part + (size_t)c * p.d + row) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) acc += v[j];
  }
  s[r][q] = acc;
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float y = s[w][lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
  if (lane == 0) p.y[(size_t)blockIdx.y * p.d + blockIdx.x * kYRows + w] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
}

}  // namespace

cudaError_t launch_decode_batch(const DecodeParams& p, cudaStream_t s) {
  const moe_dims dims = {p.d, p.E, p.k, p.inter, p.inter, kGroup};
  const int parts = p.inter / kDecPartRows, n_parts = decode_parts(dims);
  const int smem = b_smem(p.d).total;
  static cudaError_t attr = [] {  // two blocks per SM: the largest shared-memory carveout
    cudaError_t e = cudaFuncSetAttribute(decode_batch_expert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         b_smem(kBatchMaxD).total);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_batch_expert_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  // the distinct-expert list lives in the routing part of the workspace: after topk_w
  int32_t* dexp = reinterpret_cast<int32_t*>(p.topk_w + (size_t)p.T * p.k);
  int32_t* n_distinct = dexp + p.T * p.k;
  cudaError_t err = launch_pdl(decode_router_kernel, (p.E + 1) / 2, kRThreads, 0, 1, s, p);
  if (err != cudaSuccess) return err;
  err = launch_pdl(decode_batch_select_kernel, 1, kMaxDecodeBatch * 32, 0, 1, s, p, dexp, n_distinct);
  if (err != cudaSuccess) return err;
  if ((err = launch_pdl(decode_batch_expert_kernel, (p.T * p.k + 1) * parts, kXThreads, (size_t)smem, 1, s, p,
                        (const int32_t*)dexp, (const int32_t*)n_distinct)) != cudaSuccess)
    return err;
  return launch_pdl(decode_reduce_kernel, dim3(p.d / kYRows, p.T), kYThreads, 0, 1, s, p, n_parts);
}

}  // namespace moe
