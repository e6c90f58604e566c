// Batch-1 decode path: Q4 GEMVs that stream only the selected experts' packed weights.
//
// Page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model":
// section "Prefill and decode are different problems" (decode at batch 1 is a matrix-vector
// product bound by memory bandwidth; "minimize bytes moved per token"), section "Decode:
// minimize bytes per token" (the input projections fused with the gate activation, the output
// projection with the routing scores and the shared expert; dependency-aware overlap of
// kernels), section "What didn't work" (the GEMV runs near the weight-read rate).
//
// Three launches chained with programmatic dependent launch (PDL): each kernel lets its
// successor start at once, and does everything that does not depend on its predecessor's
// results (loading static weights) before waiting for it. (Folding the router or the combine into
// the expert kernel behind an in-kernel release/acquire handshake was measured slower: each
// handshake costs more than the hand-off between two dependent launches.)
//   decode_router_kernel  (decode_common.cuh) two experts per CTA: logit = W_r[e] . x (+ b_e);
//                         the router weight slice is loaded before the wait
//   decode_expert_kernel  one CTA per (selected or shared expert, 32 intermediate rows): routed
//                         CTAs select the top k from the logits themselves (all 512 threads: a
//                         threshold from the maxima of 16-thread groups, then exact ranks of the
//                         few experts above it; ties to the lower index); each CTA bulk-copies its
//                         gate/up rows to shared memory as soon as the expert is known (the shared
//                         expert's CTAs before routing is known); gate/up GEMV + SwiGLU, scaled by
//                         the routing weight, written as the CTA's h record
//   decode_down_kernel    one CTA per 16 output rows: started once the router is complete, it
//                         selects the experts itself and copies its 16 down rows of every slot
//                         before waiting for the expert kernel; then every (slot, 64-column group)
//                         unit against the h records, summed in a fixed order -> bf16 y (the
//                         combine needs no partial rows)
// The GEMV inner products run on the tensor cores (mma.sync m16n8k16, fp16 in, fp32
// accumulate): the packed nibble pairs of a row map directly onto the MMA fragment layout, so
// the weights cost about one ALU operation per two values instead of an fp32 FMA each, which on
// GB300 would otherwise take as long as streaming the weights. The order of the reduction index
// inside an MMA is free as long as A and B agree: lane (g, tig) takes the four column pairs of
// its own code word tig of each row (and B the matching pairs of the vector), so a warp reads
// a tile's codes as contiguous 128-byte lines, with no lanes reading the same word. The GEMV
// vector occupies one column of B (x for gate/up; the SwiGLU output as an fp16 leading part and
// remainder in two columns for down), and each 64-column group's scale and bias are applied to
// the fp32 accumulator: sum (s*q + b) v = s * sum(q v) + b * sum(v). The codes enter the MMA as
// (base + q) with base 1024 or 64 depending on the column (one byte permute and four LOP3s per
// eight codes), and the bases are removed with the group's sums of x (gate/up) or of h (down)
// over the columns of each base; the fp32 accumulation keeps sum(q v) to about 1e-5 relative,
// far below the rounding of the fp16 operands.
// An fp16 operand range check on x and on h reports MOE_ERR_OUT_OF_RANGE; a bounded wait that
// gives up reports MOE_ERR_DEVICE_TIMEOUT, skips the CTA's arithmetic and stores (its outputs are
// then undefined) and lets the CTA's copies land before it exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "topk.cuh"


namespace moe {
namespace {

// Shared memory of the expert kernel (offsets in bytes, each 16-aligned).
struct XSmem {
  int gu, dn, x16, xsum, red, h, topk, misc, bars, total;
};

// Block-wide top-k scratch: the 16-lane groups' largest keys, the threshold, per-warp candidate
// counts, the candidate keys, the selected keys and weights.
struct TopkSmem {
  unsigned long long gmax[kXThreads / 16];
  unsigned long long tau;
  int wcnt[kXWarps];
  unsigned long long sel[kMaxTopK];
  float w[kMaxTopK];
  unsigned long long cand[kMaxExperts];
};

__host__ __device__ inline XSmem x_smem(int d) {
  const int KB = d / kGroup, DM = d / kBlockRows;
  XSmem L;
  L.gu = 0;                                           // KB entries of gate/up rows
  L.dn = L.gu + KB * kGUStage;                        // read-only probe: DM code halves, DM scale runs
  L.x16 = up16(L.dn + DM * kDnStage);                 // x as fp16 pairs
  L.xsum = up16(L.x16 + d * 2);                       // per-64-group sums of x, two column classes
  L.red = up16(L.xsum + KB * 8);                      // [warp][gate/up][32 rows] partial dots
  L.topk = up16(L.red + kXWarps * 2 * kDecPartRows * 4);
  L.misc = up16(L.topk + (int)sizeof(TopkSmem));      // abort flag
  L.bars = up16(L.misc + 16);
  L.total = L.bars + (kXMaxGUChunks + 1) * 8;         // gate/up pieces, down
  return L;
}

// Top k (k <= 16) of the E <= 1024 router logits, by all kXThreads threads of the block, with
// the same selection as warp_topk_softmax (largest logit first, equal logits to the lower
// index). Every expert has the unique key (orderable logit << 32) | ~index. Thread t reads the
// logits t and t + 512 (coalesced); the largest keys of the 32 groups of 16 consecutive threads
// belong to different experts, so the k-th largest key overall is at least tau, the k-th largest
// of those group maxima (once k groups hold experts; tau = 0 otherwise). Only the experts with a
// key >= tau (about k + 2 for Gaussian logits; all of them when the logits tie) are gathered,
// without atomics (per-warp counts and a prefix over the warps), and ranked by counting the
// larger candidate keys. Leaves the selected keys in s->sel[0..k) in slot order. Returns true on
// every thread if a logit was NaN or infinite (the selection is then meaningless but stays within
// [0, E)). Contains barriers: the whole block calls it.
__device__ bool block_select_topk(const float* logits, int E, int k, TopkSmem* s) {
  static_assert(kXWarps == 16 && kXThreads * 2 == kMaxExperts, "two experts per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = kMaxExperts / kXThreads;
  unsigned long long u[kPer];
  bool bad = false;
  unsigned long long best = 0ull;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid + kXThreads * i;
    u[i] = 0ull;  // below every real key
    if (e < E) {
      const float v = __ldcg(logits + e);
      bad |= !isfinite(v);
      u[i] = ((unsigned long long)max(orderable_f32(v), 1u) << 32) | (uint32_t)~(uint32_t)e;
    }
    best = u[i] > best ? u[i] : best;
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {  // the largest key of these 16 lanes
    const unsigned long long b = __shfl_xor_sync(0xFFFFFFFFu, best, o);
    best = b > best ? b : best;
  }
  if ((lane & 15) == 0) s->gmax[tid >> 4] = best;
  __syncthreads();
  if (warp == 0) {  // tau: the k-th largest group maximum (0 if fewer than k groups hold experts)
    const unsigned long long v = s->gmax[lane];
    int r = 0;
#pragma unroll 8
    for (int j = 0; j < kXThreads / 16; ++j) r += s->gmax[j] > v ? 1 : 0;
    const unsigned nz = __ballot_sync(0xFFFFFFFFu, v != 0ull);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, v != 0ull && r == k - 1);
    const unsigned long long tv = __shfl_sync(0xFFFFFFFFu, v, hit ? __ffs(hit) - 1 : 0);
    if (lane == 0) s->tau = (k <= __popc(nz) && hit) ? tv : 0ull;
  }
  __syncthreads();
  const unsigned long long tau = s->tau;
  unsigned bal[kPer];
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    bal[i] = __ballot_sync(0xFFFFFFFFu, u[i] != 0ull && u[i] >= tau);
    cnt += __popc(bal[i]);
  }
  if (lane == 0) s->wcnt[warp] = cnt;
  __syncthreads();
  int base = 0, n = 0;
#pragma unroll
  for (int w = 0; w < kXWarps; ++w) {
    const int c = s->wcnt[w];
    base += w < warp ? c : 0;
    n += c;
  }
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    if ((bal[i] >> lane) & 1u) s->cand[base + __popc(bal[i] & lt)] = u[i];
    base += __popc(bal[i]);
  }
  __syncthreads();
  for (int c = tid; c < n; c += kXThreads) {
    const unsigned long long K = s->cand[c];
    int rank = 0;
#pragma unroll 4
    for (int j = 0; j < n; ++j) rank += s->cand[j] > K ? 1 : 0;
    if (rank < k) s->sel[rank] = K;
  }
  return __syncthreads_or(bad) != 0;
}

// Softmax restricted to the selected experts (slot 0 holds the largest logit), by one warp, in
// the same arithmetic as warp_topk_softmax. Lane j < k returns slot j's expert and weight.
__device__ __forceinline__ void warp_selected_softmax(const TopkSmem* s, int E, int k, int* e_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  const unsigned long long K = lane < k ? s->sel[lane] : s->sel[0];
  const float my_v = from_orderable_f32((uint32_t)(K >> 32));
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const float ex = lane < k ? expf(my_v - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  *e_out = min(max((int)~(uint32_t)K, 0), E - 1);
  *w_out = ex / sum;
}

// kMode 0: the decode expert kernel. Diagnostics (the ablations the pages use to locate the
// decode bound, section "What didn't work"): kMode 1 deletes the GEMV arithmetic (same copies,
// waits and stores; the h records are zeros, and the down kernel's kMode 1 writes y = 0); kMode 2
// is a read-only probe of the layer's weight reads (each CTA copies its gate/up rows and the down
// slice of its part, for expert `slot` (< k) or the shared expert, waits for them and exits;
// launched alone).
template <int kMode>
__global__ void __launch_bounds__(kXThreads, 1) decode_expert_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t xs[];
  const XSmem L = x_smem(p.d);
  const int KB = p.d / kGroup, DM = p.d / kBlockRows, KBI = p.inter / kGroup;
  const int parts = p.inter / kDecPartRows;
  const int slot = blockIdx.x / parts, part = blockIdx.x % parts;
  const bool shared = (slot == p.k);
  const int m = part / (kBlockRows / kDecPartRows);          // gate/up row block
  const int kbd = part / 2, hd = part % 2;                    // down: column group of I and its half
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bars = smem_u32(xs + L.bars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(xs + L.misc);
  TopkSmem* tk = reinterpret_cast<TopkSmem*>(xs + L.topk);
  const int NGU = min(kXMaxGUChunks, KB);  // barriers 0..NGU-1: gate/up pieces; NGU: down
  if (tid == 0) {
    for (int i = 0; i <= NGU; ++i) mbar_init(bars + 8u * i, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // Lanes of warp 0 issue this CTA's copies, one each (a thread's TMA copies to different barriers
  // go out one after another, ~0.25 us apart): lanes 0..NGU-1 the contiguous run of its 32 gate
  // and up rows for every column block (KB * 2304 bytes, in NGU pieces). The read-only probe also
  // copies what the down kernel reads for this CTA's part, on the down barrier: lane NGU its
  // 32-column half of every down row block (DM * 2048 bytes of codes), lane NGU + 1 the matching
  // scale/bias rows.
  auto issue = [&](int expert) {
    const uint8_t* eb = p.packed + (size_t)expert * p.expert_stride;
    if (lane < NGU) {
      const int kb0 = lane * KB / NGU, kb1 = (lane + 1) * KB / NGU;
      const uint32_t bytes = (uint32_t)(kb1 - kb0) * kGUStage;
      mbar_arrive_expect_tx(bars + 8u * lane, bytes);
      tma_bulk_g2s(smem_u32(xs + L.gu + kb0 * kGUStage),
                   eb + gu_offset(m, part % (kBlockRows / kDecPartRows), 0, KB) + (size_t)kb0 * kGUStage, bytes,
                   bars + 8u * lane);
    } else if (kMode == 2 && lane <= NGU + 1) {
      const bool codes = lane == NGU;
      const uint8_t* src = eb + p.gu_bytes + (codes ? dn_code_offset(kbd, hd, 0, DM) : dn_sb_offset(kbd, 0, DM, KBI));
      if (codes) mbar_arrive_expect_tx(bars + 8u * NGU, (uint32_t)(DM * (kHalfBytes + kSBBytes)));
      tma_bulk_g2s(smem_u32(xs + L.dn + (codes ? 0 : DM * kHalfBytes)), src, codes ? DM * kHalfBytes : DM * kSBBytes,
                   bars + 8u * NGU);
    }
  };

  if constexpr (kMode == 2) {
    if (warp == 0) issue(shared ? p.E : min(slot, p.E - 1));
    bool ok = true;
    for (int i = 0; i <= NGU && ok; ++i) ok = mbar_wait(bars + 8u * i, 0, s_abort);
    __syncthreads();
    if (tid == 0 && *s_abort) {
      for (int i = 0; i <= NGU; ++i) mbar_drain(bars + 8u * i, 0);
      set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
    }
    return;
  }
  if (shared && warp == 0) issue(p.E);  // static weights: before waiting on the router
  pdl_wait();
  // The down kernel may start once every CTA of this kernel is past its wait: the router's logits,
  // which it reads before its own wait, are complete by then.
  pdl_launch_dependents();

  // x (one 8-value chunk per thread of warps 2..15) is loaded before the selection so both loads
  // overlap.
  static_assert(kDecodeMaxD / 8 <= kXThreads - 64, "warps 2..15 hold one 8-value chunk of x each");
  const int nch = p.d / 8, cx = tid - 64;
  const uint4 xv = cx >= 0 && cx < nch ? __ldcg(reinterpret_cast<const uint4*>(p.x) + cx) : make_uint4(0u, 0u, 0u, 0u);
  // Routed blocks select the top k themselves from the router's logits (every block gets the same,
  // deterministic answer); then warp 0 issues this block's copies at once while warp 1 computes the
  // routing weights (block 0 also publishes the routing) and the other warps stage x. The branch
  // is uniform over the block.
  if (!shared || blockIdx.x == 0) {
    const bool bad = block_select_topk(p.logits, p.E, p.k, tk);
    if (warp == 0 && !shared) issue((int)~(uint32_t)tk->sel[slot]);
    if (warp == 1) {
      int my_e;
      float my_w;
      warp_selected_softmax(tk, p.E, p.k, &my_e, &my_w);
      if (lane < p.k) tk->w[lane] = my_w;
      if (blockIdx.x == 0) {
        if (lane < p.k) {
          p.topk_idx[lane] = my_e;
          p.topk_w[lane] = my_w;
        }
        if (bad && lane == 0) set_device_status(p.hdr, MOE_ERR_NONFINITE);
      }
    }
  }
  if (warp >= 2) {
    // x as fp16 pairs, and per 64-column group the sums of x over the columns whose codes enter
    // the MMA with base 1024 (columns 0,1,4,5 of every 8) and base 64 (columns 2,3,6,7); x must lie
    // in the fp16 operand range (block 0 reports it once per call).
    uint32_t* x2w = reinterpret_cast<uint32_t*>(xs + L.x16);
    float* xsw = reinterpret_cast<float*>(xs + L.xsum);
    const uint32_t in[4] = {xv.x, xv.y, xv.z, xv.w};
    float sa = 0.f, sb = 0.f;
    bool over = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = bf16lo(in[j]), hi = bf16hi(in[j]);
      over |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
      if (j == 0 || j == 2) sa += lo + hi; else sb += lo + hi;
      const __half2 h2 = __floats2half2_rn(lo, hi);
      if (cx < nch) x2w[4 * cx + j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      sa += __shfl_xor_sync(0xFFFFFFFFu, sa, o);
      sb += __shfl_xor_sync(0xFFFFFFFFu, sb, o);
    }
    if (cx < nch && (cx & 7) == 0) {
      xsw[2 * (cx >> 3)] = sa;
      xsw[2 * (cx >> 3) + 1] = sb;
    }
    if (blockIdx.x == 0 && __any_sync(0xFFFFFFFFu, over && cx < nch) && lane == 0)
      set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }
  __syncthreads();
  const float wslot = shared ? 1.f : tk->w[slot];
  const uint32_t* x2 = reinterpret_cast<const uint32_t*>(xs + L.x16);
  const float* xsum = reinterpret_cast<const float*>(xs + L.xsum);

  // ---- gate/up: warp w takes K blocks w, w+16, ...; 2 row tiles of 16 per matrix
  const int g = lane >> 2, tig = lane & 3;
  float acc[2][2][2] = {};  // [gate/up][row tile][row g, row g+8] (meaningful on tig == 0)
  bool gu_ok = true;
  for (int kb = warp; kb < KB; kb += kXWarps) {
    int chunk = 0;
    while (kb >= (chunk + 1) * KB / NGU) ++chunk;
    if (!(gu_ok = mbar_wait(bars + 8u * chunk, 0, s_abort))) break;
    if constexpr (kMode == 1) continue;  // arithmetic deleted
    const uint8_t* st = xs + L.gu + kb * kGUStage;
    // B: x for the columns of this lane's two code words (tig and tig + 4): 4 consecutive pairs each
    uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
    if (g == 0) {
      xa = *reinterpret_cast<const uint4*>(x2 + kb * (kGroup / 2) + 4 * tig);
      xb = *reinterpret_cast<const uint4*>(x2 + kb * (kGroup / 2) + 16 + 4 * tig);
    }
    const float sa = xsum[2 * kb], sb = xsum[2 * kb + 1];
#pragma unroll
    for (int mat = 0; mat < 2; ++mat) {
      const uint8_t* ms = st + mat * (kGUStage / 2);
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        const int R0 = rt * 16 + g, R1 = R0 + 8;
        // lane (g, tig) reads word tig (columns 8 tig..8 tig+7) and word tig + 4 of rows R0 and R1;
        // a warp's read of one word per row is one contiguous 128-byte line
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
        // d = sum (base + q) x over the group: s*q + b weights give
        // s*d + (b - 1024 s) * (sum of x over base-1024 columns) + (b - 64 s) * (the others)
        const uint32_t sb0 = *reinterpret_cast<const uint32_t*>(ms + 2 * kDecPartRows * 16 + R0 * 4);
        const uint32_t sb1 = *reinterpret_cast<const uint32_t*>(ms + 2 * kDecPartRows * 16 + R1 * 4);
        acc[mat][rt][0] += bf16lo(sb0) * d[0] + (bf16hi(sb0) - 1024.f * bf16lo(sb0)) * sa +
                           (bf16hi(sb0) - 64.f * bf16lo(sb0)) * sb;
        acc[mat][rt][1] += bf16lo(sb1) * d[2] + (bf16hi(sb1) - 1024.f * bf16lo(sb1)) * sa +
                           (bf16hi(sb1) - 64.f * bf16lo(sb1)) * sb;
      }
    }
  }
  float* red = reinterpret_cast<float*>(xs + L.red);
  if (tig == 0) {
#pragma unroll
    for (int mat = 0; mat < 2; ++mat)
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        red[(warp * 2 + mat) * kDecPartRows + rt * 16 + g] = acc[mat][rt][0];
        red[(warp * 2 + mat) * kDecPartRows + rt * 16 + g + 8] = acc[mat][rt][1];
      }
  }
  __syncthreads();
  if (warp == 0 && !*s_abort) {
    // SwiGLU of this CTA's 32 rows, scaled by the routing weight, into its h record: the fp16
    // leading parts, the fp16 remainders, and the sums of h over the base-1024 columns (0,1,4,5 of
    // every 8) and the base-64 columns of the down projection's codes
    float gs = 0.f, us = 0.f;
    for (int w = 0; w < kXWarps; ++w) {
      gs += red[(w * 2 + 0) * kDecPartRows + lane];
      us += red[(w * 2 + 1) * kDecPartRows + lane];
    }
    const float h = gs / (1.f + expf(-gs)) * us * wslot;
    const __half hi = __float2half_rn(h);
    uint8_t* rec = p.hrec + (size_t)blockIdx.x * kHRecBytes;  // blockIdx.x = slot * parts + part
    reinterpret_cast<__half*>(rec)[lane] = hi;
    reinterpret_cast<__half*>(rec + 2 * kDecPartRows)[lane] = __float2half_rn(h - __half2float(hi));
    const bool base1024 = (lane & 2) == 0;
    float ta = base1024 ? h : 0.f, tb = base1024 ? 0.f : h;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ta += __shfl_xor_sync(0xFFFFFFFFu, ta, o);
      tb += __shfl_xor_sync(0xFFFFFFFFu, tb, o);
    }
    if (lane == 0) *reinterpret_cast<float2*>(rec + 4 * kDecPartRows) = make_float2(ta, tb);
    if (__any_sync(0xFFFFFFFFu, !(fabsf(h) <= 65504.f)) && lane == 0) set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }
  if (tid == 0 && *s_abort) {  // outputs are undefined; let this CTA's copies land before exiting
    for (int i = 0; i < NGU; ++i) mbar_drain(bars + 8u * i, 0);
    set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
  }
}

// y[r0 .. r0 + 16) for r0 = 16 blockIdx.x: the sum over every (expert slot j <= k, 32-column part
// pp) of W_down_e[rows, 32 pp .. 32 pp + 32) . h_{j,pp} (slot k: the shared expert; the routing
// weights are already in h). The kernel starts once every expert-kernel CTA is past its own wait,
// so the router's logits are complete: it selects the experts itself (the same deterministic
// selection as the expert kernel) and, before waiting for the expert kernel, warp 0 issues two
// tensor copies per slot for the first 16 parts (the CTA's 16 code rows of each part and their
// scale/bias rows), which stream from HBM while the expert kernel runs. After the wait every
// thread copies the parts' h records to shared memory. Each unit (slot, 64-column group: two
// parts sharing their scale/bias rows) is four MMAs and one epilogue; every warp takes its units
// in a fixed order, and the 16 warp sums are then added in warp order, so the result does not
// depend on timing. kMode 1 (arithmetic deleted) makes the same copies and writes y = 0.
template <int kMode>
__global__ void __launch_bounds__(kDThreads, 2) decode_down_kernel(const DecodeParams p,
                                                                   const __grid_constant__ DecodeMaps maps) {
  static_assert(kDThreads == kXThreads, "the block-wide top-k runs on 512 threads");
  extern __shared__ uint8_t ds_raw[];
  uint8_t* ds = ds_raw + ((128u - (smem_u32(ds_raw) & 127u)) & 127u);  // tensor copies land 128-aligned
  __shared__ float s_red[kDWarps][kDRows];
  __shared__ TopkSmem s_tk;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int r0 = blockIdx.x * kDRows, mm = r0 / kBlockRows, ro = r0 % kBlockRows;
  const int parts = p.inter / kDecPartRows, k1 = p.k + 1;
  uint8_t* s_codes = ds;                               // [slot][16 parts][16 rows][16 B]
  uint8_t* s_sb = ds + k1 * kDCodeSlot;                // [slot][8 K blocks][16 rows][4 B]
  uint8_t* s_h = s_sb + k1 * kDSBSlot;                 // [slot][16 parts] h records
  const uint32_t bar = smem_u32(&s_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < 2) prefetch_tmap(lane ? &maps.sb : &maps.codes);
  __syncthreads();
  block_select_topk(p.logits, p.E, p.k, &s_tk);  // non-finite logits are reported by the expert kernel
  // lane j < k of warp 0: slot j's expert; lane k: the shared expert
  const int e = lane < p.k ? min(max((int)~(uint32_t)s_tk.sel[lane], 0), p.E - 1) : p.E;
  const int pieces = min(parts, kDWarps);
  auto issue = [&](int pc) {  // warp 0: every slot's codes and scale/bias rows for parts pc .. pc + 15
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(k1 * (pieces * kDPieceBytes + pieces / 2 * kDSBBytes)));
      __syncwarp();
      if (lane < k1) {
        tma_load_4d(smem_u32(s_codes + lane * kDCodeSlot), &maps.codes, 2 * ro, mm, pc, e, bar);
        tma_load_4d(smem_u32(s_sb + lane * kDSBSlot), &maps.sb, ro / 2, mm, pc / 2, e, bar);
      }
    }
  };
  issue(0);
  pdl_launch_dependents();
  pdl_wait();
  float acc0 = 0.f, acc1 = 0.f;  // rows g and g + 8 (meaningful on tig == 0)
  uint32_t phase = 0;
  for (int pc = 0; pc < parts; pc += kDWarps, phase ^= 1u) {
    if (pc > 0) issue(pc);
    // the h records of parts pc .. pc + 15, every slot (k1 * 16 records of 9 16-byte words)
    const int n16 = k1 * kDWarps * (kHRecBytes / 16);
    for (int q = tid; q < n16; q += kDThreads) {
      const int r = q / (kHRecBytes / 16), pq = pc + r % kDWarps;
      if (pq < parts)
        cp_async_16(smem_u32(s_h + (size_t)q * 16),
                    p.hrec + (size_t)((r / kDWarps) * parts + pq) * kHRecBytes + (q % (kHRecBytes / 16)) * 16);
    }
    cp_async_wait_all();
    mbar_wait(bar, phase, &s_abort);
    __syncthreads();
    if (s_abort) break;  // uniform: read after the barrier
    if (kMode == 0) {
      // units (slot j, column group kb) of this chunk: both 32-column halves of the group share its
      // scale/bias rows, so one unit is four chained MMAs (K = 64) and one epilogue. Warp w takes
      // column group w % npk and the slots w / npk, w / npk + 16 / npk, ... in order (warps past
      // npk * (16 / npk) idle). The loop is bound by shared-memory and issue throughput, not by
      // latency, so it is not unrolled.
      const int npk = min(parts - pc, kDWarps) / 2, jstep = kDWarps / npk, kb = warp % npk;
      const uint8_t* cw = s_codes + 2 * kb * kDPieceBytes + g * 16 + 4 * tig;
      const uint8_t* sw = s_sb + kb * kDSBBytes + g * 4;
      const uint8_t* rw = s_h + 2 * kb * kHRecBytes;
      const int ho = 2 * kDecPartRows * (g & 1) + 16 * tig;
#pragma unroll 1
      for (int j = warp < npk * jstep ? warp / npk : k1; j < k1; j += jstep) {
        // A: lane (g, tig) takes code word tig of rows g and g + 8 of both halves; B: column 0
        // the leading part of h, column 1 its remainder, for that word's 8 columns (columns 2..7
        // of B and of the product are not used)
        const uint8_t* c = cw + j * kDCodeSlot;
        const uint8_t* r = rw + j * (kDWarps * kHRecBytes);
        const uint32_t c0a = *reinterpret_cast<const uint32_t*>(c);
        const uint32_t c1a = *reinterpret_cast<const uint32_t*>(c + 8 * 16);
        const uint32_t c0b = *reinterpret_cast<const uint32_t*>(c + kDPieceBytes);
        const uint32_t c1b = *reinterpret_cast<const uint32_t*>(c + kDPieceBytes + 8 * 16);
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(sw + j * kDSBSlot);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(sw + j * kDSBSlot + 8 * 4);
        uint4 hva = make_uint4(0u, 0u, 0u, 0u), hvb = hva;
        if (g < 2) {
          hva = *reinterpret_cast<const uint4*>(r + ho);
          hvb = *reinterpret_cast<const uint4*>(r + kHRecBytes + ho);
        }
        const float2 ha = *reinterpret_cast<const float2*>(r + 4 * kDecPartRows);
        const float2 hb = *reinterpret_cast<const float2*>(r + kHRecBytes + 4 * kDecPartRows);
        uint32_t qa0[4], qa1[4], qb0[4], qb1[4];
        q_pairs(c0a, qa0);
        q_pairs(c1a, qa1);
        q_pairs(c0b, qb0);
        q_pairs(c1b, qb1);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816_acc(d, qa0[0], qa1[0], qa0[1], qa1[1], hva.x, hva.y);
        mma16816_acc(d, qa0[2], qa1[2], qa0[3], qa1[3], hva.z, hva.w);
        mma16816_acc(d, qb0[0], qb1[0], qb0[1], qb1[1], hvb.x, hvb.y);
        mma16816_acc(d, qb0[2], qb1[2], qb0[3], qb1[3], hvb.z, hvb.w);
        // d = sum (base + q) h over the 64 columns: s*q + b weights give
        // s * (d - 1024 sa - 64 sb) + b * (sa + sb), with sa, sb the sums of h over the base-1024
        // and base-64 columns
        const float sa = ha.x + hb.x, sb = ha.y + hb.y, h0 = sa + sb, h1 = 1024.f * sa + 64.f * sb;
        acc0 = fmaf(bf16lo(w0), (d[0] + d[1]) - h1, fmaf(bf16hi(w0), h0, acc0));
        acc1 = fmaf(bf16lo(w1), (d[2] + d[3]) - h1, fmaf(bf16hi(w1), h0, acc1));
      }
    }
    __syncthreads();  // before the next parts' copies overwrite shared memory
  }
  if (s_abort) {  // y is undefined; let this CTA's copies land before exiting
    if (tid == 0) {
      mbar_drain(bar, phase);
      set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
    }
    return;
  }
  if (tig == 0) {
    s_red[warp][g] = acc0;
    s_red[warp][g + 8] = acc1;
  }
  __syncthreads();
  if (tid < kDRows) {
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) y += s_red[w][tid];
    p.y[r0 + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, const DecodeMaps& maps, cudaStream_t s, void* const* events,
                          int mode) {
  const moe_dims dims = {p.d, p.E, p.k, p.inter, p.inter, kGroup};
  const int n_parts = decode_parts(dims);
  const int smem = x_smem(p.d).total;
  const size_t down_smem = (size_t)(p.k + 1) * kDSlotBytes + 128;
  // The router and down kernels ask for the largest shared-memory carveout, so that the SMs they
  // run on can take an expert-kernel CTA (~120 KB of shared memory) as soon as PDL lets it start,
  // instead of waiting for the SM to drain and change its L1/shared split.
  static cudaError_t attr = [] {
    cudaError_t e = cudaSuccess;
    for (auto kernel : {decode_expert_kernel<0>, decode_expert_kernel<1>, decode_expert_kernel<2>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, x_smem(kDecodeMaxD).total);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_router_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    for (auto kernel : {decode_down_kernel<0>, decode_down_kernel<1>}) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (kMaxTopK + 1) * kDSlotBytes + 128);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    }
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  if (mode == kDecodeDiagReadOnly) {  // the layer's weight copies alone, no chain
    decode_expert_kernel<2><<<n_parts, kXThreads, (size_t)smem, s>>>(p);
    return cudaGetLastError();
  }
  cudaError_t err = record_event(events, 0, s);
  if (err != cudaSuccess) return err;
  if ((err = launch_pdl(decode_router_kernel, (p.E + 1) / 2, kRThreads, 0, 1, s, p)) != cudaSuccess) return err;
  if ((err = record_event(events, 1, s)) != cudaSuccess) return err;
  err = mode == kDecodeDiagNoMath ? launch_pdl(decode_expert_kernel<1>, n_parts, kXThreads, (size_t)smem, 1, s, p)
                                  : launch_pdl(decode_expert_kernel<0>, n_parts, kXThreads, (size_t)smem, 1, s, p);
  if (err != cudaSuccess) return err;
  if ((err = record_event(events, 2, s)) != cudaSuccess) return err;
  err = mode == kDecodeDiagNoMath
            ? launch_pdl(decode_down_kernel<1>, p.d / kDRows, kDThreads, down_smem, 1, s, p, maps)
            : launch_pdl(decode_down_kernel<0>, p.d / kDRows, kDThreads, down_smem, 1, s, p, maps);
  if (err != cudaSuccess) return err;
  return record_event(events, 3, s);
}

}  // namespace moe
