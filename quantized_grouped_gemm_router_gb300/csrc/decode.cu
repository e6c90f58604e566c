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
// results (loading static weights) before waiting for it.
//   decode_router_kernel  two experts per CTA: logit = W_r[e] . x (+ b_e); the router weight
//                         slice is loaded before the wait
//   decode_expert_kernel  one CTA per (selected or shared expert, 32 intermediate rows): routed
//                         CTAs select the top k from the logits themselves (all 512 threads: a
//                         threshold from the warp maxima, then exact ranks of the few experts
//                         above it; ties to the lower index); all of a CTA's gate/up rows and its
//                         32-column slice of the down projection are bulk-copied to shared memory
//                         as soon as the expert is known (the shared expert's CTAs before routing
//                         is known); gate/up + SwiGLU, scaled by the routing weight, then this
//                         slice's contribution to every output row (split-K over the intermediate
//                         dimension), written as the CTA's partial row
//   decode_reduce_kernel  y = sum of the partial rows in a fixed order -> bf16
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

#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"
#include "topk.cuh"


namespace moe {
namespace {

constexpr int kRThreads = 256;         // router: two experts per CTA, 128 threads each
constexpr int kRMaxChunks = kDecodeMaxD / 8 / 128;
constexpr int kXThreads = 512;         // expert kernel: 16 warps to hide MMA and smem latency
constexpr int kXWarps = kXThreads / 32;
constexpr int kYThreads = 512;         // reduce: 16 output rows x 32 groups of partial rows
constexpr int kYRows = 16;
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

__global__ void __launch_bounds__(kRThreads) decode_router_kernel(const DecodeParams p) {
  __shared__ float s_part[kRThreads / 32];
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
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kRMaxChunks; ++i) {
    const int c = t + 128 * i;
    if (e < p.E && c < nch) {
      const uint4 xv = __ldcg(reinterpret_cast<const uint4*>(p.x) + c);
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
  if (lane == 0) s_part[warp] = acc;
  __syncthreads();
  if (t == 0 && e < p.E) {
    const float* sp = s_part + 4 * half;
    p.logits[e] = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + (p.router_bias ? p.router_bias[e] : 0.f);
  }
}

// Shared memory of the expert kernel (offsets in bytes, each 16-aligned).
struct XSmem {
  int gu, dn, x16, xsum, red, h, topk, misc, bars, total;
};
__host__ __device__ inline int up16(int v) { return (v + 15) & ~15; }

// The routing of this call as warp 0 selected it: slot j's expert and weight.
struct SelSmem {
  int e[kMaxTopK];
  float w[kMaxTopK];
};

__host__ __device__ inline XSmem x_smem(int d) {
  const int KB = d / kGroup, DM = d / kBlockRows;
  XSmem L;
  L.gu = 0;                                           // KB entries of gate/up rows
  L.dn = L.gu + KB * kGUStage;                        // DM code halves, then DM scale runs
  L.x16 = up16(L.dn + DM * kDnStage);                 // x as fp16 pairs
  L.xsum = up16(L.x16 + d * 2);                       // per-64-group sums of x, two column classes
  L.red = up16(L.xsum + KB * 8);                      // [warp][gate/up][32 rows] partial dots
  L.h = up16(L.red + kXWarps * 2 * kDecPartRows * 4); // h leading part, remainder (fp16), two sums
  L.topk = up16(L.h + 2 * kDecPartRows * 2 + 16);
  L.misc = up16(L.topk + (int)sizeof(SelSmem));       // abort flag
  L.bars = up16(L.misc + 16);
  L.total = L.bars + (kXMaxGUChunks + 1) * 8;
  return L;
}

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

// kMode 0: the decode expert kernel. Diagnostics (the ablations the pages use to locate the
// decode bound, section "What didn't work"): kMode 1 deletes the GEMV arithmetic (same copies,
// waits and stores; the partial rows are zeros); kMode 2 is a read-only probe of the same access
// pattern (each CTA copies the pieces it would copy for expert `slot` (< k) or the shared expert,
// waits for them and exits; launched alone).
// kSlots: router logits per lane of the top-k warp (8 for up to 256 experts, 32 for up to 1024),
// a template parameter so the common shapes keep the register footprint of the 8-slot selection.
template <int kMode, int kSlots>
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
  SelSmem* sel = reinterpret_cast<SelSmem*>(xs + L.topk);
  const int NGU = min(kXMaxGUChunks, KB);  // barriers 0..NGU-1: gate/up pieces; NGU: down
  if (tid == 0) {
    for (int i = 0; i <= NGU; ++i) mbar_init(bars + 8u * i, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // Lanes 0..NGU of warp 0 issue this CTA's copies, one piece each (a thread's TMA copies to
  // different barriers are issued one after another, ~0.25 us apart): the contiguous run of its 32
  // gate and up rows for every column block (KB * 2304 bytes, in NGU pieces), then its 32-column
  // half of every down row block (DM * 2048 bytes of codes) and the matching scale/bias rows.
  auto issue = [&](int expert) {
    const uint8_t* eb = p.packed + (size_t)expert * p.expert_stride;
    if (lane < NGU) {
      const uint8_t* gu = eb + gu_offset(m, part % (kBlockRows / kDecPartRows), 0, KB);
      const int c = lane, kb0 = c * KB / NGU, kb1 = (c + 1) * KB / NGU;
      const uint32_t bytes = (uint32_t)(kb1 - kb0) * kGUStage;
      mbar_arrive_expect_tx(bars + 8u * c, bytes);
      tma_bulk_g2s(smem_u32(xs + L.gu + kb0 * kGUStage), gu + (size_t)kb0 * kGUStage, bytes, bars + 8u * c);
    } else if (lane == NGU) {
      const uint8_t* dn = eb + p.gu_bytes;
      mbar_arrive_expect_tx(bars + 8u * NGU, (uint32_t)(DM * (kHalfBytes + kSBBytes)));
      tma_bulk_g2s(smem_u32(xs + L.dn), dn + dn_code_offset(kbd, hd, 0, DM), DM * kHalfBytes, bars + 8u * NGU);
      tma_bulk_g2s(smem_u32(xs + L.dn + DM * kHalfBytes), dn + dn_sb_offset(kbd, 0, DM, KBI), DM * kSBBytes,
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
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    // Routed blocks select the top k themselves from the router's logits (every block gets the
    // same, deterministic answer), then issue this block's copies at once; block 0 also publishes
    // the routing.
    if (!shared || blockIdx.x == 0) {
      int rank, my_e;
      float my_w;
      const bool bad = warp_select_topk<kSlots>(p.logits, p.E, p.k, &rank, &my_e, &my_w);
      if (rank >= 0) {
        sel->e[rank] = my_e;
        sel->w[rank] = my_w;
      }
      __syncwarp();
      if (!shared) issue(sel->e[slot]);
      if (blockIdx.x == 0) {
        if (rank >= 0) {
          p.topk_idx[rank] = my_e;
          p.topk_w[rank] = my_w;
        }
        if (bad && lane == 0) set_device_status(p.hdr, MOE_ERR_NONFINITE);
      }
    }
  } else {
    // Meanwhile the other warps stage x as fp16 pairs, and per 64-column group the sums of x over
    // the columns whose codes enter the MMA with base 1024 (columns 0,1,4,5 of every 8) and base 64
    // (columns 2,3,6,7); x must lie in the fp16 operand range (block 0 reports it once per call).
    uint32_t* x2w = reinterpret_cast<uint32_t*>(xs + L.x16);
    float* xsw = reinterpret_cast<float*>(xs + L.xsum);
    const int nch = p.d / 8, t = tid - 32, nt = kXThreads - 32;
    bool over = false;
    for (int base = 0; base < nch; base += nt) {
      const int c = base + t;
      float sa = 0.f, sb = 0.f;
      if (c < nch) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p.x) + c);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = bf16lo(in[j]), hi = bf16hi(in[j]);
          over |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
          if (j == 0 || j == 2) sa += lo + hi; else sb += lo + hi;
          const __half2 h2 = __floats2half2_rn(lo, hi);
          x2w[4 * c + j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        sa += __shfl_xor_sync(0xFFFFFFFFu, sa, o);
        sb += __shfl_xor_sync(0xFFFFFFFFu, sb, o);
      }
      if (c < nch && (c & 7) == 0) {
        xsw[2 * (c >> 3)] = sa;
        xsw[2 * (c >> 3) + 1] = sb;
      }
    }
    if (blockIdx.x == 0 && __any_sync(0xFFFFFFFFu, over) && lane == 0) set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }
  __syncthreads();
  const float wslot = shared ? 1.f : sel->w[slot];
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
  gu_ok = __all_sync(0xFFFFFFFFu, gu_ok);
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
  __half* hh = reinterpret_cast<__half*>(xs + L.h);
  __half* hl = hh + kDecPartRows;
  float* hsum = reinterpret_cast<float*>(xs + L.h + 2 * kDecPartRows * 2);
  if (warp == 0) {  // SwiGLU of this CTA's 32 rows, scaled by the routing weight
    float gs = 0.f, us = 0.f;
    for (int w = 0; w < kXWarps; ++w) {
      gs += red[(w * 2 + 0) * kDecPartRows + lane];
      us += red[(w * 2 + 1) * kDecPartRows + lane];
    }
    const float h = gs / (1.f + expf(-gs)) * us * wslot;
    const __half hi = __float2half_rn(h);
    hh[lane] = hi;
    hl[lane] = __float2half_rn(h - __half2float(hi));
    // sums of h over the base-1024 columns (0,1,4,5 of every 8) and the base-64 columns
    const bool base1024 = (lane & 2) == 0;
    float ta = base1024 ? h : 0.f, tb = base1024 ? 0.f : h;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ta += __shfl_xor_sync(0xFFFFFFFFu, ta, o);
      tb += __shfl_xor_sync(0xFFFFFFFFu, tb, o);
    }
    if (lane == 0) {
      hsum[0] = ta;
      hsum[1] = tb;
    }
    if (__any_sync(0xFFFFFFFFu, !(fabsf(h) <= 65504.f)) && lane == 0) set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }
  __syncthreads();

  // ---- down: this CTA's 32 columns of W_down against every output row (split-K partial)
  const bool down_ok = mbar_wait(bars + 8u * NGU, 0, s_abort);
  const bool ok = !*s_abort && down_ok && gu_ok;  // after an abort nothing is computed or stored
  const uint32_t* hh2 = reinterpret_cast<const uint32_t*>(hh);
  const uint32_t* hl2 = reinterpret_cast<const uint32_t*>(hl);
  // B: column 0 the leading part of h, column 1 its remainder, for this lane's code word (columns
  // 8 tig..8 tig+7 of the CTA's 32): 4 consecutive pairs
  uint4 hb = make_uint4(0u, 0u, 0u, 0u);
  if (g < 2) hb = *reinterpret_cast<const uint4*>((g == 0 ? hh2 : hl2) + 4 * tig);
  const float ha = hsum[0], hb64 = hsum[1];
  // Each warp owns DM * 8 / 16 row tiles of 16; all of its code words are read first so the
  // shared-memory latency overlaps, then the MMAs run back to back. Row results go straight to
  // this CTA's partial row in global memory (16 consecutive floats per tile).
  float* gout = p.partials + (size_t)blockIdx.x * p.d;
  constexpr int kMaxTilesPerWarp = kDecodeMaxD / 16 / kXWarps;  // 12 for d = 3072
  const int ntw = DM * 8 / kXWarps;                              // tiles per warp (exact: d % 128 == 0)
  uint32_t c0[kMaxTilesPerWarp], c1[kMaxTilesPerWarp];
#pragma unroll
  for (int i = 0; i < kMaxTilesPerWarp; ++i) {
    if (ok && i < ntw) {  // lane (g, tig): word tig of rows R0 and R0 + 8 of the tile
      const int tile = warp + i * kXWarps, mm = tile >> 3, R0 = (tile & 7) * 16 + g;
      const uint8_t* ds = xs + L.dn + mm * kHalfBytes;
      c0[i] = *reinterpret_cast<const uint32_t*>(ds + R0 * 16 + 4 * tig);
      c1[i] = *reinterpret_cast<const uint32_t*>(ds + (R0 + 8) * 16 + 4 * tig);
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxTilesPerWarp; ++i) {
    if (ok && i < ntw) {
      const int tile = warp + i * kXWarps, mm = tile >> 3, R0 = (tile & 7) * 16 + g, R1 = R0 + 8;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (kMode == 0) {
        uint32_t q0[4], q1[4];
        q_pairs(c0[i], q0);
        q_pairs(c1[i], q1);
        mma16816(d, q0[0], q1[0], q0[1], q1[1], hb.x, hb.y);
        mma16816(d, q0[2], q1[2], q0[3], q1[3], hb.z, hb.w);
      }
      if (tig == 0) {
        const uint8_t* dsb = xs + L.dn + DM * kHalfBytes + mm * kSBBytes;
        const uint32_t sb0 = *reinterpret_cast<const uint32_t*>(dsb + R0 * 4);
        const uint32_t sb1 = *reinterpret_cast<const uint32_t*>(dsb + R1 * 4);
        // d = sum (base + q) h over the 32 columns: s*q + b weights give
        // s*d + (b - 1024 s) * (sum of h over base-1024 columns) + (b - 64 s) * (the others)
        if constexpr (kMode == 0) {
          gout[mm * kBlockRows + R0] = bf16lo(sb0) * (d[0] + d[1]) + (bf16hi(sb0) - 1024.f * bf16lo(sb0)) * ha +
                                       (bf16hi(sb0) - 64.f * bf16lo(sb0)) * hb64;
          gout[mm * kBlockRows + R1] = bf16lo(sb1) * (d[2] + d[3]) + (bf16hi(sb1) - 1024.f * bf16lo(sb1)) * ha +
                                       (bf16hi(sb1) - 64.f * bf16lo(sb1)) * hb64;
        } else {
          gout[mm * kBlockRows + R0] = 0.f;
          gout[mm * kBlockRows + R1] = 0.f;
        }
      }
    }
  }
  if (!down_ok && tid == 0) *s_abort = 1;
  __syncthreads();
  if (tid == 0 && *s_abort) {  // outputs are undefined; let this CTA's copies land before exiting
    for (int i = 0; i <= NGU; ++i) mbar_drain(bars + 8u * i, 0);
    set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
  }
}

// y[i] = sum over the expert-kernel CTAs c (ascending) of partials[c][i], rounded to bf16.
// Thread (row r, group q) sums a contiguous range of c with batched loads; the 32 group sums of
// a row are then added in group order, so the result does not depend on timing.
__global__ void __launch_bounds__(kYThreads) decode_reduce_kernel(const DecodeParams p, int n_parts) {
  constexpr int kGroups = kYThreads / kYRows;
  __shared__ float s[kGroups][kYRows];
  pdl_launch_dependents();
  pdl_wait();
  const int r = threadIdx.x % kYRows, q = threadIdx.x / kYRows;
  const int row = blockIdx.x * kYRows + r;
  const int per = (n_parts + kGroups - 1) / kGroups, c_end = min(n_parts, (q + 1) * per);
  float acc = 0.f;
  for (int c0 = q * per; c0 < c_end; c0 += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (c0 + j < c_end) ? __ldcg(p.partials + (size_t)(c0 + j) * p.d + row) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc += v[j];
  }
  s[q][r] = acc;
  __syncthreads();
  if (q == 0) {
    float y = 0.f;
    for (int i = 0; i < kGroups; ++i) y += s[i][r];
    p.y[row] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s, void* const* events, int mode) {
  const moe_dims dims = {p.d, p.E, p.k, p.inter, p.inter, kGroup};
  const int n_parts = decode_parts(dims);
  const int smem = x_smem(p.d).total;
  // The router and reduce kernels ask for the largest shared-memory carveout, so that the SMs
  // they run on can take an expert-kernel CTA (~160 KB of shared memory) as soon as PDL lets it
  // start, instead of waiting for the SM to drain and change its L1/shared split.
  static cudaError_t attr = [] {
    cudaError_t e = cudaSuccess;
    for (auto kernel : {decode_expert_kernel<0, 8>, decode_expert_kernel<1, 8>, decode_expert_kernel<2, 8>,
                        decode_expert_kernel<0, 32>, decode_expert_kernel<1, 32>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, x_smem(kDecodeMaxD).total);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_router_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_reduce_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  if (mode == kDecodeDiagReadOnly) {  // the expert kernel's weight copies alone, no chain
    decode_expert_kernel<2, 8><<<n_parts, kXThreads, (size_t)smem, s>>>(p);
    return cudaGetLastError();
  }
  cudaError_t err = record_event(events, 0, s);
  if (err != cudaSuccess) return err;
  if ((err = launch_pdl(decode_router_kernel, (p.E + 1) / 2, kRThreads, 0, 1, s, p)) != cudaSuccess) return err;
  if ((err = record_event(events, 1, s)) != cudaSuccess) return err;
  if (p.E <= 256)
    err = mode == kDecodeDiagNoMath ? launch_pdl(decode_expert_kernel<1, 8>, n_parts, kXThreads, (size_t)smem, 1, s, p)
                                    : launch_pdl(decode_expert_kernel<0, 8>, n_parts, kXThreads, (size_t)smem, 1, s, p);
  else
    err = mode == kDecodeDiagNoMath ? launch_pdl(decode_expert_kernel<1, 32>, n_parts, kXThreads, (size_t)smem, 1, s, p)
                                    : launch_pdl(decode_expert_kernel<0, 32>, n_parts, kXThreads, (size_t)smem, 1, s, p);
  if (err != cudaSuccess) return err;
  if ((err = record_event(events, 2, s)) != cudaSuccess) return err;
  if ((err = launch_pdl(decode_reduce_kernel, p.d / kYRows, kYThreads, 0, 1, s, p, n_parts)) != cudaSuccess)
    return err;
  return record_event(events, 3, s);
}

}  // namespace moe
