// Grouped GEMMs of the prefill path on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model", section
// "Prefill: keep routing on the GPU, dequantize in flight": the grouped GEMM dequantizes one
// small tile of groupwise-affine Q4 weights at a time in on-chip memory, accumulates in FP32,
// writes bf16 and never materialises the expanded weights; section "Decode: minimize bytes per
// token" (fusion): input projections fused with the gate activation, output projection fused
// with the routing scores and the shared expert.
//
// GB300 design (swap-AB): the dequantized weight slab is MMA operand A (M = 128 output rows),
// the expert's token rows are operand B (N = rows of the tile rounded up to 16, chosen per tile
// at run time, <= 256), so an expert with few rows still issues dense MMAs and an expert with
// up to 256 rows dequantizes each weight exactly once.
//
// One CTA = 6 warps:
//   warp 0     producer: TMA bulk copies of packed weight blocks; TMA gather4 (token rows of x
//              picked through the scatter permutation) or tiled loads (contiguous rows) of B
//   warp 1     allocates TMEM; lane 0 issues tcgen05.mma and the commits
//   warps 2-5  dequantize packed nibbles into 128-byte-swizzled bf16 A tiles in shared memory,
//              then run the epilogue from TMEM: SwiGLU -> bf16 hidden rows (gate/up), routing
//              weight x accumulator -> fp32 red.add into the token's output row (down), or
//              logits + bias (router)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kRouterRows = 64;  // token rows per router tile

template <int MODE>
struct Cfg;
// kNumA: weight operands per K step (gate and up share the B tile); kNumB: B operands per K step
// (the down projection reads the hidden rows as two fp16 planes into one accumulator);
// kFp16: fp16 operands (expert GEMMs) or bf16 operands (router).
template <>
struct Cfg<kModeGateUp> {
  static constexpr int kNumA = 2, kNumB = 1, kStagesW = 4, kStagesA = 2, kStagesB = 3, kRows = kTileRows;
  static constexpr int kTmemCols = 512, kWBytes = 2 * kBlockBytes;
  static constexpr bool kFp16 = true;
};
template <>
struct Cfg<kModeDown> {
  static constexpr int kNumA = 1, kNumB = 2, kStagesW = 6, kStagesA = 2, kStagesB = 2, kRows = kTileRows;
  static constexpr int kTmemCols = 256, kWBytes = kBlockBytes;
  static constexpr bool kFp16 = true;
};
template <>
struct Cfg<kModeRouter> {
  static constexpr int kNumA = 1, kNumB = 1, kStagesW = 0, kStagesA = 4, kStagesB = 4, kRows = kRouterRows;
  static constexpr int kTmemCols = 64, kWBytes = 0;
  static constexpr bool kFp16 = false;
};

constexpr int kATileBytes = kBlockRows * 128;  // 128 rows x 64 bf16

template <int MODE>
struct Smem {
  using C = Cfg<MODE>;
  static constexpr int kBTile = C::kRows * 128;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + C::kStagesA * C::kNumA * kATileBytes;
  static constexpr int w_off = b_off + C::kStagesB * C::kNumB * kBTile;
  static constexpr int tok_off = w_off + C::kStagesW * C::kWBytes;
  static constexpr int wgt_off = tok_off + C::kRows * 4;
  static constexpr int bar_off = wgt_off + C::kRows * 4;
  static constexpr int n_bars = 2 * (C::kStagesW + C::kStagesA + C::kStagesB) + 1;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int bytes = misc_off + 16;
  static constexpr int alloc = bytes + 1024;  // slack for 1024-byte alignment of the base
};

// 8 packed codes (one word, nibble order of the packed layout) -> 8 fp16 weights
// w = scale * q + bias as one fused multiply-add rounded once to fp16 (exact whenever the value
// has at most 11 significant bits, e.g. bias = -8 * scale).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2, __half2 b2) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;  // fp16 pair (1024 + q)
    __half2 v = *reinterpret_cast<__half2*>(&t);
    v = __hsub2(v, k1024);                                        // exact: q
    v = __hfma2(v, s2, b2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_a) {
  using C = Cfg<MODE>;
  using S = Smem<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- which tile is ours
  const int tile = blockIdx.x / p.m_tiles, m = blockIdx.x % p.m_tiles;
  int expert = 0, r0, nrows, row0;
  bool shared_tile = false;
  if (MODE == kModeRouter) {
    r0 = tile * kRouterRows;
    if (r0 >= p.T) return;
    nrows = min(kRouterRows, p.T - r0);
    row0 = r0;
  } else {
    const int n_routed = *p.n_tiles;
    if (tile < n_routed) {
      expert = p.tile_map[3 * tile];
      r0 = p.tile_map[3 * tile + 1];
      nrows = p.tile_map[3 * tile + 2];
      row0 = p.offsets[expert] + r0;
    } else {
      r0 = (tile - n_routed) * kTileRows;
      if (r0 >= p.T) return;  // beyond the shared expert's tiles: nothing to do
      expert = p.E;
      shared_tile = true;
      nrows = min(kTileRows, p.T - r0);
      row0 = p.T * p.k + r0;
    }
  }
  const int n16 = (nrows + 15) & ~15;

  int32_t* s_tok = reinterpret_cast<int32_t*>(smem + S::tok_off);
  float* s_wgt = reinterpret_cast<float*>(smem + S::wgt_off);
  const uint32_t bars = base + S::bar_off;
  auto full_w = [&](int s) { return bars + 8u * s; };
  auto empty_w = [&](int s) { return bars + 8u * (C::kStagesW + s); };
  auto full_a = [&](int s) { return bars + 8u * (2 * C::kStagesW + s); };
  auto empty_a = [&](int s) { return bars + 8u * (2 * C::kStagesW + C::kStagesA + s); };
  auto full_b = [&](int s) { return bars + 8u * (2 * C::kStagesW + 2 * C::kStagesA + s); };
  auto empty_b = [&](int s) { return bars + 8u * (2 * C::kStagesW + 2 * C::kStagesA + C::kStagesB + s); };
  const uint32_t tmem_full = bars + 8u * (S::n_bars - 1);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::misc_off);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::misc_off + 4);
  auto a_tile = [&](int stage, int which) { return base + S::a_off + (stage * C::kNumA + which) * kATileBytes; };
  auto b_tile = [&](int stage, int plane) { return base + S::b_off + (stage * C::kNumB + plane) * S::kBTile; };
  auto w_tile = [&](int stage) { return smem + S::w_off + stage * C::kWBytes; };

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesW; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(empty_w(s), 128);
    }
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(full_a(s), MODE == kModeRouter ? 1 : 128);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(tmem_full, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0) {
    prefetch_tmap(&tmap_b);
    if (MODE == kModeRouter) prefetch_tmap(&tmap_a);
    // Per-row token index (and routing weight for the down projection). Padding rows up to
    // the MMA's N repeat the tile's last valid row; their results are discarded.
    for (int j = lane; j < n16; j += 32) {
      const int jj = min(j, nrows - 1);
      int tok;
      float wgt = 1.f;
      if (MODE == kModeRouter || shared_tile) {
        tok = r0 + jj;
      } else {
        const int a = p.perm[row0 + jj];
        tok = a / p.k;
        if (MODE == kModeDown) wgt = p.topk_w[a];
      }
      s_tok[j] = tok;
      s_wgt[j] = wgt;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int KB = p.k_blocks;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    const uint8_t* ebase = p.packed + (size_t)expert * p.expert_stride + p.region_offset;
    for (int kb = 0; kb < KB; ++kb) {
      if constexpr (MODE != kModeRouter) {
        const int s = kb % C::kStagesW;
        if (!mbar_wait(empty_w(s), ((kb / C::kStagesW) & 1) ^ 1, s_abort)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_w(s), C::kWBytes);
          const uint32_t dst = smem_u32(w_tile(s));
          if (MODE == kModeGateUp) {  // four 32-row quarters: [gate | up] each
            for (int q = 0; q < 4; ++q)
              tma_bulk_g2s(dst + q * kGUQuarter, ebase + gu_offset(m, q, kb, KB), kGUQuarter, full_w(s));
          } else {                    // code halves of columns 0..31 and 32..63, then scale/bias
            const int DM = p.m_tiles;
            tma_bulk_g2s(dst, ebase + dn_code_offset(kb, 0, m, DM), kHalfBytes, full_w(s));
            tma_bulk_g2s(dst + kHalfBytes, ebase + dn_code_offset(kb, 1, m, DM), kHalfBytes, full_w(s));
            tma_bulk_g2s(dst + kCodeBytes, ebase + dn_sb_offset(kb, m, DM, KB), kSBBytes, full_w(s));
          }
        }
      } else {
        const int s = kb % C::kStagesA;
        if (!mbar_wait(empty_a(s), ((kb / C::kStagesA) & 1) ^ 1, s_abort)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_a(s), kATileBytes);
          tma_load_2d(a_tile(s, 0), &tmap_a, kb * kGroup, m * kBlockRows, full_a(s));
        }
      }
      const int sb = kb % C::kStagesB;
      if (!mbar_wait(empty_b(sb), ((kb / C::kStagesB) & 1) ^ 1, s_abort)) break;
      if (lane == 0) mbar_arrive_expect_tx(full_b(sb), (uint32_t)(C::kNumB * n16 * 128));
      __syncwarp();
      if (MODE == kModeGateUp) {
        for (int g = lane; g < n16 / 4; g += 32)
          tma_gather4(b_tile(sb, 0) + g * 512, &tmap_b, kb * kGroup, s_tok[4 * g], s_tok[4 * g + 1],
                      s_tok[4 * g + 2], s_tok[4 * g + 3], full_b(sb));
      } else {
        for (int g = lane; g < n16 / 16; g += 32) {
          tma_load_2d(b_tile(sb, 0) + g * 2048, &tmap_b, kb * kGroup, row0 + 16 * g, full_b(sb));
          if (C::kNumB == 2)
            tma_load_2d(b_tile(sb, 1) + g * 2048, &tmap_b, kb * kGroup, p.hidden_rows + row0 + 16 * g, full_b(sb));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBlockRows, n16, C::kFp16);
      bool ok = true;
      for (int kb = 0; kb < KB && ok; ++kb) {
        const int sa = kb % C::kStagesA, sb = kb % C::kStagesB;
        ok = mbar_wait(full_a(sa), (kb / C::kStagesA) & 1, s_abort) &&
             mbar_wait(full_b(sb), (kb / C::kStagesB) & 1, s_abort);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kGroup / 16; ++ks) {
#pragma unroll
          for (int b = 0; b < C::kNumB; ++b) {
            const uint64_t bdesc = sw128_desc(b_tile(sb, b) + ks * 32);
#pragma unroll
            for (int a = 0; a < C::kNumA; ++a)
              umma_f16_ss(tmem_base + a * kTileRows, sw128_desc(a_tile(sa, a) + ks * 32), bdesc, idesc,
                          (kb | ks | b) != 0);
          }
        }
        umma_commit(empty_a(sa));
        umma_commit(empty_b(sb));
      }
      if (ok) umma_commit(tmem_full);
    }
  } else {
    // ---------------------------------------------------------------- dequant (Q4 modes)
    const int r = threadIdx.x - 64;  // row of the 128-row block this thread dequantizes
    if constexpr (MODE != kModeRouter) {
      for (int kb = 0; kb < KB; ++kb) {
        const int sw = kb % C::kStagesW, sa = kb % C::kStagesA;
        if (!mbar_wait(full_w(sw), (kb / C::kStagesW) & 1, s_abort)) break;
        if (!mbar_wait(empty_a(sa), ((kb / C::kStagesA) & 1) ^ 1, s_abort)) break;
#pragma unroll
        for (int a = 0; a < C::kNumA; ++a) {
          // stage layout: gate/up = 4 quarters x [gate rows | up rows], each (half 0, half 1,
          // scale/bias) for 32 rows; down = (half 0, half 1, scale/bias) for 128 rows
          const uint8_t* blk;
          int rr, half_stride;
          if (MODE == kModeGateUp) {
            blk = w_tile(sw) + (r / kQuarterRows) * kGUQuarter + a * kGUMat;
            rr = r % kQuarterRows;
            half_stride = kQuarterRows * 16;
          } else {
            blk = w_tile(sw);
            rr = r;
            half_stride = kHalfBytes;
          }
          const uint4 c0 = *reinterpret_cast<const uint4*>(blk + rr * 16);
          const uint4 c1 = *reinterpret_cast<const uint4*>(blk + half_stride + rr * 16);
          const uint32_t sbw = *reinterpret_cast<const uint32_t*>(blk + 2 * half_stride + rr * 4);
          // bf16 scale and bias -> fp16 (exact inside the fp16 range)
          const __half sh = __float2half_rn(__uint_as_float(sbw << 16));
          const __half bh = __float2half_rn(__uint_as_float(sbw & 0xFFFF0000u));
          const __half2 s2 = __halves2half2(sh, sh), b2 = __halves2half2(bh, bh);
          const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint8_t* arow = smem + (a_tile(sa, a) - base) + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = dequant8(words[c], s2, b2);
        }
        fence_proxy_async_smem();
        mbar_arrive(full_a(sa));
        mbar_arrive(empty_w(sw));
      }
    }
    // ---------------------------------------------------------------- epilogue
    bool over = false;
    if (mbar_wait(tmem_full, 0, s_abort)) {
      tc_fence_after();
      const int q = warp & 3;                 // TMEM lane quadrant this warp may access
      const int orow = m * kBlockRows + q * 32 + lane;  // output row (feature / expert)
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
      for (int j0 = 0; j0 < n16; j0 += 16) {
        uint32_t acc0[16], acc1[16];
        tmem_ld16(taddr + j0, acc0);
        if (C::kNumA == 2) tmem_ld16(taddr + kTileRows + j0, acc1);
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = j0 + jj;
          if (j >= nrows) break;
          const float v0 = __uint_as_float(acc0[jj]);
          if (MODE == kModeGateUp) {
            const float u = __uint_as_float(acc1[jj]);
            const float h = v0 / (1.f + expf(-v0)) * u;
            const __half hi = __float2half_rn(h);
            const __half lo = __float2half_rn(h - __half2float(hi));
            over |= !(fabsf(h) <= 65504.f);
            const size_t o = (size_t)(row0 + j) * p.inter + orow;
            p.hidden[o] = __half_as_ushort(hi);
            p.hidden[o + (size_t)p.hidden_rows * p.inter] = __half_as_ushort(lo);
          } else if (MODE == kModeDown) {
            atomicAdd(p.yacc + (size_t)s_tok[j] * p.d + orow, v0 * s_wgt[j]);
          } else {
            if (orow < p.E)
              p.logits[(size_t)(r0 + j) * p.E + orow] = v0 + (p.router_bias ? p.router_bias[orow] : 0.f);
          }
        }
      }
    }
    if (MODE == kModeGateUp && __any_sync(0xFFFFFFFFu, over) && lane == 0)
      set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }

  // ---------------------------------------------------------------- tear-down
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *s_abort) set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
}

template <int MODE>
cudaError_t launch_mode(const GemmParams& p, const CUtensorMap* tb, const CUtensorMap* ta, int grid, cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(moe_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Smem<MODE>::alloc);
  if (attr != cudaSuccess) return attr;
  moe_gemm_kernel<MODE><<<grid, kThreads, Smem<MODE>::alloc, s>>>(p, *tb, *ta);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(int mode, const GemmParams& p, const CUtensorMap* tmap_b, const CUtensorMap* tmap_a, int grid,
                        cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  switch (mode) {
    case kModeRouter: return launch_mode<kModeRouter>(p, tmap_b, tmap_a, grid, s);
    case kModeGateUp: return launch_mode<kModeGateUp>(p, tmap_b, tmap_a, grid, s);
    default: return launch_mode<kModeDown>(p, tmap_b, tmap_a, grid, s);
  }
}

int router_tile_rows() { return kRouterRows; }

}  // namespace moe
