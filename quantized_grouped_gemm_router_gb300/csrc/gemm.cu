// Grouped GEMMs of the prefill path on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model", section
// "Prefill: keep routing on the GPU, dequantize in flight": the grouped GEMM dequantizes one
// small tile of groupwise-affine Q4 weights at a time in on-chip memory, accumulates in FP32,
// and never materialises the expanded weights; section "Decode: minimize bytes per token"
// (fusion): input projections fused with the gate activation, output projection fused with the
// routing scores and the shared expert.
//
// GB300 design (swap-AB): the dequantized weight slab is MMA operand A (M = 128 output rows),
// the expert's token rows are operand B (N = rows of the tile rounded up to 16, <= 128, set
// per tile at run time), so an expert with few rows still issues dense MMAs.
//
// Persistent, warp-specialised CTAs (one per SM) walk the work items (block-map tile x 128
// output rows) in a fixed stride; every ring of stages keeps running across items:
//   warp 0      weight producer: TMA bulk copies of packed Q4 blocks into a deep ring (router
//               mode: 2-D tiles of the bf16 router weight)
//   warp 1      activation producer: a tile's rows are contiguous (expert-sorted fp16 x, hidden
//               rows, or token rows), fetched by 2-D TMA boxes of 128/64/32/16 rows
//   warp 2      allocates TMEM; lane 0 issues tcgen05.mma into one of two accumulator buffers
//   warps 3-10  dequantize nibbles into 128-byte-swizzled fp16 A tiles in shared memory
//   warps 11-14 epilogue from the other accumulator buffer while the next tile accumulates:
//               SwiGLU -> hidden rows (gate/up), routing weight x accumulator -> fp32 red.add
//               into the token's output row (down), or logits + bias (router)
// Every mbarrier wait is bounded; a timeout raises a CTA-wide abort flag, every role leaves its
// loop, TMEM is freed and MOE_ERR_DEVICE_TIMEOUT is recorded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRouterRows = 64;    // token rows per router tile
constexpr int kWarpW = 0, kWarpB = 1, kWarpMMA = 2, kWarpDq0 = 3, kNumDqWarps = 8;
constexpr int kWarpEpi0 = kWarpDq0 + kNumDqWarps, kNumEpiWarps = 4;
constexpr int kThreads = (kWarpEpi0 + kNumEpiWarps) * 32;  // 480
constexpr int kDqThreads = kNumDqWarps * 32;               // 256
constexpr int kEpiThreads = kNumEpiWarps * 32;             // 128

// kNumA: weight operands per K step (gate and up share the B tile); kNumB: B operands per K step
// (the down projection reads the hidden rows as two fp16 planes into one accumulator);
// kFp16: fp16 operands (expert GEMMs) or bf16 operands (router).
template <int MODE>
struct Cfg;
template <>
struct Cfg<kModeGateUp> {
  static constexpr int kNumA = 2, kNumB = 1, kStagesW = 9, kStagesA = 2, kStagesB = 4, kRows = kTileRows;
  static constexpr int kWBytes = 4 * kGUQuarter;  // the 4 quarters of a 128-row block: gate + up
  static constexpr bool kFp16 = true;
};
template <>
struct Cfg<kModeDown> {
  static constexpr int kNumA = 1, kNumB = 2, kStagesW = 16, kStagesA = 2, kStagesB = 3, kRows = kTileRows;
  static constexpr int kWBytes = kBlockBytes;     // two code halves + scale/bias of one block
  static constexpr bool kFp16 = true;
};
template <>
struct Cfg<kModeRouter> {
  static constexpr int kNumA = 1, kNumB = 1, kStagesW = 0, kStagesA = 4, kStagesB = 4, kRows = kRouterRows;
  static constexpr int kWBytes = 0;
  static constexpr bool kFp16 = false;
};

constexpr int kATileBytes = kBlockRows * 128;  // 128 rows x 64 16-bit values

constexpr int tmem_cols_for(int cols) {
  return cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
}

template <int MODE>
struct Smem {
  using C = Cfg<MODE>;
  static constexpr int kBTile = C::kRows * 128;
  static constexpr int kAccCols = C::kNumA * C::kRows;  // one accumulator buffer
  static constexpr int kTmemCols = tmem_cols_for(2 * kAccCols);
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + C::kStagesA * C::kNumA * kATileBytes;
  static constexpr int w_off = b_off + C::kStagesB * C::kNumB * kBTile;
  // down projection: each epilogue warp keeps its own copy of the tile's (token, weight) list
  static constexpr int kListRows = MODE == kModeDown ? C::kRows : 0;
  static constexpr int tok_off = w_off + C::kStagesW * C::kWBytes;
  static constexpr int wgt_off = tok_off + kNumEpiWarps * kListRows * 4;
  static constexpr int bar_off = wgt_off + kNumEpiWarps * kListRows * 4;
  // full/empty per ring stage, then acc_full[2], acc_empty[2]
  static constexpr int n_bars = 2 * (C::kStagesW + C::kStagesA + C::kStagesB) + 4;
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

// bf16 (scale, bias) pair -> two fp16x2 broadcasts (exact inside the fp16 range).
__device__ __forceinline__ void scale_bias(uint32_t sbw, __half2& s2, __half2& b2) {
  const __half sh = __float2half_rn(__uint_as_float(sbw << 16));
  const __half bh = __float2half_rn(__uint_as_float(sbw & 0xFFFF0000u));
  s2 = __halves2half2(sh, sh);
  b2 = __halves2half2(bh, bh);
}

// One work item: a block-map tile (or a shared-expert / router row tile) x one 128-row block of
// the output features.
struct Item {
  int expert, r0, nrows, row0, m, n16;
  bool shared;
};

template <int MODE>
__device__ __forceinline__ Item decode_item(const GemmParams& p, int item, int n_routed) {
  Item it;
  const int tile = item / p.m_tiles;
  it.m = item % p.m_tiles;
  it.shared = false;
  it.expert = 0;
  if (MODE == kModeRouter) {
    it.r0 = tile * kRouterRows;
    it.nrows = min(kRouterRows, p.T - it.r0);
    it.row0 = it.r0;
  } else if (tile < n_routed) {
    it.expert = p.tile_map[3 * tile];
    it.r0 = p.tile_map[3 * tile + 1];
    it.nrows = p.tile_map[3 * tile + 2];
    it.row0 = p.offsets[it.expert] + it.r0;
  } else {
    it.r0 = (tile - n_routed) * kTileRows;
    it.expert = p.E;
    it.shared = true;
    it.nrows = min(kTileRows, p.T - it.r0);
    it.row0 = p.T * p.k + it.r0;
  }
  it.n16 = (it.nrows + 15) & ~15;
  return it;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const GemmParams p, const __grid_constant__ RowMaps maps_b,
                    const __grid_constant__ CUtensorMap tmap_a) {
  using C = Cfg<MODE>;
  using S = Smem<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- work list
  int n_routed = 0, n_tile_total;
  if (MODE == kModeRouter) {
    n_tile_total = (p.T + kRouterRows - 1) / kRouterRows;
  } else {
    n_routed = *p.n_tiles;
    n_tile_total = n_routed + (p.T + kTileRows - 1) / kTileRows;  // routed tiles, then shared
  }
  const int n_items = n_tile_total * p.m_tiles;
  if ((int)blockIdx.x >= n_items) return;  // nothing for this CTA (uniform: before any set-up)
  const int KB = p.k_blocks;

  int32_t* s_tok = reinterpret_cast<int32_t*>(smem + S::tok_off);  // [epilogue warp][kListRows]
  float* s_wgt = reinterpret_cast<float*>(smem + S::wgt_off);      // [epilogue warp][kListRows]
  const uint32_t bars = base + S::bar_off;
  auto full_w = [&](int s) { return bars + 8u * s; };
  auto empty_w = [&](int s) { return bars + 8u * (C::kStagesW + s); };
  auto full_a = [&](int s) { return bars + 8u * (2 * C::kStagesW + s); };
  auto empty_a = [&](int s) { return bars + 8u * (2 * C::kStagesW + C::kStagesA + s); };
  auto full_b = [&](int s) { return bars + 8u * (2 * C::kStagesW + 2 * C::kStagesA + s); };
  auto empty_b = [&](int s) { return bars + 8u * (2 * C::kStagesW + 2 * C::kStagesA + C::kStagesB + s); };
  const uint32_t acc_bars = bars + 8u * (2 * (C::kStagesW + C::kStagesA + C::kStagesB));
  auto acc_full = [&](int b) { return acc_bars + 8u * b; };
  auto acc_empty = [&](int b) { return acc_bars + 8u * (2 + b); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::misc_off);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::misc_off + 4);
  auto a_tile = [&](int stage, int which) { return base + S::a_off + (stage * C::kNumA + which) * kATileBytes; };
  auto b_tile = [&](int stage, int plane) { return base + S::b_off + (stage * C::kNumB + plane) * S::kBTile; };
  auto w_tile = [&](int stage) { return smem + S::w_off + stage * C::kWBytes; };

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesW; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(empty_w(s), kDqThreads);
    }
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(full_a(s), MODE == kModeRouter ? 1 : kDqThreads);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiThreads);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(s_tmem), S::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpB && lane < 4) prefetch_tmap(&maps_b.box[lane]);
  if (warp == kWarpW && lane == 0 && MODE == kModeRouter) prefetch_tmap(&tmap_a);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (warp == kWarpW) {
    // ------------------------------------------------------------ weight (A) producer
    if (lane == 0) {
      uint32_t g = 0;  // running K-block counter across this CTA's items
      for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const Item it = decode_item<MODE>(p, item, n_routed);
        const uint8_t* ebase = p.packed + (size_t)it.expert * p.expert_stride + p.region_offset;
        bool ok = true;
        for (int kb = 0; kb < KB && ok; ++kb, ++g) {
          if constexpr (MODE != kModeRouter) {
            const int s = g % C::kStagesW;
            if (!(ok = mbar_wait(empty_w(s), ((g / C::kStagesW) & 1) ^ 1, s_abort))) break;
            mbar_arrive_expect_tx(full_w(s), C::kWBytes);
            const uint32_t dst = smem_u32(w_tile(s));
            if (MODE == kModeGateUp) {  // four 32-row quarters: [gate | up] each
              for (int q = 0; q < 4; ++q)
                tma_bulk_g2s(dst + q * kGUQuarter, ebase + gu_offset(it.m, q, kb, KB), kGUQuarter, full_w(s));
            } else {                    // code halves of columns 0..31 and 32..63, then scale/bias
              const int DM = p.m_tiles;
              tma_bulk_g2s(dst, ebase + dn_code_offset(kb, 0, it.m, DM), kHalfBytes, full_w(s));
              tma_bulk_g2s(dst + kHalfBytes, ebase + dn_code_offset(kb, 1, it.m, DM), kHalfBytes, full_w(s));
              tma_bulk_g2s(dst + kCodeBytes, ebase + dn_sb_offset(kb, it.m, DM, KB), kSBBytes, full_w(s));
            }
          } else {
            const int s = g % C::kStagesA;
            if (!(ok = mbar_wait(empty_a(s), ((g / C::kStagesA) & 1) ^ 1, s_abort))) break;
            mbar_arrive_expect_tx(full_a(s), kATileBytes);
            tma_load_2d(a_tile(s, 0), &tmap_a, kb * kGroup, it.m * kBlockRows, full_a(s));
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == kWarpB) {
    // ------------------------------------------------------------ activation (B) producer
    // Rows of the tile: the padded rows up to n16 belong to the next tile or lie beyond the
    // tensor (zero fill); their accumulator columns are never read.
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const Item it = decode_item<MODE>(p, item, n_routed);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int sb = g % C::kStagesB;
          if (!(ok = mbar_wait(empty_b(sb), ((g / C::kStagesB) & 1) ^ 1, s_abort))) break;
          mbar_arrive_expect_tx(full_b(sb), (uint32_t)(C::kNumB * it.n16 * 128));
          int row = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int h = 128 >> i;
            if (it.n16 - row >= h) {
#pragma unroll
              for (int plane = 0; plane < C::kNumB; ++plane)
                tma_load_2d(b_tile(sb, plane) + row * 128, &maps_b.box[i], kb * kGroup,
                            plane * p.hidden_rows + it.row0 + row, full_b(sb));
              row += h;
            }
          }
        }
      }
    }
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0;
      int n = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
        const Item it = decode_item<MODE>(p, item, n_routed);
        const int buf = n & 1;
        if (!(ok = mbar_wait(acc_empty(buf), ((n >> 1) & 1) ^ 1, s_abort))) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(kBlockRows, it.n16, C::kFp16);
        const uint32_t acc = tmem_base + buf * S::kAccCols;
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int sa = g % C::kStagesA, sb = g % C::kStagesB;
          ok = mbar_wait(full_a(sa), (g / C::kStagesA) & 1, s_abort) &&
               mbar_wait(full_b(sb), (g / C::kStagesB) & 1, s_abort);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kGroup / 16; ++ks) {
#pragma unroll
            for (int b = 0; b < C::kNumB; ++b) {
              const uint64_t bdesc = sw128_desc(b_tile(sb, b) + ks * 32);
#pragma unroll
              for (int a = 0; a < C::kNumA; ++a)
                umma_f16_ss(acc + a * C::kRows, sw128_desc(a_tile(sa, a) + ks * 32), bdesc, idesc,
                            (kb | ks | b) != 0);
            }
          }
          umma_commit(empty_a(sa));
          umma_commit(empty_b(sb));
        }
        if (ok) umma_commit(acc_full(buf));
      }
    }
  } else if (warp < kWarpEpi0) {
    // ------------------------------------------------------------ dequant (Q4 modes)
    if constexpr (MODE != kModeRouter) {
      const int t = threadIdx.x - kWarpDq0 * 32;  // 0..255
      uint32_t g = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int sw = g % C::kStagesW, sa = g % C::kStagesA;
          ok = mbar_wait(full_w(sw), (g / C::kStagesW) & 1, s_abort) &&
               mbar_wait(empty_a(sa), ((g / C::kStagesA) & 1) ^ 1, s_abort);
          if (!ok) break;
          if (MODE == kModeGateUp) {
            // thread = (matrix, row): the row's 8 words -> 8 swizzled 16-byte chunks
            const int mat = t >> 7, r = t & 127, rr = r & (kQuarterRows - 1);
            const uint8_t* src = w_tile(sw) + (r / kQuarterRows) * kGUQuarter + mat * kGUMat;
            const uint4 c0 = *reinterpret_cast<const uint4*>(src + rr * 16);
            const uint4 c1 = *reinterpret_cast<const uint4*>(src + kQuarterRows * 16 + rr * 16);
            __half2 s2, b2;
            scale_bias(*reinterpret_cast<const uint32_t*>(src + 2 * kQuarterRows * 16 + rr * 4), s2, b2);
            const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint8_t* arow = smem + (a_tile(sa, mat) - base) + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = dequant8(words[c], s2, b2);
          } else {
            // thread = (row, half): the 4 words of one 32-column half
            const int r = t & 127, h = t >> 7;
            const uint8_t* src = w_tile(sw);
            const uint4 cw = *reinterpret_cast<const uint4*>(src + h * kHalfBytes + r * 16);
            __half2 s2, b2;
            scale_bias(*reinterpret_cast<const uint32_t*>(src + kCodeBytes + r * 4), s2, b2);
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
            uint8_t* arow = smem + (a_tile(sa, 0) - base) + r * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(arow + (((4 * h + c) ^ (r & 7)) << 4)) = dequant8(words[c], s2, b2);
          }
          fence_proxy_async_smem();
          mbar_arrive(full_a(sa));
          mbar_arrive(empty_w(sw));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                          // TMEM lane quadrant this warp may access
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    bool over = false;
    int n = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
      const Item it = decode_item<MODE>(p, item, n_routed);
      const int buf = n & 1;
      int32_t* tok = s_tok + (warp - kWarpEpi0) * S::kListRows;
      float* wgt = s_wgt + (warp - kWarpEpi0) * S::kListRows;
      if (MODE == kModeDown) {  // this warp's (token, routing weight) list, read before the wait
        __syncwarp();
        for (int j = lane; j < it.nrows; j += 32) {
          if (it.shared) {
            tok[j] = it.r0 + j;
            wgt[j] = 1.f;
          } else {
            const int a = p.perm[it.row0 + j];
            tok[j] = a / p.k;
            wgt[j] = p.topk_w[a];
          }
        }
        __syncwarp();
      }
      if (!mbar_wait(acc_full(buf), (n >> 1) & 1, s_abort)) break;
      tc_fence_after();
      const int orow = it.m * kBlockRows + q * 32 + lane;  // output row (feature / expert)
      const uint32_t taddr = tmem_base + lane_addr + buf * S::kAccCols;
      for (int j0 = 0; j0 < it.n16; j0 += 16) {
        uint32_t acc0[16], acc1[16];
        tmem_ld16(taddr + j0, acc0);
        if (C::kNumA == 2) tmem_ld16(taddr + C::kRows + j0, acc1);
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = j0 + jj;
          if (j >= it.nrows) break;
          const float v0 = __uint_as_float(acc0[jj]);
          if (MODE == kModeGateUp) {
            const float u = __uint_as_float(acc1[jj]);
            const float h = v0 / (1.f + expf(-v0)) * u;
            const __half hi = __float2half_rn(h);
            const __half lo = __float2half_rn(h - __half2float(hi));
            over |= !(fabsf(h) <= 65504.f);
            const size_t o = (size_t)(it.row0 + j) * p.inter + orow;
            p.hidden[o] = __half_as_ushort(hi);
            p.hidden[o + (size_t)p.hidden_rows * p.inter] = __half_as_ushort(lo);
          } else if (MODE == kModeDown) {
            atomicAdd(p.yacc + (size_t)tok[j] * p.d + orow, v0 * wgt[j]);
          } else {
            if (orow < p.E)
              p.logits[(size_t)(it.r0 + j) * p.E + orow] = v0 + (p.router_bias ? p.router_bias[orow] : 0.f);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty(buf));  // the accumulator buffer is free again
    }
    if (MODE == kModeGateUp && __any_sync(0xFFFFFFFFu, over) && lane == 0)
      set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
  }

  // ---------------------------------------------------------------- tear-down
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
  if (threadIdx.x == 0 && *s_abort) set_device_status(p.hdr, MOE_ERR_DEVICE_TIMEOUT);
}

int num_sms() {
  static int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      v = 1;
    return v > 0 ? v : 1;
  }();
  return n;
}

template <int MODE>
cudaError_t launch_mode(const GemmParams& p, const RowMaps* tb, const CUtensorMap* ta, int max_items,
                        cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(moe_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Smem<MODE>::alloc);
  if (attr != cudaSuccess) return attr;
  const int grid = max_items < num_sms() ? max_items : num_sms();  // persistent: one CTA per SM
  moe_gemm_kernel<MODE><<<grid, kThreads, Smem<MODE>::alloc, s>>>(p, *tb, *ta);
  return cudaGetLastError();
}

}  // namespace

// `grid` is an upper bound on the number of work items; the persistent grid is at most one CTA
// per SM, and each CTA reads the actual work list size on the device.
cudaError_t launch_gemm(int mode, const GemmParams& p, const RowMaps* tmap_b, const CUtensorMap* tmap_a, int grid,
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
