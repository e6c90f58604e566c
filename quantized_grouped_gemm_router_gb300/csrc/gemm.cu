// Grouped GEMMs of the prefill path on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model", section
// "Prefill: keep routing on the GPU, dequantize in flight": the grouped GEMM dequantizes one
// small tile of groupwise-affine Q4 weights at a time on chip, accumulates in FP32, and never
// materialises the expanded weights; section "Decode: minimize bytes per token" (fusion): input
// projections fused with the gate activation, output projection fused with the routing scores
// and the shared expert.
//
// GB300 design (swap-AB): the dequantized weight slab is MMA operand A (M = 128 rows), the
// tile's token rows are operand B (N = rows of the tile rounded up to 16, up to 192, set per
// tile at run time), so an expert with few rows still issues dense MMAs. Dequantized A tiles go
// from registers straight into tensor memory (tcgen05.st) and the MMA reads A from there; shared
// memory only carries the packed codes and the B rows. One accumulator per tile:
//   gate/up: A stacks 64 gate rows over the same 64 features' up rows, so gate and up of a tile
//            share one M=128 accumulator and a tile can be 192 rows with two accumulator
//            buffers in TMEM (2 x 192 + 4 A tiles x 32 = 512 columns);
//   down:    the hidden rows' leading and remainder fp16 planes accumulate into the same
//            accumulator (two MMAs per K step).
// Fewer, taller tiles mean each weight is dequantized fewer times per FLOP.
//
// Three GB300 facts shape the pipeline (measured on this part):
//   * a TMA copy costs a roughly fixed ~0.2-0.3 us of issue time however small it is, so every
//     copy here moves several K steps at once (3-D / 4-D tensor maps, bulk copies of >= 9 KB);
//   * one thread issues at most one tcgen05.mma per ~40-60 cycles, so two warps issue, each
//     into its own column range of the accumulator (the tile's rows split in two);
//   * integer ALU ops issue at half the rate of fp16x2 ops; the dequant uses few of them.
//
// Persistent, warp-specialised CTAs (one per SM) walk the work items (block-map tile x output
// row block) in a fixed stride; every ring keeps running across items:
//   warp 0       weight producer: packed Q4 stages (kSW K blocks) by bulk / tensor copies
//                (router mode: bf16 router weight tiles, which the MMA reads from shared memory)
//   warp 1       activation producer: the tile's contiguous rows (expert-sorted fp16 x, hidden
//                rows of both planes, or token rows) for kSB K blocks in one tensor copy
//   warps 2, 11  MMA issuers (whole warp runs the loop, one elected lane issues), each for one
//                half of the tile's rows, or for tiles of at most 96 rows, each for one of a
//                stage's two K blocks into its own half of the accumulator buffer (the epilogue
//                adds the halves); warp 2 also owns the TMEM allocation
//   warps 3-10   dequantize nibbles into fp16 A tiles in tensor memory (each warp writes the 32
//                TMEM lanes its index may access)
//   warps 12-19  epilogue (two warps per TMEM lane quadrant, alternate 16-column chunks) from
//                one of two accumulator buffers while the next tile accumulates: SwiGLU ->
//                hidden rows (gate/up; the up-lane warp hands its values to the gate-lane warp
//                through shared memory), routing weight x accumulator -> fp32 red.add into the
//                token's output row (down), or logits + bias (router)
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
constexpr int kWarpMMA2 = kWarpDq0 + kNumDqWarps;          // second MMA issuer (warp 11)
constexpr int kWarpEpi0 = kWarpMMA2 + 1, kNumEpiWarps = 8;  // warps 12-19
constexpr int kThreads = (kWarpEpi0 + kNumEpiWarps) * 32;  // 640
constexpr int kATileBytes = kBlockRows * 128;              // 128 rows x 64 16-bit values

// kIssuers: MMA-issuing warps (each takes a column range of the one accumulator); kSW / kSB: K
// blocks per weight / activation stage; kStagesW / kStagesB: stages of the weight and activation
// rings; kStagesA: TMEM A stages (kAK K blocks each, matching the activation stages, so the MMA
// warps wait and commit once per kAK K blocks); kWStage: bytes of one weight stage;
// kPlanes: B operand planes per K block (down: leading and remainder fp16 parts of the hidden
// rows); kRows: maximum tile rows (MMA N); kMRows: output rows of one work item; kAcc: TMEM
// columns of one accumulator buffer.
template <int MODE>
struct Cfg;
// kEpi: the work list and epilogue the mode shares (the dense ablation modes reuse the gate/up and
// down ones; only their A operand differs); kW: the packed-weight layout the producer copies and
// the dequant warps read (kModeGateUp / kModeDown for the Q4 modes, else the mode itself).
template <>
struct Cfg<kModeGateUp> {
  static constexpr int kIssuers = 2, kSW = 4, kSB = 2, kStagesW = 3, kStagesB = 3, kStagesA = 2, kPlanes = 1;
  static constexpr int kRows = kTileRows, kMRows = 64, kAcc = kRows, kAK = 2;  // 64 features: gate over up rows
  static constexpr int kWStage = 2 * kSW * kGUQuarter;               // two row quarters x kSW blocks
  static constexpr bool kFp16 = true, kQ4 = true;
  static constexpr int kEpi = kModeGateUp, kW = kModeGateUp;
};
template <>
struct Cfg<kModeDown> {
  static constexpr int kIssuers = 2, kSW = 2, kSB = 2, kStagesW = 3, kStagesB = 2, kStagesA = 2, kPlanes = 2;
  static constexpr int kRows = kTileRows, kMRows = kBlockRows, kAcc = kRows, kAK = 2;
  static constexpr int kWStage = kSW * kBlockBytes;                // codes (2 kSW halves), then kSW sb
  static constexpr bool kFp16 = true, kQ4 = true;
  static constexpr int kEpi = kModeDown, kW = kModeDown;
};
// Narrow tiles (at most 32 rows: a short prompt spread over many experts): accumulator buffers of
// 64 columns, so every tile splits its K blocks over the two issuers, and the room the 192-row
// operands took goes to deeper rings and larger stages: 7 (gate/up) or 6 (down) weight stages of
// 18 KB in flight per SM instead of 3 x 18 KB / 3 x 9 KB, and dequantized A stages of 4 K blocks
// (half the barrier round trips per K block).
template <>
struct Cfg<kModeGateUpNarrow> {
  static constexpr int kIssuers = 2, kSW = 4, kSB = 4, kStagesW = 7, kStagesB = 4, kStagesA = 3, kPlanes = 1;
  static constexpr int kRows = kNarrowTileRows, kMRows = 64, kAcc = 2 * kRows, kAK = 4;
  static constexpr int kWStage = 2 * kSW * kGUQuarter;
  static constexpr bool kFp16 = true, kQ4 = true;
  static constexpr int kEpi = kModeGateUp, kW = kModeGateUp;
};
template <>
struct Cfg<kModeDownNarrow> {
  static constexpr int kIssuers = 2, kSW = 4, kSB = 4, kStagesW = 6, kStagesB = 3, kStagesA = 3, kPlanes = 2;
  static constexpr int kRows = kNarrowTileRows, kMRows = kBlockRows, kAcc = 2 * kRows, kAK = 4;
  static constexpr int kWStage = kSW * kBlockBytes;
  static constexpr bool kFp16 = true, kQ4 = true;
  static constexpr int kEpi = kModeDown, kW = kModeDown;
};
template <>
struct Cfg<kModeRouter> {
  static constexpr int kIssuers = 1, kSW = 4, kSB = 4, kStagesW = 2, kStagesB = 2, kStagesA = 0, kPlanes = 1;
  static constexpr int kRows = kRouterRows, kMRows = kBlockRows, kAcc = kRows, kAK = 2;
  static constexpr int kWStage = kSW * kATileBytes;                // bf16 A tiles, read by the MMA
  static constexpr bool kFp16 = false, kQ4 = false;
  static constexpr int kEpi = kModeRouter, kW = kModeRouter;
};
// Materialised-dequantization ablation: fp16 weight tiles from the dense buffer, read by the MMA
// from shared memory like the router's.
template <>
struct Cfg<kModeGateUpDense> {
  static constexpr int kIssuers = 2, kSW = 2, kSB = 2, kStagesW = 3, kStagesB = 2, kStagesA = 0, kPlanes = 1;
  static constexpr int kRows = kTileRows, kMRows = 64, kAcc = kRows, kAK = 2;
  static constexpr int kWStage = kSW * kATileBytes;
  static constexpr bool kFp16 = true, kQ4 = false;
  static constexpr int kEpi = kModeGateUp, kW = kModeGateUpDense;
};
template <>
struct Cfg<kModeDownDense> {
  static constexpr int kIssuers = 2, kSW = 2, kSB = 1, kStagesW = 3, kStagesB = 2, kStagesA = 0, kPlanes = 2;
  static constexpr int kRows = kTileRows, kMRows = kBlockRows, kAcc = kRows, kAK = 2;
  static constexpr int kWStage = kSW * kATileBytes;
  static constexpr bool kFp16 = true, kQ4 = false;
  static constexpr int kEpi = kModeDown, kW = kModeDownDense;
};

constexpr int tmem_cols_for(int cols) {
  return cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
}

constexpr int kXPairs = 4, kXSlots = 2;  // gate/up epilogue exchange: warp pairs x buffered chunks

template <int MODE>
struct Smem {
  using C = Cfg<MODE>;
  static constexpr int kBStage = C::kSB * C::kPlanes * C::kRows * 128;  // [kb][plane][rows][128 B]
  static constexpr int kAccCols = C::kAcc;                              // one accumulator buffer
  // TMEM columns: two accumulator buffers, then (Q4 modes) the A tiles, 32 columns per 128x64 tile
  static constexpr int kACol = 2 * kAccCols;
  static constexpr int kTmemNeed = kACol + C::kStagesA * C::kAK * 32;
  static_assert(!C::kQ4 || (C::kSB == C::kAK && C::kSW % C::kAK == 0 && C::kStagesB >= C::kStagesA),
                "A stages follow the activation stages");
  static constexpr int kTmemCols = tmem_cols_for(kTmemNeed);
  static_assert(kTmemNeed <= 512, "tensor memory budget");
  // down: each epilogue warp keeps the (token, weight) list of its own chunks (half the rows)
  static constexpr int kListRows = C::kEpi == kModeDown ? C::kRows / 2 : 0;
  static constexpr int kXBytes = C::kEpi == kModeGateUp ? kXPairs * kXSlots * 16 * 32 * 4 : 0;
  static constexpr int w_off = 0;
  static constexpr int b_off = w_off + C::kStagesW * C::kWStage;
  static constexpr int x_off = b_off + C::kStagesB * kBStage;
  static constexpr int tok_off = x_off + kXBytes;
  static constexpr int wgt_off = tok_off + kNumEpiWarps * kListRows * 4;
  static_assert(tok_off % 16 == 0 && kListRows % 16 == 0, "16-byte loads of a chunk's list entries");
  static constexpr int bar_off = wgt_off + kNumEpiWarps * kListRows * 4;
  // full/empty per ring stage, acc_full[2], acc_empty[2], xfull/xempty[pairs][slots]
  static constexpr int n_bars = 2 * (C::kStagesW + C::kStagesA + C::kStagesB) + 4 + 2 * kXPairs * kXSlots;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int bytes = misc_off + 16;
  static constexpr int alloc = bytes + 1024;  // slack for 1024-byte alignment of the base
  static_assert(alloc <= 232448, "shared memory budget");
  static_assert(C::kWStage % 1024 == 0 && kBStage % 1024 == 0, "stage alignment");
};

// 8 packed codes (one word, nibble order of the packed layout) -> 8 fp16 weights, pairs of
// columns (2i, 2i+1) = nibbles (i, i+4). Integer ops issue at half the fp16x2 rate, so the
// fields are taken where they lie: nibbles 0/4 sit in mantissa bits [3:0] of 1024.0 and nibbles
// 1/5 in bits [7:4] of 64.0 (ulp 1/16), then one byte swap brings nibbles 2/6 and 3/7 to the
// same places: 1 PRMT + 4 LOP3 per word. Each pair becomes (base + q) exactly, base is
// subtracted exactly, and w = scale * q + bias is one fused multiply-add rounded once to fp16
// (exact whenever the value has at most 11 significant bits, e.g. bias = -8 * scale).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2, __half2 b2) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const __half2 k64 = __halves2half2(__ushort_as_half(0x5400), __ushort_as_half(0x5400));
  const uint32_t sw = __byte_perm(w, 0, 0x2301);  // swap the bytes inside each 16-bit half
  uint32_t t[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x54005400u,
                   (sw & 0x000F000Fu) | 0x64006400u, (sw & 0x00F000F0u) | 0x54005400u};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = __hsub2(*reinterpret_cast<__half2*>(&t[i]), (i & 1) ? k64 : k1024);  // exact: q
    v = __hfma2(v, s2, b2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The same 8 weights without the base subtraction for the pairs of nibbles 1/5 and 3/7: masked
// to mantissa bits [7:4] with a zero exponent field, such a pair is the fp16 subnormal q * 2^-20
// exactly, so w = (q * 2^-20) * (scale * 2^20) + bias is one fused multiply-add with the exact
// product q * scale, the result the base path rounds once too (bit-identical). Valid while
// scale * 2^20 is an fp16 number (|scale| <= 0.0624); the caller picks the path per warp.
__device__ __forceinline__ uint4 dequant8_sub(uint32_t w, __half2 s2, __half2 s2x, __half2 b2) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const uint32_t sw = __byte_perm(w, 0, 0x2301);
  uint32_t t[4] = {(w & 0x000F000Fu) | 0x64006400u, w & 0x00F000F0u, (sw & 0x000F000Fu) | 0x64006400u,
                   sw & 0x00F000F0u};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = *reinterpret_cast<__half2*>(&t[i]);
    v = (i & 1) ? __hfma2(v, s2x, b2) : __hfma2(__hsub2(v, k1024), s2, b2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// A (scale, bias) pair the fp16 dequantization cannot carry exactly: a nonzero scale or bias below
// the normal fp16 range (2^-14, where fp16 starts losing significant bits), or a weight
// scale * q + bias that could exceed 65504 (q <= 15); NaN and infinity included.
__device__ __forceinline__ bool sb_out_of_range(uint32_t sbw) {
  const float as = fabsf(__uint_as_float(sbw << 16)), ab = fabsf(__uint_as_float(sbw & 0xFFFF0000u));
  return !((as == 0.f || as >= 0x1p-14f) && (ab == 0.f || ab >= 0x1p-14f) && 15.f * as + ab <= 65504.f);
}

// bf16 (scale, bias) pair -> two fp16x2 broadcasts (exact inside the range sb_out_of_range checks).
__device__ __forceinline__ void scale_bias(uint32_t sbw, __half2& s2, __half2& b2) {
  const __half sh = __float2half_rn(__uint_as_float(sbw << 16));
  const __half bh = __float2half_rn(__uint_as_float(sbw & 0xFFFF0000u));
  s2 = __halves2half2(sh, sh);
  b2 = __halves2half2(bh, bh);
}

// One work item: a block-map tile (or a shared-expert / router row tile) x one block of output
// rows (gate/up: 64 features, stacked gate over up; down / router: 128 rows).
struct Item {
  int expert, r0, nrows, row0, m, n16;
  int ks, kbo;  // router: K slice and its first K block (0 otherwise)
  bool shared;
};

// Work order: the shared expert's tiles (every one full but the last) first, then the routed tiles
// in block-map order, so that the CTAs that run one item more than the others (the work list is
// rarely a multiple of the grid) end on the light tiles of the last, least popular experts rather
// than on the shared expert's full ones (same-box A/B, per-layer us: 512 tokens 202.5 -> 199.7,
// skewed 2048 tokens 205.2 -> 198.5, 4096 tokens 381.2 -> 377.9).
template <int MODE>
__device__ __forceinline__ Item decode_item(const GemmParams& p, int item, int n_routed) {
  Item it;
  const int tq = item / p.m_tiles, n_shared = (p.T + p.tile_rows - 1) / p.tile_rows;
  const int tile = MODE == kModeRouter ? tq : tq < n_shared ? n_routed + tq : tq - n_shared;
  it.m = item % p.m_tiles;
  it.shared = false;
  it.expert = 0;
  it.ks = it.kbo = 0;
  if (MODE == kModeRouter) {  // item = (token tile, m block, K slice), the slice fastest
    const int rest = item / p.ksplit;
    it.ks = item % p.ksplit;
    it.kbo = it.ks * p.k_blocks;
    it.m = rest % p.m_tiles;
    it.r0 = rest / p.m_tiles * kRouterRows;
    it.nrows = min(kRouterRows, p.T - it.r0);
    it.row0 = it.r0;
  } else if (tile < n_routed) {
    it.expert = p.tile_map[3 * tile];
    it.r0 = p.tile_map[3 * tile + 1];
    it.nrows = p.tile_map[3 * tile + 2];
    it.row0 = p.tile_row0[tile];  // no dependent load: the router stored offsets[expert] + r0
  } else {
    it.r0 = (tile - n_routed) * p.tile_rows;
    it.expert = p.E;
    it.shared = true;
    it.nrows = min(p.tile_rows, p.T - it.r0);
    it.row0 = p.T * p.k + it.r0;
  }
  it.n16 = (it.nrows + 15) & ~15;
  return it;
}

// RO: the read-only probe of the same access pattern. The two producers run unchanged (the same
// work list, copies, stage sizes and ring depths); warps 2 and 11 release each weight / activation
// stage as soon as it has landed; nothing is dequantized, multiplied or written.
template <int MODE, bool RO = false>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const GemmParams p, const __grid_constant__ GemmMaps maps) {
  using C = Cfg<MODE>;
  using S = Smem<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int KB = p.k_blocks;

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
  auto xfull = [&](int pr, int sl) { return acc_bars + 8u * (4 + pr * kXSlots + sl); };
  auto xempty = [&](int pr, int sl) { return acc_bars + 8u * (4 + kXPairs * kXSlots + pr * kXSlots + sl); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::misc_off);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::misc_off + 4);
  auto w_stage = [&](int s) { return smem + S::w_off + s * C::kWStage; };
  auto b_stage = [&](int s) { return base + S::b_off + s * S::kBStage; };
  auto a_tmem = [&](uint32_t tbase, int stage) { return tbase + S::kACol + stage * C::kAK * 32; };

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesW; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(empty_w(s), RO ? 1 : C::kQ4 ? kNumDqWarps : C::kIssuers);
    }
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(full_a(s), kNumDqWarps);
      mbar_init(empty_a(s), C::kIssuers);
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), RO ? 1 : C::kIssuers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), C::kIssuers);
      mbar_init(acc_empty(b), kNumEpiWarps);
    }
    for (int pr = 0; pr < kXPairs; ++pr)
      for (int sl = 0; sl < kXSlots; ++sl) {
        mbar_init(xfull(pr, sl), 1);
        mbar_init(xempty(pr, sl), 1);
      }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(s_tmem), S::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpB && lane < 12) prefetch_tmap(&maps.rows[lane]);
  if (warp == kWarpW && lane == 0 && C::kW != kModeGateUp) prefetch_tmap(&maps.a);
  if (warp == kWarpW && lane == 1 && C::kW == kModeDown) prefetch_tmap(&maps.a2);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  // ---------------------------------------------------------------- work list
  // Everything above touched only this CTA's shared and tensor memory, so it overlaps the
  // predecessor kernel (programmatic dependent launch); the tile count and every activation are
  // read after it has completed. A CTA past the end of the work list runs empty loops.
  pdl_wait();
  pdl_launch_dependents();
  int n_routed = 0, n_tile_total;
  if (MODE == kModeRouter) {
    n_tile_total = (p.T + kRouterRows - 1) / kRouterRows;
  } else {
    n_routed = *p.n_tiles;
    n_tile_total = n_routed + (p.T + p.tile_rows - 1) / p.tile_rows;  // routed tiles, then shared
  }
  const int n_items = n_tile_total * p.m_tiles * (MODE == kModeRouter ? p.ksplit : 1);

  if (warp == kWarpW) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      uint32_t gw = 0;  // running weight-stage counter across this CTA's items
      bool ok = true;
      Item nxt = decode_item<MODE>(p, blockIdx.x, n_routed);
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const Item it = nxt;
        if (item + (int)gridDim.x < n_items) nxt = decode_item<MODE>(p, item + gridDim.x, n_routed);
        const uint8_t* ebase = p.packed + (size_t)it.expert * p.expert_stride + p.region_offset;
        for (int kb0 = 0; kb0 < KB; kb0 += C::kSW, ++gw) {
          const int s = gw % C::kStagesW;
          if (!(ok = mbar_wait(empty_w(s), ((gw / C::kStagesW) & 1) ^ 1, s_abort))) break;
          const uint32_t dst = smem_u32(w_stage(s));
          if (C::kW == kModeGateUp) {
            // features 64h..64h+63 = quarters 2(h%2), 2(h%2)+1 of block h/2; K blocks kb0.. of a
            // quarter are contiguous, 2304 bytes each (gate then up)
            const int nk = min(C::kSW, KB - kb0), m = it.m >> 1, q0 = 2 * (it.m & 1);
            mbar_arrive_expect_tx(full_w(s), (uint32_t)(2 * nk * kGUQuarter));
            for (int qq = 0; qq < 2; ++qq)
              tma_bulk_g2s(dst + qq * C::kSW * kGUQuarter, ebase + gu_offset(m, q0 + qq, kb0, KB), nk * kGUQuarter,
                           full_w(s));
          } else if (C::kW == kModeDown) {
            // codes of (K block, half) pieces kb0*2 .. kb0*2+2kSW-1 of block m, then their scale/bias
            mbar_arrive_expect_tx(full_w(s), (uint32_t)C::kWStage);
            tma_load_4d(dst, &maps.a, 0, it.m, 2 * kb0, it.expert, full_w(s));
            tma_load_4d(dst + 2 * C::kSW * kHalfBytes, &maps.a2, 0, it.m, kb0, it.expert, full_w(s));
          } else {
            // 16-bit A tiles by one 3-D tensor copy: the router weight, or the dense weights of the
            // materialised-dequantization ablation ([expert][item][128 rows] / [expert][d rows])
            const int row0 = MODE == kModeRouter       ? it.m * kBlockRows
                             : MODE == kModeGateUpDense ? (it.expert * p.m_tiles + it.m) * kBlockRows
                                                        : it.expert * p.d + it.m * kBlockRows;
            mbar_arrive_expect_tx(full_w(s), (uint32_t)C::kWStage);
            tma_load_3d(dst, &maps.a, 0, row0, kb0 + it.kbo, full_w(s));
          }
        }
      }
    }
  } else if (warp == kWarpB) {
    // ------------------------------------------------------------ activation (B) producer
    // One copy brings n16 rows x kSB K blocks (x both planes), laid out [K block][plane][row][64
    // values]; rows past the tile's end belong to the next tile or lie beyond the tensor (zero
    // fill) and their accumulator columns are never read.
    if (lane == 0) {
      uint32_t gb = 0;
      bool ok = true;
      Item nxt = decode_item<MODE>(p, blockIdx.x, n_routed);
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const Item it = nxt;
        if (item + (int)gridDim.x < n_items) nxt = decode_item<MODE>(p, item + gridDim.x, n_routed);
        const CUtensorMap* map = &maps.rows[it.n16 / 16 - 1];
        for (int kb0 = 0; kb0 < KB; kb0 += C::kSB, ++gb) {
          const int s = gb % C::kStagesB;
          if (!(ok = mbar_wait(empty_b(s), ((gb / C::kStagesB) & 1) ^ 1, s_abort))) break;
          mbar_arrive_expect_tx(full_b(s), (uint32_t)(C::kSB * C::kPlanes * it.n16 * 128));
          if (C::kPlanes == 2)
            tma_load_4d(b_stage(s), map, 0, it.row0, 0, kb0, full_b(s));
          else
            tma_load_3d(b_stage(s), map, 0, it.row0, kb0 + it.kbo, full_b(s));
        }
      }
    }
  } else if constexpr (RO) {
    // ------------------------------------------------------------ read-only probe: release stages
    if ((warp == kWarpMMA || warp == kWarpMMA2) && lane == 0) {
      const bool wring = warp == kWarpMMA;
      const int per = wring ? C::kSW : C::kSB, stages = wring ? C::kStagesW : C::kStagesB;
      uint32_t g = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x)
        for (int kb0 = 0; kb0 < KB && ok; kb0 += per, ++g) {
          const int s = g % stages;
          if ((ok = mbar_wait(wring ? full_w(s) : full_b(s), (g / stages) & 1, s_abort)))
            mbar_arrive(wring ? empty_w(s) : empty_b(s));
        }
    }
  } else if (warp == kWarpMMA || warp == kWarpMMA2) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer i owns accumulator columns [c0, c0 + n) = its half of the tile's rows (n may be 0 for
    // a 16-row tile; the issuer then only keeps the barrier counts). The whole warp runs the loop
    // (uniform operands); one elected lane issues each instruction.
    const int issuer = warp == kWarpMMA ? 0 : 1;
    if (issuer < C::kIssuers) {
      uint32_t gb = 0, gw = 0;
      int n = 0;
      bool ok = true;
      Item nxt = decode_item<MODE>(p, blockIdx.x, n_routed);
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
        const Item it = nxt;
        if (item + (int)gridDim.x < n_items) nxt = decode_item<MODE>(p, item + gridDim.x, n_routed);
        const int buf = n & 1;
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_empty(buf), ((n >> 1) & 1) ^ 1, s_abort)))) break;
        tc_fence_after();
        // A tile of at most half a buffer splits the K blocks instead of the rows: issuer i takes
        // the K blocks j of every stage with j % 2 == i over all of the tile's rows, into its own
        // half of the buffer, and the epilogue adds the halves. Each tcgen05.mma costs its issuing
        // thread tens of cycles however narrow the tile, so a narrow tile left to one issuer would
        // bound the kernel (K blocks per stage: an even kSB; every K extent is a multiple of 128).
        const bool split_k = C::kIssuers == 2 && C::kSB % 2 == 0 && it.n16 <= S::kAccCols / 2;
        const int half16 = C::kIssuers == 2 ? 16 * ((it.n16 / 16 + 1) / 2) : it.n16;
        const int c0 = split_k || issuer == 0 ? 0 : half16;
        const int ncols = split_k ? it.n16 : issuer == 0 ? half16 : it.n16 - half16;
        const uint32_t idesc = idesc_f16(kBlockRows, ncols > 0 ? ncols : 16, C::kFp16);
        const uint32_t acc = tmem_base + buf * S::kAccCols + (split_k ? issuer * (S::kAccCols / 2) : c0);
        int kb = 0;  // K block of this item
        for (int s0 = 0; s0 < KB && ok; s0 += C::kSB, ++gb) {
          const int nkb = min(C::kSB, KB - s0);
          constexpr int kSA = C::kStagesA > 0 ? C::kStagesA : 1;  // router mode has no A stages
          const int sb = gb % C::kStagesB, sa = C::kQ4 ? (int)(gb % kSA) : 0;
          // Q4 modes: the dequant warps see the activation stage land before they mark the A
          // stage full, so one wait covers both operands (each wait costs the issuing warp ~100
          // cycles even when the barrier is already complete)
          ok = __all_sync(0xFFFFFFFFu, C::kQ4 ? mbar_wait(full_a(sa), (gb / kSA) & 1, s_abort)
                                              : mbar_wait(full_b(sb), (gb / C::kStagesB) & 1, s_abort));
          if (!ok) break;
          for (int j = 0; j < nkb; ++j, ++kb) {
            // router weights: a shared-memory tile of the current weight stage
            const int sw = C::kQ4 ? 0 : (int)(gw % C::kStagesW), jw = C::kQ4 ? 0 : kb % C::kSW;
            if constexpr (!C::kQ4) {
              if (jw == 0 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(full_w(sw), (gw / C::kStagesW) & 1, s_abort))))
                break;
            }
            tc_fence_after();
            if (ncols > 0 && (!split_k || (j & 1) == issuer)) {
              const int kfirst = split_k ? s0 + j - issuer : kb;  // 0 on this issuer's first K block
              // B operand of (K block j, plane b, K step ks): the descriptor's start-address field
              // (16-byte units, 14 bits; every shared-memory address here is below 2^18) advanced
              // from the stage's first row instead of rebuilt per instruction
              const uint64_t bdj = sw128_desc(b_stage(sb) + c0 * 128) + (uint64_t)(j * C::kPlanes * it.n16 * 8);
              if constexpr (C::kQ4) {
                // the K block's 4 K steps (x 2 planes for down) under one elected lane: fewer
                // instructions per MMA on a scheduler the dequant warps share (measured: 512 tokens
                // 199.4 -> 196.2 us per layer, 4096 tokens 373.9 -> 371.8)
                if constexpr (C::kPlanes == 1)
                  umma_f16_ts_k64_elect(acc, a_tmem(tmem_base, sa) + j * 32, bdj, idesc, kfirst != 0);
                else
                  umma_f16_ts_k64x2_elect(acc, a_tmem(tmem_base, sa) + j * 32, bdj, bdj + (uint64_t)(it.n16 * 8), idesc,
                                          kfirst != 0);
              } else {
#pragma unroll
                for (int ks = 0; ks < kGroup / 16; ++ks) {
#pragma unroll
                  for (int b = 0; b < C::kPlanes; ++b) {
                    const uint64_t bdesc = bdj + (uint64_t)(b * it.n16 * 8 + ks * 2);
                    const uint32_t accumulate = (kfirst | ks | b) != 0;
                    umma_f16_ss_elect(acc, sw128_desc(smem_u32(w_stage(sw)) + jw * kATileBytes + ks * 32), bdesc, idesc,
                                      accumulate);
                  }
                }
              }
            }
            if constexpr (!C::kQ4) {
              if (jw == C::kSW - 1 || kb == KB - 1) {
                umma_commit_elect(empty_w(sw));
                ++gw;
              }
            }
          }
          if (!ok) break;
          if constexpr (C::kQ4) umma_commit_elect(empty_a(sa));
          umma_commit_elect(empty_b(sb));
        }
        if (ok) umma_commit_elect(acc_full(buf));
      }
    }
  } else if (warp < kWarpEpi0) {
    // ------------------------------------------------------------ dequant (Q4 modes)
    // Warp -> (TMEM lane quadrant, part): with A stages of 2 K blocks a thread converts one K
    // half (32 values, 16 columns) of its A row in every block of the stage (part = K half); with
    // stages of 4 blocks it converts whole blocks, every other one (part = block parity), with
    // one scale/bias conversion and one 32-column tensor-memory store per block (measured: gate/up
    // 4.8% faster at 512 tokens; no gain with 2-block stages). gate/up rows 0..63 are gate
    // features, 64..127 the same features' up rows.
    if constexpr (C::kQ4) {
      constexpr bool kWhole = C::kAK >= 4;
      constexpr int kPer = kWhole ? C::kAK / 2 : C::kAK, kHalves = kWhole ? 2 : 1;  // blocks, K halves per block
      static_assert(C::kAK % 2 == 0, "two warps per lane quadrant share a stage's blocks");
      const int quad = warp & 3, part = (warp - kWarpDq0) >> 2;
      const int r = quad * 32 + lane;  // A row
      const uint32_t lanes = (uint32_t)(quad * 32) << 16;
      uint32_t ga = 0, gw = 0;
      bool ok = true, sb_bad = false;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        for (int kb0 = 0; kb0 < KB && ok; kb0 += C::kSW, ++gw) {
          const int nk = min(C::kSW, KB - kb0);  // even: KB and kSW are
          const int sw = gw % C::kStagesW;
          // tcgen05.st is warp-collective: every lane takes the same exit on an abort
          if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(full_w(sw), (gw / C::kStagesW) & 1, s_abort)))) break;
          const uint8_t* ws = w_stage(sw);
          for (int j0 = 0; j0 < nk; j0 += C::kAK, ++ga) {
            const int sa = ga % C::kStagesA;
            uint4 cw[kPer][kHalves];
            uint32_t sbw[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {  // a ragged last stage reads stale, unused blocks
              const int j = j0 + (kWhole ? part + 2 * u : u);
#pragma unroll
              for (int h = 0; h < kHalves; ++h) {
                const int hh = kWhole ? h : part;  // K half: values 32hh .. 32hh + 31 of the block
                if constexpr (C::kW == kModeGateUp)
                  cw[u][h] = *reinterpret_cast<const uint4*>(ws + ((quad & 1) * C::kSW + j) * kGUQuarter +
                                                             (quad >> 1) * kGUMat + hh * kQuarterRows * 16 + lane * 16);
                else
                  cw[u][h] = *reinterpret_cast<const uint4*>(ws + (2 * j + hh) * kHalfBytes + r * 16);
              }
              if constexpr (C::kW == kModeGateUp)
                sbw[u] = *reinterpret_cast<const uint32_t*>(ws + ((quad & 1) * C::kSW + j) * kGUQuarter +
                                                            (quad >> 1) * kGUMat + 2 * kQuarterRows * 16 + lane * 4);
              else
                sbw[u] = *reinterpret_cast<const uint32_t*>(ws + 2 * C::kSW * kHalfBytes + j * kSBBytes + r * 4);
            }
            if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty_a(sa), ((ga / C::kStagesA) & 1) ^ 1, s_abort)))) break;
            tc_fence_after();
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
              const int t = kWhole ? part + 2 * u : u;
              __half2 s2, b2;
              if ((kWhole || part == 0) && j0 + t < nk) sb_bad |= sb_out_of_range(sbw[u]);  // once per word
              scale_bias(sbw[u], s2, b2);
              uint32_t v[16 * kHalves];
              // whole blocks: the subnormal path when every lane's scale allows it (a uniform branch;
              // measured 3.3% faster at 512 tokens, 1% slower with the wide configuration's half blocks)
              bool sub = false;
              __half2 s2x;
              if constexpr (kWhole) {
                const float sf = __uint_as_float(sbw[u] << 16);
                const __half sxh = __float2half_rn(sf * 1048576.f);  // scale * 2^20, exact while sub
                s2x = __halves2half2(sxh, sxh);
                sub = __all_sync(0xFFFFFFFFu, fabsf(sf) <= 0.0624f);
              }
              if (sub) {
#pragma unroll
                for (int h = 0; h < kHalves; ++h) {
                  const uint32_t words[4] = {cw[u][h].x, cw[u][h].y, cw[u][h].z, cw[u][h].w};
#pragma unroll
                  for (int c = 0; c < 4; ++c) {
                    const uint4 o = dequant8_sub(words[c], s2, s2x, b2);
                    v[16 * h + 4 * c] = o.x, v[16 * h + 4 * c + 1] = o.y, v[16 * h + 4 * c + 2] = o.z;
                    v[16 * h + 4 * c + 3] = o.w;
                  }
                }
              } else {
#pragma unroll
                for (int h = 0; h < kHalves; ++h) {
                  const uint32_t words[4] = {cw[u][h].x, cw[u][h].y, cw[u][h].z, cw[u][h].w};
#pragma unroll
                  for (int c = 0; c < 4; ++c) {
                    const uint4 o = dequant8(words[c], s2, b2);
                    v[16 * h + 4 * c] = o.x, v[16 * h + 4 * c + 1] = o.y, v[16 * h + 4 * c + 2] = o.z;
                    v[16 * h + 4 * c + 3] = o.w;
                  }
                }
              }
              if constexpr (kWhole)
                tmem_st32(a_tmem(tmem_base, sa) + lanes + t * 32, v);
              else
                tmem_st16(a_tmem(tmem_base, sa) + lanes + t * 32 + part * 16, v);
            }
            // The weight stage is released only once every lane's codes have been consumed (the
            // values above depend on them). Arriving right after issuing the shared-memory loads
            // let the next TMA copy overwrite the stage before every load had read it: the copy is
            // an async-proxy write, which the barrier's release does not order after generic
            // reads. Barriers count warps: lane 0 arrives after the warp has synchronised (one
            // arrival instead of 32 on the same shared-memory word).
            if (j0 + C::kAK >= nk) {
              __syncwarp();
              if (lane == 0) mbar_arrive(empty_w(sw));
            }
            tmem_wait_st();
            tc_fence_before();
            // The MMA warps wait only on full_a: make it imply this stage's activation rows too.
            // full_a completes only once all the dequant warps have arrived, so it is enough that
            // one of them saw the activation stage land before arriving; the duty rotates over the
            // warps, stage by stage (a wait on a completed barrier still costs a warp ~100 cycles).
            // The activation stage cannot be refilled before this stage's MMAs complete, so the
            // waiting warp's parity is never a phase behind.
            if ((int)(ga % kNumDqWarps) == warp - kWarpDq0) {
              if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(full_b(ga % C::kStagesB), (ga / C::kStagesB) & 1, s_abort))))
                break;
            } else {
              __syncwarp();  // every lane's tensor-memory stores are complete before lane 0 arrives
            }
            if (lane == 0) mbar_arrive(full_a(sa));
          }
        }
      }
      // scales or biases the fp16 operands cannot hold exactly are reported, not hidden
      if (__any_sync(0xFFFFFFFFu, sb_bad) && lane == 0) set_device_status(p.hdr, MOE_ERR_OUT_OF_RANGE);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    static_assert(kWarpEpi0 % 4 == 0 && kNumEpiWarps == 8, "two epilogue warps per lane quadrant");
    const int q = warp & 3;                          // TMEM lane quadrant this warp may access
    const int half = (warp - kWarpEpi0) >> 2;        // this warp takes 16-column chunks half, half+2, ...
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    // down: this warp's rows in chunk order, as output-row offsets (token x d) and routing weights
    int32_t* tok = reinterpret_cast<int32_t*>(smem + S::tok_off) + (warp - kWarpEpi0) * S::kListRows;
    float* wgt = reinterpret_cast<float*>(smem + S::wgt_off) + (warp - kWarpEpi0) * S::kListRows;
    // gate/up: the gate-lane warp (quadrants 0, 1) and the up-lane warp (quadrants 2, 3) of the
    // same features and chunks form pair `pr`; the up warp passes its 16 x 32 values through slot
    // (u & 1) of the pair's exchange buffer, [value][lane] to avoid bank conflicts
    const int pr = (q & 1) + 2 * half;
    const bool gate_warp = q < 2;
    float* xbuf = reinterpret_cast<float*>(smem + S::x_off) + pr * kXSlots * 16 * 32;
    uint32_t u = 0;  // chunks exchanged so far by this pair
    bool over = false, ok = true;
    int n = 0;
    Item nxt = decode_item<MODE>(p, blockIdx.x, n_routed);
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
      const Item it = nxt;
      if (item + (int)gridDim.x < n_items) nxt = decode_item<MODE>(p, item + gridDim.x, n_routed);
      const int buf = n & 1;
      if (C::kEpi == kModeDown) {  // this warp's (token, routing weight) list, read before the wait
        constexpr int kPer = (C::kRows + 31) / 32;
        int2 tw[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {  // all loads first: they overlap
          const int j = lane + 32 * i;
          const bool mine = j < it.nrows && ((j >> 4) & 1) == half;  // only the rows of this warp's chunks
          tw[i] = mine && !it.shared ? p.row_tw[it.row0 + j]          // written by the router's scatter
                                     : make_int2(it.r0 + j, __float_as_int(1.f));
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int j = lane + 32 * i;
          if (j < it.nrows && ((j >> 4) & 1) == half) {
            const int li = ((j >> 5) << 4) | (j & 15);  // position among this warp's rows
            tok[li] = tw[i].x * p.d;
            wgt[li] = __int_as_float(tw[i].y);
          }
        }
        __syncwarp();
      }
      // tcgen05.ld is warp-collective: every lane takes the same exit on an abort
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_full(buf), (n >> 1) & 1, s_abort)))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_addr + buf * S::kAccCols;
      const bool split_k = C::kIssuers == 2 && C::kSB % 2 == 0 && it.n16 <= S::kAccCols / 2;  // the issuers' K split
      for (int j0 = 16 * half; j0 < it.n16 && ok; j0 += 32) {
        uint32_t acc[16];
        tmem_ld16(taddr + j0, acc);
        tmem_wait_ld();
        if (split_k) {  // the second issuer's partial sums over the other K blocks
          uint32_t acc2[16];
          tmem_ld16(taddr + S::kAccCols / 2 + j0, acc2);
          tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) acc[jj] = __float_as_uint(__uint_as_float(acc[jj]) + __uint_as_float(acc2[jj]));
        }
        if (C::kEpi == kModeGateUp) {
          const int sl = u & 1;
          float* xs = xbuf + sl * 16 * 32;
          if (!gate_warp) {  // hand the up values to the gate warp
            if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(xempty(pr, sl), ((u >> 1) & 1) ^ 1, s_abort)))) break;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) xs[jj * 32 + lane] = __uint_as_float(acc[jj]);
            __syncwarp();
            if (lane == 0) mbar_arrive(xfull(pr, sl));
          } else {
            if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(xfull(pr, sl), (u >> 1) & 1, s_abort)))) break;
            float up[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) up[jj] = xs[jj * 32 + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(xempty(pr, sl));
            const int f = it.m * 64 + (q & 1) * 32 + lane;  // feature
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = j0 + jj;
              // SiLU(gate) * up; the exponent is clamped so 1 + e^-g stays finite (SiLU(-80) ~ -1e-33)
              const float gv = __uint_as_float(acc[jj]);
              const float h = __fdividef(gv, 1.f + __expf(-fmaxf(gv, -80.f))) * up[jj];
              const __half hi = __float2half_rn(h);
              const __half lo = __float2half_rn(h - __half2float(hi));
              if (j < it.nrows) {
                over |= !(fabsf(h) <= 65504.f);
                const size_t o = (size_t)(it.row0 + j) * p.inter + f;
                p.hidden[o] = __half_as_ushort(hi);
                p.hidden[o + (size_t)p.hidden_rows * p.inter] = __half_as_ushort(lo);
              }
            }
          }
          ++u;
        } else if constexpr (C::kEpi == kModeDown) {
          // the chunk's 16 rows sit at 16 consecutive list positions: their offsets and weights
          // come in as four 16-byte shared loads each, and every value is one multiply and one
          // fp32 reduction into its token's output row
          float* yrow = p.yacc + it.m * kBlockRows + q * 32 + lane;  // output feature of this lane
          const int L0 = (j0 >> 5) << 4, nv = it.nrows - j0;
          const int4* ro4 = reinterpret_cast<const int4*>(tok + L0);
          const float4* w4 = reinterpret_cast<const float4*>(wgt + L0);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int4 ro = ro4[g];
            const float4 w = w4[g];
            const int o[4] = {ro.x, ro.y, ro.z, ro.w};
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * g + e < nv) atomicAdd(yrow + o[e], __uint_as_float(acc[4 * g + e]) * wv[e]);
          }
        } else {
          const int orow = it.m * kBlockRows + q * 32 + lane;  // output row (expert)
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = j0 + jj;
            if (j < it.nrows && orow < p.E)  // K slice ks: its partial logits (the bias in slice 0)
              p.logits[((size_t)it.ks * p.T + it.r0 + j) * p.E + orow] =
                  __uint_as_float(acc[jj]) + (p.router_bias && it.ks == 0 ? p.router_bias[orow] : 0.f);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(buf));  // the accumulator buffer is free again
    }
    if (C::kEpi == kModeGateUp && __any_sync(0xFFFFFFFFu, over) && lane == 0)
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

template <int MODE, bool RO = false>
cudaError_t launch_mode(const GemmParams& p, const GemmMaps* maps, int max_items, cudaStream_t s) {
  // the maps' boxes must be the stages this configuration's shared memory holds
  if (p.b_kb != Cfg<MODE>::kSB || p.w_kb != Cfg<MODE>::kSW) return cudaErrorInvalidValue;
  static cudaError_t attr = cudaFuncSetAttribute(moe_gemm_kernel<MODE, RO>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<MODE>::alloc);
  if (attr != cudaSuccess) return attr;
  const int grid = max_items < num_sms() ? max_items : num_sms();  // persistent: one CTA per SM
  return launch_pdl(moe_gemm_kernel<MODE, RO>, grid, kThreads, (size_t)Smem<MODE>::alloc, 1, s, p, *maps);
}

}  // namespace

// `grid` is an upper bound on the number of work items; the persistent grid is at most one CTA
// per SM, and each CTA reads the actual work list size on the device.
cudaError_t launch_gemm(int mode, const GemmParams& p, const GemmMaps* maps, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  switch (mode) {
    case kModeRouter: return launch_mode<kModeRouter>(p, maps, grid, s);
    case kModeGateUp: return launch_mode<kModeGateUp>(p, maps, grid, s);
    case kModeGateUpDense: return launch_mode<kModeGateUpDense>(p, maps, grid, s);
    case kModeDownDense: return launch_mode<kModeDownDense>(p, maps, grid, s);
    case kModeGateUpNarrow: return launch_mode<kModeGateUpNarrow>(p, maps, grid, s);
    case kModeDownNarrow: return launch_mode<kModeDownNarrow>(p, maps, grid, s);
    default: return launch_mode<kModeDown>(p, maps, grid, s);
  }
}

cudaError_t launch_gemm_read_probe(int mode, const GemmParams& p, const GemmMaps* maps, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (mode == kModeGateUp) return launch_mode<kModeGateUp, true>(p, maps, grid, s);
  if (mode == kModeDown) return launch_mode<kModeDown, true>(p, maps, grid, s);
  if (mode == kModeGateUpNarrow) return launch_mode<kModeGateUpNarrow, true>(p, maps, grid, s);
  if (mode == kModeDownNarrow) return launch_mode<kModeDownNarrow, true>(p, maps, grid, s);
  return cudaErrorInvalidValue;
}

template <int F, int MODE>
int cfg_field() {
  using C = Cfg<MODE>;
  return F == 0 ? C::kSB : F == 1 ? C::kSW : C::kMRows;
}
template <int F>
int cfg_value(int mode) {
  switch (mode) {
    case kModeGateUpNarrow: return cfg_field<F, kModeGateUpNarrow>();
    case kModeDownNarrow: return cfg_field<F, kModeDownNarrow>();
    case kModeRouter: return F == 0 ? Cfg<kModeRouter>::kSB : F == 1 ? Cfg<kModeRouter>::kSW : Cfg<kModeRouter>::kMRows;
    case kModeGateUp: return F == 0 ? Cfg<kModeGateUp>::kSB : F == 1 ? Cfg<kModeGateUp>::kSW : Cfg<kModeGateUp>::kMRows;
    case kModeGateUpDense:
      return F == 0 ? Cfg<kModeGateUpDense>::kSB : F == 1 ? Cfg<kModeGateUpDense>::kSW : Cfg<kModeGateUpDense>::kMRows;
    case kModeDownDense:
      return F == 0 ? Cfg<kModeDownDense>::kSB : F == 1 ? Cfg<kModeDownDense>::kSW : Cfg<kModeDownDense>::kMRows;
    default: return F == 0 ? Cfg<kModeDown>::kSB : F == 1 ? Cfg<kModeDown>::kSW : Cfg<kModeDown>::kMRows;
  }
}
int gemm_kb_per_stage(int mode) { return cfg_value<0>(mode); }
int gemm_kw_per_stage(int mode) { return cfg_value<1>(mode); }
int gemm_out_rows(int mode) { return cfg_value<2>(mode); }

int router_tile_rows() { return kRouterRows; }

int router_split(const moe_dims& d, int T) {
  const int items = ((T + kRouterRows - 1) / kRouterRows) * ((d.n_experts + kBlockRows - 1) / kBlockRows);
  const int kb = d.d / kGroup;
  int s = 1;
  while (s < kMaxRouterSplit && 2 * s * items <= num_sms() && kb % (2 * s * Cfg<kModeRouter>::kSW) == 0) s *= 2;
  return s;
}

}  // namespace moe
