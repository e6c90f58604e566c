// Host side of the C ABI declared in include/moe_gb300.h: argument checks, workspace carve-up,
// TMA descriptor encoding and the launch sequence of each call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "moe_internal.h"

namespace moe {
int router_tile_rows();

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->group != kGroup || d->d < kBlockRows || d->d % kBlockRows || d->d > 16384 || d->inter < kBlockRows ||
      d->inter % kBlockRows || d->inter > 16384 || d->shared_inter != d->inter || d->top_k < 1 ||
      d->top_k > kMaxTopK || d->n_experts < d->top_k || d->n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int check_layer(const moe_layer* L, bool need_router) {
  if (!L) return MOE_ERR_INVALID_ARG;
  int st = check_dims(&L->dims);
  if (st) return st;
  if (!L->packed || (need_router && !L->router_w)) return MOE_ERR_INVALID_ARG;
  if (!aligned(L->packed, 128) || !aligned(L->router_w, 16) || !aligned(L->router_bias, 16)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType type, cuuint32_t rank, const void* ptr, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, type, rank, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major [rows, cols] 16-bit matrix seen as (64 columns, rows, cols / 64 column blocks), so
// that one box (64 x box_rows x kb) lands in shared memory as kb consecutive [box_rows][64] tiles,
// 128-byte swizzled.
bool make_rows_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t kb,
                   bool fp16) {
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, kb};
  return encode(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

// rows[i]: boxes of 16 (i + 1) rows x kb column blocks (tiles of up to 192 rows).
bool make_gemm_rows(GemmMaps* g, const void* ptr, uint64_t rows, uint64_t cols, uint32_t kb, bool fp16) {
  for (int i = 0; i < 12; ++i)
    if (!make_rows_map(&g->rows[i], ptr, rows, cols, 16u * (i + 1), kb, fp16)) return false;
  g->a = g->rows[0];
  g->a2 = g->rows[0];
  return true;
}

// Both fp16 planes of the hidden rows [2, rows, cols] as (64 columns, rows, plane, cols / 64):
// one box brings a tile's leading and remainder rows for kb column blocks, [kb][plane][row][64].
bool make_gemm_planes(GemmMaps* g, const void* ptr, uint64_t rows, uint64_t cols, uint32_t kb) {
  for (int i = 0; i < 12; ++i) {
    const cuuint64_t dims[4] = {64, rows, 2, cols / 64};
    const cuuint64_t strides[3] = {cols * 2, rows * cols * 2, 128};
    const cuuint32_t box[4] = {64, 16u * (i + 1), 2, kb};
    if (!encode(&g->rows[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  g->a = g->rows[0];
  g->a2 = g->rows[0];
  return true;
}

// The down region of every expert as u64 words: codes (256 words, m block, (K block, half),
// expert) and scale/bias (64 words, m block, K block, expert); one box covers kb K blocks of one
// m block (see dn_code_offset / dn_sb_offset).
bool make_down_weight_maps(GemmMaps* g, const uint8_t* packed, const PackedLayout& P, const moe_dims& d, uint32_t kb) {
  const uint64_t DM = d.d / kBlockRows, KBD = d.inter / kGroup, E1 = (uint64_t)d.n_experts + 1;
  const uint8_t* codes = packed + P.gu_bytes;
  const uint8_t* sb = codes + dn_sb_offset(0, 0, (int)DM, (int)KBD);
  const cuuint64_t cdims[4] = {kHalfBytes / 8, DM, 2 * KBD, E1};
  const cuuint64_t cstr[3] = {kHalfBytes, DM * kHalfBytes, P.expert_stride};
  const cuuint32_t cbox[4] = {kHalfBytes / 8, 1, 2 * kb, 1};
  const cuuint64_t sdims[4] = {kSBBytes / 8, DM, KBD, E1};
  const cuuint64_t sstr[3] = {kSBBytes, DM * kSBBytes, P.expert_stride};
  const cuuint32_t sbox[4] = {kSBBytes / 8, 1, kb, 1};
  return encode(&g->a, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, codes, cdims, cstr, cbox, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode(&g->a2, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, sb, sdims, sstr, sbox, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

bool moe::make_decode_down_maps(DecodeMaps* m, const uint8_t* packed, const moe_dims& d) {
  const PackedLayout P = packed_layout(d);
  const uint64_t DM = d.d / kBlockRows, KBD = d.inter / kGroup, E1 = (uint64_t)d.n_experts + 1;
  const uint32_t pieces = KBD * 2 < 16 ? (uint32_t)KBD * 2 : 16u;  // I is a multiple of 128: >= 4
  const uint8_t* codes = packed + P.gu_bytes;
  const uint8_t* sb = codes + dn_sb_offset(0, 0, (int)DM, (int)KBD);
  const cuuint64_t cdims[4] = {kHalfBytes / 8, DM, 2 * KBD, E1};
  const cuuint64_t cstr[3] = {kHalfBytes, DM * kHalfBytes, P.expert_stride};
  const cuuint32_t cbox[4] = {16 * 16 / 8, 1, pieces, 1};
  const cuuint64_t sdims[4] = {kSBBytes / 8, DM, KBD, E1};
  const cuuint64_t sstr[3] = {kSBBytes, DM * kSBBytes, P.expert_stride};
  const cuuint32_t sbox[4] = {16 * 4 / 8, 1, pieces / 2, 1};
  return encode(&m->codes, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, codes, cdims, cstr, cbox, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode(&m->sb, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, sb, sdims, sstr, sbox, CU_TENSOR_MAP_SWIZZLE_NONE);
}

namespace {

int check_ws(void* ws, size_t ws_bytes, const moe_dims& d, int T) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 128)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < ws_layout(d, T).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

int check_out(const moe_route_out* o) {
  if (!o) return MOE_OK;
  const void* ps[] = {o->logits, o->topk_idx, o->topk_w, o->counts, o->offsets, o->perm,
                      o->inv_perm, o->tile_map, o->n_tiles, o->hidden};
  for (const void* p : ps)
    if (!aligned(p, 16)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

struct Ws {
  uint8_t* base;
  WsLayout L;
  template <class T>
  T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

int copy_out(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (!dst || bytes == 0) return MOE_OK;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

RouteParams route_params(const moe_dims& d, const float* logits, int T, const Ws& w, float* yacc, const uint16_t* x,
                         int tile_rows, int ksplit) {
  RouteParams p;
  p.logits = logits;
  p.topk_idx = w.at<int32_t>(w.L.topk_idx);
  p.topk_w = w.at<float>(w.L.topk_w);
  p.chunk_counts = w.at<int32_t>(w.L.chunk_counts);
  p.totals = w.at<int32_t>(w.L.totals);
  p.counts = w.at<int32_t>(w.L.counts);
  p.offsets = w.at<int32_t>(w.L.offsets);
  p.perm = w.at<int32_t>(w.L.perm);
  p.inv_perm = w.at<int32_t>(w.L.inv_perm);
  p.row_tw = w.at<int2>(w.L.row_tw);
  p.tile_map = w.at<int32_t>(w.L.tile_map);
  p.tile_row0 = w.at<int32_t>(w.L.tile_row0);
  p.n_tiles = w.at<int32_t>(w.L.n_tiles);
  p.tile_rows = tile_rows;
  p.ksplit = ksplit;
  p.yacc = yacc;
  p.x = x;
  p.x16 = w.at<uint16_t>(w.L.x16);
  p.hdr = w.at<WsHeader>(w.L.header);
  p.T = T;
  p.E = d.n_experts;
  p.k = d.top_k;
  p.d = d.d;
  p.n_chunks = w.L.n_chunks;
  p.chunk = w.L.chunk;
  return p;
}

// Routing on top of logits already in the workspace (or caller-given): top-k, histogram, scan,
// scatter and block map. `yacc` non-NULL also zeroes the combine accumulator rows.
// `x` non-NULL also writes its fp16 copy (the expert GEMMs' operand) into the workspace.
// ksplit: the router GEMM's K slices whose partial logits the top-k kernel sums (1: final logits).
int run_route(const moe_dims& d, const float* logits, int T, const Ws& w, float* yacc, const uint16_t* x,
              cudaStream_t s, int tile_rows, int ksplit) {
  return launch_route(route_params(d, logits, T, w, yacc, x, tile_rows, ksplit), s) == cudaSuccess ? MOE_OK
                                                                                                  : MOE_ERR_CUDA;
}

// The host round trip the GPU-resident routing removes (ablation): after the top-k kernel, the
// selection is copied to the host and the stream synchronised; the host computes the histogram,
// the exclusive scan, the stable scatter and the block map exactly as the device kernels define
// them and copies them back; then the fp16 rows are placed as usual.
int run_route_host(const moe_dims& d, const float* logits, int T, const Ws& w, float* yacc, const uint16_t* x,
                   cudaStream_t s, int tile_rows, int ksplit) {
  const RouteParams p = route_params(d, logits, T, w, yacc, x, tile_rows, ksplit);
  if (launch_route_topk(p, s) != cudaSuccess || launch_route_streams(p, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int E = d.n_experts, k = d.top_k, A = T * k;
  std::vector<int32_t> idx(A), counts(E, 0), offsets(E + 1, 0), perm(A), inv(A), tile_map, tile_row0;
  std::vector<float> wt(A);
  std::vector<int2> row_tw(A);
  if (cudaMemcpyAsync(idx.data(), p.topk_idx, (size_t)A * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(wt.data(), p.topk_w, (size_t)A * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int a = 0; a < A; ++a) ++counts[std::min(std::max(idx[a], 0), E - 1)];
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> next(offsets.begin(), offsets.end() - 1);
  for (int a = 0; a < A; ++a) {  // stable: ascending assignment within each expert
    const int pos = next[std::min(std::max(idx[a], 0), E - 1)]++;
    perm[pos] = a;
    inv[a] = pos;
    int32_t wbits;
    std::memcpy(&wbits, &wt[a], 4);
    row_tw[pos] = make_int2(a / k, wbits);
  }
  for (int e = 0; e < E; ++e)
    for (int r = 0; r < counts[e]; r += tile_rows) {
      tile_map.insert(tile_map.end(), {e, r, std::min(tile_rows, counts[e] - r)});
      tile_row0.push_back(offsets[e] + r);
    }
  const int32_t n_tiles = (int32_t)tile_row0.size();
  int st = cudaMemcpyAsync(p.counts, counts.data(), (size_t)E * 4, cudaMemcpyHostToDevice, s) |
           cudaMemcpyAsync(p.offsets, offsets.data(), (size_t)(E + 1) * 4, cudaMemcpyHostToDevice, s) |
           cudaMemcpyAsync(p.perm, perm.data(), (size_t)A * 4, cudaMemcpyHostToDevice, s) |
           cudaMemcpyAsync(p.inv_perm, inv.data(), (size_t)A * 4, cudaMemcpyHostToDevice, s) |
           cudaMemcpyAsync(p.row_tw, row_tw.data(), (size_t)A * 8, cudaMemcpyHostToDevice, s) |
           cudaMemcpyAsync(p.n_tiles, &n_tiles, 4, cudaMemcpyHostToDevice, s);
  if (n_tiles)
    st |= cudaMemcpyAsync(p.tile_map, tile_map.data(), tile_map.size() * 4, cudaMemcpyHostToDevice, s) |
          cudaMemcpyAsync(p.tile_row0, tile_row0.data(), tile_row0.size() * 4, cudaMemcpyHostToDevice, s);
  if (st != cudaSuccess) return MOE_ERR_CUDA;
  // pageable host buffers: wait for the copies before the vectors go out of scope
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_route_rows(p, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int run_router_gemm(const moe_layer* L, const uint16_t* x, int T, const Ws& w, cudaStream_t s) {
  const moe_dims& d = L->dims;
  GemmMaps maps;
  if (!make_gemm_rows(&maps, x, T, d.d, gemm_kb_per_stage(kModeRouter), false) ||
      !make_rows_map(&maps.a, L->router_w, d.n_experts, d.d, kBlockRows, gemm_kw_per_stage(kModeRouter), false))
    return MOE_ERR_CUDA;
  GemmParams p = {};
  p.b_kb = gemm_kb_per_stage(kModeRouter);
  p.w_kb = gemm_kw_per_stage(kModeRouter);
  p.ksplit = router_split(d, T);
  p.k_blocks = d.d / kGroup / p.ksplit;
  p.m_tiles = (d.n_experts + kBlockRows - 1) / kBlockRows;
  p.logits = w.at<float>(w.L.logits);
  p.router_bias = L->router_bias;
  p.hdr = w.at<WsHeader>(w.L.header);
  p.T = T;
  p.k = d.top_k;
  p.E = d.n_experts;
  p.d = d.d;
  p.inter = d.inter;
  const int rt = router_tile_rows();
  const int grid = ((T + rt - 1) / rt) * p.m_tiles * p.ksplit;
  return launch_gemm(kModeRouter, p, &maps, grid, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int copy_route_out(const moe_dims& d, int T, const Ws& w, const moe_route_out* o, cudaStream_t s) {
  if (!o) return MOE_OK;
  const size_t A = (size_t)T * d.top_k, E = d.n_experts;
  int st = MOE_OK;
  st |= copy_out(o->logits, w.base + w.L.logits, (size_t)T * E * 4, s);
  st |= copy_out(o->topk_idx, w.base + w.L.topk_idx, A * 4, s);
  st |= copy_out(o->topk_w, w.base + w.L.topk_w, A * 4, s);
  st |= copy_out(o->counts, w.base + w.L.counts, E * 4, s);
  st |= copy_out(o->offsets, w.base + w.L.offsets, (E + 1) * 4, s);
  st |= copy_out(o->perm, w.base + w.L.perm, A * 4, s);
  st |= copy_out(o->inv_perm, w.base + w.L.inv_perm, A * 4, s);
  st |= copy_out(o->tile_map, w.base + w.L.tile_map,
                 (size_t)max_routed_tiles(T, d.top_k, d.n_experts, prefill_tile_rows(d, T)) * 12, s);
  st |= copy_out(o->n_tiles, w.base + w.L.n_tiles, 4, s);
  return st ? MOE_ERR_CUDA : MOE_OK;
}

// moe_decode_timed (mode 0) and moe_decode_diag: argument checks, parameter block, launch.
int decode_common(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_route_out* out, void* ws,
                  size_t ws_bytes, moe_stream_t stream, void* const* events, int mode) {
  int st = check_layer(layer, true);
  if (st) return st;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_MISALIGNED;
  if (layer->dims.d > kDecodeMaxD) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((st = check_out(out)) || (st = check_ws(ws, ws_bytes, layer->dims, 1))) return st;
  const moe_dims& d = layer->dims;
  Ws w{static_cast<uint8_t*>(ws), ws_layout(d, 1)};
  const PackedLayout P = packed_layout(d);
  DecodeParams p;
  p.x = x;
  p.router_w = layer->router_w;
  p.router_bias = layer->router_bias;
  p.packed = static_cast<const uint8_t*>(layer->packed);
  p.expert_stride = P.expert_stride;
  p.gu_bytes = P.gu_bytes;
  p.logits = w.at<float>(w.L.logits);
  p.topk_idx = w.at<int32_t>(w.L.topk_idx);
  p.topk_w = w.at<float>(w.L.topk_w);
  p.partials = nullptr;
  p.hrec = w.at<uint8_t>(w.L.dec_part);
  p.y = y;
  p.hdr = w.at<WsHeader>(w.L.header);
  p.d = d.d;
  p.E = d.n_experts;
  p.k = d.top_k;
  p.inter = d.inter;
  p.T = 1;
  DecodeMaps maps;
  if (!make_decode_down_maps(&maps, p.packed, d)) return MOE_ERR_CUDA;
  if (launch_decode(p, maps, stream, events, mode) != cudaSuccess) return MOE_ERR_CUDA;
  if (!out) return MOE_OK;
  st = copy_out(out->logits, p.logits, (size_t)d.n_experts * 4, stream);
  st |= copy_out(out->topk_idx, p.topk_idx, (size_t)d.top_k * 4, stream);
  st |= copy_out(out->topk_w, p.topk_w, (size_t)d.top_k * 4, stream);
  return st ? MOE_ERR_CUDA : MOE_OK;
}
}  // namespace

extern "C" {

size_t moe_packed_bytes(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return packed_layout(*dims).total;
}

int moe_pack_weights(const moe_dims* dims, moe_q4_view gate, moe_q4_view up, moe_q4_view down, moe_q4_view sh_gate,
                     moe_q4_view sh_up, moe_q4_view sh_down, void* packed_out, moe_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  const moe_q4_view v[6] = {gate, up, down, sh_gate, sh_up, sh_down};
  for (const moe_q4_view& m : v) {
    if (!m.q || !m.scale || !m.bias) return MOE_ERR_INVALID_ARG;
    if (!aligned(m.q, 16) || !aligned(m.scale, 2) || !aligned(m.bias, 2)) return MOE_ERR_MISALIGNED;
  }
  if (!packed_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(packed_out, 128)) return MOE_ERR_MISALIGNED;
  return launch_pack(*dims, v, static_cast<uint8_t*>(packed_out), stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_workspace_bytes(const moe_dims* dims, int32_t max_tokens) {
  if (check_dims(dims) != MOE_OK || max_tokens < 1 || max_tokens > kMaxTokens) return 0;
  return ws_layout(*dims, max_tokens).total;
}

int moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < sizeof(WsHeader)) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 128)) return MOE_ERR_MISALIGNED;
  return cudaMemsetAsync(ws, 0, sizeof(WsHeader), stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int32_t moe_tile_rows(void) { return kTileRows; }

int32_t moe_prefill_tile_rows(const moe_dims* dims, int32_t T) {
  if (check_dims(dims) != MOE_OK || T < 1) return 0;
  return prefill_tile_rows(*dims, T);
}

int moe_route(const moe_layer* layer, const uint16_t* x, const float* logits_in, int32_t T, moe_route_out* out,
              void* ws, size_t ws_bytes, moe_stream_t stream) {
  int st = check_layer(layer, logits_in == nullptr);
  if (st) return st;
  if (T < 1 || T > kMaxTokens) return T < 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  if (!logits_in && !x) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(logits_in, 16)) return MOE_ERR_MISALIGNED;
  if ((st = check_out(out)) || (st = check_ws(ws, ws_bytes, layer->dims, T))) return st;
  const moe_dims& d = layer->dims;
  Ws w{static_cast<uint8_t*>(ws), ws_layout(d, T)};
  const float* logits = w.at<float>(w.L.logits);
  if (logits_in) {
    if (cudaMemcpyAsync(w.at<float>(w.L.logits), logits_in, (size_t)T * d.n_experts * 4, cudaMemcpyDeviceToDevice,
                        stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if ((st = run_router_gemm(layer, x, T, w, stream))) {
    return st;
  }
  if ((st = run_route(d, logits, T, w, nullptr, nullptr, stream, prefill_tile_rows(d, T),
                       logits_in ? 1 : router_split(d, T))))
    return st;
  return copy_route_out(d, T, w, out, stream);
}

// The prefill sequence. arm: 0 the product path; MOE_PREFILL_ARM_HOST_ROUTING the block map built
// on the host after a synchronisation; MOE_PREFILL_ARM_TILE32 block-map tiles of 32 rows for the
// wide GEMM configuration; MOE_PREFILL_ARM_DENSE the selected experts' weights expanded into `aux`
// first; MOE_PREFILL_ARM_WIDE_TILES / MOE_PREFILL_ARM_NARROW_TILES one GEMM configuration at any
// T; kArmReadProbe the read-only probes in place of the two grouped GEMMs (y = 0).
constexpr int kArmReadProbe = 100;

static int prefill_impl(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, moe_route_out* out,
                        void* ws, size_t ws_bytes, moe_stream_t stream, void* const* events, int arm,
                        void* aux = nullptr) {
  int st = check_layer(layer, true);
  if (st) return st;
  if (T < 1 || !x || !y) return MOE_ERR_INVALID_ARG;
  if (T > kMaxTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_MISALIGNED;
  if ((st = check_out(out)) || (st = check_ws(ws, ws_bytes, layer->dims, T))) return st;
  const moe_dims& d = layer->dims;
  Ws w{static_cast<uint8_t*>(ws), ws_layout(d, T)};
  const PackedLayout P = packed_layout(d);
  float* yacc = w.at<float>(w.L.yacc);
  uint16_t* hidden = w.at<uint16_t>(w.L.hidden);
  const int A = T * d.top_k;

  // 1. router logits (tensor cores), 2. top-k + grouping (+ zero the combine accumulator)
  if (record_event(events, 0, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = run_router_gemm(layer, x, T, w, stream))) return st;
  if (record_event(events, 1, stream) != cudaSuccess) return MOE_ERR_CUDA;
  // block-map tile height and GEMM configuration: narrow (32-row tiles, deeper rings) while the
  // experts average few rows, else wide (tiles of up to 192 rows)
  const int tile_rows = arm == MOE_PREFILL_ARM_TILE32        ? kMinTileRows
                        : arm == MOE_PREFILL_ARM_WIDE_TILES   ? kTileRows
                        : arm == MOE_PREFILL_ARM_NARROW_TILES ? kNarrowTileRows
                                                              : prefill_tile_rows(d, T);
  const bool narrow = tile_rows == kNarrowTileRows && arm != MOE_PREFILL_ARM_TILE32 && arm != MOE_PREFILL_ARM_DENSE;
  if (arm == MOE_PREFILL_ARM_HOST_ROUTING) {
    if ((st = run_route_host(d, w.at<float>(w.L.logits), T, w, yacc, x, stream, tile_rows, router_split(d, T))))
      return st;
  } else if ((st = run_route(d, w.at<float>(w.L.logits), T, w, yacc, x, stream, tile_rows, router_split(d, T)))) {
    return st;
  }

  // 3. gate|up grouped GEMM + SwiGLU -> hidden; 4. down grouped GEMM + weighted combine -> yacc.
  // Every tensor map is built with the stage sizes of the configuration that reads it (a box
  // wider than the kernel's stage would overrun its shared memory; launch_gemm checks the match).
  const bool dense = arm == MOE_PREFILL_ARM_DENSE;
  const int mode_gu = dense ? kModeGateUpDense : narrow ? kModeGateUpNarrow : kModeGateUp;
  const int mode_dn = dense ? kModeDownDense : narrow ? kModeDownNarrow : kModeDown;
  GemmMaps x_maps, h_maps;
  if (!make_gemm_rows(&x_maps, w.at<uint16_t>(w.L.x16), (uint64_t)A + T, d.d, gemm_kb_per_stage(mode_gu), true) ||
      !make_gemm_planes(&h_maps, hidden, (uint64_t)A + T, d.inter, gemm_kb_per_stage(mode_dn)) ||
      (!dense && !make_down_weight_maps(&h_maps, static_cast<const uint8_t*>(layer->packed), P, d,
                                        gemm_kw_per_stage(mode_dn))))
    return MOE_ERR_CUDA;
  GemmParams p = {};
  p.packed = static_cast<const uint8_t*>(layer->packed);
  p.expert_stride = P.expert_stride;
  p.tile_map = w.at<int32_t>(w.L.tile_map);
  p.tile_row0 = w.at<int32_t>(w.L.tile_row0);
  p.n_tiles = w.at<int32_t>(w.L.n_tiles);
  p.row_tw = w.at<int2>(w.L.row_tw);
  p.hidden = hidden;
  p.yacc = yacc;
  p.hdr = w.at<WsHeader>(w.L.header);
  p.T = T;
  p.k = d.top_k;
  p.E = d.n_experts;
  p.d = d.d;
  p.inter = d.inter;
  p.hidden_rows = A + T;
  p.tile_rows = tile_rows;
  p.b_kb = gemm_kb_per_stage(mode_gu);
  p.w_kb = gemm_kw_per_stage(mode_gu);
  const int tiles = max_routed_tiles(T, d.top_k, d.n_experts, tile_rows) + (T + tile_rows - 1) / tile_rows;

  if (dense) {  // expand the selected experts' weights, then dense GEMMs on them
    uint16_t* dgu = static_cast<uint16_t*>(aux);
    uint16_t* ddn = dgu + dense_gu_bytes(d) / 2;
    if (launch_dense_dequant(d, p.packed, w.at<int32_t>(w.L.counts), dgu, ddn, stream) != cudaSuccess ||
        !make_rows_map(&x_maps.a, dgu, (uint64_t)(d.n_experts + 1) * 2 * d.inter, d.d, kBlockRows,
                       gemm_kw_per_stage(kModeGateUpDense), true) ||
        !make_rows_map(&h_maps.a, ddn, (uint64_t)(d.n_experts + 1) * d.d, d.inter, kBlockRows,
                       gemm_kw_per_stage(kModeDownDense), true))
      return MOE_ERR_CUDA;
  }
  p.region_offset = 0;
  p.m_tiles = d.inter / gemm_out_rows(mode_gu);
  p.k_blocks = d.d / kGroup;
  if (record_event(events, 2, stream) != cudaSuccess) return MOE_ERR_CUDA;
  const bool probe = arm == kArmReadProbe;
  if ((probe ? launch_gemm_read_probe(mode_gu, p, &x_maps, tiles * p.m_tiles, stream)
             : launch_gemm(mode_gu, p, &x_maps, tiles * p.m_tiles, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;

  p.region_offset = P.gu_bytes;
  p.m_tiles = d.d / kBlockRows;
  p.k_blocks = d.inter / kGroup;
  p.b_kb = gemm_kb_per_stage(mode_dn);
  p.w_kb = gemm_kw_per_stage(mode_dn);
  if (record_event(events, 3, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if ((probe ? launch_gemm_read_probe(mode_dn, p, &h_maps, tiles * p.m_tiles, stream)
             : launch_gemm(mode_dn, p, &h_maps, tiles * p.m_tiles, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;

  // 5. fp32 accumulator -> bf16 output
  if (record_event(events, 4, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_cast(yacc, y, (size_t)T * d.d, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (record_event(events, 5, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = copy_route_out(d, T, w, out, stream))) return st;
  if (out && out->hidden) return copy_out(out->hidden, hidden, 2 * ((size_t)A + T) * d.inter * 2, stream);
  return MOE_OK;
}

int moe_prefill_timed(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, moe_route_out* out,
                      void* ws, size_t ws_bytes, moe_stream_t stream, void* const* events) {
  return prefill_impl(layer, x, T, y, out, ws, ws_bytes, stream, events, 0);
}

int moe_prefill(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, moe_route_out* out, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
  return prefill_impl(layer, x, T, y, out, ws, ws_bytes, stream, nullptr, 0);
}

size_t moe_prefill_ablation_aux_bytes(const moe_dims* dims, int arm) {
  if (check_dims(dims) != MOE_OK || arm != MOE_PREFILL_ARM_DENSE) return 0;
  return dense_gu_bytes(*dims) + dense_dn_bytes(*dims);
}

int moe_prefill_ablation(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, int arm, void* ws,
                         size_t ws_bytes, void* aux, size_t aux_bytes, moe_stream_t stream) {
  if (arm != MOE_PREFILL_ARM_HOST_ROUTING && arm != MOE_PREFILL_ARM_TILE32 && arm != MOE_PREFILL_ARM_DENSE &&
      arm != MOE_PREFILL_ARM_WIDE_TILES && arm != MOE_PREFILL_ARM_NARROW_TILES)
    return MOE_ERR_INVALID_ARG;
  if (arm == MOE_PREFILL_ARM_DENSE) {
    int st = check_layer(layer, true);
    if (st) return st;
    if (!aux) return MOE_ERR_INVALID_ARG;
    if (!aligned(aux, 128)) return MOE_ERR_MISALIGNED;
    if (aux_bytes < moe_prefill_ablation_aux_bytes(&layer->dims, arm)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  }
  return prefill_impl(layer, x, T, y, nullptr, ws, ws_bytes, stream, nullptr, arm, aux);
}

int moe_prefill_diag(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, int mode, void* ws,
                     size_t ws_bytes, moe_stream_t stream, void* const* events) {
  if (mode != MOE_PREFILL_DIAG_READ_ONLY) return MOE_ERR_INVALID_ARG;
  return prefill_impl(layer, x, T, y, nullptr, ws, ws_bytes, stream, events, kArmReadProbe);
}

int moe_prefill_chunked(const moe_layer* layer, const uint16_t* x, int64_t T, uint16_t* y, int32_t chunk_tokens,
                        void* ws, size_t ws_bytes, moe_stream_t stream) {
  int st = check_layer(layer, true);
  if (st) return st;
  if (T < 1 || chunk_tokens < 1 || !x || !y) return MOE_ERR_INVALID_ARG;
  if (chunk_tokens > kMaxTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_MISALIGNED;
  const int32_t chunk = (int32_t)std::min<int64_t>(chunk_tokens, T);
  // Workspaces only grow with the token count, so the first (largest) chunk's check covers all.
  if ((st = check_ws(ws, ws_bytes, layer->dims, chunk))) return st;
  const size_t d = (size_t)layer->dims.d;
  for (int64_t c = 0; c < T; c += chunk) {
    const int32_t n = (int32_t)std::min<int64_t>(chunk, T - c);
    if ((st = prefill_impl(layer, x + c * d, n, y + c * d, nullptr, ws, ws_bytes, stream, nullptr, 0))) return st;
  }
  return MOE_OK;
}

int moe_decode_batch(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, moe_route_out* out, void* ws,
                     size_t ws_bytes, moe_stream_t stream) {
  int st = check_layer(layer, true);
  if (st) return st;
  if (!x || !y || T < 1) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_MISALIGNED;
  const moe_dims& d = layer->dims;
  if (T > kMaxDecodeBatch || d.d > kBatchMaxD) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 1) return decode_common(layer, x, y, out, ws, ws_bytes, stream, nullptr, 0);  // the batch-1 chain
  if ((st = check_out(out)) || (st = check_ws(ws, ws_bytes, d, T))) return st;
  Ws w{static_cast<uint8_t*>(ws), ws_layout(d, T)};
  const PackedLayout P = packed_layout(d);
  DecodeParams p;
  p.x = x;
  p.router_w = layer->router_w;
  p.router_bias = layer->router_bias;
  p.packed = static_cast<const uint8_t*>(layer->packed);
  p.expert_stride = P.expert_stride;
  p.gu_bytes = P.gu_bytes;
  p.logits = w.at<float>(w.L.logits);
  p.topk_idx = w.at<int32_t>(w.L.topk_idx);
  p.topk_w = w.at<float>(w.L.topk_w);   // followed by room for the distinct-expert list (T*k + 1 ints)
  p.partials = w.at<float>(w.L.dec_part);
  p.hrec = nullptr;
  p.y = y;
  p.hdr = w.at<WsHeader>(w.L.header);
  p.d = d.d;
  p.E = d.n_experts;
  p.k = d.top_k;
  p.inter = d.inter;
  p.T = T;
  if (launch_decode_batch(p, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (!out) return MOE_OK;
  st = copy_out(out->logits, p.logits, (size_t)T * d.n_experts * 4, stream);
  st |= copy_out(out->topk_idx, p.topk_idx, (size_t)T * d.top_k * 4, stream);
  st |= copy_out(out->topk_w, p.topk_w, (size_t)T * d.top_k * 4, stream);
  return st ? MOE_ERR_CUDA : MOE_OK;
}

int moe_decode_timed(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_route_out* out, void* ws,
                     size_t ws_bytes, moe_stream_t stream, void* const* events) {
  return decode_common(layer, x, y, out, ws, ws_bytes, stream, events, 0);
}

int moe_decode_diag(const moe_layer* layer, const uint16_t* x, uint16_t* y, void* ws, size_t ws_bytes, int mode,
                    moe_stream_t stream) {
  if (mode != MOE_DECODE_DIAG_NO_MATH && mode != MOE_DECODE_DIAG_READ_ONLY) return MOE_ERR_INVALID_ARG;
  return decode_common(layer, x, y, nullptr, ws, ws_bytes, stream, nullptr,
                       mode == MOE_DECODE_DIAG_NO_MATH ? kDecodeDiagNoMath : kDecodeDiagReadOnly);
}


int moe_decode(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_route_out* out, void* ws, size_t ws_bytes,
               moe_stream_t stream) {
  return moe_decode_timed(layer, x, y, out, ws, ws_bytes, stream, nullptr);
}

int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < sizeof(WsHeader)) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 128)) return MOE_ERR_MISALIGNED;
  return launch_wait_timeout_selftest(static_cast<WsHeader*>(ws), stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_read_device_status(void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int bits = 0;
  WsHeader* h = static_cast<WsHeader*>(ws);
  if (cudaMemcpy(&bits, &h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(&h->status, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  for (int code = MOE_ERR_NONFINITE; code <= MOE_ERR_OUT_OF_RANGE; ++code)
    if (bits & status_bit(code)) return code;
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or copy failed";
    case MOE_ERR_NONFINITE: return "non-finite router logit";
    case MOE_ERR_DEVICE_TIMEOUT: return "bounded device wait gave up";
    case MOE_ERR_OUT_OF_RANGE: return "activation outside the fp16 operand range";
    default: return "unknown status";
  }
}

}  // extern "C"
