// Internal layouts and kernel parameter blocks of the GB300 Q4 MoE library (host + device).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

// ------------------------------------------------------------------------------------------
// Packed expert layout.
//
// Every quantized matrix is cut into blocks of 128 output rows x 64 input columns (one
// quantization group wide). Inside a block, the codes of each row are two 16-byte halves
// (columns 0..31 and 32..63, four uint32 words each, word w = columns 8w..8w+7) and each row has
// one (scale, bias) bf16 pair (scale in the low half). Inside a word, the code of column c sits
// in nibble slot (c/2) + 4*(c%2): slots 0..3 hold columns 0,2,4,6 and slots 4..7 hold columns
// 1,3,5,7, so (word >> 4i) & 0x000F000F yields the columns (2i, 2i+1) as the two 16-bit halves.
//
// The blocks are stored so that both consumers read long contiguous runs:
//   gate|up region (I/128 row blocks m, 4 quarters q of 32 rows, d/64 column blocks kb):
//     entry (m, q, kb) at ((m*4 + q) * KB + kb) * 2304 holds the gate rows of the quarter
//     (half 0: 32 x 16 B, half 1: 32 x 16 B, scale/bias: 32 x 4 B = 1152 B) then the up rows
//     (1152 B). A decode block reading 32 intermediate rows streams one contiguous
//     KB * 2304-byte run; a prefill CTA reading a 128-row block gathers 4 quarter entries.
//   down region (I/64 column groups kbd, 2 halves hd, d/128 row blocks mm):
//     codes (kbd, hd, mm) at ((kbd*2 + hd) * DM + mm) * 2048: 128 rows x 16 B;
//     then scale/bias (kbd, mm) at codes_end + (kbd * DM + mm) * 512: 128 rows x 4 B.
//     A decode block reading a 32-column slice of W_down streams DM * 2048 contiguous bytes
//     of codes plus DM * 512 bytes of scales; a prefill CTA gathers 2 halves + 1 scale run.
// Per expert (routed e = 0..E-1, then the shared expert at index E): gate|up then down.
// ------------------------------------------------------------------------------------------
constexpr int kGroup = 64;          // quantization group (input columns per block)
constexpr int kBlockRows = 128;     // output rows per block (= MMA M)
constexpr int kHalfBytes = kBlockRows * 16;          // 2048: codes of one 32-column half
constexpr int kCodeBytes = 2 * kHalfBytes;           // 4096
constexpr int kBlockBytes = kCodeBytes + kBlockRows * 4;  // 4608
constexpr int kQuarterRows = 32;
constexpr int kGUMat = 2 * kQuarterRows * 16 + kQuarterRows * 4;  // 1152: one matrix's quarter
constexpr int kGUQuarter = 2 * kGUMat;                             // 2304: gate + up quarter
constexpr int kSBBytes = kBlockRows * 4;                           // 512
constexpr int kTileRows = 192;      // block-map tile height (max MMA N of the prefill GEMMs)
constexpr int kMinTileRows = 32;    // smallest tile height a call may ask for (fixed-tile ablation)
constexpr int kNarrowTileRows = 32; // tile height of the narrow GEMM configuration (few rows per expert)
constexpr int kNarrowMaxAvgRows = 24;  // narrow configuration while T * k <= this * E
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTokens = 65536;

__host__ __device__ inline size_t gu_offset(int m, int q, int kb, int KB) {
  return ((size_t)(m * 4 + q) * KB + kb) * kGUQuarter;
}
__host__ __device__ inline size_t dn_code_offset(int kbd, int hd, int mm, int DM) {
  return ((size_t)(kbd * 2 + hd) * DM + mm) * kHalfBytes;
}
__host__ __device__ inline size_t dn_sb_offset(int kbd, int mm, int DM, int KBI) {
  return (size_t)KBI * 2 * DM * kHalfBytes + ((size_t)kbd * DM + mm) * kSBBytes;
}

struct PackedLayout {
  size_t gu_bytes;       // gate|up region of one expert
  size_t down_bytes;     // down region of one expert
  size_t expert_stride;  // bytes per expert
  size_t total;          // (E + 1) experts
};

inline PackedLayout packed_layout(const moe_dims& d) {
  PackedLayout L;
  L.gu_bytes = (size_t)(d.inter / kBlockRows) * (d.d / kGroup) * 2 * kBlockBytes;
  L.down_bytes = (size_t)(d.d / kBlockRows) * (d.inter / kGroup) * kBlockBytes;
  L.expert_stride = L.gu_bytes + L.down_bytes;
  L.total = L.expert_stride * (size_t)(d.n_experts + 1);
  return L;
}

// ------------------------------------------------------------------------------------------
// Workspace layout (one call with T tokens, A = T*k assignments). Every region 256-aligned.
// The header words must be zero before the first use of a workspace; the kernels return the
// counters to zero at the end of every call, and the status word is sticky until read.
// ------------------------------------------------------------------------------------------
constexpr int kMaxRouterSplit = 4;  // K slices of the prefill router GEMM at most (partial logits)
constexpr int kRouteChunk = 64;     // tokens per routing chunk (histogram / scatter CTA), at least
constexpr int kMaxRouteChunks = 64; // chunks per call at most (a scatter CTA sums its predecessors' counts)

// Tokens per routing chunk of a T-token call: 64, or more (a multiple of 64) so that a call has at
// most kMaxRouteChunks chunks. Non-decreasing in T, so the workspace grows with the token count.
inline int route_chunk_tokens(int T) {
  const int per = (T + kMaxRouteChunks - 1) / kMaxRouteChunks;
  return per <= kRouteChunk ? kRouteChunk : (per + kRouteChunk - 1) / kRouteChunk * kRouteChunk;
}

struct WsHeader {
  int status;        // sticky device status (moe_status codes ORed as bits 1 << code)
  unsigned ticket;   // last-CTA ticket of the routing histogram kernel
  int pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header size");

struct WsLayout {
  size_t header, logits, topk_idx, topk_w, chunk_counts, totals, counts, offsets, perm,
      inv_perm, row_tw, tile_map, tile_row0, n_tiles, x16, hidden, yacc, dec_part, total;
  int n_chunks, chunk, max_tiles;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Decode: one expert-kernel CTA per (selected or shared expert, 32 intermediate rows); each
// writes an h record (the 32 SwiGLU values of its rows as fp16 leading parts and remainders, and
// their sums over the two code-base column classes) that the down kernel reads. The small-batch
// decode writes partial output rows of d floats instead, summed in a fixed order.
constexpr int kDecPartRows = 32;
constexpr int kHRecBytes = 144;     // 32 fp16 leading parts, 32 fp16 remainders, 2 floats, padding
constexpr int kDecodeMaxD = 3072;   // the expert kernel keeps all its weight slices in smem
constexpr int kMaxDecodeBatch = 8;  // tokens of one moe_decode_batch call (the MMA's 8 columns)
constexpr int kBatchMaxD = 2048;    // the batch expert kernel also keeps 8 tokens' x in smem
inline int decode_parts(const moe_dims& d) { return (d.top_k + 1) * (d.inter / kDecPartRows); }
inline size_t decode_partial_bytes(const moe_dims& d) { return (size_t)decode_parts(d) * d.d * 4; }
inline size_t decode_hrec_bytes(const moe_dims& d) { return (size_t)decode_parts(d) * kHRecBytes; }

// Upper bound on the routed block-map tiles of T tokens with tiles of tile_rows rows: every hit
// expert has a ragged last tile, and the whole tiles are at most A / tile_rows.
inline int max_routed_tiles(int T, int k, int E, int tile_rows = kTileRows) {
  long long A = (long long)T * k;
  return (int)((A < E ? A : E) + A / tile_rows);
}

// Block-map tile height of a T-token prefill (and of moe_route): the narrow GEMM configuration's
// 32-row tiles while the experts average at most kNarrowMaxAvgRows rows, else tiles of up to 192.
inline int prefill_tile_rows(const moe_dims& d, int T) {
  return (long long)T * d.top_k <= (long long)kNarrowMaxAvgRows * d.n_experts ? kNarrowTileRows : kTileRows;
}

inline WsLayout ws_layout(const moe_dims& d, int T) {
  WsLayout L;
  const size_t A = (size_t)T * d.top_k, E = (size_t)d.n_experts;
  L.chunk = route_chunk_tokens(T);
  L.n_chunks = (T + L.chunk - 1) / L.chunk;
  L.max_tiles = max_routed_tiles(T, d.top_k, d.n_experts, kMinTileRows);  // room for any tile height
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
  L.header = take(sizeof(WsHeader));
  L.logits = take((size_t)kMaxRouterSplit * T * E * 4);  // [K slice][T][E]: slice 0 the logits
  L.topk_idx = take(A * 4);
  L.topk_w = take(A * 4 + (A + 1) * 4);  // + the batch decode's distinct-expert list
  L.chunk_counts = take((size_t)L.n_chunks * E * 4);
  L.totals = take(E * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(A * 4);
  L.inv_perm = take(A * 4);
  L.row_tw = take(A * 8);
  L.tile_map = take((size_t)L.max_tiles * 3 * 4);
  L.tile_row0 = take((size_t)L.max_tiles * 4);
  L.n_tiles = take(4);
  L.x16 = take((A + T) * (size_t)d.d * 2);             // fp16 x: A expert-sorted rows, then T token rows
  L.hidden = take(2 * (A + T) * (size_t)d.inter * 2);  // SwiGLU rows: fp16 leading part, fp16 remainder
  L.yacc = take((size_t)T * d.d * 4);
  L.dec_part = take(decode_partial_bytes(d) * (size_t)(T < kMaxDecodeBatch ? T : kMaxDecodeBatch));
  L.total = o;
  return L;
}

// Status bits stored in WsHeader::status.
__host__ __device__ inline int status_bit(int code) { return 1 << code; }

// ------------------------------------------------------------------------------------------
// Kernel parameter blocks
// ------------------------------------------------------------------------------------------
struct RouteParams {
  const float* logits;   // [T, E] fp32 (computed or caller-given); with ksplit > 1 the router's
                         // K slices [ksplit][T][E], summed by the top-k kernel into slice 0
  int32_t* topk_idx;     // [T, k]
  float* topk_w;         // [T, k]
  int32_t* chunk_counts; // [n_chunks, E]
  int32_t* totals;       // [E] assignments per expert, summed over the chunks (zeroed by the top-k kernel)
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E + 1]
  int32_t* perm;         // [A]
  int32_t* inv_perm;     // [A]
  int2* row_tw;          // [A] (token, routing weight bits) of each expert-sorted row
  int32_t* tile_map;     // [max_tiles, 3]
  int32_t* tile_row0;    // [max_tiles] sorted row of each tile's first row (offsets[expert] + row)
  int32_t* n_tiles;      // [1]
  int tile_rows;         // block-map tile height (kTileRows, or smaller for the fixed-tile ablation)
  float* yacc;           // [T, d] zeroed by the top-k kernel (NULL: skip)
  const uint16_t* x;     // [T, d] bf16 input (NULL: no conversion)
  uint16_t* x16;         // [A + T, d] fp16 x: rows A.. in token order (top-k kernel), rows 0..A-1 in
                         // expert-sorted order (row gather after the scatter)
  WsHeader* hdr;
  int T, E, k, d, n_chunks, chunk;  // chunk: tokens per routing chunk
  int ksplit;                        // router K slices: the top-k kernel sums their partial logits
};

// kModeGateUpDense / kModeDownDense: the materialised-dequantization ablation, the same GEMMs on
// fp16 weights expanded beforehand into a dense buffer (gate/up: [E + 1][I / 64][128 rows: 64 gate
// then the same 64 features' up][d]; down: [E + 1][d][I]).
// kModeGateUpNarrow / kModeDownNarrow: the same GEMMs for tiles of at most kNarrowTileRows rows,
// with the shared memory and tensor memory the wide tiles' operands take given to deeper weight,
// activation and dequantized-operand rings.
enum GemmMode {
  kModeRouter = 0,
  kModeGateUp = 1,
  kModeDown = 2,
  kModeGateUpDense = 3,
  kModeDownDense = 4,
  kModeGateUpNarrow = 5,
  kModeDownNarrow = 6
};

struct GemmParams {
  // weights
  const uint8_t* packed;      // packed experts (gate/up or down modes)
  size_t expert_stride;       // bytes per expert
  size_t region_offset;       // 0 (gate|up) or gu_bytes (down)
  int m_tiles;                // output-row tiles of 128 per expert
  int k_blocks;               // input-column blocks of 64
  // routing
  const int32_t* tile_map;    // [max_tiles, 3]
  const int32_t* tile_row0;   // [max_tiles]
  const int32_t* n_tiles;     // device count of routed tiles
  const int2* row_tw;         // [A] (token, routing weight bits) of each expert-sorted row
  // activations
  uint16_t* hidden;           // [2, A + T, I] fp16: leading part, then remainder (gate/up writes,
                              // down reads both planes via TMA)
  float* yacc;                // [T, d] fp32 combine accumulator (down)
  float* logits;              // [ksplit][T][E] (router): partial logits per K slice
  const float* router_bias;   // [E] or NULL (router)
  WsHeader* hdr;
  int T, k, E, d, inter;
  int tile_rows;              // block-map tile height (shared-expert tiles use the same)
  int ksplit;                 // router: K slices (k_blocks each); slice s writes logits + s * T * E
  int b_kb, w_kb;             // K blocks per box of the activation / weight tensor maps (launch_gemm
                              // refuses a launch whose maps do not match the mode's stages)
  int hidden_rows;            // A + T: row offset of the remainder plane of `hidden`
};

struct DecodeParams {
  const uint16_t* x;          // [T, d] bf16
  const uint16_t* router_w;   // [E, d] bf16
  const float* router_bias;   // [E] or NULL
  const uint8_t* packed;
  size_t expert_stride, gu_bytes;
  float* logits;              // [T, E]
  int32_t* topk_idx;          // [T, k]
  float* topk_w;              // [T, k]
  float* partials;            // [T, k + 1, I / 32, d] fp32 partial outputs (small-batch decode)
  uint8_t* hrec;              // [k + 1, I / 32] h records of kHRecBytes (batch-1 decode)
  uint16_t* y;                // [T, d] bf16
  WsHeader* hdr;
  int d, E, k, inter;
  int T;                      // tokens: 1 (moe_decode), up to kMaxDecodeBatch (moe_decode_batch)
};

// Argument checks shared by every entry point (csrc/api.cu): supported dims, and a layer's
// pointers (non-NULL where required, 128-byte aligned packed weights, 16-byte aligned router).
bool aligned(const void* p, size_t a);
int check_dims(const moe_dims* d);
int check_layer(const moe_layer* L, bool need_router);

// Launchers (each returns cudaGetLastError()).
cudaError_t launch_wait_timeout_selftest(WsHeader* hdr, cudaStream_t s);
cudaError_t launch_pack(const moe_dims& d, const moe_q4_view* views, uint8_t* packed, cudaStream_t s);
// Expands the packed weights of the experts with counts[e] > 0 and of the shared expert into the
// dense fp16 layouts of the materialised-dequantization ablation (see GemmMode).
size_t dense_gu_bytes(const moe_dims& d);
size_t dense_dn_bytes(const moe_dims& d);
cudaError_t launch_dense_dequant(const moe_dims& d, const uint8_t* packed, const int32_t* counts, uint16_t* dense_gu,
                                 uint16_t* dense_dn, cudaStream_t s);
cudaError_t launch_route(const RouteParams& p, cudaStream_t s);        // all of the routing below
cudaError_t launch_route_topk(const RouteParams& p, cudaStream_t s);   // top-k
cudaError_t launch_route_group(const RouteParams& p, cudaStream_t s);  // histogram, scan, block map, scatter
                                                                       // (+ fp16 x, zero Yacc)
cudaError_t launch_route_streams(const RouteParams& p, cudaStream_t s);  // fp16 x, zero Yacc alone
cudaError_t launch_route_rows(const RouteParams& p, cudaStream_t s);   // expert-sorted fp16 x rows
// Tensor maps of the prefill GEMMs.
//   rows[i]: the activation operand for tiles of 16 (i + 1) rows, box = 64 columns x 16 (i + 1)
//            rows x kSB column blocks: gate/up and router see a row-major [rows, cols] 16-bit
//            matrix as (64 columns, rows, cols / 64); down sees both fp16 planes of the hidden
//            rows as (64 columns, rows, plane, cols / 64). One copy lands as consecutive
//            [rows][64] tiles (128-byte swizzled), a whole tile's rows for several K steps.
//   a:  router mode: the bf16 router weight [E, d] in the 3-D form (box 128 rows);
//       down mode: the packed down codes of every expert as u64 words (256 words, m block,
//       (K block, half), expert), box = one m block x 2 kSW (K block, half) pieces.
//   a2: down mode: the down scale/bias words (64 words, m block, K block, expert).
struct GemmMaps {
  CUtensorMap rows[12];
  CUtensorMap a, a2;
};
cudaError_t launch_gemm(int mode, const GemmParams& p, const GemmMaps* maps, int grid, cudaStream_t s);
// The read-only probe of a gate/up or down GEMM (the Q4 modes): the same grid, work list,
// weight and activation copies and ring depths, each stage released as soon as it lands; no
// dequantization, MMA or epilogue (hidden and yacc are not written).
cudaError_t launch_gemm_read_probe(int mode, const GemmParams& p, const GemmMaps* maps, int grid, cudaStream_t s);
int gemm_kb_per_stage(int mode);  // K blocks that one activation copy covers
int gemm_kw_per_stage(int mode);  // K blocks that one weight stage covers
int gemm_out_rows(int mode);      // output rows of one work item (gate/up: 64 features)
// K slices of the prefill router GEMM for T tokens: more than one only while the token tiles
// leave SMs idle (each slice a CTA of its own; the top-k kernel sums the partial logits).
int router_split(const moe_dims& d, int T);
cudaError_t launch_cast(const float* yacc, uint16_t* y, size_t n, cudaStream_t s);
// mode: 0 the decode path; kDecodeDiagNoMath the same chain with the GEMV arithmetic deleted
// (y = 0); kDecodeDiagReadOnly one kernel that copies every weight the layer reads, alone.
constexpr int kDecodeDiagNoMath = 1, kDecodeDiagReadOnly = 2;
// Tensor maps of the decode down kernel: the down codes of every expert as u64 words (256 words,
// m block, 32-column part, expert), box = the 16 rows (32 words) of one m block for 16 parts; the
// down scale/bias words (64 words, m block, K block, expert), box = the 16 rows (8 words) for 8 K
// blocks.
struct DecodeMaps {
  CUtensorMap codes, sb;
};
bool make_decode_down_maps(DecodeMaps* m, const uint8_t* packed, const moe_dims& d);
cudaError_t launch_decode(const DecodeParams& p, const DecodeMaps& maps, cudaStream_t s, void* const* events,
                          int mode = 0);
// p.T tokens (2..kMaxDecodeBatch): the union of their selected experts is read once.
cudaError_t launch_decode_batch(const DecodeParams& p, cudaStream_t s);

// Records events[i] (if the array and the entry are non-NULL) on the stream: as an external event
// node while the stream is being captured (so the graph records it at replay), else a plain record
// (the external flag is refused outside a capture).
inline cudaError_t record_event(void* const* events, int i, cudaStream_t s) {
  if (!events || !events[i]) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  const cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

}  // namespace moe
