/*
 * moe_gb300.h - C ABI of the GB300 (sm_103a) 4-bit quantized Mixture-of-Experts layer forward.
 *
 * The layer (page "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model",
 * agentnative.dev):
 *   - section "Why Qwen3.6-35B-A3B is a weird workload": a router scores E experts, each token
 *     picks top_k of them, and one shared expert sees every token;
 *   - section "Prefill and decode are different problems": prefill runs the expert projections
 *     as matrix-matrix products, batch-1 decode as a bandwidth-bound matrix-vector product;
 *   - section "Prefill: keep routing on the GPU, dequantize in flight": weights are groupwise
 *     affine 4-bit (group 64, one bf16 scale and one bf16 bias per group), dequantized tile by
 *     tile on chip with fp32 accumulation and bf16 output; routing after top-k is histogram,
 *     prefix scan, scatter and block map, all on the GPU with no host round trip;
 *   - section "Decode: minimize bytes per token" (fusion): the expert input projections are
 *     fused with the gate activation, the output projection with the routing scores and the
 *     shared expert.
 *
 * For one token x (d values):
 *   l_e     = W_r[e] . x (+ b_e)                         router logits, fp32
 *   S       = the top_k experts by l (ties -> lower index), w_e = softmax of l over S
 *   FFN_e(x)= W_down_e ( silu(W_gate_e x) * (W_up_e x) ),  silu(z) = z / (1 + exp(-z))
 *   y       = sum_{e in S} w_e FFN_e(x) + FFN_shared(x)
 *
 * Conventions shared by every call:
 *   - Every pointer is a DEVICE pointer to memory the caller owns (allocated, kept alive and
 *     freed by the caller), except where a comment says "host". The library never allocates,
 *     frees or synchronises a stream, except moe_read_device_status (which synchronises).
 *   - Every compute call is asynchronous on `stream` (NULL = the legacy default stream).
 *   - bf16 values are passed as their uint16 bit patterns.
 *   - Alignment: 16 bytes for every device pointer, 128 bytes for `packed` and `ws`.
 *   - Argument errors are returned before anything is launched (MOE_ERR_INVALID_ARG,
 *     MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_MISALIGNED, MOE_ERR_WORKSPACE_TOO_SMALL). A failed
 *     launch returns MOE_ERR_CUDA. Errors detected on the device (non-finite router logits,
 *     a value outside the fp16 operand range, a bounded wait that gave up) are ORed into a
 *     sticky status word inside `ws`; read them with moe_read_device_status. After
 *     MOE_ERR_DEVICE_TIMEOUT the call's outputs are undefined.
 *   - Numerics of prefill: the expert GEMMs take fp16 operands with fp32 accumulation. A
 *     dequantized weight scale*q + bias is one fused multiply-add rounded once to fp16, exact
 *     whenever its exact value has at most 11 significant bits (e.g. bias = -8*scale). bf16 x
 *     converts to fp16 exactly for 2^-14 <= |x| <= 65504 and for zero; smaller magnitudes round
 *     to fp16 subnormals (absolute error at most 2^-25). The SwiGLU output reaches the down
 *     projection as an fp16 pair (about 22 significant bits). Routing weights and the combine are
 *     fp32; y is rounded once to bf16. Decode keeps the weights exact (scale and bias applied in
 *     fp32) and x, h in fp16 operands (h as a leading part and remainder).
 *   - Supported shapes: group == 64, d % 128 == 0, inter % 128 == 0, shared_inter == inter,
 *     1 <= top_k <= 16, top_k <= n_experts <= 1024, 1 <= T <= 65536 (MOE_ERR_UNSUPPORTED_SHAPE).
 *   - State kept across calls: per-process caches set once (the driver entry point that encodes
 *     TMA descriptors, the SM count of the device, the kernels' shared-memory attributes) and,
 *     for moe_decode_noalloc only, a fixed device array; no call result depends on an earlier
 *     call. Calls on different streams with different workspaces may run concurrently
 *     (moe_decode_noalloc excepted: see there).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(MOE_BUILD) && defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object type as cudaStream_t / CUstream. */
typedef struct CUstream_st* moe_stream_t;

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer where one is required, T < 1, ...         */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* dims outside the supported set listed above            */
  MOE_ERR_MISALIGNED = 3,         /* a pointer breaks the alignment rule above              */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,/* ws_bytes < moe_workspace_bytes(dims, T)                */
  MOE_ERR_CUDA = 5,               /* a CUDA launch or copy failed                           */
  MOE_ERR_NONFINITE = 6,          /* device: a router logit was NaN or infinite             */
  MOE_ERR_DEVICE_TIMEOUT = 7,     /* device: a bounded wait inside a kernel gave up         */
  MOE_ERR_OUT_OF_RANGE = 8        /* device: a value outside what the fp16 operands of the expert
                                     GEMMs hold: an activation (x or a SwiGLU output) with
                                     |v| > 65504, or (prefill) a nonzero scale or bias below
                                     2^-14 in magnitude or with 15*|scale| + |bias| > 65504  */
};

/* Layer dimensions. `group` is the quantization group along the input dimension (64). */
typedef struct moe_dims {
  int32_t d;             /* hidden size                                  */
  int32_t n_experts;     /* routed experts E                             */
  int32_t top_k;         /* experts picked per token                     */
  int32_t inter;         /* routed-expert intermediate size I            */
  int32_t shared_inter;  /* shared-expert intermediate size (== inter)   */
  int32_t group;         /* quantization group (== 64)                   */
} moe_dims;

/*
 * One groupwise-affine 4-bit matrix W[rows, cols] in the canonical (MLX affine) layout,
 * cols = input dimension (page: section "Setup", "MLX affine 4-bit checkpoint with group
 * size 64"; section "Prefill: keep routing on the GPU, dequantize in flight"):
 *   q      uint32[rows, cols/8]: code of column c in bits 4*(c%8) of word c/8 (low nibble first)
 *   scale  bf16  [rows, cols/64], bias bf16 [rows, cols/64]
 *   W[r][c] = scale[r][c/64] * code(r, c) + bias[r][c/64],  code in 0..15.
 * Routed experts are stacked: gate/up are [E, I, d], down is [E, d, I] (leading expert axis).
 */
typedef struct moe_q4_view {
  const uint32_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
} moe_q4_view;

/* Bytes of the packed weight buffer written by moe_pack_weights (E routed + 1 shared expert).
 * Returns 0 for unsupported dims. Host-only, no CUDA call. */
MOE_API size_t moe_packed_bytes(const moe_dims* dims);

/*
 * Re-lays the canonical weights of all experts and the shared expert into the library's
 * packed layout (tile-contiguous 128-row x 64-column blocks, nibbles ordered for cheap
 * unpacking, scale and bias interleaved). The values are unchanged: packing is a pure
 * permutation of codes plus a copy of scales and biases.
 * packed_out: device buffer of moe_packed_bytes(dims) bytes, 128-byte aligned, caller-owned.
 * Inputs may be freed once the stream has passed this call.
 */
MOE_API int moe_pack_weights(const moe_dims* dims, moe_q4_view gate, moe_q4_view up, moe_q4_view down,
                     moe_q4_view sh_gate, moe_q4_view sh_up, moe_q4_view sh_down,
                     void* packed_out, moe_stream_t stream);

/* One layer: router weight bf16 [E, d] (row e scores expert e), optional fp32 router bias [E]
 * (NULL = none), and the buffer filled by moe_pack_weights. All device pointers. */
typedef struct moe_layer {
  moe_dims dims;
  const uint16_t* router_w;
  const float* router_bias;
  const void* packed;
} moe_layer;

/*
 * Optional copies of the routing results (every field may be NULL; non-NULL fields receive a
 * device-to-device copy at the end of the call). A = T * top_k assignments, a = t*top_k + j.
 *   logits   fp32 [T, E]
 *   topk_idx int32[T, top_k]  experts of token t, largest logit first, ties -> lower index
 *   topk_w   fp32 [T, top_k]  softmax of the logits restricted to the selected experts
 *   counts   int32[E]         histogram of assignments per expert
 *   offsets  int32[E + 1]     exclusive prefix scan of counts
 *   perm     int32[A]         sorted position p -> assignment a (stable: ascending a within e)
 *   inv_perm int32[A]         assignment a -> sorted position p
 *   tile_map int32[max_tiles, 3] rows (expert, first row within the expert, rows), experts
 *                             ascending, tiles of R = moe_prefill_tile_rows(dims, T) rows;
 *                             max_tiles = min(E, A) + A / R
 *   n_tiles  int32[1]         number of valid tile_map rows
 *   hidden   fp16 [2, A + T, I] (prefill only) SwiGLU outputs h in sorted order as a pair of
 *                             fp16 planes, h = plane0 + plane1 (leading part and remainder);
 *                             rows A + t hold the shared expert on token t
 * Decode (T = 1) fills logits, topk_idx and topk_w only.
 */
typedef struct moe_route_out {
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* tile_map;
  int32_t* n_tiles;
  uint16_t* hidden;
} moe_route_out;

/* Workspace bytes a call with up to max_tokens tokens needs (0 for unsupported dims). The
 * workspace is caller-owned device memory, 128-byte aligned, used only while the stream runs
 * the call; one workspace must not be shared by calls that may overlap on the GPU. Its first
 * 256 bytes hold counters and the sticky status word: zero them once before the first call
 * (moe_workspace_init, or zero-filled allocation); every call leaves the counters at zero. */
MOE_API size_t moe_workspace_bytes(const moe_dims* dims, int32_t max_tokens);

/* Zeroes the counters and the status word of a workspace (asynchronous on `stream`). */
MOE_API int moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Largest block-map tile height (rows of one expert per tile): 192. */
MOE_API int32_t moe_tile_rows(void);

/* Block-map tile height of a T-token moe_route / moe_prefill call, so a checker can rebuild
 * tile_map: 32 while T * top_k <= 24 * n_experts (few rows per expert: the grouped GEMMs run
 * their narrow configuration, with deeper copy rings), else moe_tile_rows(). 0 for unsupported
 * dims or T < 1. */
MOE_API int32_t moe_prefill_tile_rows(const moe_dims* dims, int32_t T);

/*
 * Routing only (section "Prefill: keep routing on the GPU, dequantize in flight"):
 * router logits, top-k with renormalised softmax weights, histogram, exclusive scan, stable
 * scatter and block map, all on the device with no host round trip.
 * x: bf16 [T, d]. logits_in: NULL, or fp32 [T, E] logits to route instead of computing
 * x . W_r^T (+ bias) (x may then be NULL). Results go to the non-NULL fields of `out`.
 */
MOE_API int moe_route(const moe_layer* layer, const uint16_t* x, const float* logits_in, int32_t T,
              moe_route_out* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Prefill forward of one layer on T tokens (sections "Prefill and decode are different
 * problems" and "Prefill: keep routing on the GPU, dequantize in flight"): routing as in
 * moe_route, then the grouped gate/up GEMM with in-tile Q4 dequantization fused with SwiGLU,
 * then the grouped down GEMM fused with the routing-weighted combine and the shared expert.
 * x: bf16 [T, d]; y: bf16 [T, d] (may not alias x). `out` may be NULL.
 */
MOE_API int moe_prefill(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                moe_route_out* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Bounded-chunk prefill (section "Prefill: keep routing on the GPU, dequantize in flight":
 * long prompts run in chunks of bounded size so that temporary activations stay small next to
 * the weights): moe_prefill on rows [c, c + chunk_tokens) of x for c = 0, chunk_tokens, ...,
 * the last chunk ragged, all queued on `stream` in order. Every token's output depends only on
 * its own row, so y is the single-call result for any chunking, up to fp32 summation order (the
 * expert tiles, and with them the order of the GEMMs' K sums, follow the chunk's routing). Only
 * the workspace of one chunk is needed, however long the prompt:
 * ws_bytes >= moe_workspace_bytes(dims, min(chunk_tokens, T)); T may exceed the single-call
 * limit of 65536 tokens.
 * x: bf16 [T, d]; y: bf16 [T, d] (may not alias x). chunk_tokens: 1..65536.
 * Errors (returned before anything is queued): INVALID_ARG for T < 1, chunk_tokens < 1 or a NULL
 * pointer; UNSUPPORTED_SHAPE for chunk_tokens > 65536; the argument errors of moe_prefill.
 * A launch failure in a later chunk returns MOE_ERR_CUDA with the earlier chunks queued.
 */
MOE_API int moe_prefill_chunked(const moe_layer* layer, const uint16_t* x, int64_t T, uint16_t* y,
                                int32_t chunk_tokens, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Prefill ablations: the three design choices the page measures one at a time (section "Prefill:
 * keep routing on the GPU, dequantize in flight": in-tile dequantization +77.4% and GPU-resident
 * routing +89% at 512 tokens, 32-row tiles +13.2% at 2K tokens), each undone in an otherwise
 * unchanged moe_prefill, so that the benchmark can time what each buys on this GPU, plus the two
 * GEMM configurations moe_prefill chooses between, each forced. Arguments, checks and results as
 * moe_prefill (no routing outputs); `arm`:
 *   MOE_PREFILL_ARM_HOST_ROUTING  after the top-k kernel the selection is copied to the host and
 *                                 the stream is synchronised; the host computes the histogram,
 *                                 scan, stable scatter and block map and copies them back (the
 *                                 round trip the GPU-resident routing removes). This arm
 *                                 synchronises `stream` and allocates host memory; it cannot be
 *                                 captured in a CUDA graph.
 *   MOE_PREFILL_ARM_TILE32        block-map tiles of 32 rows in the wide GEMM configuration
 *                                 (fixed narrow tiles, as on the page, instead of tiles as tall
 *                                 as the expert's rows allow); the workspace of
 *                                 moe_workspace_bytes holds any tiling.
 *   MOE_PREFILL_ARM_WIDE_TILES    the wide GEMM configuration (tiles of up to moe_tile_rows()
 *                                 rows) whatever the token count.
 *   MOE_PREFILL_ARM_NARROW_TILES  the narrow GEMM configuration (32-row tiles, deeper weight,
 *                                 activation and dequantized-operand rings) whatever the token
 *                                 count. moe_prefill picks one of the two by
 *                                 moe_prefill_tile_rows; these two arms time the other.
 *   MOE_PREFILL_ARM_DENSE         materialised dequantization: the weights of every selected
 *                                 expert and of the shared expert are first expanded to fp16
 *                                 (scale * q + bias rounded once, the values the in-tile path
 *                                 computes) into `aux`, then the grouped GEMMs (wide
 *                                 configuration, moe_prefill's block map) read those dense
 *                                 weights instead of the packed codes. aux: device buffer of at
 *                                 least moe_prefill_ablation_aux_bytes(dims, arm) bytes, 128-byte
 *                                 aligned (NULL and 0 for the other arms).
 * MOE_ERR_INVALID_ARG for another arm or a missing aux buffer, MOE_ERR_WORKSPACE_TOO_SMALL for a
 * short one.
 */
#define MOE_PREFILL_ARM_HOST_ROUTING 1
#define MOE_PREFILL_ARM_TILE32 2
#define MOE_PREFILL_ARM_DENSE 3
#define MOE_PREFILL_ARM_WIDE_TILES 4
#define MOE_PREFILL_ARM_NARROW_TILES 5
MOE_API size_t moe_prefill_ablation_aux_bytes(const moe_dims* dims, int arm);
MOE_API int moe_prefill_ablation(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, int arm,
                                 void* ws, size_t ws_bytes, void* aux, size_t aux_bytes, moe_stream_t stream);

/*
 * Prefill diagnostic: the read-rate ceiling of the two grouped GEMMs (section "What didn't work":
 * a kernel's rate is placed against the fastest sustained read rate of its own access pattern).
 *   MOE_PREFILL_DIAG_READ_ONLY  moe_prefill with each grouped GEMM replaced by its read-only probe:
 *                               the same grid, work list (router GEMM and routing run as usual),
 *                               packed-weight and activation copies, stage sizes and ring depths,
 *                               every stage released as soon as it has landed; nothing is
 *                               dequantized, multiplied or written, so the hidden rows are left
 *                               as they were and y becomes zeros.
 * Arguments, checks and errors as moe_prefill_timed (no routing outputs; `events` may be NULL, or 6
 * entries recorded at the same kernel boundaries), plus MOE_ERR_INVALID_ARG for an unknown mode.
 */
#define MOE_PREFILL_DIAG_READ_ONLY 1
MOE_API int moe_prefill_diag(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y, int mode,
                             void* ws, size_t ws_bytes, moe_stream_t stream, void* const* events);

/*
 * Batch-1 decode forward (sections "Prefill and decode are different problems" and
 * "Decode: minimize bytes per token"): router GEMV and top-k, then Q4 GEMVs that stream only
 * the top_k selected experts and the shared expert, gate activation fused into the input
 * projections, routing weights and the shared expert fused into the output projection.
 * x: bf16 [1, d]; y: bf16 [1, d]. ws: at least moe_workspace_bytes(dims, 1). `out` may be NULL.
 * Decode supports d <= 3072 (MOE_ERR_UNSUPPORTED_SHAPE otherwise). The kernels are chained with
 * programmatic dependent launch: each loads the static weights it needs (router rows, the
 * shared expert, and in the last kernel the selected experts' down rows) before waiting for the
 * work that precedes it in the stream, so `layer`'s weights must not be written by that
 * preceding work. The result is deterministic (fixed summation order).
 */
MOE_API int moe_decode(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_route_out* out,
               void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Small-batch decode of T = 1..8 tokens at once (page, section "What didn't work": verifying 2 to
 * 5 draft tokens at once, whose rows route to different experts): the router and the selection
 * of every token, then one pass over the union of the experts the T tokens selected (each
 * distinct expert's weights are streamed once and applied to every token that chose it, the
 * tokens filling the columns of the MMAs), the shared expert likewise, and a fixed-order combine
 * per token. Each token's y equals what moe_decode gives for it alone, up to fp32 summation order.
 * x, y: bf16 [T, d]. ws: at least moe_workspace_bytes(dims, T). `out` may be NULL; it receives
 * logits [T, E], topk_idx [T, k] and topk_w [T, k].
 * Supports d <= 2048 and T <= 8 (MOE_ERR_UNSUPPORTED_SHAPE otherwise); INVALID_ARG for T < 1.
 * T = 1 runs moe_decode's kernels (bit-identical to it). Kernels chained by programmatic
 * dependent launch, as moe_decode.
 */
MOE_API int moe_decode_batch(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                             moe_route_out* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Allocation-free batch-1 decode. The paper has no counterpart to this call; it exists for
 * callers that cannot allocate device memory: code embedded in a host application that owns
 * every device allocation and only lends it input and output buffers, and code that must not
 * allocate after start-up because cudaMalloc can synchronise the device and can fail under
 * memory pressure. It computes exactly what moe_decode computes, with the same kernels, but its
 * scratch (logits, selected experts and weights, the expert kernel's per-block SwiGLU records,
 * status) lives in a fixed 512 KiB device array inside the library instead of a caller workspace.
 *   - x, y: bf16 [1, d] device buffers owned by the caller, as for moe_decode.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *   - The 512 KiB array is held on every device that loads the library until the process
 *     exits. A shape needs 256 + 4E + 8k + 144(k+1)I/32 bytes of it (each part rounded up to
 *     256; d=2048, E=256, k=8, I=512 needs 22 KiB); shapes whose scratch does not fit return
 *     MOE_ERR_UNSUPPORTED_SHAPE before anything is launched.
 *   - The first call on a device looks up the array's device address (once per device, with
 *     that device current); make that first call before any stream capture.
 *   - Every call uses the same array, which keeps the last call's contents; each call writes
 *     everything it later reads, so nothing has to start at zero. Calls that overlap on the GPU
 *     (other streams or host threads) race on the array: serialise them.
 *   - Device-side errors (non-finite logits, an activation outside the fp16 range, a bounded
 *     wait that gave up) are not reported by this variant: it has no status word the caller can
 *     read, and y may then be non-finite or wrong. Callers that need these errors use
 *     moe_decode with a workspace and moe_read_device_status. Argument errors are returned as
 *     for moe_decode.
 */
MOE_API int moe_decode_noalloc(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_stream_t stream);

/*
 * Timed variants of moe_prefill and moe_decode for measurement: identical work, plus an event
 * record at each kernel boundary: cudaEventRecordWithFlags(events[i], stream,
 * cudaEventRecordExternal) while `stream` is being captured, so the events become nodes of the
 * CUDA graph captured from the call, and a plain cudaEventRecord otherwise. `events` is a host
 * array of cudaEvent_t (created by the caller with timing enabled); any entry may be NULL.
 *   prefill: events[0] before the router GEMM, [1] before the routing kernels (top-k and
 *            scatter), [2] before the gate/up GEMM, [3] before the down GEMM, [4] before the
 *            output cast, [5] after it (6 entries).
 *   decode:  events[0] before the router GEMV, [1] before the expert kernel (top-k, gate/up
 *            GEMV + SwiGLU), [2] before the down kernel (down GEMVs and the weighted combine),
 *            [3] after it (4 entries). Events between the kernels also stop them from
 *            overlapping through programmatic dependent launch.
 */
MOE_API int moe_prefill_timed(const moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                              moe_route_out* out, void* ws, size_t ws_bytes, moe_stream_t stream,
                              void* const* events);
MOE_API int moe_decode_timed(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_route_out* out,
                             void* ws, size_t ws_bytes, moe_stream_t stream, void* const* events);

/*
 * Decode diagnostics: the two ablations the page uses to locate the decode bound (section
 * "What didn't work": the GEMV's rate against the fastest sustained weight-read rate of its access
 * pattern, and the effect of deleting its arithmetic). Arguments as for moe_decode (no routing
 * outputs); the same checks and error codes, plus MOE_ERR_INVALID_ARG for an unknown mode.
 *   MOE_DECODE_DIAG_NO_MATH    the full kernel chain with the GEMV arithmetic deleted: router,
 *                              top-k, the same weight copies, prefetches, loads and waits; y
 *                              becomes zeros.
 *   MOE_DECODE_DIAG_READ_ONLY  one kernel that copies every expert weight byte the layer reads
 *                              (gate/up and down of experts 0..k-1 and of the shared expert) into
 *                              shared memory, each block waiting for its own; no router, no
 *                              chaining; x and y are not accessed (they must still be valid,
 *                              16-byte aligned pointers).
 */
#define MOE_DECODE_DIAG_NO_MATH 1
#define MOE_DECODE_DIAG_READ_ONLY 2
MOE_API int moe_decode_diag(const moe_layer* layer, const uint16_t* x, uint16_t* y, void* ws, size_t ws_bytes,
                            int mode, moe_stream_t stream);

/*
 * Failure-detection self-test: launches one thread block whose bounded mbarrier wait (the routine
 * the prefill GEMM and decode kernels wait with) is never satisfied. It gives up after about 2e9 SM cycles
 * (roughly one second), records MOE_ERR_DEVICE_TIMEOUT in the sticky status word of `ws`
 * (read it with moe_read_device_status) and returns: no fault, trap or hang, and the context
 * stays usable. ws: at least 256 bytes, 128-byte aligned. Returns INVALID_ARG, MISALIGNED or
 * CUDA synchronously.
 */
MOE_API int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronises `stream`, returns the sticky device status of `ws` (MOE_OK or a device error
 * code) and clears it. */
MOE_API int moe_read_device_status(void* ws, moe_stream_t stream);

/* Static, human-readable name of a status code. */
MOE_API const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
