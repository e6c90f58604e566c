// Allocation-free batch-1 decode: moe_decode without a caller-supplied workspace.
//
// Some callers cannot allocate device memory themselves: code embedded in a host application
// that owns every device allocation and only lends it input and output buffers, and code that
// forbids device allocation after start-up because cudaMalloc can synchronise the whole device
// and can fail under memory pressure in the middle of serving. For them this entry point runs
// the same decode kernels as moe_decode with its scratch (router logits, the selected experts and
// weights, the expert kernel's per-block SwiGLU records and the status word) held in a fixed
// file-scope device array.
//
// That array lives as long as the library stays loaded, on every device that loads it, and
// every call shares it: two calls that overlap on the GPU (different streams, or different
// host threads) race on it and may return wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

// Largest scratch this entry point can use. A shape needs
//   256 (status) + 4 E + 8 k + 144 (k + 1) I / 32 bytes, each part rounded up to 256;
// d=2048, E=256, k=8, I=512 needs 22 KiB.
constexpr size_t kNoAllocScratchBytes = 512 * 1024;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

struct ScratchLayout {
  size_t header, logits, topk_idx, topk_w, hrec, total;
};

ScratchLayout scratch_layout(const moe_dims& d) {
  ScratchLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
  L.header = take(sizeof(WsHeader));
  L.logits = take((size_t)d.n_experts * 4);
  L.topk_idx = take((size_t)d.top_k * 4);
  L.topk_w = take((size_t)d.top_k * 4);
  L.hrec = take(decode_hrec_bytes(d));
  L.total = o;
  return L;
}

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_decode_noalloc(const moe_layer* layer, const uint16_t* x, uint16_t* y, moe_stream_t stream) {
  // the same checks as moe_decode, then the limits of this variant
  int st = check_layer(layer, true);
  if (st) return st;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_MISALIGNED;
  const moe_dims& d = layer->dims;
  if (d.d > kDecodeMaxD) return MOE_ERR_UNSUPPORTED_SHAPE;
  const ScratchLayout L = scratch_layout(d);
  if (L.total > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;  // shape needs more scratch
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  uint8_t* s = static_cast<uint8_t*>(base);
  // Nothing in the scratch must start at zero: every call writes the logits, the routing and
  // the SwiGLU records before it reads them; the status word is written only on device errors.
  WsHeader* hdr = reinterpret_cast<WsHeader*>(s + L.header);
  const PackedLayout P = packed_layout(d);
  DecodeParams p;
  p.x = x;
  p.router_w = layer->router_w;
  p.router_bias = layer->router_bias;
  p.packed = static_cast<const uint8_t*>(layer->packed);
  p.expert_stride = P.expert_stride;
  p.gu_bytes = P.gu_bytes;
  p.logits = reinterpret_cast<float*>(s + L.logits);
  p.topk_idx = reinterpret_cast<int32_t*>(s + L.topk_idx);
  p.topk_w = reinterpret_cast<float*>(s + L.topk_w);
  p.partials = nullptr;
  p.hrec = s + L.hrec;
  p.y = y;
  p.hdr = hdr;
  p.d = d.d;
  p.E = d.n_experts;
  p.k = d.top_k;
  p.inter = d.inter;
  p.T = 1;
  DecodeMaps maps;
  if (!make_decode_down_maps(&maps, p.packed, d)) return MOE_ERR_CUDA;
  return launch_decode(p, maps, stream, nullptr) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
