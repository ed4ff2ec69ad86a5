// noalloc.cu -- paged_decode_attn_noalloc: paged_decode_attn with its scratch
// workspace taken from a fixed device array compiled into the library, for
// callers that cannot allocate device memory.
//
// Who needs it: some hosts of this library own every byte of device memory
// themselves -- for example a serving runtime that reserves the GPU's memory
// up front and hands out no scratch buffers, or a plug-in that runs inside
// such a runtime -- and so can neither call cudaMalloc nor pass a workspace.
// For them the decode scratch (split-K partials and the batch plan) lives in
// one file-scope __device__ array.  Nothing here calls cudaMalloc, cudaFree or
// any allocating routine.
//
// The array's host-side name is only a stand-in for the symbol; its device
// address comes from cudaGetSymbolAddress with the device current.  A call
// made outside stream capture looks it up again (cheap once the module is
// loaded), so a device reset, after which the module may load at another
// address, leaves no stale pointer behind; a call made while its stream is
// being captured uses the address found by the last uncaptured call on that
// device (or looks it up, if there was none).
#include <mutex>

#include "internal.h"

namespace {

// Capacity of the static scratch.  Every GPU that loads the library keeps
// this much device memory until the process exits.  Enough for GQA batches of
// up to a few thousand (request, kv head) pairs at head dim 128.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device.
kv_status scratch_address(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KV_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone || g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return KV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KV_OK;
}

}  // namespace

extern "C" kv_status paged_decode_attn_noalloc(kv_pool* pool, void* stream, int32_t B,
                                               int32_t num_q_heads, int32_t q_tokens,
                                               const void* q, const int32_t* page_table,
                                               int32_t max_pages_per_req,
                                               const int32_t* seq_lens,
                                               const uint8_t* abort_mask, float sm_scale,
                                               void* out) {
  if (!pool || B < 0) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  kvfp8::DecodeConfig cfg;
  const kv_status shape = kvfp8::decode_config(pool, B, num_q_heads, q_tokens, &cfg);
  if (shape != KV_OK) return shape;
  const size_t need = paged_decode_workspace_size(pool, B, num_q_heads, q_tokens);
  if (need > kStaticScratchBytes) return KV_ERR_UNSUPPORTED;  // batch too large for the array
  void* ws = nullptr;
  const kv_status st = scratch_address(static_cast<cudaStream_t>(stream), &ws);
  if (st != KV_OK) return st;
  // Nothing in the scratch needs clearing: each call's plan kernel rewrites
  // every word of it that the later kernels read.
  return paged_decode_attn(pool, stream, B, num_q_heads, q_tokens, q, page_table,
                           max_pages_per_req, seq_lens, abort_mask, sm_scale, out, ws,
                           kStaticScratchBytes);
}
