// kvq_static.cu — decode attention whose scratch lives in a static device array.
//
// kvq_decode_attn keeps its split-K partials in the workspace part of the
// caller's cache buffer.  Some callers cannot provide device memory for that:
// a host runtime whose device memory is planned once up front by another
// component (an inference server's arena, a plugin inside someone else's
// engine) must not call cudaMalloc, and memory it did not plan may not exist.
// This entry point runs the same kernel with its scratch (partials + combine
// tickets) in a fixed-size array compiled into the library.  It allocates
// nothing: no cudaMalloc / cudaFree and no allocating library routine.
#include <cmath>
#include <mutex>
#include <string>

#include "kvq_internal.h"

namespace {

// Largest scratch this entry point can use (every GPU that loads the library
// keeps this array resident until the process exits).
constexpr size_t kStaticScratchBytes = 16u << 20;

// Partials first, then the per-(sequence, kv head) tickets.
static __device__ __align__(256) unsigned char g_kvq_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of the array, per device

// Set-up, once per device, with that device current: the host-side symbol is a
// stand-in, not a device address, so the kernel gets the address from the runtime.
cudaError_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_kvq_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" kvq_status kvq_decode_attn_static(kvq_cache_t C, int layer, const void* q, int q_dtype,
                                             float softmax_scale, float* out, void* stream) {
  if (!C || layer < 0 || layer >= C->cfg.layers) return KVQ_ERR_INVALID_ARG;
  if (!q || !out || (q_dtype != KVQ_F16 && q_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f)) softmax_scale = 1.0f / std::sqrt((float)C->cfg.head_dim);
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  const kvq_config& c = C->cfg;
  const size_t work_bytes = align256(kvq::decode_work_floats(c.batch, c.q_heads, c.head_dim, C->max_chunks) * 4);
  const size_t ticket_bytes = kvq::decode_ticket_words(c.batch, c.kv_heads, C->max_chunks) * 4;
  if (work_bytes + ticket_bytes > kStaticScratchBytes) {
    C->last_error = "kvq_decode_attn_static: needs " + std::to_string(work_bytes + ticket_bytes) +
                    " bytes of scratch, the static array holds " + std::to_string(kStaticScratchBytes);
    return KVQ_ERR_BUFFER_TOO_SMALL;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  void* base = nullptr;
  if (e == cudaSuccess) e = scratch_address(dev, &base);
  if (e != cudaSuccess) {
    C->last_error = cudaGetErrorString(e);
    return KVQ_ERR_CUDA;
  }
  float* work = static_cast<float*>(base);
  uint32_t* tickets = reinterpret_cast<uint32_t*>(static_cast<char*>(base) + work_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The tickets must start at zero.  A completed call leaves them at zero
  // (the merging CTA resets each ticket it used), but the array keeps whatever
  // the last call left, and a call that did not complete (a launch that failed
  // or was aborted) can leave counts behind: clear them on every call.
  e = cudaMemsetAsync(tickets, 0, ticket_bytes, st);
  C->last_launches = 0;
  if (e == cudaSuccess)
    e = kvq::launch_decode_scratch(C, layer, q, q_dtype == KVQ_F32, softmax_scale, out, st, &C->last_launches,
                                   work, tickets);
  if (e != cudaSuccess) {
    C->last_error = cudaGetErrorString(e);
    return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}
