// hfa_noalloc.cu -- the attention step for callers that cannot allocate device memory.
//
// hfa_attention_decode needs a scratch workspace (a status word, one counter per
// (sequence, KV head) and one (m, l, O) record per key chunk) that its caller allocates.
// Some callers cannot allocate at the point where they run attention: a serving engine
// that plans all device memory at start-up and forbids allocation on the request path,
// a plugin whose host application owns the allocator, or code that must not let
// cudaMalloc/cudaFree synchronise the device while other streams are working.
// hfa_attention_decode_noalloc serves them: its scratch is the file-scope array below,
// a fixed 4 MiB that every GPU loading this library holds until the process exits.
//
// Set-up: the first call on each device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress; later calls reuse it.  Make that
// first call before any stream capture.  Each call clears the status word and the
// counters (cudaMemsetAsync on the caller's stream) and then runs the same kernel as
// hfa_attention_decode.  All calls share the one array: calls that overlap on the GPU
// (different streams, no ordering between them) race on it and give wrong results.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "hfa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// device address of g_attn_scratch on the current device (set-up on first use)
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" hfa_status hfa_attention_decode_noalloc(const hfa_attn_desc* d, void* stream,
                                                   const float* q_dev,
                                                   const int32_t* seq_pos_dev,
                                                   const int32_t* seq_pos_host, int batch,
                                                   const void* k_cache_dev,
                                                   const void* v_cache_dev, float* o_dev) {
  char msg[256];
  if (!d || batch < 1) {
    hfa::set_thread_error(!d ? "desc is NULL" : "batch must be >= 1");
    return HFA_EINVAL;
  }
  const size_t need = hfa_attention_workspace_bytes(d, batch);
  if (need == 0) {
    // invalid descriptor or no device: let the workspace entry point report which
    return hfa_attention_decode(d, stream, q_dev, seq_pos_dev, seq_pos_host, batch, k_cache_dev,
                                v_cache_dev, nullptr, 0, o_dev);
  }
  if (need > kStaticScratchBytes) {
    snprintf(msg, sizeof msg,
             "batch %d x %d KV heads needs %zu bytes of scratch; the static scratch of "
             "hfa_attention_decode_noalloc holds %zu bytes (use hfa_attention_decode)",
             batch, d->num_kv_heads, need, kStaticScratchBytes);
    hfa::set_thread_error(msg);
    return HFA_ERANGE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch: %s",
             cudaGetErrorString(e));
    hfa::set_thread_error(msg);
    return HFA_ECUDA;
  }
  // the status word and the per-(sequence, KV head) counters must start at zero
  const size_t head = ((size_t)(batch * d->num_kv_heads + 1) * 4 + 255) / 256 * 256;
  e = cudaMemsetAsync(scratch, 0, head, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "clearing the static scratch: %s", cudaGetErrorString(e));
    hfa::set_thread_error(msg);
    return HFA_ECUDA;
  }
  return hfa_attention_decode(d, stream, q_dev, seq_pos_dev, seq_pos_host, batch, k_cache_dev,
                              v_cache_dev, scratch, kStaticScratchBytes, o_dev);
}
