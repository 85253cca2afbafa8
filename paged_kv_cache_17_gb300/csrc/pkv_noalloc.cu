// pkv_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc when they run a decode step: an allocator that has
// reserved all of the device's memory for itself and hands none out, a serving loop that
// forbids allocation after start-up (cudaMalloc can synchronise the device and stall other
// streams), or a plain C caller with no allocator at hand.  For them this file keeps the
// decode workspace in a fixed array in the library's own device memory, present on every
// GPU that loads the library, so a call needs nothing from the caller beyond its inputs
// and its output.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/pkv.h"

namespace {

// Largest workspace this entry point can serve: 32 MiB per device (for example the
// 8B-shaped step at batch 64 needs under 5 MiB and the 70B-shaped 128K step under 18 MiB).
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Device-side scratch.  In host code this name only stands for the symbol: its device
// address must be obtained with cudaGetSymbolAddress on each device (see scratch_ptr).
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

void* g_ptr[kMaxDevices] = {};
std::mutex g_mu;

// Device address of this device's copy of the scratch array; looked up once per device,
// with that device current.
cudaError_t scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace

// Sets the message pkv_last_error() returns (defined next to it, not exported).
extern "C" void pkv_internal_set_error(const char* msg);

extern "C" pkv_status pkv_paged_decode_attention_noalloc(const pkv_cache_desc* cache, const void* q,
                                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                         const int32_t* context_lens, int32_t batch,
                                                         int32_t num_q_heads, int32_t max_context_len,
                                                         float softmax_scale, void* out, pkv_out_dtype out_dtype,
                                                         pkv_stream_t stream) {
  // Without a usable descriptor, for an empty batch, or when the sizes themselves are
  // refused, the regular entry point (given no workspace) makes the same checks and returns
  // the same status and message as it would for this call; nothing is enqueued.
  auto regular_without_workspace = [&]() {
    return pkv_paged_decode_attention(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                                      max_context_len, softmax_scale, out, out_dtype, nullptr, 0, stream);
  };
  if (!cache || batch == 0) return regular_without_workspace();
  const size_t need = pkv_decode_workspace_size(batch, num_q_heads, cache->num_kv_heads, cache->head_dim,
                                                max_context_len);
  if (need == 0 && pkv_last_error()[0] != '\0') return regular_without_workspace();
  if (need > kScratchBytes) {
    const std::string msg = "this call needs " + std::to_string(need) + " bytes of decode scratch; the "
                            "no-allocation entry point holds at most " + std::to_string(kScratchBytes) +
                            " bytes -- use pkv_paged_decode_attention with a caller-provided workspace";
    pkv_internal_set_error(msg.c_str());
    return PKV_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  cudaError_t e = scratch_ptr(&ws);
  if (e != cudaSuccess) {
    pkv_internal_set_error((std::string("cudaGetSymbolAddress(decode scratch): ") + cudaGetErrorString(e)).c_str());
    return PKV_ERR_CUDA;
  }
  // The scratch keeps whatever the previous call left; the decode needs nothing in it
  // initialised (every record it reads was written by the same call).
  return pkv_paged_decode_attention(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                                    max_context_len, softmax_scale, out, out_dtype, ws, kScratchBytes, stream);
}
