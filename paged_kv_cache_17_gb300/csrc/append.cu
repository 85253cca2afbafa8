// append.cu -- scatter one decode step's new K/V rows into the paged pool.
//
// habr.com/ru/articles/1021832, section 1 "Prefill и Decode": each decode step computes
// K, V for the new token only and appends them to the cache; section 4 "Вспомним
// PagedAttention", worked example: the new token goes to the next slot of the sequence's
// current block (or slot 0 of a freshly allocated block).  The slot of every new token is
// given by the caller's slot mapping (slot = physical block * 16 + offset).
//
// One thread moves one 16-byte piece (8 bf16) of one (token, kv head) row of K and the
// same piece of V.  For an E4M3 pool the piece is divided by the head's scale (IEEE
// binary32 division) and rounded to nearest-even E4M3 with saturation (hardware cvt
// with .satfinite), 8 bytes out.
#include <cuda_runtime.h>

#include "decode_launch.cuh"

namespace pkv {

template <bool FP8>
__global__ void __launch_bounds__(256) paged_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                           const int64_t* __restrict__ slots, int64_t num_tokens,
                                                           int hkv, int pieces_per_row, uint8_t* k_cache,
                                                           uint8_t* v_cache, int64_t pool_slots,
                                                           const float* __restrict__ scales, uint32_t* status) {
  pdl_launch_dependents();  // the decode kernel may start its launch; it waits for us to finish
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_token = static_cast<int64_t>(hkv) * pieces_per_row;
  if (idx >= num_tokens * per_token) return;
  const int64_t t = idx / per_token;
  const int rem = static_cast<int>(idx - t * per_token);
  const int h = rem / pieces_per_row;
  const int c = rem - h * pieces_per_row;
  const int64_t slot = slots[t];
  if (slot < 0) return;  // padding token
  if (slot >= pool_slots) {
    set_flag(status, PKV_DEVFLAG_BAD_SLOT);
    return;
  }
  const int64_t row = slot * hkv + h;  // [block][offset] flattened == slot
  const uint4 kw = k[idx];
  const uint4 vw = v[idx];
  if constexpr (!FP8) {
    reinterpret_cast<uint4*>(k_cache)[row * pieces_per_row + c] = kw;
    reinterpret_cast<uint4*>(v_cache)[row * pieces_per_row + c] = vw;
  } else {
    const float ks = scales[h];
    const float vs = scales[hkv + h];
    reinterpret_cast<uint2*>(k_cache)[row * pieces_per_row + c] = e4m3_quant8(kw, ks);
    reinterpret_cast<uint2*>(v_cache)[row * pieces_per_row + c] = e4m3_quant8(vw, vs);
  }
}

cudaError_t launch_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, int hkv,
                          int d, bool fp8, void* k_cache, void* v_cache, int64_t pool_slots, const float* scales,
                          uint32_t* status, cudaStream_t stream) {
  const int pieces = d / 8;
  const int64_t total = num_tokens * hkv * pieces;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  auto* kk = static_cast<const uint4*>(k);
  auto* vv = static_cast<const uint4*>(v);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  if (fp8)
    return cudaLaunchKernelEx(&cfg, paged_append_kernel<true>, kk, vv, slot_mapping, num_tokens, hkv, pieces, kc, vc,
                              pool_slots, scales, status);
  return cudaLaunchKernelEx(&cfg, paged_append_kernel<false>, kk, vv, slot_mapping, num_tokens, hkv, pieces, kc, vc,
                            pool_slots, scales, status);
}

}  // namespace pkv
