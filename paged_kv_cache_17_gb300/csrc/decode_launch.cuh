// decode_launch.cuh -- launch of one decode-kernel instantiation (shared by the TUs that
// instantiate the bf16 and the E4M3 variants, and by the C-ABI layer that picks one).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "decode_kernel.cuh"
#include "decode_mma.cuh"

namespace pkv {

// Consumer warps and ring depth of each variant: 4 consumer warps + 1 producer warp,
// and as many stages as fit in 64 KiB (4..16), so that two to three CTAs share an SM.
template <int D, bool FP8>
struct DecodeShape {
  static constexpr int kNWC = 4;
  static constexpr int kTile = 16 * D * (FP8 ? 1 : 2);
  static constexpr int kStagesRaw = 65536 / (2 * kTile);
  static constexpr int kStages = kStagesRaw < 4 ? 4 : (kStagesRaw > 16 ? 16 : kStagesRaw);
};

struct DecodeLaunchInfo {
  int threads;
  int smem_bytes;
  int tile_area_bytes;  // bytes usable by the cross-partition merge weights
};

template <int D, int G, bool FP8, bool CAS>
DecodeLaunchInfo decode_launch_info() {
  using S = DecodeShape<D, FP8>;
  using C = DecodeCfg<D, G, FP8, S::kNWC, S::kStages>;
  return DecodeLaunchInfo{C::kThreads, C::kSmemBytes, C::kTilesBytes};
}

template <int D, int G, bool FP8, bool CAS>
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, dim3 grid,
                          cudaStream_t stream, int device) {
  using S = DecodeShape<D, FP8>;
  using C = DecodeCfg<D, G, FP8, S::kNWC, S::kStages>;
  auto kern = paged_decode_kernel<D, G, FP8, S::kNWC, S::kStages, CAS>;
  // set once per device; concurrent first calls may both set it (the call is idempotent)
  static std::atomic<bool> configured[64] = {};
  if (device >= 0 && device < 64 && !configured[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[device].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

// The tensor-core form: same grid and launch, 2 consumer warps and a 32 KiB ring of K and V
// tiles (bf16: 4 stages at D = 128; E4M3: 8), six CTAs per SM (shared-memory limit).  bf16
// measured against 4/8, 2/6, 1/2 and 1/4 (warps/stages) on the 8B-shaped, 70B-shaped and
// short-suffix steps; E4M3 against 4 warps (fork decode 127.0 against 94.2 us), 1 warp,
// and 16 or 64 KiB rings.
template <int D, bool FP8>
struct MmaShape {
  static constexpr int kNWC = 2;
  static constexpr int kRingTile = FP8 ? 16 * D : 16 * D * 2;
  static constexpr int kStages = 32768 / (2 * kRingTile);
};

template <int D, int G, bool FP8, bool CAS>
DecodeLaunchInfo decode_mma_launch_info() {
  using S = MmaShape<D, FP8>;
  using C = MmaCfg<D, G, FP8, S::kNWC, S::kStages>;
  return DecodeLaunchInfo{C::kThreads, C::kSmemBytes, C::kTilesBytes};
}

template <int D, int G, bool FP8, bool CAS>
cudaError_t launch_decode_mma(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream, int device) {
  using S = MmaShape<D, FP8>;
  using C = MmaCfg<D, G, FP8, S::kNWC, S::kStages>;
  auto kern = paged_decode_mma_kernel<D, G, FP8, S::kNWC, S::kStages, CAS>;
  // set once per device; concurrent first calls may both set it (the call is idempotent)
  static std::atomic<bool> configured[64] = {};
  if (device >= 0 && device < 64 && !configured[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[device].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

#define PKV_DECLARE_DECODE_MMA(D, G, FP8, CAS)                                                              \
  extern template DecodeLaunchInfo decode_mma_launch_info<D, G, FP8, CAS>();                                \
  extern template cudaError_t launch_decode_mma<D, G, FP8, CAS>(const CUtensorMap&, const CUtensorMap&,    \
                                                                const DecodeParams&, dim3, cudaStream_t, int);
#define PKV_DEFINE_DECODE_MMA(D, G, FP8, CAS)                                                        \
  template DecodeLaunchInfo decode_mma_launch_info<D, G, FP8, CAS>();                                \
  template cudaError_t launch_decode_mma<D, G, FP8, CAS>(const CUtensorMap&, const CUtensorMap&,    \
                                                         const DecodeParams&, dim3, cudaStream_t, int);
#define PKV_FOR_EACH_GROUP_MMA(M, D, FP8, CAS) M(D, 1, FP8, CAS) M(D, 2, FP8, CAS) M(D, 4, FP8, CAS) M(D, 8, FP8, CAS)
#define PKV_FOR_EACH_MMA(M)                                                                          \
  PKV_FOR_EACH_GROUP_MMA(M, 64, false, false) PKV_FOR_EACH_GROUP_MMA(M, 128, false, false)          \
  PKV_FOR_EACH_GROUP_MMA(M, 64, false, true) PKV_FOR_EACH_GROUP_MMA(M, 128, false, true)            \
  PKV_FOR_EACH_GROUP_MMA(M, 64, true, false) PKV_FOR_EACH_GROUP_MMA(M, 128, true, false)            \
  PKV_FOR_EACH_GROUP_MMA(M, 64, true, true) PKV_FOR_EACH_GROUP_MMA(M, 128, true, true)
PKV_FOR_EACH_MMA(PKV_DECLARE_DECODE_MMA)

// Explicit instantiations live in decode_bf16.cu / decode_e4m3.cu (plain) and
// cascade_bf16.cu / cascade_e4m3.cu (cascade variants).
#define PKV_DECLARE_DECODE(D, G, FP8, CAS)                                                              \
  extern template DecodeLaunchInfo decode_launch_info<D, G, FP8, CAS>();                                \
  extern template cudaError_t launch_decode<D, G, FP8, CAS>(const CUtensorMap&, const CUtensorMap&,    \
                                                            const DecodeParams&, dim3, cudaStream_t, int);
#define PKV_DEFINE_DECODE(D, G, FP8, CAS)                                                        \
  template DecodeLaunchInfo decode_launch_info<D, G, FP8, CAS>();                                \
  template cudaError_t launch_decode<D, G, FP8, CAS>(const CUtensorMap&, const CUtensorMap&,    \
                                                     const DecodeParams&, dim3, cudaStream_t, int);

#define PKV_FOR_EACH_GROUP(M, D, FP8, CAS) M(D, 1, FP8, CAS) M(D, 2, FP8, CAS) M(D, 4, FP8, CAS) M(D, 8, FP8, CAS)

PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 64, false, false)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 128, false, false)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 64, true, false)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 128, true, false)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 64, false, true)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 128, false, true)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 64, true, true)
PKV_FOR_EACH_GROUP(PKV_DECLARE_DECODE, 128, true, true)

// merge of the partition (and prefix) records into the output (merge_partitions.cu):
// grid (kv heads, batch), launched right after the decode kernel
cudaError_t launch_merge_partitions(int d, int g, bool fp8, const DecodeParams& p, dim3 grid, cudaStream_t stream);

// copy-on-write block copy (copy_blocks.cu)
cudaError_t launch_copy_blocks(const int64_t* pairs, int64_t num_pairs, int64_t block_bytes, void* k_cache,
                               void* v_cache, int64_t num_blocks, uint32_t* status, int sm_count,
                               cudaStream_t stream);

// read-only checksum pass over the cached K/V (kv_checksum.cu): grid (kv heads, batch,
// partitions), the decode's tables, lengths and partition length
struct ChecksumParams {
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  uint32_t* out;                // [B][Hkv][2], zeroed before the launch
  uint32_t* status;
  int max_blocks;
  int hkv;
  int num_blocks;
  int max_context_len;
  int split_blocks;
};
// copy `bytes` (a multiple of 16) with the SMs; either side may be page-locked host memory
cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, int sm_count, cudaStream_t stream);

cudaError_t launch_kv_checksum(int row_bytes, const CUtensorMap& tk, const CUtensorMap& tv, const ChecksumParams& p,
                               dim3 grid, cudaStream_t stream);

// append (append.cu)
cudaError_t launch_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                          int hkv, int d, bool fp8, void* k_cache, void* v_cache, int64_t pool_slots,
                          const float* scales, uint32_t* status, cudaStream_t stream);

}  // namespace pkv
