// cascade.cuh -- parameters and launch of the shared-prefix pass of cascade decode.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {

struct PrefixParams {
  const uint16_t* q;             // [B][Hq][D] bf16
  const int32_t* prefix_tables;  // [P][max_prefix_blocks]
  const int32_t* prefix_lens;    // [P], tokens, multiples of 16
  const int32_t* indptr;         // [P + 1]: members of prefix p are seqs[indptr[p] .. indptr[p+1])
  const int32_t* seqs;           // member sequence ids
  float* part_ml;                // records [B][Hkv][rec_slots][G][2]
  float* part_acc;               // records [B][Hkv][rec_slots][G][D]
  uint32_t* status;
  int max_prefix_blocks;
  int max_members;  // grid coverage: members per prefix
  int batch;
  int hq;
  int hkv;
  int group;        // G = Hq / Hkv
  int num_blocks;   // pool size in blocks
  int split_blocks; // prefix blocks per split (a multiple of 4)
  int pre_slots;    // splits per prefix = prefix records per (sequence, kv head)
  int rec_slots;    // records per (sequence, kv head): pre_slots + decode partitions
  float score_scale;  // softmax_scale * log2(e)
  const float* scales;  // [2][Hkv] (E4M3 pools) or nullptr
  const uint8_t* k_codes;  // the pools (read by the mma.sync pass without tensor maps)
  const uint8_t* v_codes;
};


// The prefix pass on the tcgen05 tensor cores (cascade_prefix_tc.cu): 128-row query tiles;
// bf16 pools are read through the 128-byte-swizzled 64-column tensor maps, E4M3 pools
// through the plain ones.
template <int D, bool FP8>
int cascade_prefix_tc_ctas_per_sm(int device);  // CTAs of the pass resident per SM; 0 on error
template <int D, bool FP8>
cudaError_t launch_cascade_prefix_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixParams& p, dim3 grid,
                                     cudaStream_t stream, int device);
#define PKV_DECLARE_PREFIX_TC(D, FP8)                                                                        \
  extern template int cascade_prefix_tc_ctas_per_sm<D, FP8>(int);                                           \
  extern template cudaError_t launch_cascade_prefix_tc<D, FP8>(const CUtensorMap&, const CUtensorMap&,      \
                                                               const PrefixParams&, dim3, cudaStream_t, int);
PKV_DECLARE_PREFIX_TC(64, false)
PKV_DECLARE_PREFIX_TC(128, false)
PKV_DECLARE_PREFIX_TC(64, true)
PKV_DECLARE_PREFIX_TC(128, true)
#undef PKV_DECLARE_PREFIX_TC

// The prefix pass for small member groups of an E4M3 pool on mma.sync
// (cascade_prefix_mma.cu): at most 16 MT query rows per (prefix, kv head), grid.x = 1; the
// warps copy the pool's codes (k_codes / v_codes) into their rings themselves.
template <int D, int MT>
int cascade_prefix_mma_ctas_per_sm(int device);  // CTAs of the pass resident per SM; 0 on error
template <int D, int MT>
cudaError_t launch_cascade_prefix_mma(const PrefixParams& p, dim3 grid, cudaStream_t stream, int device);
#define PKV_DECLARE_PREFIX_MMA(D, MT)                                              \
  extern template int cascade_prefix_mma_ctas_per_sm<D, MT>(int);                 \
  extern template cudaError_t launch_cascade_prefix_mma<D, MT>(const PrefixParams&, dim3, cudaStream_t, int);
PKV_DECLARE_PREFIX_MMA(64, 1)
PKV_DECLARE_PREFIX_MMA(64, 2)
PKV_DECLARE_PREFIX_MMA(128, 1)
PKV_DECLARE_PREFIX_MMA(128, 2)
#undef PKV_DECLARE_PREFIX_MMA

}  // namespace pkv
