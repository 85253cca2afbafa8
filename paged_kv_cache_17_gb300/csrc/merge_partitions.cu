// merge_partitions.cu -- combine the partial results of a split context (and of a shared
// prefix) into the decode output.
//
// habr.com/ru/articles/1021832, section 3 "Вспомним FlashAttention": attention over a set
// of keys split into parts is recovered exactly from each part's running max m, running
// sum l and unnormalised output o: with M the largest m, out = sum 2^(m_j - M) o_j /
// sum 2^(m_j - M) l_j (scores in log2 units).  The decode kernels write one record
// (m, l, o) per context partition (and the prefix pass one per prefix split) and exit;
// this kernel, launched right after them, merges the records of every (sequence, kv head)
// that has more than one partition.  One CTA per (kv head, sequence), one warp per query
// head; the records are taken in record order and the sums reduced in a fixed lane order,
// so the result does not depend on timing.
#include <cuda_runtime.h>

#include "decode_launch.cuh"

namespace pkv {

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(256) merge_partitions_kernel(const DecodeParams p) {
  constexpr int DPL = D / 32;
  pdl_wait();  // the decode grid (and, through it, a prefix pass) has completed
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int len = p.context_lens[b];
  const int cap = min(p.max_context_len, p.max_blocks * kBlockSize);
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int nblk = (len + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  if (nsplit <= 1) return;  // one partition: the decode kernel wrote the output itself
  const int npre = (p.seq_prefix != nullptr && p.seq_prefix[b] >= 0) ? p.pre_slots : 0;
  const int lo = p.pre_slots - npre, hi = p.pre_slots + nsplit;
  const int g = warp;
  if (g >= G) return;
  const size_t rec0 = (static_cast<size_t>(b) * p.hkv + h) * p.rec_slots;
  const float* ml = p.part_ml + (rec0 * G + g) * 2;  // record j: ml[j * G * 2 + {0, 1}]
  const float* acc = p.part_acc + (rec0 * G + g) * D + lane * DPL;

  float M = -INFINITY;
  for (int j = lo + lane; j < hi; j += 32) M = fmaxf(M, __ldcg(ml + static_cast<size_t>(j) * G * 2));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, shfl_xor(M, m));
  float den = 0.f;
  if (M != -INFINITY)
    for (int j = lo + lane; j < hi; j += 32) {
      const float* r = ml + static_cast<size_t>(j) * G * 2;
      den = fmaf(fast_exp2(__ldcg(r) - M), __ldcg(r + 1), den);
    }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) den += shfl_xor(den, m);
  const float inv = den > 0.f ? 1.0f / den : 0.f;

  float num[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) num[i] = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int j = lo; j < hi; ++j) {
      const float w = fast_exp2(__ldcg(ml + static_cast<size_t>(j) * G * 2) - M);
      const float* a = acc + static_cast<size_t>(j) * G * D;
      if constexpr (DPL == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a));
        num[0] = fmaf(w, v.x, num[0]);
        num[1] = fmaf(w, v.y, num[1]);
        num[2] = fmaf(w, v.z, num[2]);
        num[3] = fmaf(w, v.w, num[3]);
      } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(a));
        num[0] = fmaf(w, v.x, num[0]);
        num[1] = fmaf(w, v.y, num[1]);
      }
    }
  }
  float fix = 1.0f;  // E4M3 records carry V * 2^-120 without V's scale
  if constexpr (FP8) fix = p.scales[p.hkv + h];
  const size_t oi = ((static_cast<size_t>(b) * p.hq + h * G + g) * D) + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    float o = num[i] * inv;
    if constexpr (FP8) o = (o * 1152921504606846976.0f) * (fix * 1152921504606846976.0f);  // 2^60 * 2^60
    if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi + i] = o;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[oi + i] = __float2bfloat16_rn(o);
  }
}

template <int D, bool FP8>
static cudaError_t launch_merge_d(int g, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (g) {
    case 1: return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<D, 1, FP8>, p);
    case 2: return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<D, 2, FP8>, p);
    case 4: return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<D, 4, FP8>, p);
    case 8: return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<D, 8, FP8>, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge_partitions(int d, int g, bool fp8, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  if (d == 64) return fp8 ? launch_merge_d<64, true>(g, p, grid, stream) : launch_merge_d<64, false>(g, p, grid, stream);
  return fp8 ? launch_merge_d<128, true>(g, p, grid, stream) : launch_merge_d<128, false>(g, p, grid, stream);
}

}  // namespace pkv
