// merge_partitions.cu -- combine the partial results of a split context (and of a shared
// prefix) into the decode output.
//
// habr.com/ru/articles/1021832, section 3 "Вспомним FlashAttention": attention over a set
// of keys split into parts is recovered exactly from each part's running max m, running
// sum l and unnormalised output o: with M the largest m, out = sum 2^(m_j - M) o_j /
// sum 2^(m_j - M) l_j (scores in log2 units).  The decode kernels write one record
// (m, l, o) per context partition (and the prefix pass one per prefix split) and exit;
// this kernel, launched right after them, merges the records of every (sequence, kv head)
// that has more than one partition.  One CTA of up to 8 warps per (kv head, sequence, group of
// query heads), W warps per query head (W grows with the record count, so that a warp
// takes at most about 8 records); every load is issued before its value is needed.  The
// records are taken in record order within a warp, the warps' partial sums are added in
// warp order and the lane sums reduced in a fixed order, so the result does not depend on
// timing.
#include <cuda_runtime.h>

#include <type_traits>

#include "decode_launch.cuh"

namespace pkv {

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(256) merge_partitions_kernel(const DecodeParams p) {
  constexpr int DPL = D / 32;
  constexpr int kBatch = 8;  // records whose outputs one warp loads at a time
  using VecT = typename std::conditional<DPL == 4, float4, float2>::type;
  __shared__ VecT red[8][32];  // the warps' partial sums
  pdl_wait();  // the decode grid (and, through it, a prefix pass) has completed
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int len = p.context_lens[b];
  const int cap = min(p.max_context_len, p.max_blocks * kBlockSize);
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int nblk = (len + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  const int npre = (p.seq_prefix != nullptr && p.seq_prefix[b] >= 0) ? p.pre_slots : 0;
  // one partition and no deferred prefix records: the decode kernel wrote the output itself
  // (CTA-uniform)
  if (nsplit <= 1 && !(p.defer_prefix && npre > 0)) return;
  const int lo = p.pre_slots - npre, hi = p.pre_slots + nsplit;
  const int W = p.merge_warps;          // warps per query head
  const int gl = warp / W, wk = warp % W;
  const int g = blockIdx.z * (8 / W) + gl;
  const bool active = g < G;
  const int gg = active ? g : 0;
  const size_t rec0 = (static_cast<size_t>(b) * p.hkv + h) * p.rec_slots;
  const float* ml = p.part_ml + (rec0 * G + gg) * 2;  // record j: ml[j * G * 2 + {0, 1}]
  const float* acc = p.part_acc + (rec0 * G + gg) * D + lane * DPL;
  auto rec_ml = [&](int j) { return __ldcg(reinterpret_cast<const float2*>(ml + static_cast<size_t>(j) * G * 2)); };
  auto rec_acc = [&](int j) { return __ldcg(reinterpret_cast<const VecT*>(acc + static_cast<size_t>(j) * G * D)); };

  VecT part = VecT{};  // this warp's sum over its records
  float inv = 0.f;
  if (active) {
    // lane k holds (m, l) of records lo + k and lo + 32 + k; the outputs of this warp's first
    // batch (records lo + kBatch * wk ..) are loaded before the max is known
    const float2 none = make_float2(-INFINITY, 0.f);
    const float2 r0 = lo + lane < hi ? rec_ml(lo + lane) : none;
    const float2 r1 = lo + 32 + lane < hi ? rec_ml(lo + 32 + lane) : none;
    VecT v[kBatch];
    const int first = lo + kBatch * wk;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (first + u < hi) v[u] = rec_acc(first + u);
      else v[u] = VecT{};
    }
    float M = fmaxf(r0.x, r1.x);
    for (int j = lo + 64 + lane; j < hi; j += 32) M = fmaxf(M, rec_ml(j).x);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, shfl_xor(M, m));
    float den = 0.f, w0 = 0.f, w1 = 0.f;
    if (M != -INFINITY) {
      if (lo + lane < hi) {
        w0 = fast_exp2(r0.x - M);
        den = fmaf(w0, r0.y, den);
      }
      if (lo + 32 + lane < hi) {
        w1 = fast_exp2(r1.x - M);
        den = fmaf(w1, r1.y, den);
      }
      for (int j = lo + 64 + lane; j < hi; j += 32) {
        const float2 r = rec_ml(j);
        den = fmaf(fast_exp2(r.x - M), r.y, den);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) den += shfl_xor(den, m);
    inv = den > 0.f ? 1.0f / den : 0.f;
    if (M != -INFINITY) {
      for (int j0 = first; j0 < hi; j0 += kBatch * W) {
        if (j0 != first) {
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
            if (j0 + u < hi) v[u] = rec_acc(j0 + u);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u, k = j - lo;  // warp-uniform
          if (j >= hi) break;
          const float w = k < 32 ? __shfl_sync(kFull, w0, k)
                                 : (k < 64 ? __shfl_sync(kFull, w1, k - 32) : fast_exp2(rec_ml(j).x - M));
          if constexpr (DPL == 4) {
            part.x = fmaf(w, v[u].x, part.x);
            part.y = fmaf(w, v[u].y, part.y);
            part.z = fmaf(w, v[u].z, part.z);
            part.w = fmaf(w, v[u].w, part.w);
          } else {
            part.x = fmaf(w, v[u].x, part.x);
            part.y = fmaf(w, v[u].y, part.y);
          }
        }
      }
    }
  }
  if (W > 1) {  // the partial sums of a query head's warps, added in warp order
    red[warp][lane] = part;
    __syncthreads();
    if (wk == 0) {
      for (int k = 1; k < W; ++k) {
        const VecT q = red[warp + k][lane];
        part.x += q.x;
        part.y += q.y;
        if constexpr (DPL == 4) {
          part.z += q.z;
          part.w += q.w;
        }
      }
    }
  }
  if (!active || wk != 0) return;
  float num[DPL];
  num[0] = part.x;
  num[1] = part.y;
  if constexpr (DPL == 4) {
    num[2] = part.z;
    num[3] = part.w;
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
static cudaError_t launch_merge_d(int g, const DecodeParams& p0, dim3 grid, cudaStream_t stream) {
  // W warps per query head: at most about 8 records per warp (more warps for short record
  // lists only left the 8B-shaped step slower)
  DecodeParams p = p0;
  int w = 1;
  while (w < 8 && w * 8 < p.rec_slots) w *= 2;
  p.merge_warps = w;
  grid.z = static_cast<unsigned>((g + 8 / w - 1) / (8 / w));
  // the warps a CTA uses: g * w when that is below 8 (a query group of 4 with one warp per
  // head: 4 warps, so that twice as many CTAs fit an SM)
  const int warps = g * w < 8 ? g * w : 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(32 * warps), 1, 1);
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
