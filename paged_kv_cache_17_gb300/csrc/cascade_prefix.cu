// cascade_prefix.cu -- the shared-prefix pass of two-level (cascade) decode attention.
//
// habr.com/ru/articles/1021832, section 7 "Тот самый Cache Read": requests that start with
// the same prompt share that prompt's KV blocks (read through the same physical ids), and
// ml-canon.vercel.app/54-prefix-caching-cacheblend.html, "Идея и механизм": the prefix's
// K/V are identical for every request that shares it.  Decode attention of such a request
// is softmax over (prefix keys) u (own keys); section 3 of the habr article ("Вспомним
// FlashAttention") gives the exact split: attention over a part of the keys yields a
// running max m, a running sum l and an unnormalised output, and parts combine with the
// rescale exp(m_part - m_total).  So the prefix part is computed once for all the
// requests that share it: queries (every member sequence x every query head of kv head h)
// against the prefix keys is a dense [rows x prefix] contraction, done here on the tensor
// cores (mma.sync bf16 -> fp32); each request's own blocks are handled by the decode
// kernel, which merges these partial results as extra partitions.
//
// CTA = 4 warps = 64 query rows (row r: member r / G of prefix p, query head h*G + r % G),
// one kv head h, one split (a run of whole prefix blocks).  K and V arrive by TMA in
// 64-key stages (four 16-token blocks), 128-byte-swizzled so that ldmatrix reads them
// without bank conflicts; every warp computes S = Q K^T for its 16 rows, the online
// softmax (log2 units), and O += P V with P taken straight from the S registers.
// E4M3 pools: the raw codes land by TMA in a separate ring and every thread expands its
// share of a stage to fp16 (exact: 3-bit mantissas, exponents within fp16's range) into
// the same swizzled layout, and the products run as fp16 MMAs; q is rounded to fp16 (exact
// for bf16 values of magnitude 2^-14 .. 65504), the K scale goes into the score scale and
// the records carry V / v_scale * 2^-120, the units the decode kernel's E4M3 records use.
#include <cuda.h>
#include <cuda_runtime.h>

#include "cascade.cuh"
#include "mma_ops.cuh"
#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kRowsPerWarp = 16;
constexpr int kWarps = 4;
constexpr int kRowsPerCta = kRowsPerWarp * kWarps;  // 64
constexpr int kStageBlocks = 4;                       // 16-token blocks per stage
constexpr int kStageKeys = kStageBlocks * kBlockSize;  // 64
constexpr int kStages = 3;
constexpr int kBoxBytes = kBlockSize * 128;           // one 16 x 64 bf16 box, swizzled

// Shared address of key row kr (0..63 of a stage) and 16-byte chunk c (8 elements of the
// head dim) in a stage laid out as [block][half][16 rows][128 B], 128-byte swizzled.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int kr, int c) {
  return swz_addr<D>(base, kr, c);
}

}  // namespace

// Shared-memory plan of one variant: the TMA ring (bf16 tiles already in the swizzled
// layout; E4M3 tiles raw), plus for E4M3 one converted stage of fp16 tiles.
template <int D, bool FP8>
struct PrefixSmem {
  static constexpr int kHalves = D / 64;
  static constexpr int kStageBytes = kStageBlocks * kHalves * kBoxBytes;     // one pool, 16-bit
  static constexpr int kRingStage = FP8 ? kStageKeys * D : kStageBytes;     // one pool, as loaded
  static constexpr int kRingBytes = 2 * kStages * kRingStage;
  static constexpr int kConvBytes = FP8 ? 2 * kStageBytes : 0;
  static constexpr int kBarOffset = kRingBytes + kConvBytes;
  static constexpr int kBytes = 1024 + kBarOffset + kStages * 8;  // 1024: alignment slack
  static_assert(kRingStage % 1024 == 0 && kStageBytes % 1024 == 0, "1024-byte aligned stages");
};

template <int D, bool FP8>
__global__ void __launch_bounds__(kWarps * 32) cascade_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                     const __grid_constant__ CUtensorMap tm_v,
                                                                     const PrefixParams p) {
  using SM = PrefixSmem<D, FP8>;
  constexpr int kHalves = SM::kHalves;
  constexpr int kStageBytes = SM::kStageBytes;
  constexpr int kRingStage = SM::kRingStage;
  constexpr int kNT = D / 8;  // n-tiles of the output
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of every box keeps the swizzle pattern aligned with the rows
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + SM::kBarOffset);

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int pfx = blockIdx.z / p.pre_slots;
  const int split = blockIdx.z % p.pre_slots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  pdl_wait();
  // the decode kernel that follows may start now: what it reads before waiting for this
  // grid (the pool after the append) is complete once every CTA is past the wait above
  pdl_launch_dependents();

  const int m0 = p.indptr[pfx], m1 = p.indptr[pfx + 1];
  int members = m1 - m0;
  if (members < 0 || members > p.max_members) {  // the grid covers max_members members
    if (threadIdx.x == 0 && tile == 0 && split == 0 && h == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    members = max(0, min(members, p.max_members));
  }
  const int G = p.group;
  const int rows = members * G;
  if (tile * kRowsPerCta >= rows) return;
  int plen = p.prefix_lens[pfx];
  if (plen < 0 || plen > p.max_prefix_blocks * kBlockSize || (plen & (kBlockSize - 1))) {
    if (threadIdx.x == 0 && tile == 0 && split == 0 && h == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    plen = max(0, min(plen, p.max_prefix_blocks * kBlockSize)) & ~(kBlockSize - 1);
  }
  const int pblocks = plen / kBlockSize;
  const int blk0 = min(pblocks, split * p.split_blocks);
  const int blk1 = min(pblocks, blk0 + p.split_blocks);
  const int nstage = (blk1 - blk0 + kStageBlocks - 1) / kStageBlocks;
  const int32_t* table = p.prefix_tables + static_cast<size_t>(pfx) * p.max_prefix_blocks;

  // ---- this warp's two rows per thread: r = tile*64 + warp*16 + gid (+8)
  int rb[2], rg[2];
  bool rv[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = tile * kRowsPerCta + warp * kRowsPerWarp + gid + 8 * i;
    rv[i] = r < rows;
    const int mem = rv[i] ? r / G : 0;
    rg[i] = rv[i] ? r % G : 0;
    int b = rv[i] ? p.seqs[m0 + mem] : 0;
    if (rv[i] && (b < 0 || b >= p.batch)) {
      set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
      rv[i] = false;
      b = 0;
    }
    rb[i] = b;
  }
  // Q fragments (A operand, row-major 16 x 16 per k-step) straight from global memory
  uint32_t qa[D / 16][4];
  {
    const uint32_t* q0 =
        reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(rb[0]) * p.hq + h * G + rg[0]) * D);
    const uint32_t* q1 =
        reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(rb[1]) * p.hq + h * G + rg[1]) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int w = kk * 8 + tig;  // 32-bit word: elements 16kk + 2tig, +1
      qa[kk][0] = rv[0] ? q0[w] : 0u;
      qa[kk][1] = rv[1] ? q1[w] : 0u;
      qa[kk][2] = rv[0] ? q0[w + 4] : 0u;
      qa[kk][3] = rv[1] ? q1[w + 4] : 0u;
      if constexpr (FP8) {  // bf16 pairs -> fp16 pairs
#pragma unroll
        for (int e = 0; e < 4; ++e) qa[kk][e] = pack_f16(bf16_lo(qa[kk][e]), bf16_hi(qa[kk][e]));
      }
    }
  }

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int i = 0; i < kStages; ++i) mbar_init(&full_bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const uint32_t k_base = smem_u32(smem);
  const uint32_t v_base = k_base + kStages * kRingStage;
  const uint32_t kc_base = k_base + SM::kRingBytes;  // converted stage (E4M3 only)
  const uint32_t vc_base = kc_base + kStageBytes;
  // thread 0 loads stage t (keys [blk0 + 4t, +4) blocks) into ring slot t % kStages; blocks
  // past the split read zeros (a box entirely outside the tensor)
  auto issue = [&](int t) {
    const int st = t % kStages;
    mbar_arrive_expect_tx(&full_bar[st], 2 * kRingStage);
#pragma unroll
    for (int j = 0; j < kStageBlocks; ++j) {
      const int blk = blk0 + t * kStageBlocks + j;
      int row0 = -kBlockSize;
      if (blk < blk1) {
        const int pb = table[blk];
        if (pb >= 0 && pb < p.num_blocks) row0 = pb * kBlockSize;
        else set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
      }
      if constexpr (FP8) {  // one box of 16 rows x D codes per block
        const int off = st * kRingStage + j * kBlockSize * D;
        tma_load_3d(smem + off, &tm_k, 0, h, row0, &full_bar[st]);
        tma_load_3d(smem + kStages * kRingStage + off, &tm_v, 0, h, row0, &full_bar[st]);
      } else {
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) {
          const int off = st * kStageBytes + (j * kHalves + hf) * kBoxBytes;
          tma_load_3d(smem + off, &tm_k, hf * 64, h, row0, &full_bar[st]);
          tma_load_3d(smem + kStages * kStageBytes + off, &tm_v, hf * 64, h, row0, &full_bar[st]);
        }
      }
    }
  };
  int n_issued = 0;  // meaningful in thread 0, the only issuer
  if (threadIdx.x == 0) {
    n_issued = min(kStages, nstage);
    for (int t = 0; t < n_issued; ++t) issue(t);
  }

  float o[kNT][4];
#pragma unroll
  for (int n = 0; n < kNT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sscale = FP8 ? p.score_scale * p.scales[h] : p.score_scale;
  bool ok = true;
  int t_fail = 0;

  for (int t = 0; t < nstage; ++t) {
    t_fail = t;
    const int st = t % kStages;
    if (!__all_sync(kFull, mbar_wait(&full_bar[st], (t / kStages) & 1))) {
      if (lane == 0) set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
      ok = false;
    }
    // a CTA-uniform verdict: thread 0 must not refill a ring slot that some warp gave up on
    ok = __syncthreads_and(ok);
    if (!ok) break;
    uint32_t kb = k_base + st * kStageBytes;
    uint32_t vb = v_base + st * kStageBytes;
    if constexpr (FP8) {
      // expand the raw stage to fp16 tiles: 8 codes -> one swizzled 16-byte chunk
      const uint8_t* rk = smem + st * kRingStage;
      const uint8_t* rvv = smem + kStages * kRingStage + st * kRingStage;
      constexpr int kChunks = kStageKeys * (D / 8);
      for (int ci = threadIdx.x; ci < 2 * kChunks; ci += kWarps * 32) {
        const bool isv = ci >= kChunks;
        const int cj = isv ? ci - kChunks : ci;
        const int kr = cj / (D / 8), c = cj % (D / 8);
        const uint2 raw = *reinterpret_cast<const uint2*>((isv ? rvv : rk) + kr * D + c * 8);
        uint4 h4;
        h4.x = e4m3x2_to_f16x2(static_cast<uint16_t>(raw.x & 0xffffu));
        h4.y = e4m3x2_to_f16x2(static_cast<uint16_t>(raw.x >> 16));
        h4.z = e4m3x2_to_f16x2(static_cast<uint16_t>(raw.y & 0xffffu));
        h4.w = e4m3x2_to_f16x2(static_cast<uint16_t>(raw.y >> 16));
        const uint32_t dst = tile_addr<D>(isv ? vc_base : kc_base, kr, c);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(h4.x), "r"(h4.y), "r"(h4.z),
                     "r"(h4.w)
                     : "memory");
      }
      // the raw slot is read: refill it with stage t + kStages while this stage computes
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0 && t + kStages < nstage) issue(t + kStages), n_issued = t + kStages + 1;
      kb = kc_base;
      vb = vc_base;
    }
    const int nkeys = min(kStageKeys, (blk1 - blk0 - t * kStageBlocks) * kBlockSize);

    // ---- S = Q K^T: 16 rows x 64 keys per warp (8 n-tiles of 8 keys)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const int mi = lane >> 3;
        const int kr = 8 * j + 8 * (mi >> 1) + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tile_addr<D>(kb, kr, 2 * kk + (mi & 1)), b0, b1, b2, b3);
        mma16<FP8>(s[j], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma16<FP8>(s[j + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }
    // ---- online softmax in log2 units; keys past the split are -inf
    float mnew[2] = {mrow[0], mrow[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int key = 8 * j + 2 * tig;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = (key + (e & 1)) < nkeys;
        s[j][e] = in ? s[j][e] * sscale : -INFINITY;
        mnew[e >> 1] = fmaxf(mnew[e >> 1], s[j][e]);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mnew[i] = fmaxf(mnew[i], shfl_xor(mnew[i], 1));
      mnew[i] = fmaxf(mnew[i], shfl_xor(mnew[i], 2));
    }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      // an all -inf row so far keeps alpha 1 (its sums are still zero)
      alpha[i] = (mnew[i] == -INFINITY) ? 1.f : fast_exp2(mrow[i] - mnew[i]);
      mrow[i] = mnew[i];
      lrow[i] *= alpha[i];
    }
#pragma unroll
    for (int n = 0; n < kNT; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    uint32_t pa[4][4];  // P as the A operand of the four 16-key k-steps
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float e0 = fast_exp2(s[j][0] - mrow[0]);
      const float e1 = fast_exp2(s[j][1] - mrow[0]);
      const float e2 = fast_exp2(s[j][2] - mrow[1]);
      const float e3 = fast_exp2(s[j][3] - mrow[1]);
      lrow[0] += e0 + e1;
      lrow[1] += e2 + e3;
      pa[j >> 1][(j & 1) * 2 + 0] = FP8 ? pack_f16(e0, e1) : pack_bf16(e0, e1);
      pa[j >> 1][(j & 1) * 2 + 1] = FP8 ? pack_f16(e2, e3) : pack_bf16(e2, e3);
    }
    // ---- O += P V: four 16-key k-steps x kNT n-tiles of 8 dims
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int n = 0; n < kNT; n += 2) {
        const int mi = lane >> 3;
        const int kr = 16 * kk + 8 * (mi & 1) + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tile_addr<D>(vb, kr, n + (mi >> 1)), b0, b1, b2, b3);
        mma16<FP8>(o[n], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        mma16<FP8>(o[n + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
    if constexpr (FP8) {
      __syncthreads();  // the converted stage is rewritten next
    } else {
      // ---- the slot is read: refill it with stage t + kStages
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0 && t + kStages < nstage) issue(t + kStages), n_issued = t + kStages + 1;
    }
  }
  if (!ok) {
    // let every copy still in flight (stages t_fail .. n_issued-1) land, bounded, before the
    // CTA exits
    if (threadIdx.x == 0)
      for (int t = t_fail; t < n_issued; ++t)
        if (!mbar_wait(&full_bar[t % kStages], (t / kStages) & 1)) break;
    __syncthreads();
    return;
  }

  // ---- the record of each row: m, l (summed over the quad), unnormalised O
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lrow[i] += shfl_xor(lrow[i], 1);
    lrow[i] += shfl_xor(lrow[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!rv[i]) continue;
    const size_t rec = (static_cast<size_t>(rb[i]) * p.hkv + h) * p.rec_slots + split;
    const size_t base = rec * G + rg[i];
    if (tig == 0) {
      p.part_ml[base * 2 + 0] = mrow[i];
      p.part_ml[base * 2 + 1] = lrow[i];
    }
    float* acc = p.part_acc + base * D;
    const float vunit = FP8 ? 7.52316384526264e-37f : 1.0f;  // 2^-120: the decode kernel's E4M3 units
#pragma unroll
    for (int n = 0; n < kNT; ++n)
      *reinterpret_cast<float2*>(acc + 8 * n + 2 * tig) = make_float2(o[n][2 * i] * vunit, o[n][2 * i + 1] * vunit);
  }
}

template <int D, bool FP8>
cudaError_t launch_cascade_prefix(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixParams& p, dim3 grid,
                                  cudaStream_t stream, int device) {
  const int smem = PrefixSmem<D, FP8>::kBytes;
  auto kern = cascade_prefix_kernel<D, FP8>;
  static bool configured[64] = {};
  if (device >= 0 && device < 64 && !configured[device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[device] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

#define PKV_DEFINE_PREFIX(D, FP8)                                                                          \
  template cudaError_t launch_cascade_prefix<D, FP8>(const CUtensorMap&, const CUtensorMap&, const PrefixParams&, \
                                                     dim3, cudaStream_t, int);
PKV_DEFINE_PREFIX(64, false)
PKV_DEFINE_PREFIX(128, false)
PKV_DEFINE_PREFIX(64, true)
PKV_DEFINE_PREFIX(128, true)
#undef PKV_DEFINE_PREFIX

}  // namespace pkv
