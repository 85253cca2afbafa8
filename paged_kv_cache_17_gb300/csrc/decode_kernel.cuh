// decode_kernel.cuh -- paged GQA decode attention with split-K over the context.
//
// What it computes (habr.com/ru/articles/1021832, section 3 "Вспомним FlashAttention":
// softmax(q K^T * scale) V, evaluated tile by tile with a running max m, a running sum l
// and the rescale exp(m_old - m_new), which gives the exact result; section 4 "Вспомним
// PagedAttention": K/V live in 16-token blocks scattered in a flat pool, found through a
// per-sequence block table; section 5: the cache layout [blocks][16][kv heads][head dim]).
//
// Work decomposition (one CTA = one (sequence b, kv head h, context partition s)):
//   * the partition is a run of `split_blocks` logical 16-token blocks of sequence b;
//   * warp NWC (the producer) reads the block-table entries 32 at a time and issues one
//     TMA tensor load per K tile and per V tile (16 tokens x head_dim of kv head h) into a
//     ring of STAGES shared-memory stages, completing on per-stage mbarriers;
//   * warps 0..NWC-1 (consumers) serve all G query heads of the group and take the
//     partition's blocks round-robin, each with its own online-softmax state, so every K/V
//     element is widened to fp32 once and used by all G heads;
//   * scores: lane l owns head_dim elements [l*D/32, (l+1)*D/32); per chunk of TC = 16/GW
//     tokens it forms the 16 partial dot products (GW heads x TC tokens) over its slice and
//     sums them across the warp with a transposing butterfly (each level halves the values
//     a lane holds; the last level is a plain butterfly), so lanes 2k and 2k+1 end with the
//     same finished score; the registers are permuted per lane so that every level adds the
//     same register half on every lane (no selects);
//   * P V: the weights go through a per-warp shared buffer; lane l accumulates its
//     head_dim slice for its heads with packed fp32x2 FMAs into (even token, odd token)
//     accumulator pairs, so neither operand of a packed FMA needs duplicating; full blocks
//     take a branch-free path, the one partial block of a sequence a masked one; the
//     rescale by exp(m_old - m_new) runs only when a running max actually moved;
//   * the consumer warps' states are merged in shared memory; a single-partition sequence
//     writes its output directly, otherwise the partition's (m, l, unnormalised acc) go to
//     the workspace and the merge kernel that follows (merge_partitions.cu) combines the
//     partitions in partition order with their log-sum-exp weights.
// Scores are kept in log2 units (q is pre-multiplied by scale*log2(e)), so every
// exponential is one ex2.approx.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

// Shared-prefix records a sequence's decode merges at most (splits of the prefix pass).
constexpr int kMaxPrefixRecords = 16;

struct DecodeParams {
  const uint16_t* q;            // [B][Hq][D] bf16
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  const float* scales;          // [2][Hkv] (E4M3) or nullptr
  void* out;                    // [B][Hq][D] bf16 or fp32
  float* part_ml;               // [B][Hkv][rec_slots][G][2]
  float* part_acc;              // [B][Hkv][rec_slots][G][D]
  const int32_t* seq_prefix;    // [B]: >= 0 if the sequence has shared-prefix records, or nullptr
  uint32_t* status;
  int max_blocks;
  int hq;
  int hkv;
  int num_blocks;       // pool size in blocks
  int max_context_len;  // launch bound on context_lens
  int split_blocks;     // blocks per partition
  int max_splits;       // gridDim.z
  int pre_slots;        // shared-prefix records per (b, h) ahead of the partitions' (0: none)
  int rec_slots;        // records per (b, h): pre_slots + max_splits
  float score_scale;    // softmax_scale * log2(e)
  int out_fp32;
  int merge_warps;      // merge kernel: warps per query head (1, 2, 4 or 8; set by its launch)
  int defer_prefix;     // cascade: the decode writes a record for every prefixed sequence and
                        // the merge kernel combines it with the prefix records (tensor-core form)
  // Failure-detection tests only (tensor-core form; 0 = off, the default): the consumer
  // warps give up waiting for a K/V stage after this many cycles instead of about a second,
  // and the producer warp waits this many cycles before its first load, so that the
  // consumers' wait runs out while the loads are still to come.
  long long test_consumer_wait_cycles;
  long long test_producer_delay_cycles;
  // Fused append (tensor-core form, plain decode): sequence b's new token, at position
  // context_lens[b] - 1, is k_new / v_new [B][Hkv][D] bf16 for slot new_slots[b] (< 0: none);
  // the CTA holding the sequence's last block writes it into the pool (k_pool / v_pool) and
  // into its copy of that block.  fused == 0: none of this.
  int fused;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int64_t* new_slots;
  void* k_pool;
  void* v_pool;
};

template <int D, int G, bool FP8, int NWC, int STAGES>
struct DecodeCfg {
  // query heads per consumer warp: the whole group, so every K/V element is widened to
  // fp32 once and used by all G heads (splitting a group of 8 over two warps that read the
  // same tiles costs a second widening and was 12 % slower on the 70B-shaped step)
  static constexpr int kGW = G;
  static constexpr int kHG = G / kGW;                  // head groups (warps sharing a tile)
  static constexpr int kWPH = NWC / kHG;               // consumer warps per head group
  static constexpr int kDPL = D / 32;                  // head_dim elements per lane
  static constexpr int kTC = 16 / kGW;                 // tokens per score chunk
  static constexpr int kNCH = kBlockSize / kTC;        // chunks per block (== kGW)
  static constexpr int kESZ = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kESZ;
  static constexpr int kTileBytes = kBlockSize * kRowBytes;
  static constexpr int kThreads = (NWC + 1) * 32;
  // per consumer warp: P[GW][16] weights and GW (alpha, alpha) pairs, rounded to 16 bytes
  // so that every warp's P rows stay aligned for 16-byte shared loads
  static constexpr int kPWarpFloats = (kGW * kBlockSize + 2 * kGW + 3) / 4 * 4;
  static constexpr int kPBytes = NWC * kPWarpFloats * 4;
  static constexpr int kTilesBytes = 2 * STAGES * kTileBytes;
  static constexpr int kBarOffset = ((kTilesBytes + kPBytes) + 15) / 16 * 16;
  static constexpr int kSmemBytes = kBarOffset + 2 * STAGES * 8;
  // merge scratch in the tile area: per warp m[GW], l[GW], acc[GW][D]
  static constexpr int kMergeBytes = NWC * (2 * kGW + kGW * D) * 4;
  static_assert(kMergeBytes <= kTilesBytes, "merge scratch must fit in the tile ring");
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size");
  static_assert(NWC % kHG == 0, "consumer warps per head group");
  // Each stage must always be consumed by the same warps: a warp then waits on a stage
  // barrier only after consuming that stage's previous phase itself, so a phase parity can
  // never be mistaken for the one two phases back.
  static_assert(STAGES % kWPH == 0, "ring depth must be a multiple of the warps per head group");
  static_assert(kPWarpFloats % 4 == 0 && kTilesBytes % 16 == 0, "16-byte aligned P buffers");
};

// Widen kDPL consecutive elements at p (this lane's slice of one tile row) to fp32.
// E4M3 values come out times 2^-120; the factor is folded into q and the output scale.
template <int D, bool FP8>
__device__ __forceinline__ void load_slice(const uint8_t* p, float (&x)[D / 32]) {
  constexpr int DPL = D / 32;
  if constexpr (!FP8) {
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = bf16_lo(w); x[1] = bf16_hi(w);
    }
  } else {
    if constexpr (DPL == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = e4m3_x2m120<0>(w); x[1] = e4m3_x2m120<1>(w); x[2] = e4m3_x2m120<2>(w); x[3] = e4m3_x2m120<3>(w);
    } else {
      const uint32_t w = *reinterpret_cast<const uint16_t*>(p);
      x[0] = e4m3_x2m120<0>(w); x[1] = e4m3_x2m120<1>(w);
    }
  }
}

// Online-softmax state of one consumer warp for its GW query heads.
template <int D, int GW>
struct WarpState {
  float2 acc[GW][D / 32];  // (even-token, odd-token) partial sums of P V, this lane's slice
  float m;                 // running max (log2 units) of head sig_g
  float l;                 // this lane's share of the running sum of head sig_g
};

// One 16-token block: scores, online-softmax update, P V.  `valid` tokens (1..16) count.
template <int D, int GW, bool FP8, bool FULL>
__device__ __forceinline__ void consume_block(const uint8_t* kt, const uint8_t* vt, int valid, float smul,
                                              const float2 (&qd)[GW][D / 32], const int (&rowoff)[16 / GW],
                                              int sig_g, int sig_t, int lane, float* pbuf, float2* abuf,
                                              WarpState<D, GW>& st) {
  constexpr int DPL = D / 32, TC = 16 / GW, NCH = kBlockSize / TC;
  constexpr int ROW = D * (FP8 ? 1 : 2);
  const int slice = lane * DPL * (FP8 ? 1 : 2);

  // ---- scores: one finished score per lane pair per chunk
  float sc[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    float kx[TC][DPL];
#pragma unroll
    for (int ts = 0; ts < TC; ++ts) load_slice<D, FP8>(kt + c * TC * ROW + rowoff[ts], kx[ts]);
    float part[16];
#pragma unroll
    for (int gs = 0; gs < GW; ++gs)
#pragma unroll
      for (int tp = 0; tp < TC; tp += 2) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < DPL; ++i) a = ffma2(qd[gs][i], make_float2(kx[tp][i], kx[tp + 1][i]), a);
        part[gs * TC + tp] = a.x;
        part[gs * TC + tp + 1] = a.y;
      }
    // transposing butterfly over 16 values: lane bit 4..1 select the half kept at each level
    {
      float r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = shfl_xor(part[i + 8], 16);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const float2 s2 = fadd2(make_float2(part[i], part[i + 1]), make_float2(r[i], r[i + 1]));
        part[i] = s2.x; part[i + 1] = s2.y;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = shfl_xor(part[i + 4], 8);
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const float2 s2 = fadd2(make_float2(part[i], part[i + 1]), make_float2(r[i], r[i + 1]));
        part[i] = s2.x; part[i + 1] = s2.y;
      }
      r[0] = shfl_xor(part[2], 4);
      r[1] = shfl_xor(part[3], 4);
      {
        const float2 s2 = fadd2(make_float2(part[0], part[1]), make_float2(r[0], r[1]));
        part[0] = s2.x; part[1] = s2.y;
      }
      part[0] += shfl_xor(part[1], 2);
      part[0] += shfl_xor(part[0], 1);
    }
    if constexpr (FULL) {
      sc[c] = part[0] * smul;
    } else {
      sc[c] = (c * TC + sig_t) < valid ? part[0] * smul : -INFINITY;
    }
  }

  // ---- online softmax for head sig_g (lanes 2k, 2k+1 hold the same scores)
  float bmax = sc[0];
#pragma unroll
  for (int c = 1; c < NCH; ++c) bmax = fmaxf(bmax, sc[c]);
#pragma unroll
  for (int m = 2; m <= TC; m <<= 1) bmax = fmaxf(bmax, shfl_xor(bmax, m));
  const bool moved = __any_sync(kFull, bmax > st.m);
  if (moved) {
    const float m_new = fmaxf(st.m, bmax);
    const float alpha = (m_new == st.m) ? 1.0f : fast_exp2(st.m - m_new);
    st.l *= alpha;
    st.m = m_new;
    if ((lane & (2 * TC - 1)) == 0) abuf[sig_g] = make_float2(alpha, alpha);
  }
  float psum = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const float pv = fast_exp2(sc[c] - st.m);
    psum += pv;
    pbuf[sig_g * kBlockSize + c * TC + sig_t] = pv;
  }
  st.l += psum;
  __syncwarp();
  if (moved) {
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      const float2 a2 = abuf[g];
#pragma unroll
      for (int i = 0; i < DPL; ++i) st.acc[g][i] = fmul2(st.acc[g][i], a2);
    }
  }

  // ---- P V over this lane's head_dim slice, tokens in (even, odd) pairs
#pragma unroll
  for (int t4 = 0; t4 < kBlockSize; t4 += 4) {
    float4 pq[GW];
#pragma unroll
    for (int g = 0; g < GW; ++g) pq[g] = *reinterpret_cast<const float4*>(pbuf + g * kBlockSize + t4);
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const int t0 = t4 + 2 * pr;
      float v0[DPL], v1[DPL];
      load_slice<D, FP8>(vt + t0 * ROW + slice, v0);
      load_slice<D, FP8>(vt + (t0 + 1) * ROW + slice, v1);
      if constexpr (!FULL) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) {  // rows past the sequence may hold anything (even NaN)
          v0[i] = t0 < valid ? v0[i] : 0.f;
          v1[i] = t0 + 1 < valid ? v1[i] : 0.f;
        }
      }
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        const float2 pp = pr == 0 ? make_float2(pq[g].x, pq[g].y) : make_float2(pq[g].z, pq[g].w);
#pragma unroll
        for (int i = 0; i < DPL; ++i) st.acc[g][i] = ffma2(pp, make_float2(v0[i], v1[i]), st.acc[g][i]);
      }
    }
  }
  __syncwarp();  // the next block rewrites pbuf
}

// Final output of (b, h) from its partial records lo .. hi-1 (log2-domain max, sum and
// unnormalised output per query head), combined in record order with their log-sum-exp
// weights (deterministic).  All threads of the CTA take part; wts is shared scratch of
// G * (rec_slots + 1) floats.  A head whose records are all empty gets zeros.
template <int D, int G, bool FP8>
__device__ __forceinline__ void merge_records(const DecodeParams& p, int b, int h, int lo, int hi, float* wts,
                                              int nthreads) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = nthreads >> 5;
  const size_t rec0 = (static_cast<size_t>(b) * p.hkv + h) * p.rec_slots;
  const int R = p.rec_slots;
  for (int g = warp; g < G; g += nwarps) {
    float M = -INFINITY;
    for (int j = lo + lane; j < hi; j += 32) M = fmaxf(M, __ldcg(&p.part_ml[((rec0 + j) * G + g) * 2]));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, shfl_xor(M, m));
    for (int j = lo + lane; j < hi; j += 32)
      wts[g * R + j] = M == -INFINITY ? 0.f : fast_exp2(__ldcg(&p.part_ml[((rec0 + j) * G + g) * 2]) - M);
    __syncwarp();
    if (lane == 0) {  // the denominator is summed in record order (deterministic)
      float den = 0.f;
      for (int j = lo; j < hi; ++j) den = fmaf(wts[g * R + j], __ldcg(&p.part_ml[((rec0 + j) * G + g) * 2 + 1]), den);
      wts[G * R + g] = den > 0.f ? 1.0f / den : 0.f;
    }
  }
  __syncthreads();
  float vfix = 1.0f;  // E4M3 values carry 2^-120; V's scale and that factor go to the output
  if constexpr (FP8) vfix = p.scales[p.hkv + h];
  const size_t out_row0 = static_cast<size_t>(b) * p.hq + h * G;
  for (int e = threadIdx.x; e < G * D; e += nthreads) {
    const int g = e / D, d = e % D;
    float num = 0.f;
    for (int j = lo; j < hi; ++j) num = fmaf(wts[g * R + j], __ldcg(&p.part_acc[((rec0 + j) * G + g) * D + d]), num);
    float o = num * wts[G * R + g];
    if constexpr (FP8) o = (o * 1152921504606846976.0f) * (vfix * 1152921504606846976.0f);  // 2^60 * 2^60
    const size_t oi = (out_row0 + g) * D + d;
    if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
  }
}

// CAS: the cascade variant, which merges shared-prefix records (seq_prefix, pre_slots);
// the plain variant carries none of that code.
// Register cap of the CUDA-core kernel: CTAs of NWC + 1 warps share an SM only while
// ceil(n (NWC + 1) / 4) warps x regs x 32 fit one scheduler's 16K registers.  The G = 8,
// D = 128 form aims at two CTAs per SM (168 registers; uncapped it takes 172 and drops to
// one), every other form at three (128), which their shared memory allows.
template <int D, int G, int NWC>
struct DecodeRegCap {
  static constexpr int kCtas = (D == 128 && G == 8) ? 2 : 3;
  static constexpr int kWarpsPerScheduler = (kCtas * (NWC + 1) + 3) / 4;
  static constexpr int kRegs = (16384 / (kWarpsPerScheduler * 32)) / 8 * 8;
};

template <int D, int G, bool FP8, int NWC, int STAGES, bool CAS>
__global__ void __launch_bounds__((NWC + 1) * 32) __maxnreg__((DecodeRegCap<D, G, NWC>::kRegs))
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p) {
  using C = DecodeCfg<D, G, FP8, NWC, STAGES>;
  constexpr int DPL = C::kDPL, TC = C::kTC, GW = C::kGW, HG = C::kHG, WPH = C::kWPH;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* k_tiles = smem;
  uint8_t* v_tiles = smem + STAGES * C::kTileBytes;
  float* p_all = reinterpret_cast<float*>(smem + C::kTilesBytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;

  // grid (kv head, sequence, partition): the block scheduler hands out every sequence's first
  // partition before any second one, so the long sequences' last partitions come last
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // No global reads before the preceding kernel (e.g. the append) completed.  In a cascade
  // call the preceding kernel is the prefix pass, which lets this grid start once all its
  // CTAs are past their own wait (so the append's results are visible); this kernel then
  // waits for the prefix pass itself only before it reads the prefix records.
  if constexpr (!CAS) pdl_wait();

  // ---- sequence length (checked, clamped) and this CTA's share of it
  int len = p.context_lens[b];
  // the first 32 block ids of this partition, loaded beside the length (the row has
  // max_blocks valid entries; ids past the context are never used or checked)
  const int blk0 = s * p.split_blocks;
  const int32_t* row = p.block_tables + static_cast<size_t>(b) * p.max_blocks + blk0;
  int ids = (warp == NWC && blk0 + lane < p.max_blocks) ? row[lane] : 0;
  {
    const int cap = min(p.max_context_len, p.max_blocks * kBlockSize);
    if (len < 0 || len > cap) {
      if (threadIdx.x == 0 && s == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
      len = len < 0 ? 0 : cap;
    }
  }
  const int nblk = (len + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  const int hq0 = h * G;

  // shared-prefix records (written by the prefix pass) come first among this (b, h)'s records
  int npre = 0;
  if constexpr (CAS) npre = p.seq_prefix[b] >= 0 ? p.pre_slots : 0;
  if (nblk == 0) {  // no own blocks: partition 0 writes zeros, or the prefix result alone
    if (s == 0) {
      if (CAS && npre > 0) {
        pdl_wait();
        merge_records<D, G, FP8>(p, b, h, 0, npre, reinterpret_cast<float*>(smem), C::kThreads);
      } else {
        for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
          const size_t o = (static_cast<size_t>(b) * p.hq + hq0) * D + e;
          if (p.out_fp32) reinterpret_cast<float*>(p.out)[o] = 0.f;
          else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
        }
      }
    }
    if constexpr (CAS) pdl_wait();
    return;
  }
  if (s >= nsplit) {
    if constexpr (CAS) pdl_wait();
    return;
  }
  const int nloc = min(nblk, blk0 + p.split_blocks) - blk0;

  // issue the first global loads now, so their latency overlaps the barrier set-up
  const int hg = warp % HG;  // head group of a consumer warp
  uint32_t qbits[GW][DPL / 2];
  if (warp < NWC) {
    const int sig_g0 = (lane >> 1) / TC;
    const uint16_t* qrow = p.q + (static_cast<size_t>(b) * p.hq + hq0 + hg * GW) * D + lane * DPL;
#pragma unroll
    for (int gs = 0; gs < GW; ++gs) {
      const uint32_t* qq = reinterpret_cast<const uint32_t*>(qrow + static_cast<size_t>(gs ^ sig_g0) * D);
#pragma unroll
      for (int i = 0; i < DPL / 2; ++i) qbits[gs][i] = qq[i];
    }
  }
  if (threadIdx.x == NWC * 32) tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], HG);  // every head group's warp releases the stage
    }
    fence_mbar_init();
  }
  __syncthreads();

  // log2-domain score scale; E4M3 keys carry 2^-120, compensated in two exact steps
  // (q * 2^64 keeps every product a normal number, the rest goes into the score scale).
  float qmul = p.score_scale, smul = 1.0f;
  if constexpr (FP8) {
    qmul = 18446744073709551616.0f;                             // 2^64
    smul = p.score_scale * p.scales[h] * 72057594037927936.0f;  // * 2^56
  }

  bool timed_out = false;

  if (warp == NWC) {
    // ================================================================ producer warp
    int issued = 0;
    for (int base = 0; base < nloc && !timed_out; base += 32) {
      const int next = (base + 32 + lane < nloc) ? row[base + 32 + lane] : 0;  // prefetch
      if ((ids < 0 || ids >= p.num_blocks) && base + lane < nloc) set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
      const int cnt = min(32, nloc - base);
      for (int k = 0; k < cnt; ++k) {
        const int pb = __shfl_sync(kFull, ids, k);
        const int it = base + k;
        const int st = it % STAGES;
        if (lane == 0) {
          if (it >= STAGES && !mbar_wait(&empty_bar[st], ((it / STAGES) - 1) & 1)) {
            set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
            timed_out = true;
          }
          if (!timed_out) {
            mbar_arrive_expect_tx(&full_bar[st], 2 * C::kTileBytes);
            // out-of-range ids read zeros (tensor-map bounds), never outside the pool
            tma_load_3d(k_tiles + st * C::kTileBytes, &tm_k, 0, h, pb * kBlockSize, &full_bar[st]);
            tma_load_3d(v_tiles + st * C::kTileBytes, &tm_v, 0, h, pb * kBlockSize, &full_bar[st]);
          }
        }
        timed_out = __shfl_sync(kFull, timed_out, 0);
        if (timed_out) break;
        issued = it + 1;
      }
      ids = next;
    }
    // Before the CTA may reuse or release the ring, every issued copy must have landed.
    if (lane == 0) {
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        if (!mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1)) {
          set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
          break;
        }
    }
    __syncwarp();
  }

  // consumer lane roles: after the butterfly lanes 2k, 2k+1 hold head sig_g, token sig_t
  const int sigma = lane >> 1;
  const int sig_g = sigma / TC;
  const int sig_t = sigma % TC;
  WarpState<D, GW> st;
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int g = 0; g < GW; ++g)
#pragma unroll
    for (int i = 0; i < DPL; ++i) st.acc[g][i] = make_float2(0.f, 0.f);

  if (warp < NWC) {
    // ================================================================ consumer warps
    float* pbuf = p_all + warp * C::kPWarpFloats;  // P[g][t]
    float2* abuf = reinterpret_cast<float2*>(pbuf + GW * kBlockSize);
    int rowoff[TC];
#pragma unroll
    for (int ts = 0; ts < TC; ++ts) rowoff[ts] = (ts ^ sig_t) * C::kRowBytes + lane * DPL * C::kESZ;
    // q slice of the warp's heads, permuted: slot gs holds head hg*GW + (gs ^ sig_g), as (q, q)
    float2 qd[GW][DPL];
#pragma unroll
    for (int gs = 0; gs < GW; ++gs)
#pragma unroll
      for (int i = 0; i < DPL / 2; ++i) {
        const float lo = bf16_lo(qbits[gs][i]) * qmul, hi = bf16_hi(qbits[gs][i]) * qmul;
        qd[gs][2 * i] = make_float2(lo, lo);
        qd[gs][2 * i + 1] = make_float2(hi, hi);
      }

    for (int it = warp / HG; it < nloc; it += WPH) {
      const int sg = it % STAGES;
      if (!mbar_wait(&full_bar[sg], (it / STAGES) & 1)) {
        if (lane == 0) set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
        timed_out = true;
        break;
      }
      const uint8_t* kt = k_tiles + sg * C::kTileBytes;
      const uint8_t* vt = v_tiles + sg * C::kTileBytes;
      const int valid = min(kBlockSize, len - (blk0 + it) * kBlockSize);  // >= 1
      if (valid == kBlockSize)
        consume_block<D, GW, FP8, true>(kt, vt, valid, smul, qd, rowoff, sig_g, sig_t, lane, pbuf, abuf, st);
      else
        consume_block<D, GW, FP8, false>(kt, vt, valid, smul, qd, rowoff, sig_g, sig_t, lane, pbuf, abuf, st);
      // read through the generic proxy, refilled by TMA (async proxy): order the reads first
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[sg]);
    }
  }

  // ================================================================ merge the consumer warps
  __syncthreads();  // ring drained (every issued copy landed and was consumed)
  float* mw = reinterpret_cast<float*>(smem);  // [NWC][GW] max
  float* lw = mw + NWC * GW;                   // [NWC][GW] sum
  float* aw = lw + NWC * GW;                   // [NWC][GW][D] unnormalised output
  if (warp < NWC) {
    float lsum = st.l;
#pragma unroll
    for (int m = 2; m <= TC; m <<= 1) lsum += shfl_xor(lsum, m);  // lane 2k+1 duplicates 2k
    if ((lane & (2 * TC - 1)) == 0) {
      mw[warp * GW + sig_g] = st.m;
      lw[warp * GW + sig_g] = lsum;
    }
#pragma unroll
    for (int g = 0; g < GW; ++g)
#pragma unroll
      for (int i = 0; i < DPL; ++i) aw[(warp * GW + g) * D + lane * DPL + i] = st.acc[g][i].x + st.acc[g][i].y;
  }
  __syncthreads();

  // per query head: max over the head group's warps, weights 2^(m_w - M); then each element
  const size_t out_row0 = static_cast<size_t>(b) * p.hq + hq0;
  float vfix = 1.0f;  // E4M3 values carry 2^-120; V's scale and that factor go to the output
  if constexpr (FP8) vfix = p.scales[p.hkv + h];
  const bool single = (nsplit == 1 && npre == 0);
  // one partition and prefix records: merge them right here (no record to write)
  const bool with_prefix = CAS && (nsplit == 1 && npre > 0);
  if (with_prefix) pdl_wait();
  const size_t prec0 = (static_cast<size_t>(b) * p.hkv + h) * p.rec_slots;
  for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
    const int g = e / D, d = e % D;
    const int ghg = g / GW, gw = g % GW;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < WPH; ++k) M = fmaxf(M, mw[(ghg + HG * k) * GW + gw]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int k = 0; k < WPH; ++k) {
      const int w = ghg + HG * k;
      const float wt = fast_exp2(mw[w * GW + gw] - M);  // warps without blocks: 2^-inf = 0
      num = fmaf(wt, aw[(w * GW + gw) * D + d], num);
      den = fmaf(wt, lw[w * GW + gw], den);
    }
    if (CAS && with_prefix) {
      // combine with the prefix records in record order: theirs, then this partition's
      float Mt = M;
      for (int j = 0; j < npre; ++j) Mt = fmaxf(Mt, __ldcg(&p.part_ml[((prec0 + j) * G + g) * 2]));
      float num2 = 0.f, den2 = 0.f;
      if (Mt != -INFINITY) {
        for (int j = 0; j < npre; ++j) {
          const float wj = fast_exp2(__ldcg(&p.part_ml[((prec0 + j) * G + g) * 2]) - Mt);
          num2 = fmaf(wj, __ldcg(&p.part_acc[((prec0 + j) * G + g) * D + d]), num2);
          den2 = fmaf(wj, __ldcg(&p.part_ml[((prec0 + j) * G + g) * 2 + 1]), den2);
        }
        const float ws = fast_exp2(M - Mt);
        num2 = fmaf(ws, num, num2);
        den2 = fmaf(ws, den, den2);
      }
      float o = den2 > 0.f ? num2 / den2 : 0.f;
      if constexpr (FP8) o = (o * 1152921504606846976.0f) * (vfix * 1152921504606846976.0f);  // 2^60 * 2^60
      const size_t oi = (out_row0 + g) * D + d;
      if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
      else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
    } else if (single) {
      float o = num / den;
      if constexpr (FP8) o = (o * 1152921504606846976.0f) * (vfix * 1152921504606846976.0f);  // 2^60 * 2^60
      const size_t oi = (out_row0 + g) * D + d;
      if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
      else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
    } else {
      const size_t rec = CAS ? (static_cast<size_t>(b) * p.hkv + h) * p.rec_slots + p.pre_slots + s
                             : (static_cast<size_t>(b) * p.hkv + h) * p.max_splits + s;
      p.part_acc[(rec * G + g) * D + d] = num;
      if (d == 0) {
        p.part_ml[(rec * G + g) * 2 + 0] = M;
        p.part_ml[(rec * G + g) * 2 + 1] = den;
      }
    }
  }
  // A record was written (or, for one partition, the output): the merge kernel that
  // follows combines the records.  A cascade grid completes only after the prefix pass,
  // whose records the merge kernel also reads.
  if constexpr (CAS) pdl_wait();
}

}  // namespace pkv
