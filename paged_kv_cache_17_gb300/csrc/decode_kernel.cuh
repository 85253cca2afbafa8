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
//   * warps 0..NWC-1 (consumers) take the partition's blocks round-robin; each keeps its
//     own online-softmax state for all G = Hq/Hkv query heads of the group, so every K/V
//     element is widened to fp32 once and used by all G heads;
//   * scores: lane l owns head_dim elements [l*D/32, (l+1)*D/32); per chunk of TC tokens it
//     forms the G*TC partial dot products over its slice and sums them across the warp
//     with a transposing butterfly (each level halves the values a lane holds), so a lane
//     ends with one finished score; the registers are permuted per lane so that every
//     level adds the same register half on every lane (no selects);
//   * P V: the weights go through a per-warp shared buffer; lane l accumulates its
//     head_dim slice for all G heads with packed fp32x2 FMAs;
//   * the consumer warps' states are merged in shared memory; a single-partition sequence
//     writes its output directly, otherwise the partition's (m, l, unnormalised acc) go to
//     the workspace and the last CTA of (b, h) to finish -- found with an atomic ticket, no
//     waiting -- merges the partitions in partition order with their log-sum-exp weights.
// Scores are kept in log2 units (q is pre-multiplied by scale*log2(e)), so every
// exponential is one ex2.approx.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

struct DecodeParams {
  const uint16_t* q;            // [B][Hq][D] bf16
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  const float* scales;          // [2][Hkv] (E4M3) or nullptr
  void* out;                    // [B][Hq][D] bf16 or fp32
  int32_t* tickets;             // [B][Hkv]        (multi-partition only)
  float* part_ml;               // [B][Hkv][S][G][2]
  float* part_acc;              // [B][Hkv][S][G][D]
  uint32_t* status;
  int max_blocks;
  int hq;
  int hkv;
  int num_blocks;       // pool size in blocks
  int max_context_len;  // launch bound on context_lens
  int split_blocks;     // blocks per partition
  int max_splits;       // gridDim.y
  float score_scale;    // softmax_scale * log2(e)
  int out_fp32;
};

template <int D, int G, bool FP8, int NWC, int STAGES>
struct DecodeCfg {
  static constexpr int kDPL = D / 32;                 // head_dim elements per lane
  static constexpr int kTC = (G >= 2) ? 32 / G : 16;  // tokens per score chunk (G*TC values)
  static constexpr int kN = G * kTC;                  // partial dot products per chunk (32, or 16 for G=1)
  static constexpr int kLogN = (kN == 32) ? 5 : 4;
  static constexpr int kNCH = kBlockSize / kTC;       // chunks per block
  static constexpr int kLPG = 32 / G;                 // lanes holding scores of one query head
  static constexpr int kESZ = FP8 ? 1 : 2;
  static constexpr int kTileBytes = kBlockSize * D * kESZ;
  static constexpr int kThreads = (NWC + 1) * 32;
  // shared memory: [STAGES] K tiles, [STAGES] V tiles, per-warp P (16 x G) + alpha (G),
  // then mbarriers.  The end-of-CTA merge reuses the tile area.
  static constexpr int kPBytes = NWC * (kBlockSize * G + G) * 4;
  static constexpr int kTilesBytes = 2 * STAGES * kTileBytes;
  static constexpr int kBarOffset = ((kTilesBytes + kPBytes) + 15) / 16 * 16;
  static constexpr int kSmemBytes = kBarOffset + 2 * STAGES * 8;
  // merge scratch in the tile area: per warp m[G], l[G], acc[G][D]
  static constexpr int kMergeBytes = NWC * (2 * G + G * D) * 4;
  static_assert(kMergeBytes <= kTilesBytes, "merge scratch must fit in the tile ring");
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size");
};

// Load this lane's slice of row `row` of a K/V tile and widen it to fp32 (E4M3 values
// come out times 2^-120; the factor is folded into q and into the output scale).
template <int D, bool FP8>
__device__ __forceinline__ void load_row(const uint8_t* tile, int row, int lane, float (&x)[D / 32]) {
  constexpr int DPL = D / 32;
  if constexpr (!FP8) {
    const uint8_t* p = tile + (row * D + lane * DPL) * 2;
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = bf16_lo(w); x[1] = bf16_hi(w);
    }
  } else {
    const uint8_t* p = tile + row * D + lane * DPL;
    if constexpr (DPL == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = e4m3_x2m120<0>(w); x[1] = e4m3_x2m120<1>(w); x[2] = e4m3_x2m120<2>(w); x[3] = e4m3_x2m120<3>(w);
    } else {
      const uint32_t w = *reinterpret_cast<const uint16_t*>(p);
      x[0] = e4m3_x2m120<0>(w); x[1] = e4m3_x2m120<1>(w);
    }
  }
}

template <int D, int G, bool FP8, int NWC, int STAGES>
__global__ void __launch_bounds__((NWC + 1) * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p) {
  using C = DecodeCfg<D, G, FP8, NWC, STAGES>;
  constexpr int DPL = C::kDPL, TC = C::kTC, N = C::kN, NCH = C::kNCH, LPG = C::kLPG;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* k_tiles = smem;
  uint8_t* v_tiles = smem + STAGES * C::kTileBytes;
  float* p_all = reinterpret_cast<float*>(smem + C::kTilesBytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;

  const int h = blockIdx.x;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  pdl_wait();  // no global reads before the preceding kernel (e.g. the append) completed

  // ---- sequence length (checked, clamped) and this CTA's share of it
  int len = p.context_lens[b];
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

  if (nblk == 0) {  // empty sequence: zero output, written by partition 0
    if (s == 0) {
      for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
        const size_t o = (static_cast<size_t>(b) * p.hq + hq0) * D + e;
        if (p.out_fp32) reinterpret_cast<float*>(p.out)[o] = 0.f;
        else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
      }
    }
    return;
  }
  if (s >= nsplit) return;
  const int blk0 = s * p.split_blocks;
  const int nloc = min(nblk, blk0 + p.split_blocks) - blk0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // log2-domain score scale; E4M3 keys carry 2^-120, compensated in two exact steps
  // (q * 2^64 keeps every product a normal number, the rest goes into the score scale).
  float qmul = p.score_scale, smul = 1.0f;
  if constexpr (FP8) {
    qmul = 18446744073709551616.0f;                               // 2^64
    smul = p.score_scale * p.scales[h] * 72057594037927936.0f;    // * 2^56
  }

  bool timed_out = false;

  if (warp == NWC) {
    // ================================================================ producer warp
    const int32_t* row = p.block_tables + static_cast<size_t>(b) * p.max_blocks + blk0;
    int ids = (lane < nloc) ? row[lane] : 0;
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

  // consumer state (the producer warp keeps the neutral values)
  const int sigma = lane >> (5 - C::kLogN);  // value index this lane ends up holding
  const int sig_g = sigma / TC;               // == this lane's query head within the group
  const int sig_t = sigma % TC;               // == this lane's token within a chunk
  float m_run = -INFINITY;                    // running max (log2 units) of head sig_g
  float l_run = 0.f;                          // this lane's share of the running sum
  float2 acc[G][DPL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) acc[g][i] = make_float2(0.f, 0.f);

  if (warp < NWC) {
    // ================================================================ consumer warps
    float* pbuf = p_all + warp * (kBlockSize * G + G);  // P[t][g], then alpha[g]
    float* abuf = pbuf + kBlockSize * G;
    // q slice, permuted: register slot gs holds query head gs ^ sig_g (see header)
    float2 qd[G][DPL];
    {
      const uint16_t* qrow = p.q + (static_cast<size_t>(b) * p.hq + hq0) * D + lane * DPL;
#pragma unroll
      for (int gs = 0; gs < G; ++gs) {
        const uint16_t* qq = qrow + static_cast<size_t>(gs ^ sig_g) * D;
        float x[DPL];
        if constexpr (DPL == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(qq);
          x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(qq);
          x[0] = bf16_lo(w); x[1] = bf16_hi(w);
        }
#pragma unroll
        for (int i = 0; i < DPL; ++i) qd[gs][i] = make_float2(x[i] * qmul, x[i] * qmul);
      }
    }

    for (int it = warp; it < nloc; it += NWC) {
      const int st = it % STAGES;
      if (!mbar_wait(&full_bar[st], (it / STAGES) & 1)) {
        if (lane == 0) set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
        timed_out = true;
        break;
      }
      const uint8_t* kt = k_tiles + st * C::kTileBytes;
      const uint8_t* vt = v_tiles + st * C::kTileBytes;
      const int valid = min(kBlockSize, len - (blk0 + it) * kBlockSize);  // >= 1

      // ---- scores: one finished score per lane per chunk
      float sc[NCH];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float kx[TC][DPL];
#pragma unroll
        for (int ts = 0; ts < TC; ++ts) load_row<D, FP8>(kt, c * TC + (ts ^ sig_t), lane, kx[ts]);
        float part[N];
        static_assert(TC % 2 == 0, "token pairs");
#pragma unroll
        for (int gs = 0; gs < G; ++gs)
#pragma unroll
          for (int tp = 0; tp < TC; tp += 2) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < DPL; ++i) a = ffma2(qd[gs][i], make_float2(kx[tp][i], kx[tp + 1][i]), a);
            part[gs * TC + tp] = a.x;
            part[gs * TC + tp + 1] = a.y;
          }
        // transposing butterfly: after level j a lane holds half as many partial sums
        int n = N;
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
          if (n >= 2) {
            const int half = n >> 1;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i < half) part[i] += shfl_xor(part[i + half], m);
            n = half;
          } else {
            part[0] += shfl_xor(part[0], m);
          }
        }
        const bool ok = (c * TC + sig_t) < valid;
        sc[c] = ok ? part[0] * smul : -INFINITY;
      }

      // ---- online softmax for head sig_g (all lanes of the head agree on the max)
      float bmax = sc[0];
#pragma unroll
      for (int c = 1; c < NCH; ++c) bmax = fmaxf(bmax, sc[c]);
#pragma unroll
      for (int m = 1; m < LPG; m <<= 1) bmax = fmaxf(bmax, shfl_xor(bmax, m));
      const float m_new = fmaxf(m_run, bmax);
      const float alpha = fast_exp2(m_run - m_new);
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const float pv = fast_exp2(sc[c] - m_new);
        psum += pv;
        pbuf[(c * TC + sig_t) * G + sig_g] = pv;
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if ((lane & (LPG - 1)) == 0) abuf[sig_g] = alpha;
      __syncwarp();

      // ---- rescale and accumulate P V over this lane's head_dim slice
      {
        float al[G];
#pragma unroll
        for (int g = 0; g < G; ++g) al[g] = abuf[g];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int i = 0; i < DPL / 2; ++i) acc[g][i] = fmul2(acc[g][i], make_float2(al[g], al[g]));
      }
#pragma unroll
      for (int t = 0; t < kBlockSize; ++t) {
        if (t < valid) {
          float vx[DPL];
          load_row<D, FP8>(vt, t, lane, vx);
          float pw[G];
          if constexpr (G >= 4) {
#pragma unroll
            for (int g4 = 0; g4 < G; g4 += 4) {
              const float4 f = *reinterpret_cast<const float4*>(pbuf + t * G + g4);
              pw[g4] = f.x; pw[g4 + 1] = f.y; pw[g4 + 2] = f.z; pw[g4 + 3] = f.w;
            }
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) pw[g] = pbuf[t * G + g];
          }
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int i = 0; i < DPL / 2; ++i)
              acc[g][i] = ffma2(make_float2(pw[g], pw[g]), make_float2(vx[2 * i], vx[2 * i + 1]), acc[g][i]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
    }
  }

  // ================================================================ merge the consumer warps
  __syncthreads();  // ring drained (every issued copy landed and was consumed)
  float* mw = reinterpret_cast<float*>(smem);  // [NWC][G] max
  float* lw = mw + NWC * G;                    // [NWC][G] sum
  float* aw = lw + NWC * G;                    // [NWC][G][D] unnormalised output
  if (warp < NWC) {
    float lsum = l_run;
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) lsum += shfl_xor(lsum, m);
    if (G == 1) lsum *= 0.5f;  // with G == 1 every score is held by two lanes
    if ((lane & (LPG - 1)) == 0) {
      mw[warp * G + sig_g] = m_run;
      lw[warp * G + sig_g] = lsum;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < DPL / 2; ++i)
        *reinterpret_cast<float2*>(aw + (warp * G + g) * D + lane * DPL + 2 * i) = acc[g][i];
  }
  __syncthreads();

  // per query head: max over warps, weights 2^(m_w - M); then each element
  const size_t out_row0 = static_cast<size_t>(b) * p.hq + hq0;
  float vfix = 1.0f;  // E4M3 values carry 2^-120; V's scale and that factor go to the output
  if constexpr (FP8) vfix = p.scales[p.hkv + h];
  const bool single = (nsplit == 1);
  for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
    const int g = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWC; ++w) M = fmaxf(M, mw[w * G + g]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < NWC; ++w) {
      const float wt = fast_exp2(mw[w * G + g] - M);  // empty warps: 2^-inf = 0
      num = fmaf(wt, aw[(w * G + g) * D + d], num);
      den = fmaf(wt, lw[w * G + g], den);
    }
    if (single) {
      float o = num / den;
      if constexpr (FP8) o = (o * 1152921504606846976.0f) * (vfix * 1152921504606846976.0f);  // 2^60 * 2^60
      const size_t oi = (out_row0 + g) * D + d;
      if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
      else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
    } else {
      const size_t rec = (static_cast<size_t>(b) * p.hkv + h) * p.max_splits + s;
      p.part_acc[(rec * G + g) * D + d] = num;
      if (d == 0) {
        p.part_ml[(rec * G + g) * 2 + 0] = M;
        p.part_ml[(rec * G + g) * 2 + 1] = den;
      }
    }
  }
  if (single) return;

  // ================================================================ cross-partition merge
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.tickets[b * p.hkv + h], 1);
    s_last = (prev == nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // weights per (g, partition) in the tile area: w[g][s] = 2^(m_s - M_g) / sum_s 2^(m_s - M_g) l_s
  float* wts = reinterpret_cast<float*>(smem);
  const size_t rec0 = (static_cast<size_t>(b) * p.hkv + h) * p.max_splits;
  for (int g = warp; g < G; g += NWC + 1) {
    float M = -INFINITY;
    for (int j = lane; j < nsplit; j += 32) M = fmaxf(M, __ldcg(&p.part_ml[((rec0 + j) * G + g) * 2]));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, shfl_xor(M, m));
    // the denominator is summed in partition order by lane 0 (deterministic)
    for (int j = lane; j < nsplit; j += 32)
      wts[g * p.max_splits + j] = fast_exp2(__ldcg(&p.part_ml[((rec0 + j) * G + g) * 2]) - M);
    __syncwarp();
    if (lane == 0) {
      float den = 0.f;
      for (int j = 0; j < nsplit; ++j)
        den = fmaf(wts[g * p.max_splits + j], __ldcg(&p.part_ml[((rec0 + j) * G + g) * 2 + 1]), den);
      wts[G * p.max_splits + g] = 1.0f / den;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
    const int g = e / D, d = e % D;
    float num = 0.f;
    for (int j = 0; j < nsplit; ++j)
      num = fmaf(wts[g * p.max_splits + j], __ldcg(&p.part_acc[((rec0 + j) * G + g) * D + d]), num);
    float o = num * wts[G * p.max_splits + g];
    if constexpr (FP8) o = (o * 1152921504606846976.0f) * (vfix * 1152921504606846976.0f);
    const size_t oi = (out_row0 + g) * D + d;
    if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
  }
  if (threadIdx.x == 0) p.tickets[b * p.hkv + h] = 0;  // leave the ticket region zero
}

}  // namespace pkv
