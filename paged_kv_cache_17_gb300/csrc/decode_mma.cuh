// decode_mma.cuh -- paged GQA decode attention with the per-block products on the tensor
// cores.
//
// What it computes is exactly what decode_kernel.cuh computes (habr.com/ru/articles/1021832,
// section 3: softmax(q K^T * scale) V evaluated block by block with a running max, a
// running sum and the rescale exp(m_old - m_new); section 4: K/V in 16-token blocks found
// through the block table), with the same grid, producer warp, TMA ring, split-K records
// and log-sum-exp merge.  Only the per-block arithmetic differs.  On GB300 the CUDA-core
// form of that arithmetic costs about as much time as streaming the KV for a query group
// of 4 and 1.7 times as much for a group of 8, so the decode is not purely bandwidth bound
// there; here each 16-token block is two small matrix products per consumer warp:
//
//   S^T [16 tokens x 8] = K [16 x D] . q^T [D x 8]        (the group's G <= 8 heads as N)
//   O^T [D x 8]        += V^T [D x 16] . P^T [16 x 8]
//
// as mma.sync.m16n8k16 (bf16 in, fp32 accumulate): D/16 MMAs for the scores, 2 x D/16 for
// P V.  Tokens are the M dimension, so no row of the MMA is padding for a group of 8.  K
// and V tiles arrive by TMA as 128-byte-swizzled 64-column boxes and are read with
// ldmatrix (V transposed); q stays in registers as B fragments; the weights P leave the S
// accumulators through movmatrix (an 8x8 transpose inside the warp) as the B operand of
// the second product, split into bf16 hi + lo so that P V keeps fp32-level accuracy.
// E4M3 pools: the raw codes arrive in the ring (128-byte swizzle at D = 128, 64-byte at
// D = 64) and go straight into the MMA fragments, expanded exactly to fp16 in registers
// (cvt.rn.f16x2.e4m3x2), with no expanded copy in shared memory.  The score product
// contracts over the head dimension, so any permutation applied to K and q alike leaves it
// unchanged: lane (gid, tig) takes dims tig*D/4 .. +D/4 of every k-step's pairs, and its K
// operand is D/4 consecutive codes of tokens gid and gid + 8 (16-byte loads).  In the
// output product, row r of m-tile mt is dim (r mod 8)*D/8 + 2 mt + r/8, so a lane's V
// operand is D/8 consecutive codes of each of its four tokens, paired by byte permutes
// before the expansion; the output rows come back with the same map.  The products run in
// fp16 -- q scaled per head by a power of two into fp16's range (the factor is folded into
// that head's score scale), the K scale into the score scale, the V scale into the output.
#pragma once

#include "decode_kernel.cuh"
#include "mma_ops.cuh"

namespace pkv {

template <int D, int G, bool FP8, int NWC, int STAGES>
struct MmaCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kBlockSize * D * 2;   // one 16-bit tile, as kHalves swizzled boxes
  static constexpr int kRingTile = FP8 ? kBlockSize * D : kTileBytes;  // as loaded by TMA
  static constexpr int kKS = D / 16;                      // k-steps of the score product
  static constexpr int kMT = D / 16;                      // m-tiles of the output product
  static constexpr int kThreads = (NWC + 1) * 32;
  static constexpr int kRingBytes = 2 * STAGES * kRingTile;
  static constexpr int kTilesBytes = kRingBytes;
  static constexpr int kBarOffset = kRingBytes;
  static constexpr int kSmemBytes = 1024 + kBarOffset + 2 * STAGES * 8;  // 1024: alignment slack
  // merge scratch: the warps' states, then (cascade) the prefix records' (m, l) pairs and
  // the weights of every part
  static constexpr int kMergeBytes =
      (NWC * (2 * G + G * D) + kMaxPrefixRecords * G * 2 + (NWC + kMaxPrefixRecords + 1) * G) * 4;
  static_assert(kMergeBytes <= kRingBytes, "merge scratch must fit in the tile ring");
  static_assert(G >= 1 && G <= 8, "a query group of at most 8 heads (the MMA's N)");
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(STAGES % NWC == 0, "each stage is always consumed by the same warp");
  static_assert(kTileBytes % 1024 == 0 && kRingTile % 1024 == 0, "1024-byte aligned tiles");
};

template <int D, int G, bool FP8, int NWC, int STAGES, bool CAS>
__global__ void __launch_bounds__((NWC + 1) * 32)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const DecodeParams p) {
  using C = MmaCfg<D, G, FP8, NWC, STAGES>;
  constexpr int KS = C::kKS, MT = C::kMT;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* k_tiles = smem;
  uint8_t* v_tiles = smem + STAGES * C::kRingTile;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;

  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  if constexpr (!CAS) pdl_wait();

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
  int npre = 0;
  if constexpr (CAS) npre = p.seq_prefix[b] >= 0 ? p.pre_slots : 0;
  // Deferred cascade merge: a prefixed sequence's result goes out as a record, which the
  // merge kernel combines with the prefix records, so no CTA waits here for the prefix pass
  // but one, which keeps this grid from completing before the prefix grid (the merge kernel
  // waits for this grid).  Otherwise every cascade CTA waits before it exits.
  const bool defer = CAS && p.defer_prefix != 0;
  auto end_wait = [&]() {
    if constexpr (CAS) {
      if (!defer || (blockIdx.x | blockIdx.y | blockIdx.z) == 0) pdl_wait();
    }
  };
  if (nblk == 0) {  // no own blocks: partition 0 writes zeros, or the prefix result alone
    if (s == 0) {
      if (CAS && npre > 0) {
        if (!defer) {  // deferred: the merge kernel takes the prefix records alone
          pdl_wait();
          merge_records<D, G, FP8>(p, b, h, 0, npre, reinterpret_cast<float*>(smem), C::kThreads);
        }
      } else {
        for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
          const size_t o = (static_cast<size_t>(b) * p.hq + hq0) * D + e;
          if (p.out_fp32) reinterpret_cast<float*>(p.out)[o] = 0.f;
          else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
        }
      }
    }
    end_wait();
    return;
  }
  if (s >= nsplit) {
    end_wait();
    return;
  }
  const int nloc = min(nblk, blk0 + p.split_blocks) - blk0;

  // Fused append: the CTA holding sequence b's last block stores the step's new token (kv
  // head h) into the pool -- what the append kernel would store -- and writes it into its
  // copy of that block before reading it, so the block need not be re-read after the store.
  // A slot that is not position len - 1 of the sequence's table is stored but not patched in
  // (the decode then reads the pool as the TMA found it) and flagged.
  constexpr int kRowChunks = D / 8;  // 16-byte chunks of a bf16 row
  int patch_it = -1;                 // local index of the block to patch
  uint4 newrow = make_uint4(0u, 0u, 0u, 0u);  // lanes < 2 kRowChunks: chunk (lane mod kRowChunks)
                                              // of the new K (lane < kRowChunks) or V row, as stored
  if constexpr (!CAS) {
    if (p.fused && (nblk - 1) / p.split_blocks == s) {
      const int64_t slot = p.new_slots[b];
      if (slot >= 0) {
        const int lastit = nblk - 1 - blk0;
        const int64_t want = static_cast<int64_t>(p.block_tables[static_cast<size_t>(b) * p.max_blocks + nblk - 1]) *
                                 kBlockSize + (len - 1) % kBlockSize;
        const bool in_pool = slot < static_cast<int64_t>(p.num_blocks) * kBlockSize;
        if (warp == lastit % NWC && lane < 2 * kRowChunks) {
          const bool isv = lane >= kRowChunks;
          const int c = lane % kRowChunks;
          const size_t src = (static_cast<size_t>(b) * p.hkv + h) * kRowChunks + c;
          newrow = reinterpret_cast<const uint4*>(isv ? p.v_new : p.k_new)[src];
          const size_t dst = (static_cast<size_t>(slot) * p.hkv + h) * kRowChunks + c;
          if constexpr (FP8) {
            const uint2 code = e4m3_quant8(newrow, p.scales[(isv ? p.hkv : 0) + h]);
            newrow = make_uint4(code.x, code.y, 0u, 0u);
            if (in_pool) reinterpret_cast<uint2*>(isv ? p.v_pool : p.k_pool)[dst] = code;
          } else {
            if (in_pool) reinterpret_cast<uint4*>(isv ? p.v_pool : p.k_pool)[dst] = newrow;
          }
        }
        if (slot == want && in_pool) patch_it = lastit;
        else if (threadIdx.x == 0) set_flag(p.status, PKV_DEVFLAG_BAD_SLOT);
      }
    }
  }

  // q as the B operand of the score product: column n = head gid of the group (zero
  // columns past G), k = head_dim; one pair of bf16 words per k-step
  uint32_t qb[KS][2];
  int qexp = 0;  // E4M3: q of head gid scaled by 2^qexp into fp16's range
  if (warp < NWC) {
    const bool live = gid < G;
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(b) * p.hq + hq0 + (live ? gid : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      if constexpr (FP8) {  // the permuted order: dims tig*D/4 + 4kk + {0, 1} | {2, 3}
        qb[kk][0] = live ? qr[tig * (D / 8) + 2 * kk] : 0u;
        qb[kk][1] = live ? qr[tig * (D / 8) + 2 * kk + 1] : 0u;
      } else {
        qb[kk][0] = live ? qr[kk * 8 + tig] : 0u;      // dims 16kk + 2tig, +1
        qb[kk][1] = live ? qr[kk * 8 + 4 + tig] : 0u;  // dims 16kk + 8 + 2tig, +1
      }
    }
    if constexpr (FP8) {
      // the head's largest |q| (over the 4 lanes of equal gid) goes to 2^13 .. 2^14
      float amax = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qb[kk][e])), fabsf(bf16_hi(qb[kk][e]))));
      amax = fmaxf(amax, shfl_xor(amax, 1));
      amax = fmaxf(amax, shfl_xor(amax, 2));
      qexp = amax > 0.f ? 13 - ilogbf(amax) : 0;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          qb[kk][e] = pack_f16(ldexpf(bf16_lo(qb[kk][e]), qexp), ldexpf(bf16_hi(qb[kk][e]), qexp));
    }
  }
  if (threadIdx.x == NWC * 32) tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v);
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // log2-domain score scale of this thread's two heads (2tig, 2tig+1); E4M3: times the K
  // scale and 2^-qexp of that head
  float sscale0 = p.score_scale, sscale1 = p.score_scale;
  if constexpr (FP8) {
    const int e0 = __shfl_sync(kFull, qexp, 4 * (2 * tig)), e1 = __shfl_sync(kFull, qexp, 4 * (2 * tig + 1));
    const float ks = p.score_scale * p.scales[h];
    sscale0 = ldexpf(ks, -e0);
    sscale1 = ldexpf(ks, -e1);
  }
  bool timed_out = false;

  if (warp == NWC) {
    // ================================================================ producer warp
    if (p.test_producer_delay_cycles > 0) spin_cycles(p.test_producer_delay_cycles);
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
            // an id outside the pool reads a box entirely outside the tensor: zeros
            const int row0 = (pb >= 0 && pb < p.num_blocks) ? pb * kBlockSize : -kBlockSize;
            mbar_arrive_expect_tx(&full_bar[st], 2 * C::kRingTile);
            if constexpr (FP8) {  // one plain box of 16 rows x D codes per tile
              tma_load_3d(k_tiles + st * C::kRingTile, &tm_k, 0, h, row0, &full_bar[st]);
              tma_load_3d(v_tiles + st * C::kRingTile, &tm_v, 0, h, row0, &full_bar[st]);
            } else {
#pragma unroll
              for (int hf = 0; hf < C::kHalves; ++hf) {
                tma_load_3d(k_tiles + st * C::kRingTile + hf * 2048, &tm_k, hf * 64, h, row0, &full_bar[st]);
                tma_load_3d(v_tiles + st * C::kRingTile + hf * 2048, &tm_v, hf * 64, h, row0, &full_bar[st]);
              }
            }
          }
        }
        timed_out = __shfl_sync(kFull, timed_out, 0);
        if (timed_out) break;
        issued = it + 1;
      }
      ids = next;
    }
    if (lane == 0) {  // every issued copy must land before the CTA reuses or releases the ring
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        if (!mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1)) {
          set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
          break;
        }
    }
    __syncwarp();
  }

  // per thread: heads 2tig, 2tig+1 of the group (running max, this thread's share of the
  // running sum) and O^T fragments: o[mt] = dims 16mt + gid (+8) x heads 2tig, 2tig+1
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  if (warp < NWC) {
    // ================================================================ consumer warps
    const int mi = lane >> 3;
    const long long wait_limit = p.test_consumer_wait_cycles > 0 ? p.test_consumer_wait_cycles : kWaitLimitCycles;
    for (int it = warp; it < nloc; it += NWC) {
      const int sg = it % STAGES;
      if (!mbar_wait(&full_bar[sg], (it / STAGES) & 1, wait_limit)) {
        if (lane == 0) set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
        timed_out = true;
        break;
      }
      uint32_t kb = smem_u32(k_tiles + sg * C::kRingTile);
      uint32_t vb = smem_u32(v_tiles + sg * C::kRingTile);
      const int valid = min(kBlockSize, len - (blk0 + it) * kBlockSize);  // >= 1
      if (it == patch_it) {  // fused append: the new token's row (valid - 1) of this block
        if (lane < 2 * kRowChunks) {
          const bool isv = lane >= kRowChunks;
          const int c = lane % kRowChunks;
          if constexpr (FP8) {  // the raw codes (8 of them: half of a swizzled 16-byte chunk)
            uint8_t* rowp =
                (isv ? v_tiles : k_tiles) + sg * C::kRingTile + e4m3_off<D>(valid - 1, c >> 1) + (c & 1) * 8;
            *reinterpret_cast<uint2*>(rowp) = make_uint2(newrow.x, newrow.y);
          } else {
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(swz_addr<D>(isv ? vb : kb, valid - 1, c)),
                         "r"(newrow.x), "r"(newrow.y), "r"(newrow.z), "r"(newrow.w)
                         : "memory");
          }
        }
        __syncwarp();
      }
      // ---- S^T = K q^T: rows = tokens gid, gid+8; columns = heads 2tig, 2tig+1
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t vr[4][D / 32];  // E4M3: V codes gid*D/8 .. +D/8 of tokens 2tig, 2tig+1, 2tig+8, 2tig+9
      if constexpr (FP8) {
        // K codes tig*D/4 .. +D/4 of tokens gid and gid + 8, each word one k-step's pairs
        constexpr int KCH = D / 64;  // 16-byte chunks per token and lane
        uint4 kr[2][KCH];
        const uint8_t* kt = k_tiles + sg * C::kRingTile;
        const uint8_t* vt = v_tiles + sg * C::kRingTile;
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            kr[r][c] = *reinterpret_cast<const uint4*>(kt + e4m3_off<D>(gid + 8 * r, tig * KCH + c));
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint32_t w0 = u4_word(kr[0][kk / 4], kk % 4), w1 = u4_word(kr[1][kk / 4], kk % 4);
          mma16<FP8>(sc, e4m3_lo(w0), e4m3_lo(w1), e4m3_hi(w0), e4m3_hi(w1), qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int tok = 2 * tig + (t & 1) + 8 * (t >> 1);
          if constexpr (D == 128) {
            const uint4 v = *reinterpret_cast<const uint4*>(vt + e4m3_off<D>(tok, gid));
            vr[t][0] = v.x;
            vr[t][1] = v.y;
            vr[t][2] = v.z;
            vr[t][3] = v.w;
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(vt + e4m3_off<D>(tok, gid >> 1) + (gid & 1) * 8);
            vr[t][0] = v.x;
            vr[t][1] = v.y;
          }
        }
        // both tiles are in registers: the ring slot goes back (the reads went through the
        // generic proxy, the refill comes through the async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[sg]);
      } else {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(swz_addr<D>(kb, (lane & 7) + 8 * (mi & 1), 2 * kk + (mi >> 1)), a0, a1, a2, a3);
          mma16<FP8>(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = gid + 8 * (e >> 1);
        sc[e] = tok < valid ? sc[e] * ((e & 1) ? sscale1 : sscale0) : -INFINITY;
      }
      // ---- online softmax per head: block max over the 16 tokens (lanes of equal tig)
      float bm0 = fmaxf(sc[0], sc[2]), bm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) {
        bm0 = fmaxf(bm0, shfl_xor(bm0, m));
        bm1 = fmaxf(bm1, shfl_xor(bm1, m));
      }
      const float mn0 = fmaxf(mrun[0], bm0), mn1 = fmaxf(mrun[1], bm1);
      const bool moved = __any_sync(kFull, (mn0 > mrun[0]) || (mn1 > mrun[1]));
      if (moved) {
        const float al0 = fast_exp2(mrun[0] - mn0), al1 = fast_exp2(mrun[1] - mn1);  // 2^-inf = 0 at start
        mrun[0] = mn0;
        mrun[1] = mn1;
        lrun[0] *= al0;
        lrun[1] *= al1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
      }
      const float p0 = fast_exp2(sc[0] - mrun[0]), p1 = fast_exp2(sc[1] - mrun[1]);
      const float p2 = fast_exp2(sc[2] - mrun[0]), p3 = fast_exp2(sc[3] - mrun[1]);
      lrun[0] += p0 + p2;
      lrun[1] += p1 + p3;
      // ---- P^T as the B operand: transpose (token, head-pair) fragments to (head, token-pair)
      uint32_t h01, l01, h23, l23;
      split16<FP8>(p0, p1, h01, l01);  // token gid: heads 2tig, 2tig+1
      split16<FP8>(p2, p3, h23, l23);  // token gid + 8
      const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23);  // head gid: tokens 2tig.., 8 + 2tig..
      const uint32_t bl0 = movm_t(l01), bl1 = movm_t(l23);
      if constexpr (FP8) {
        // ---- O^T += V^T P^T: code word i of each token holds dims gid*D/8 + 4i .. + 3, the
        // rows gid and gid + 8 of m-tiles 2i and 2i + 1; a byte permute pairs tokens
        // (2tig, 2tig+1) and (2tig+8, 2tig+9)
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const uint32_t x01 = __byte_perm(vr[0][i], vr[1][i], 0x5140), y01 = __byte_perm(vr[0][i], vr[1][i], 0x7362);
          const uint32_t x89 = __byte_perm(vr[2][i], vr[3][i], 0x5140), y89 = __byte_perm(vr[2][i], vr[3][i], 0x7362);
          const uint32_t e0 = e4m3_lo(x01), e1 = e4m3_hi(x01), e2 = e4m3_lo(x89), e3 = e4m3_hi(x89);
          mma16<FP8>(o[2 * i], e0, e1, e2, e3, bh0, bh1);
          mma16<FP8>(o[2 * i], e0, e1, e2, e3, bl0, bl1);
          const uint32_t f0 = e4m3_lo(y01), f1 = e4m3_hi(y01), f2 = e4m3_lo(y89), f3 = e4m3_hi(y89);
          mma16<FP8>(o[2 * i + 1], f0, f1, f2, f3, bh0, bh1);
          mma16<FP8>(o[2 * i + 1], f0, f1, f2, f3, bl0, bl1);
        }
      } else {
        // ---- O^T += V^T P^T: m-tile mt = dims 16mt .. 16mt + 15
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(swz_addr<D>(vb, (lane & 7) + 8 * (mi >> 1), 2 * mt + (mi & 1)), a0, a1, a2, a3);
          mma16<FP8>(o[mt], a0, a1, a2, a3, bh0, bh1);
          mma16<FP8>(o[mt], a0, a1, a2, a3, bl0, bl1);
        }
      }
      // The ring tiles were read with ldmatrix (generic proxy) and the producer refills them
      // with TMA (async proxy): without this fence the refill can land while a read of the
      // stage is still pending (seen as wrong output dims in repeated runs).  (E4M3: the
      // slot went back right after the loads.)
      if constexpr (!FP8) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[sg]);
      }
    }
  }

  // ================================================================ merge the consumer warps
  __syncthreads();  // ring drained (every issued copy landed and was consumed)
  float* mw = reinterpret_cast<float*>(smem);  // [NWC][G] max
  float* lw = mw + NWC * G;                    // [NWC][G] sum
  float* aw = lw + NWC * G;                    // [NWC][G][D] unnormalised output
  if (warp < NWC) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = lrun[j];
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) l += shfl_xor(l, m);
      const int g = 2 * tig + j;
      if (g < G) {
        if (gid == 0) {
          mw[warp * G + g] = mrun[j];
          lw[warp * G + g] = l;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // rows gid and gid + 8 of m-tile mt: dims 16mt + gid and + 8 (E4M3: gid*D/8 + 2mt, + 1)
          const int d0 = FP8 ? gid * (D / 8) + 2 * mt : 16 * mt + gid;
          const int d1 = FP8 ? d0 + 1 : d0 + 8;
          aw[(warp * G + g) * D + d0] = o[mt][j];
          aw[(warp * G + g) * D + d1] = o[mt][2 + j];
        }
      }
    }
  }
  __syncthreads();

  const size_t out_row0 = static_cast<size_t>(b) * p.hq + hq0;
  const bool single = (nsplit == 1 && npre == 0);
  const bool with_prefix = CAS && !defer && (nsplit == 1 && npre > 0);
  const size_t prec0 = (static_cast<size_t>(b) * p.hkv + h) * p.rec_slots;
  if (CAS && with_prefix) {
    // One partition plus the shared-prefix records: per head the total max over the warps
    // and the records, each part's weight and the denominator (the records' (m, l) pairs
    // come in one round trip), then per element the weighted sum with every record's
    // output loaded independently of the others.
    pdl_wait();
    float* pml = aw + NWC * G * D;           // [npre][G][2] records' max and sum
    float* wt = pml + kMaxPrefixRecords * G * 2;  // [NWC + npre][G] weights, then [G] 1 / denominator
    for (int i = threadIdx.x; i < npre * G * 2; i += C::kThreads) pml[i] = __ldcg(&p.part_ml[prec0 * G * 2 + i]);
    __syncthreads();
    if (threadIdx.x < G) {
      const int g = threadIdx.x;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NWC; ++w) M = fmaxf(M, mw[w * G + g]);
      for (int j = 0; j < npre; ++j) M = fmaxf(M, pml[(j * G + g) * 2]);
      float den = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NWC; ++w) {
          const float x = fast_exp2(mw[w * G + g] - M);  // warps without blocks: 0
          wt[w * G + g] = x;
          den = fmaf(x, lw[w * G + g], den);
        }
        for (int j = 0; j < npre; ++j) {
          const float x = fast_exp2(pml[(j * G + g) * 2] - M);
          wt[(NWC + j) * G + g] = x;
          den = fmaf(x, pml[(j * G + g) * 2 + 1], den);
        }
      } else {
        for (int w = 0; w < NWC + npre; ++w) wt[w * G + g] = 0.f;
      }
      wt[(NWC + npre) * G + g] = den > 0.f ? 1.f / den : 0.f;
    }
    __syncthreads();
    constexpr int U = 4;  // elements per thread in flight
    for (int e0 = threadIdx.x; e0 < G * D; e0 += U * C::kThreads) {
      float num[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = e0 + u * C::kThreads;
        num[u] = 0.f;
        if (e < G * D) {
          const int g = e / D, d = e % D;
#pragma unroll
          for (int w = 0; w < NWC; ++w) num[u] = fmaf(wt[w * G + g], aw[(w * G + g) * D + d], num[u]);
          if constexpr (FP8) num[u] *= 7.52316384526264e-37f;  // 2^-120: the E4M3 record units
        }
      }
      for (int j = 0; j < npre; ++j) {
        const float* acc = p.part_acc + ((prec0 + j) * G) * D;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = e0 + u * C::kThreads;
          if (e < G * D) num[u] = fmaf(wt[(NWC + j) * G + e / D], __ldcg(&acc[e]), num[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = e0 + u * C::kThreads;
        if (e >= G * D) continue;
        const int g = e / D;
        float ov = num[u] * wt[(NWC + npre) * G + g];
        if constexpr (FP8) ov = (ov * 1152921504606846976.0f) * (p.scales[p.hkv + h] * 1152921504606846976.0f);
        const size_t oi = out_row0 * D + e;
        if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = ov;
        else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(ov);
      }
    }
  } else {
    for (int e = threadIdx.x; e < G * D; e += C::kThreads) {
      const int g = e / D, d = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NWC; ++w) M = fmaxf(M, mw[w * G + g]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < NWC; ++w) {
        const float wt = fast_exp2(mw[w * G + g] - M);  // warps without blocks: 2^-inf = 0
        num = fmaf(wt, aw[(w * G + g) * D + d], num);
        den = fmaf(wt, lw[w * G + g], den);
      }
      if constexpr (FP8) num *= 7.52316384526264e-37f;  // 2^-120: the E4M3 record units
      if (single) {
        float ov = num / den;
        if constexpr (FP8) ov = (ov * 1152921504606846976.0f) * (p.scales[p.hkv + h] * 1152921504606846976.0f);
        const size_t oi = (out_row0 + g) * D + d;
        if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = ov;
        else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(ov);
      } else {
        const size_t rec = prec0 + p.pre_slots + s;
        p.part_acc[(rec * G + g) * D + d] = num;
        if (d == 0) {
          p.part_ml[(rec * G + g) * 2 + 0] = M;
          p.part_ml[(rec * G + g) * 2 + 1] = den;
        }
      }
    }
  }
  // A record was written (or, for one partition, the output): the merge kernel that
  // follows combines the records.  A cascade grid completes only after the prefix pass,
  // whose records the merge kernel also reads.
  end_wait();
}

}  // namespace pkv
