// cascade_prefix_mma.cu -- the shared-prefix pass of cascade decode for small member groups
// over an E4M3 pool (members x G <= 32 query rows per kv head), on mma.sync.
//
// habr.com/ru/articles/1021832, section 7 "Тот самый Cache Read", and
// actionbridge.io chapter 8, the PagedAttention paragraph (parallel sampling, best-of-8: the
// samples share the prompt's blocks): every member of a group reads the same prefix blocks,
// so the prefix part of their decode attention is computed once per group, as the exact
// split of section 3 ("Вспомним FlashAttention") -- per query row a running max m (log2
// units), a running sum l and an unnormalised output -- and merged with each sequence's own
// blocks by the merge kernel.  The tcgen05 pass (cascade_prefix_tc.cu) is built for groups
// that fill its 128-row tiles; a best-of-8 fork (8 members x 4 heads = 32 rows) fills a
// quarter of one.  Here each 16-token block and each 16-row slice of the group is
//
//   S [16 rows x 16 tokens] = Q [16 x D] K^T     (mma.sync m16n8k16, fp16 in, fp32 out)
//   P = 2^(S * scale - m)                         (registers: S's accumulators are the A
//                                                  operand of the next product as they are)
//   O [16 x D]            += P [16 x 16] V [16 x D]
//
// The codes go from the staged tile straight into the MMA fragments, with no expanded copy:
//   - the score product contracts over the head dimension, which any permutation applied to
//     both q and K leaves unchanged; lane (gid, tig) takes dims tig*D/4 .. +D/4 of every
//     k-step's pairs, so its K operand is D/4 consecutive codes of token gid (one or two
//     16-byte loads), and cvt.rn.f16x2.e4m3x2 turns each code pair into one fragment
//     register; q takes the same permutation once (ready-made A fragments in shared memory);
//   - the output product's column n of n-tile j is dim n*D/8 + j, so a lane's V operand is
//     D/8 consecutive codes of each of its four tokens; byte permutes pair the codes of two
//     tokens before the expansion; the output rows come back with the same map.
// The tiles are stored with the 128-byte (D = 128) or 64-byte (D = 64) swizzle (16-byte
// chunk c of row r at chunk c ^ (r mod 8), or c ^ ((r / 2) mod 4)), under which these loads
// meet no bank conflicts.  E4M3 codes expand to fp16 exactly; q is scaled
// per row by a power of two into fp16's range (folded into the row's score scale with the
// K scale), the weights are fp16, and the V scale is applied by the merge kernel.  The
// reference max of a row moves only when a block's max exceeds it by more than 2^8, so the
// weights stay <= 256 and O is rescaled rarely.
//
// CTA = one (kv head, prefix, split of the prefix's blocks), four warps and no producer
// warp (its registers would cost a CTA per SM): warp w takes the 16-row slice w % MT of the
// group and the block stream w / MT, i.e. blocks w / MT, w / MT + 4 / MT, ...; each stream
// has four slots of a ring of 16-token K and V tiles, which the stream's own MT warps fill
// with 16-byte cp.async copies (block ids 32 at a time in every warp's lanes).  Per block:
// wait for this thread's copies of the block, meet the other slice's warp at the stream's
// named barrier (its copies have landed, and it has read the previous block), refill the
// previous block's slot with the block DEPTH - 1 ahead, then compute from the tile.  No
// thread waits on another thread's flag, and no single lane issues the copies (a loading
// lane's tensor-map copies had stood on every block's critical path).  q sits in shared
// memory as ready-made A fragments.  At the end the warps of a slice combine their (m, l, O)
// through shared memory and one of them writes the split's record per row.  128 registers
// and 40 KiB (D = 128, 32 rows): four CTAs fit an SM; the host plans two, so that decode
// CTAs stream the sequences' own blocks beside the pass.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "cascade.cuh"
#include "mma_ops.cuh"
#include "pkv_device.cuh"

namespace pkv {

template <int D, int MT>
struct MmaPrefixCfg {
  static constexpr int kStreams = 4 / MT;              // warps per 16-row slice = block streams
  static constexpr int kThreads = 128;
  static constexpr int kDepth = 4;                     // ring slots per stream
  static constexpr int kStages = kDepth * kStreams;
  static constexpr int kTile = kBlockSize * D;         // one K or V tile of codes
  static constexpr int kRowChunks = D / 16;            // 16-byte chunks of a token's codes
  static constexpr int kTileChunks = kBlockSize * kRowChunks;
  static constexpr int kCopyThreads = 32 * MT;         // the warps of a stream copy its stages
  static constexpr int kTileCopies = kTileChunks / kCopyThreads;  // per thread and tile
  static constexpr int kKS = D / 16;                   // k-steps of the score product
  static constexpr int kNT = D / 8;                    // n-tiles of the output product
  static constexpr int kDQ = D / 4;                    // score-product dims per lane
  static constexpr int kFrag = 4 * kNT + 4;            // per lane: O fragments, (m, l) of 2 rows
  static constexpr int kScratchBytes = (kStreams - 1) * MT * 32 * kFrag * 4;
  static constexpr int kRingBytes = 2 * kStages * kTile;
  static constexpr int kOffQ = kRingBytes;             // q fragments [slice][k-step][lane] x 16 B
  static constexpr int kSmemBytes = kOffQ + MT * kKS * 32 * 16;
  static constexpr int kMinCtas = 4;                   // CTAs per SM the registers are capped for
  static constexpr float kLazy = 8.f;                  // log2 of the largest weight before a rescale
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(MT == 1 || MT == 2, "16 or 32 query rows");
  static_assert(kScratchBytes <= kRingBytes, "the merge scratch reuses the ring");
  static_assert(kTileChunks % kCopyThreads == 0 && kTileCopies >= 1, "whole copies per thread");
};

namespace {

// 2^x by the hardware approximation with subnormal inputs and results flushed to zero
__device__ __forceinline__ float exp2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16 bytes global -> shared through L2 only; with valid false nothing is read and the
// destination is zero-filled
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// the warps of one block stream meet: barrier 1 + stream among its MT warps (two streams
// when MT = 2)
template <int MT>
__device__ __forceinline__ void stream_sync(int st) {
  if constexpr (MT == 1) {
    __syncwarp();
  } else {
    static_assert(MT == 2, "two streams of two warps");
    if (st == 0) asm volatile("bar.sync 1, 64;" ::: "memory");
    else asm volatile("bar.sync 2, 64;" ::: "memory");
  }
}

}  // namespace

template <int D, int MT>
__global__ void __launch_bounds__(MmaPrefixCfg<D, MT>::kThreads, MmaPrefixCfg<D, MT>::kMinCtas)
    cascade_prefix_mma_kernel(const PrefixParams p) {
  using C = MmaPrefixCfg<D, MT>;
  constexpr int KS = C::kKS, NT = C::kNT, NS = C::kStreams, DEPTH = C::kDepth;
  constexpr int KCH = C::kDQ / 16;  // 16-byte chunks of a lane's K operand per token
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* k_tiles = smem;
  uint8_t* v_tiles = smem + C::kStages * C::kTile;
  uint4* qs = reinterpret_cast<uint4*>(smem + C::kOffQ);

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
  int plen = p.prefix_lens[pfx];
  int members = m1 - m0;
  if (members < 0 || members > p.max_members) {
    if (threadIdx.x == 0 && split == 0 && h == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    members = max(0, min(members, p.max_members));
  }
  const int G = p.group;
  const int rows = min(members * G, 16 * MT);  // the host picks this pass for groups of <= 16 MT rows
  if (rows == 0) return;
  if (plen < 0 || plen > p.max_prefix_blocks * kBlockSize || (plen & (kBlockSize - 1))) {
    if (threadIdx.x == 0 && split == 0 && h == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    plen = max(0, min(plen, p.max_prefix_blocks * kBlockSize)) & ~(kBlockSize - 1);
  }
  const int pblocks = plen / kBlockSize;
  const int blk0 = min(pblocks, split * p.split_blocks);
  const int nloc = min(pblocks, blk0 + p.split_blocks) - blk0;
  const int32_t* table = p.prefix_tables + static_cast<size_t>(pfx) * p.max_prefix_blocks + blk0;

  const int mt = warp % MT, st = warp / MT;
  // ---- this warp's stream: stream-local stage k is block st + k NS of the split, in slot
  // st + (k mod DEPTH) NS of the ring, copied by the stream's MT warps together
  const int nk = nloc > st ? (nloc - st + NS - 1) / NS : 0;
  auto slot = [&](int k) { return st + (k % DEPTH) * NS; };
  int ids_cur = lane < nk ? table[st + lane * NS] : 0;  // block ids of stages 32 j + lane, 32 (j + 1) + lane
  int ids_next = 32 + lane < nk ? table[st + (32 + lane) * NS] : 0;
  // this thread's chunks of a tile: chunk c = copy thread + i * copy threads, token c / (D/16)
  const int ct = mt * 32 + lane;
  const size_t tok_stride = static_cast<size_t>(p.hkv) * D;
  // stage k of the stream (one commit group, empty past the last stage); the warps of the
  // stream call it with the same k, converged
  auto issue = [&](int k) {
    if (k < nk) {
      if (k > 0 && k % 32 == 0) {
        ids_cur = ids_next;
        ids_next = k + 32 + lane < nk ? table[st + (k + 32 + lane) * NS] : 0;
      }
      const int pb = __shfl_sync(kFull, ids_cur, k % 32);
      const bool ok = pb >= 0 && pb < p.num_blocks;
      if (!ok && ct == 0) set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
      // an id outside the pool reads nothing: the tiles are zero-filled
      const size_t row0 = (static_cast<size_t>(ok ? pb : 0) * kBlockSize * p.hkv + h) * D;
      uint8_t* kt = k_tiles + slot(k) * C::kTile;
      uint8_t* vt = v_tiles + slot(k) * C::kTile;
#pragma unroll
      for (int i = 0; i < C::kTileCopies; ++i) {
        const int c = ct + i * C::kCopyThreads;
        const int tok = c / C::kRowChunks, ch = c % C::kRowChunks;
        const size_t g = row0 + tok * tok_stride + ch * 16;
        const int so = e4m3_off<D>(tok, ch);
        cp_async16(kt + so, p.k_codes + g, ok);
        cp_async16(vt + so, p.v_codes + g, ok);
      }
    }
    cp_async_commit();
  };
  // the first DEPTH - 1 stages go out now, before the member rows and q are read (their
  // round trips overlap the copies' latency)
#pragma unroll
  for (int k = 0; k < DEPTH - 1; ++k) issue(k);

  // ---- this warp's rows: slice mt, rows 16 mt + gid and 16 mt + gid + 8
  int rb[2] = {0, 0}, rg[2] = {0, 0};
  bool rv[2] = {false, false};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = 16 * mt + gid + 8 * i;
    rv[i] = row < rows;
    if (rv[i]) {
      rg[i] = row % G;
      rb[i] = p.seqs[m0 + row / G];
      if (rb[i] < 0 || rb[i] >= p.batch) {
        set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
        rv[i] = false;
        rb[i] = 0;
      }
    }
  }
  constexpr float kVUnit = 7.52316384526264e-37f;  // 2^-120: the decode kernel's E4M3 record units
  auto record = [&](int i) { return ((static_cast<size_t>(rb[i]) * p.hkv + h) * p.rec_slots + split) * G + rg[i]; };

  if (nloc == 0) {  // an empty split: m = -inf, l = 0, o = 0 (no copies were issued)
    if (st == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (!rv[i]) continue;
        const size_t base = record(i);
        if (tig == 0) {
          p.part_ml[base * 2 + 0] = -INFINITY;
          p.part_ml[base * 2 + 1] = 0.f;
        }
        float4* dst = reinterpret_cast<float4*>(p.part_acc + base * D + tig * (D / 4));
#pragma unroll
        for (int q = 0; q < D / 16; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }

  // ---- q of the two rows as A fragments of the score product, in the permuted dim order:
  // k-step kk, lane tig: dims tig * D/4 + 4 kk + {0, 1} (a0 / a1) and + {2, 3} (a2 / a3);
  // every warp finds its rows' scales, the slice's stream-0 warp stores the fragments
  float ss[2] = {0.f, 0.f};  // log2-domain score scale of the two rows
  {
    const float ks = p.score_scale * p.scales[h];
    uint32_t qa[KS][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t w[C::kDQ / 2];
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<size_t>(rb[i]) * p.hq + h * G + rg[i]) * D + tig * C::kDQ);
#pragma unroll
      for (int c = 0; c < C::kDQ / 8; ++c) {
        const uint4 v = rv[i] ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < C::kDQ / 2; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
      amax = fmaxf(amax, shfl_xor(amax, 1));
      amax = fmaxf(amax, shfl_xor(amax, 2));
      const int qexp = amax > 0.f ? 13 - ilogbf(amax) : 0;  // the row's largest |q| to 2^13 .. 2^14
      ss[i] = ldexpf(ks, -qexp);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint32_t x0 = w[2 * kk], x1 = w[2 * kk + 1];  // dims 4kk, 4kk+1 | 4kk+2, 4kk+3
        qa[kk][i] = pack_f16(ldexpf(__uint_as_float(x0 << 16), qexp), ldexpf(__uint_as_float(x0 & 0xffff0000u), qexp));
        qa[kk][2 + i] =
            pack_f16(ldexpf(__uint_as_float(x1 << 16), qexp), ldexpf(__uint_as_float(x1 & 0xffff0000u), qexp));
      }
    }
    if (st == 0) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) qs[(mt * KS + kk) * 32 + lane] = make_uint4(qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }
  }
  __syncthreads();  // the q fragments are in shared memory

  // per lane: rows gid (e = 0, 1) and gid + 8 (e = 2, 3) of the slice; o[j] holds dims
  // (2 tig) D/8 + j (e = 0, 2) and (2 tig + 1) D/8 + j (e = 1, 3)
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mu[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const uint4* qw = qs + mt * KS * 32 + lane;
  for (int k = 0; k < nk; ++k) {
    // this thread's copies of stage k are done; past the stream's barrier so are its partner
    // warp's, and both warps have read stage k - 1, whose slot takes stage k + DEPTH - 1
    cp_async_wait<DEPTH - 2>();
    stream_sync<MT>(st);
    issue(k + DEPTH - 1);

    const int sg = slot(k);
    const uint8_t* kt = k_tiles + sg * C::kTile;
    const uint8_t* vt = v_tiles + sg * C::kTile;
    // K: token 8 nt + gid, codes tig * D/4 .. + D/4 (n-tile nt)
    uint4 kr[2][KCH];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < KCH; ++c)
        kr[nt][c] = *reinterpret_cast<const uint4*>(kt + e4m3_off<D>(8 * nt + gid, tig * KCH + c));
    // ---- scores, two independent accumulation chains per n-tile
    float acc[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const uint4 a = qw[kk * 32];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t w = u4_word(kr[nt][kk / 4], kk % 4);
        mma16<true>(acc[nt][kk & 1], a.x, a.y, a.z, a.w, e4m3_lo(w), e4m3_hi(w));
      }
    }
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = (acc[nt][0][e] + acc[nt][1][e]) * ss[e >> 1];
    // V is read once the score products are issued (fewer registers live at a time)
    asm volatile("" ::: "memory");
    uint32_t vr[4][NT / 4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int tok = 2 * tig + (t & 1) + 8 * (t >> 1);  // V codes gid * D/8 .. + D/8
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

    // ---- online softmax per row: the block max over the quad's 16 tokens
    float bm[2];
    bm[0] = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    bm[1] = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      bm[i] = fmaxf(bm[i], shfl_xor(bm[i], 1));
      bm[i] = fmaxf(bm[i], shfl_xor(bm[i], 2));
    }
    const bool up0 = bm[0] > mu[0] + C::kLazy, up1 = bm[1] > mu[1] + C::kLazy;
    if (__any_sync(kFull, up0 || up1)) {
      const float n0 = up0 ? bm[0] : mu[0], n1 = up1 ? bm[1] : mu[1];
      const float a0 = exp2_ftz(mu[0] - n0), a1 = exp2_ftz(mu[1] - n1);  // 0 at the start
      mu[0] = n0;
      mu[1] = n1;
      l[0] *= a0;
      l[1] *= a1;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[j][0] *= a0;
        o[j][1] *= a0;
        o[j][2] *= a1;
        o[j][3] *= a1;
      }
    }
    float w[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) w[nt][e] = exp2_ftz(s[nt][e] - mu[e >> 1]);
    l[0] += (w[0][0] + w[0][1]) + (w[1][0] + w[1][1]);
    l[1] += (w[0][2] + w[0][3]) + (w[1][2] + w[1][3]);
    // P as the A operand: tokens 2tig, 2tig+1 (n-tile 0) and 2tig+8, 2tig+9 (n-tile 1)
    const uint32_t pa0 = pack_f16(w[0][0], w[0][1]), pa1 = pack_f16(w[0][2], w[0][3]);
    const uint32_t pa2 = pack_f16(w[1][0], w[1][1]), pa3 = pack_f16(w[1][2], w[1][3]);
    // ---- O += P V: code word i of each token holds dims gid D/8 + 4i .. + 3 = n-tiles
    // 4i .. 4i + 3; a byte permute pairs tokens (2tig, 2tig+1) and (2tig+8, 2tig+9)
#pragma unroll
    for (int i = 0; i < NT / 4; ++i) {
      const uint32_t x01 = __byte_perm(vr[0][i], vr[1][i], 0x5140), y01 = __byte_perm(vr[0][i], vr[1][i], 0x7362);
      const uint32_t x89 = __byte_perm(vr[2][i], vr[3][i], 0x5140), y89 = __byte_perm(vr[2][i], vr[3][i], 0x7362);
      mma16<true>(o[4 * i + 0], pa0, pa1, pa2, pa3, e4m3_lo(x01), e4m3_lo(x89));
      mma16<true>(o[4 * i + 1], pa0, pa1, pa2, pa3, e4m3_hi(x01), e4m3_hi(x89));
      mma16<true>(o[4 * i + 2], pa0, pa1, pa2, pa3, e4m3_lo(y01), e4m3_lo(y89));
      mma16<true>(o[4 * i + 3], pa0, pa1, pa2, pa3, e4m3_hi(y01), e4m3_hi(y89));
    }
  }
  // the stages past the last one were empty groups: nothing is in flight once this returns
  cp_async_wait<0>();

  // ================================================================ combine the streams
  __syncthreads();  // the ring is drained: every copy landed and was read
  float* scratch = reinterpret_cast<float*>(smem);  // [stream - 1][slice][kFrag][32 lanes]
  if (st > 0) {
    float* sc = scratch + ((st - 1) * MT + mt) * C::kFrag * 32 + lane;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[(4 * j + e) * 32] = o[j][e];
    sc[(4 * NT + 0) * 32] = mu[0];
    sc[(4 * NT + 1) * 32] = mu[1];
    sc[(4 * NT + 2) * 32] = l[0];
    sc[(4 * NT + 3) * 32] = l[1];
  }
  __syncthreads();
  if (st != 0) return;
  float M[2] = {mu[0], mu[1]};
#pragma unroll
  for (int k = 1; k < NS; ++k) {
    const float* sc = scratch + ((k - 1) * MT + mt) * C::kFrag * 32 + lane;
    M[0] = fmaxf(M[0], sc[(4 * NT + 0) * 32]);
    M[1] = fmaxf(M[1], sc[(4 * NT + 1) * 32]);
  }
  {
    const float a0 = exp2_ftz(mu[0] - M[0]), a1 = exp2_ftz(mu[1] - M[1]);
    l[0] *= a0;
    l[1] *= a1;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= a0;
      o[j][1] *= a0;
      o[j][2] *= a1;
      o[j][3] *= a1;
    }
  }
#pragma unroll
  for (int k = 1; k < NS; ++k) {  // in stream order: the result does not depend on timing
    const float* sc = scratch + ((k - 1) * MT + mt) * C::kFrag * 32 + lane;
    const float a0 = exp2_ftz(sc[(4 * NT + 0) * 32] - M[0]), a1 = exp2_ftz(sc[(4 * NT + 1) * 32] - M[1]);
    l[0] = fmaf(a0, sc[(4 * NT + 2) * 32], l[0]);
    l[1] = fmaf(a1, sc[(4 * NT + 3) * 32], l[1]);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] = fmaf(a0, sc[(4 * j + 0) * 32], o[j][0]);
      o[j][1] = fmaf(a0, sc[(4 * j + 1) * 32], o[j][1]);
      o[j][2] = fmaf(a1, sc[(4 * j + 2) * 32], o[j][2]);
      o[j][3] = fmaf(a1, sc[(4 * j + 3) * 32], o[j][3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l[i] += shfl_xor(l[i], 1);
    l[i] += shfl_xor(l[i], 2);
  }
  // ---- the split's record of each row: lane tig holds dims 2 tig D/8 .. + D/4
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!rv[i]) continue;
    const size_t base = record(i);
    if (tig == 0) {
      p.part_ml[base * 2 + 0] = M[i];
      p.part_ml[base * 2 + 1] = l[i];
    }
    float4* dst = reinterpret_cast<float4*>(p.part_acc + base * D + tig * (D / 4));
#pragma unroll
    for (int q = 0; q < D / 16; ++q) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int x = 4 * q + u;  // dim 2 tig D/8 + x
        v[u] = (x < NT ? o[x][2 * i] : o[x - NT][2 * i + 1]) * kVUnit;
      }
      dst[q] = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
}

namespace {

// Shared-memory size set once per device and kernel, and the CTAs an SM holds, counted from
// the SM's shared memory (with the per-block reserve), registers (per warp, in units of 256)
// and warps.  0 on failure, with the error in *err.
template <int D, int MT>
int prefix_mma_configure(int device, cudaError_t* err) {
  using C = MmaPrefixCfg<D, MT>;
  // per device, set once; concurrent first calls may both compute it (the same value)
  static std::atomic<int> per_sm_of[64] = {};
  *err = cudaSuccess;
  if (device < 0 || device >= 64) {
    *err = cudaErrorInvalidDevice;
    return 0;
  }
  const int known = per_sm_of[device].load(std::memory_order_acquire);
  if (known > 0) return known;
  auto kern = cascade_prefix_mma_kernel<D, MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
  int smem_sm = 0, reserve = 0, regs_sm = 0, threads_sm = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserve, cudaDevAttrReservedSharedMemoryPerBlock, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, device);
  if (e != cudaSuccess) {
    *err = e;
    return 0;
  }
  const long long smem_cta = static_cast<long long>(C::kSmemBytes) + fa.sharedSizeBytes + reserve;
  const long long regs_warp = (static_cast<long long>(fa.numRegs) * 32 + 255) / 256 * 256;
  const int warps = C::kThreads / 32;
  long long per_sm = smem_sm / smem_cta;
  per_sm = std::min(per_sm, regs_sm / (regs_warp * warps));
  per_sm = std::min(per_sm, static_cast<long long>(threads_sm / 32 / warps));
  per_sm = std::min(per_sm, 32LL);  // the SM's CTA limit
  if (per_sm < 1) {
    *err = cudaErrorInvalidConfiguration;
    return 0;
  }
  per_sm_of[device].store(static_cast<int>(per_sm), std::memory_order_release);
  return static_cast<int>(per_sm);
}

}  // namespace

template <int D, int MT>
int cascade_prefix_mma_ctas_per_sm(int device) {
  cudaError_t e;
  return prefix_mma_configure<D, MT>(device, &e);
}

template <int D, int MT>
cudaError_t launch_cascade_prefix_mma(const PrefixParams& p, dim3 grid, cudaStream_t stream, int device) {
  using C = MmaPrefixCfg<D, MT>;
  cudaError_t e;
  if (prefix_mma_configure<D, MT>(device, &e) == 0) return e;
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
  return cudaLaunchKernelEx(&cfg, cascade_prefix_mma_kernel<D, MT>, p);
}

#define PKV_DEFINE_PREFIX_MMA(D, MT)                                                                               \
  template int cascade_prefix_mma_ctas_per_sm<D, MT>(int);                                                        \
  template cudaError_t launch_cascade_prefix_mma<D, MT>(const PrefixParams&, dim3, cudaStream_t, int);
PKV_DEFINE_PREFIX_MMA(64, 1)
PKV_DEFINE_PREFIX_MMA(64, 2)
PKV_DEFINE_PREFIX_MMA(128, 1)
PKV_DEFINE_PREFIX_MMA(128, 2)
#undef PKV_DEFINE_PREFIX_MMA

}  // namespace pkv

