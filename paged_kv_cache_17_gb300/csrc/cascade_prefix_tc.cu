// cascade_prefix_tc.cu -- the shared-prefix pass of cascade decode on the fifth-generation
// tensor cores (tcgen05 MMAs accumulating in tensor memory).
//
// habr.com/ru/articles/1021832, section 7 "Тот самый Cache Read", and
// ml-canon.vercel.app/54-prefix-caching-cacheblend.html, "Идея и механизм": requests that
// start with the same prompt share that prompt's KV blocks, identical for every one of
// them.  Section 3 of the habr article ("Вспомним FlashAttention") gives the exact split:
// attention over one part of the keys is a running max m, a running sum l and an
// unnormalised output, and parts combine with the rescale exp(m_part - m_total).  So the
// prefix part of every member's decode attention is computed here once per prefix group;
// each sequence's own blocks are handled by the decode kernel, and these partial results
// join its own as extra partitions (merged by the merge kernel after the decode, or in the
// decode CTA).  Per (kv head, prefix) the contraction is [member rows x
// prefix keys], dense and large enough for the 128-row MMAs:
//
//   S [128 rows x 64 keys] = Q [128 x D] K^T          (tcgen05.mma kind::f16, fp32 in TMEM)
//   P = 2^(S * scale - m)                             (one thread per row, CUDA cores)
//   O [128 x D]          += P [128 x 64] V [64 x D]   (P read from TMEM; O stays in TMEM)
//
// CTA = 128 query rows (row r: member r / G, query head h * G + r % G), one kv head, one
// split of the prefix (a run of whole 64-key stages):
//   warps 0-3  softmax: thread r owns row r (TMEM lane r); reads S, writes P as 16-bit
//              pairs back over the stage's own S columns, rescales its O row when its
//              reference max moved, and writes the record; bf16 pools write P as bf16
//              hi + lo (lo = P - hi rounded) and O += P V runs once for each, so the weights
//              keep about 16 bits;
//   warp 4     lane 0 issues every MMA;
//   warp 5     the producer: block ids of the split 32 at a time in its lanes, one TMA box
//              per (block, 64 columns) into the K and V rings as slots come free;
//   warps 6-9  (E4M3 pools) expand each raw stage exactly to fp16 into 16-bit rings.
// S is double-buffered in TMEM, so the tensor cores compute S of stage t + 2 and O of stage
// t while the softmax warps work on stage t + 1.  K and V have rings of their own: a K
// slot is free once S of its stage is done, long before O += P V of that stage, so K of
// stage t + 2 is loaded while stage t is still being weighed.  The reference max of a row
// changes only when the row max exceeds it by more than 2^8 (weights then stay <= 256,
// exact in bf16 and fp16 range), so O is rescaled rarely; the record carries the reference
// max it used.
//
// Each CTA is one chain of dependent steps (S -> weights -> O += P V) whose latency, not
// any one unit's throughput, sets its pace; so two CTAs fit on an SM (shared memory at most
// 98 KiB and 256 TMEM columns each) and their chains interleave.  The host plans E4M3
// passes for two CTAs per SM; bf16 passes for one, so that three decode CTAs share each SM
// with it and stream the sequences' own blocks meanwhile.
// Shared memory: Q (128 x D, 16-bit, 128-byte swizzled, K-major) and K and V rings ([column
// half][64 keys][128 bytes], swizzled by the TMA load; 2 stages each at D = 128, 4 at
// D = 64); E4M3 pools add rings of expanded fp16 tiles (1 stage each at D = 128, 2 at
// D = 64).  TMEM: S (then P) at columns 0 and 64, O at column 128.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "cascade.cuh"
#include "mma_ops.cuh"
#include "pkv_device.cuh"
#include "tc_ops.cuh"

namespace pkv {

template <int D, bool FP8>
struct TcPrefixCfg {
  static constexpr int kRows = 128;             // query rows per CTA: the MMA's M
  static constexpr int kKeys = 64;              // keys per stage: N of S, K of O += P V
  static constexpr int kStageBlocks = kKeys / kBlockSize;
  // stages per K ring and per V ring as loaded, and per ring of expanded 16-bit E4M3 tiles:
  // as deep as two CTAs per SM allow
  static constexpr int kRing = D == 64 ? 4 : 2;
  static constexpr int kExpRing = D == 64 ? 2 : 1;
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kRows * 128;    // one 64-column half of Q
  static constexpr int kHalf16 = kKeys * 128;   // one 64-column half of a 16-bit K or V stage
  static constexpr int kTile16 = kHalves * kHalf16;
  static constexpr int kRaw = FP8 ? kKeys * D : kTile16;  // a K or V stage as loaded
  static constexpr bool kPSplit = !FP8;         // bf16 weights as hi + lo (two P V products)
  static constexpr int kOffQ = 0;
  static constexpr int kOffRawK = kOffQ + kHalves * kQHalf;
  static constexpr int kOffRawV = kOffRawK + kRing * kRaw;
  static constexpr int kOffExpK = kOffRawV + kRing * kRaw;
  static constexpr int kOffExpV = kOffExpK + (FP8 ? kExpRing * kTile16 : 0);
  static constexpr int kOffBar = kOffExpV + (FP8 ? kExpRing * kTile16 : 0);
  static constexpr int kBarBytes = 512;
  static constexpr int kBytes = 1024 + kOffBar + kBarBytes;  // 1024: alignment slack
  static constexpr int kColS = 0, kColO = 128, kTmemCols = 256;
  static constexpr int kSoftWarps = 4, kIssuerWarp = 4, kProducerWarp = 5, kConvWarp0 = 6;
  static constexpr int kConvWarps = FP8 ? 4 : 0;
  static constexpr int kThreads = (kConvWarp0 + kConvWarps) * 32;
  static constexpr int kMinCtas = 2;            // CTAs per SM the registers are capped for
  static constexpr float kLazy = 8.f;           // log2 of the largest weight before a rescale
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(kRaw % 1024 == 0 && kTile16 % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kColO + D <= kTmemCols, "TMEM columns");
  static_assert(2 * (kBytes + 1024) <= 228 * 1024, "two CTAs per SM");
  static_assert((8 * kRing + 7) * 8 + 8 <= kBarBytes, "barriers, TMEM address and abort flag");
};

namespace {

// 2^x by the hardware approximation with subnormal inputs and results flushed to zero
__device__ __forceinline__ float exp2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// wait for a phase, giving up when the CTA has aborted or after the wait limit
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - start > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

}  // namespace

template <int D, bool FP8>
__global__ void __launch_bounds__(TcPrefixCfg<D, FP8>::kThreads, TcPrefixCfg<D, FP8>::kMinCtas)
    cascade_prefix_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const PrefixParams p) {
  using C = TcPrefixCfg<D, FP8>;
  constexpr int R = C::kRing, E = C::kExpRing;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + C::kOffBar);  // [R] K stage landed (TMA)
  uint64_t* vfull = kfull + R;    // [R] V stage landed
  uint64_t* kfree = vfull + R;    // [R] K slot reusable: bf16 S of its stage done, E4M3 expanded
  uint64_t* vfree = kfree + R;    // [R] V slot reusable: bf16 O += P V of its stage done, E4M3 expanded
  uint64_t* ekfull = vfree + R;   // [R] E4M3: K stage expanded
  uint64_t* evfull = ekfull + R;  // [R] E4M3: V stage expanded
  uint64_t* ekfree = evfull + R;  // [R] E4M3: S of the expanded slot's stage done
  uint64_t* evfree = ekfree + R;  // [R] E4M3: O += P V of the expanded slot's stage done
  uint64_t* s_full = evfree + R;  // [2] S of a stage done
  uint64_t* p_full = s_full + 2;  // [2] P of a stage written (one arrival per softmax warp)
  uint64_t* o_done = p_full + 2;  // O += P V of a stage done
  uint64_t* drain = o_done + 1;   // every MMA issued so far done (abort path)
  uint64_t* q_full = drain + 1;   // Q staged (one arrival per softmax warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int pfx = blockIdx.z / p.pre_slots;
  const int split = blockIdx.z % p.pre_slots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();
  // the decode kernel that follows may start now: what it reads before waiting for this
  // grid (the pool after the append) is complete once every CTA is past the wait above
  pdl_launch_dependents();

  // one round trip: the member range and the prefix length
  const int m0 = p.indptr[pfx], m1 = p.indptr[pfx + 1];
  int plen = p.prefix_lens[pfx];
  int members = m1 - m0;
  if (members < 0 || members > p.max_members) {  // the grid covers max_members members
    if (threadIdx.x == 0 && tile == 0 && split == 0 && h == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    members = max(0, min(members, p.max_members));
  }
  const int G = p.group;
  const int rows = members * G;
  if (tile * C::kRows >= rows) return;
  if (plen < 0 || plen > p.max_prefix_blocks * kBlockSize || (plen & (kBlockSize - 1))) {
    if (threadIdx.x == 0 && tile == 0 && split == 0 && h == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    plen = max(0, min(plen, p.max_prefix_blocks * kBlockSize)) & ~(kBlockSize - 1);
  }
  const int pblocks = plen / kBlockSize;
  const int blk0 = min(pblocks, split * p.split_blocks);
  const int blk1 = min(pblocks, blk0 + p.split_blocks);
  const int nstage = (blk1 - blk0 + C::kStageBlocks - 1) / C::kStageBlocks;
  const int32_t* table = p.prefix_tables + static_cast<size_t>(pfx) * p.max_prefix_blocks;

  // ---- the row of a softmax thread
  const bool soft = warp < C::kSoftWarps;
  const int r = threadIdx.x;  // softmax threads: row r of the tile, TMEM lane r
  bool rv = false;
  int rb = 0, rg = 0;
  // the row's sequence (softmax threads; a global load, issued once the setup below is done)
  auto load_row = [&]() {
    const int row = tile * C::kRows + r;
    rv = row < rows;
    if (rv) {
      rg = row % G;
      rb = p.seqs[m0 + row / G];
      if (rb < 0 || rb >= p.batch) {
        set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
        rv = false;
        rb = 0;
      }
    }
  };
  const float vunit = FP8 ? 7.52316384526264e-37f : 1.0f;  // 2^-120: the decode kernel's E4M3 units
  auto write_record = [&](float m, float l, int chunk, const float* o32) {
    // chunk < 0: m and l; else 32 output columns starting at 32 * chunk
    const size_t rec = (static_cast<size_t>(rb) * p.hkv + h) * p.rec_slots + split;
    const size_t base = rec * G + rg;
    if (chunk < 0) {
      p.part_ml[base * 2 + 0] = m;
      p.part_ml[base * 2 + 1] = l;
    } else {
      float4* dst = reinterpret_cast<float4*>(p.part_acc + base * D + 32 * chunk);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(o32[4 * i] * vunit, o32[4 * i + 1] * vunit, o32[4 * i + 2] * vunit,
                             o32[4 * i + 3] * vunit);
    }
  };
  if (nstage == 0) {  // an empty split: m = -inf, l = 0, o = 0
    if (soft) load_row();
    if (soft && rv) {
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.f;
      write_record(-INFINITY, 0.f, -1, z);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) write_record(0.f, 0.f, c, z);
    }
    return;
  }

  if (warp == 0) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == C::kIssuerWarp * 32) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&kfree[i], 1);
      mbar_init(&vfree[i], 1);
      mbar_init(&ekfull[i], 1);
      mbar_init(&evfull[i], 1);
      mbar_init(&ekfree[i], 1);
      mbar_init(&evfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], C::kSoftWarps);  // one arrival per softmax warp
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(q_full, C::kSoftWarps);
    *abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // the setup above reads no global memory, so the producer's first loads start one round
  // trip after the launch; the softmax warps stage Q meanwhile
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- Q rows -> shared memory, K-major 128-byte swizzle (16-bit; fp16 for E4M3 pools)
  const uint32_t q_base = smem_u32(smem + C::kOffQ);
  if (soft) {
    load_row();
    const uint4* qr = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(rb) * p.hq + h * G + rg) * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v = rv ? qr[c] : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (FP8) {
        v.x = pack_f16(bf16_lo(v.x), bf16_hi(v.x));
        v.y = pack_f16(bf16_lo(v.y), bf16_hi(v.y));
        v.z = pack_f16(bf16_lo(v.z), bf16_hi(v.z));
        v.w = pack_f16(bf16_lo(v.w), bf16_hi(v.w));
      }
      st_shared_v4(q_base + (c >> 3) * C::kQHalf + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4), v.x,
                   v.y, v.z, v.w);
    }
    fence_proxy_async_smem();  // read by the tensor cores
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);
  }

  auto fail = [&]() {
    set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
    *abort = 1;
  };
  // the 16-bit K and V tiles of stage t (the raw slots, or for E4M3 the expanded ones)
  auto k_tile = [&](int t) -> uint32_t {
    return FP8 ? smem_u32(smem + C::kOffExpK + (t % E) * C::kTile16) : smem_u32(smem + C::kOffRawK + (t % R) * C::kRaw);
  };
  auto v_tile = [&](int t) -> uint32_t {
    return FP8 ? smem_u32(smem + C::kOffExpV + (t % E) * C::kTile16) : smem_u32(smem + C::kOffRawV + (t % R) * C::kRaw);
  };

  if (warp == C::kIssuerWarp) {
    // ======================================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(C::kRows, C::kKeys, !FP8, false);
      constexpr uint32_t kIdO = idesc_f16(C::kRows, D, !FP8, true);
      // S(t) into TMEM buffer t % 2: D/16 k-steps of 16 head dims (byte 32k of a 128-byte row)
      auto issue_s = [&](int t) {
        const uint32_t kt = k_tile(t);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sdesc_sw128(q_base + (kk >> 2) * C::kQHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(kt + (kk >> 2) * C::kHalf16 + (kk & 3) * 32, 16, 1024);
          mma_f16_ss(tmem + C::kColS + 64 * (t & 1), a, b, kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t & 1]);
        tc_commit(FP8 ? &ekfree[t % E] : &kfree[t % R]);  // the K tile is read
      };
      // O += P(t) V(t): 4 k-steps of 16 keys; P (the A operand) in TMEM over the S columns of
      // stage t (hi at +0, lo at +32, two weights per column); V is MN-major (64 head dims per
      // 128-byte row).  The MMAs run in issue order, so S(t + 2), issued after these into the
      // same columns, overwrites P(t) only once these have read it.
      auto issue_o = [&](int t) {
        const uint32_t pt = tmem + C::kColS + 64 * (t & 1), vt = v_tile(t);
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < C::kKeys / 16; ++j) {
          const uint64_t b = sdesc_sw128(vt + j * 2048, C::kHalf16, 1024);
          mma_f16_ts(tmem + C::kColO, pt + 8 * j, b, kIdO, (t > 0 || j > 0) ? 1u : 0u);
          if constexpr (C::kPSplit) mma_f16_ts(tmem + C::kColO, pt + 32 + 8 * j, b, kIdO, 1u);
        }
        tc_commit(FP8 ? &evfree[t % E] : &vfree[t % R]);  // the V tile is read
        tc_commit(o_done);
      };
      auto wait_k = [&](int t) -> bool {
        return FP8 ? wait_or_abort(&ekfull[t % E], (t / E) & 1, abort) : wait_or_abort(&kfull[t % R], (t / R) & 1, abort);
      };
      auto wait_v = [&](int t) -> bool {
        return FP8 ? wait_or_abort(&evfull[t % E], (t / E) & 1, abort) : wait_or_abort(&vfull[t % R], (t / R) & 1, abort);
      };
      bool ok = wait_or_abort(q_full, 0, abort);  // Q staged by the softmax warps
      for (int t = 0; t < min(2, nstage) && ok; ++t) {
        ok = wait_k(t);
        if (ok) issue_s(t);
      }
      for (int t = 0; t < nstage && ok; ++t) {
        ok = wait_or_abort(&p_full[t & 1], (t >> 1) & 1, abort) && wait_v(t);
        if (!ok) break;
        issue_o(t);
        if (t + 2 < nstage) {
          ok = wait_k(t + 2);
          if (!ok) break;
          issue_s(t + 2);
        }
      }
      if (!ok && !*abort) fail();
      // nothing may run on the tensor cores when the CTA frees its tensor memory
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp == C::kProducerWarp) {
    // ======================================================================== TMA producer
    // block ids of the split, 32 (eight stages) at a time in the lanes, the next 32 in flight;
    // K of stage t + 1 goes before V of stage t (its slot frees earlier: when S of stage
    // t + 1 - R is done, before O += P V of stage t - R)
    const int nblk = blk1 - blk0;
    int ids = lane < nblk ? table[blk0 + lane] : 0;
    int nxt = 32 + lane < nblk ? table[blk0 + 32 + lane] : 0;
    // pool rows of the blocks of stage t (called for t = 0, 1, 2, ... in order); -16 for
    // blocks past the split: a box entirely outside the tensor reads zeros
    auto stage_rows = [&](int t, int (&row0)[C::kStageBlocks]) {
      const int w0 = (t * C::kStageBlocks) & 31;
      if (t > 0 && w0 == 0) {
        ids = nxt;
        const int k = t * C::kStageBlocks + 32 + lane;
        nxt = k < nblk ? table[blk0 + k] : 0;
      }
#pragma unroll
      for (int j = 0; j < C::kStageBlocks; ++j) {
        const int pb = __shfl_sync(kFull, ids, w0 + j);
        row0[j] = -kBlockSize;
        if (t * C::kStageBlocks + j < nblk) {
          if (pb >= 0 && pb < p.num_blocks) row0[j] = pb * kBlockSize;
          else if (lane == 0) set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
        }
      }
    };
    // TMA of one tensor's stage t into ring slot t % R (lane 0)
    auto load = [&](const CUtensorMap* tm, int off_ring, uint64_t* bar, const int (&row0)[C::kStageBlocks], int t) {
      const int st = t % R;
      mbar_arrive_expect_tx(&bar[st], C::kRaw);
#pragma unroll
      for (int j = 0; j < C::kStageBlocks; ++j) {
        if constexpr (FP8) {
          tma_load_3d(smem + off_ring + st * C::kRaw + j * kBlockSize * D, tm, 0, h, row0[j], &bar[st]);
        } else {
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem + off_ring + st * C::kRaw + hf * C::kHalf16 + j * 2048, tm, hf * 64, h, row0[j],
                        &bar[st]);
        }
      }
    };
    // the slot of stage t is free (t >= R): its previous stage is consumed
    auto slot_free = [&](uint64_t* bar, int t) -> bool {
      const bool ok = t < R || wait_or_abort(&bar[t % R], ((t / R) - 1) & 1, abort);
      return __all_sync(kFull, ok);
    };
    int kiss = 0, viss = 0;
    bool ok = true;
    int rk[C::kStageBlocks], rvw[C::kStageBlocks];
    stage_rows(0, rk);
    if (lane == 0) load(&tm_k, C::kOffRawK, kfull, rk, 0);
    kiss = 1;
    for (int t = 0; t < nstage; ++t) {
#pragma unroll
      for (int j = 0; j < C::kStageBlocks; ++j) rvw[j] = rk[j];  // rows of stage t, for V
      if (t + 1 < nstage) {
        stage_rows(t + 1, rk);
        if (!slot_free(kfree, t + 1)) {
          ok = false;
          break;
        }
        if (lane == 0) load(&tm_k, C::kOffRawK, kfull, rk, t + 1);
        kiss = t + 2;
      }
      if (!slot_free(vfree, t)) {
        ok = false;
        break;
      }
      if (lane == 0) load(&tm_v, C::kOffRawV, vfull, rvw, t);
      viss = t + 1;
    }
    if (lane == 0) {
      if (!ok && !*abort) fail();
      // nothing may be in flight when the CTA exits: the last stages issued have landed
      for (int t = max(0, kiss - R); t < kiss; ++t)
        if (!mbar_wait(&kfull[t % R], (t / R) & 1)) break;
      for (int t = max(0, viss - R); t < viss; ++t)
        if (!mbar_wait(&vfull[t % R], (t / R) & 1)) break;
    }
    __syncwarp();
  } else if (!soft) {
    // ======================================================================== E4M3 expansion
    if constexpr (FP8) {
      const int ct = threadIdx.x - C::kConvWarp0 * 32;  // 0 .. 127
      constexpr int kChunks = C::kKeys * (D / 8);  // 8-code chunks per tile
      static_assert((128 / (D / 8)) % 8 == 0, "a thread's rows keep their phase in the swizzle atom");
      // expand one raw tile of stage t into its 16-bit slot, in the producer's order (K of
      // stage t + 1 before V of stage t): K once S of the slot's previous stage is done, V once
      // O += P V of it is done; false once the CTA aborts
      auto expand = [&](int t, bool isv) -> bool {
        bool ok = wait_or_abort(isv ? &vfull[t % R] : &kfull[t % R], (t / R) & 1, abort);
        if (ok && t >= E) ok = wait_or_abort(isv ? &evfree[t % E] : &ekfree[t % E], ((t / E) - 1) & 1, abort);
        if (!ok && !*abort) fail();
        if (ok) {
          // thread ct takes the 8-code chunk c of rows k0, k0 + kRowsStep, ...: the row's phase in
          // its 8-row swizzle atom never changes, so both addresses advance by constants
          constexpr int kRowsStep = 128 / (D / 8);  // rows per pass of the 128 threads (8 or 16)
          const int c = ct % (D / 8), k0 = ct / (D / 8);
          const uint8_t* src = smem + (isv ? C::kOffRawV : C::kOffRawK) + (t % R) * C::kRaw + k0 * D + c * 8;
          const uint32_t dst0 = smem_u32(smem + (isv ? C::kOffExpV : C::kOffExpK) + (t % E) * C::kTile16) +
                                (c >> 3) * C::kHalf16 + (k0 >> 3) * 1024 + (k0 & 7) * 128 + (((c & 7) ^ (k0 & 7)) << 4);
#pragma unroll 4
          for (int i = 0; i < kChunks / 128; ++i) {
            const uint2 w = *reinterpret_cast<const uint2*>(src + i * kRowsStep * D);
            const uint32_t dst = dst0 + i * (kRowsStep / 8) * 1024;
            st_shared_v4(dst, e4m3x2_to_f16x2(static_cast<uint16_t>(w.x & 0xffffu)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.x >> 16)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.y & 0xffffu)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.y >> 16)));
          }
        }
        fence_proxy_async_smem();  // the expanded tile is read by the tensor cores
        // every converter thread reaches this, failed or not, and all leave together
        if (named_sync_or(1, 128, *abort != 0)) return false;
        if (ct == 0) {
          mbar_arrive(isv ? &vfree[t % R] : &kfree[t % R]);    // the raw slot is read
          mbar_arrive(isv ? &evfull[t % E] : &ekfull[t % E]);  // the expanded tile is complete
        }
        return true;
      };
      bool ok = expand(0, false);
      for (int t = 0; t < nstage && ok; ++t) {
        if (t + 1 < nstage) ok = expand(t + 1, false);
        if (ok) ok = expand(t, true);
      }
    }
  } else {
    // ======================================================================== softmax
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sscale = FP8 ? p.score_scale * p.scales[h] : p.score_scale;
    float m_used = -INFINITY, l = 0.f;
    for (int t = 0; t < nstage; ++t) {
      const int b = t & 1;
      bool ok = wait_or_abort(&s_full[b], (t >> 1) & 1, abort);
      if (!__all_sync(kFull, ok)) {  // tcgen05.ld is warp-collective: leave as a warp
        if (!*abort) fail();
        break;
      }
      tc_fence_after();
      const uint32_t scol = tmem + lane_base + C::kColS + 64 * b;
      float sv[64];
      tmem_ld64(scol, sv);
      const int nkeys = min(C::kKeys, (blk1 - blk0 - t * C::kStageBlocks) * kBlockSize);
      // keys past the split (the last stage only) take no part in the extreme below and get
      // weight 0; the row max of the scaled scores is the scale times the max (scale >= 0)
      // or the min (scale < 0) of the raw scores
      const bool partial = nkeys < C::kKeys;
      if (partial) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= nkeys) sv[i] = sscale >= 0.f ? -INFINITY : INFINITY;
      }
      float ext = sv[0];
      if (sscale >= 0.f) {
#pragma unroll
        for (int i = 1; i < 64; ++i) ext = fmaxf(ext, sv[i]);
      } else {
#pragma unroll
        for (int i = 1; i < 64; ++i) ext = fminf(ext, sv[i]);
      }
      const float mx = ext * sscale;
      const bool grow = mx > m_used + C::kLazy;  // always at t = 0 (every stage has a key)
      float alpha = 1.f;
      if (grow) {
        alpha = fast_exp2(m_used - mx);  // 0 at t = 0
        l *= alpha;
        m_used = mx;
      }
      const float negm = -m_used;
      // 2^x of a weight.  E4M3 pools: the flush-to-zero form, fewer instructions (fork step
      // 58.5 -> 56.7 us); exact in effect, as the fp16 weights turn everything below 2^-24
      // into zero anyway.  bf16 pools keep the weights below 2^-126 (no gain measured there).
      auto weight = [](float x) { return FP8 ? exp2_ftz(x) : fast_exp2(x); };
      // P row r: 64 weights 2^(s * scale - m) <= 2^8 as 16-bit pairs over the S columns just
      // read, 16 keys (8 columns) at a time.  bf16 pools: hi at +0, lo at +32 (about 16 bits
      // together), l sums the fp32 weights; E4M3 pools: fp16 weights, l sums the rounded ones,
      // so O / l weighs V by the weights the MMAs use
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[8], wl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int k = 16 * c + 2 * e;
          float a = weight(fmaf(sv[k], sscale, negm));
          float bb = weight(fmaf(sv[k + 1], sscale, negm));
          if (partial) {  // a zero scale makes the masked products NaN: weight 0 by selection
            a = k < nkeys ? a : 0.f;
            bb = k + 1 < nkeys ? bb : 0.f;
          }
          if constexpr (C::kPSplit) {
            w[e] = pack_bf16(a, bb);
            wl[e] = pack_bf16(a - __uint_as_float(w[e] << 16), bb - __uint_as_float(w[e] & 0xffff0000u));
            ls += a + bb;
          } else {
            w[e] = pack_f16(a, bb);
            wl[e] = 0u;
            ls += sum16<true>(w[e]);
          }
        }
        tmem_st8(scol + 8 * c, w);
        if constexpr (C::kPSplit) tmem_st8(scol + 32 + 8 * c, wl);
      }
      tmem_wait_st();
      l += ls;
      // O += P V of stage t - 1 is done.  Waited at every stage, rescale or not: a parity
      // wait is unambiguous only while the barrier is at most one phase past the waiter,
      // and O += P V of stage t cannot start before this warp's arrival below
      if (t > 0) {
        ok = wait_or_abort(o_done, (t - 1) & 1, abort);
        if (!__all_sync(kFull, ok)) {
          if (!*abort) fail();
          break;
        }
      }
      // rescale O where this warp's rows moved their reference max
      if (t > 0 && __any_sync(kFull, grow)) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float o[32];
          tmem_ld32(tmem + lane_base + C::kColO + 32 * ch, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + lane_base + C::kColO + 32 * ch, o);
        }
      }
      tc_fence_before();
      __syncwarp();  // the warp's P rows and O rescales are done
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    // ---- the record: reference max, sum, unnormalised O of the row (the stages before the
    // last were waited in the loop, so the barrier is at the last phase or one past it)
    if (__all_sync(kFull, *abort == 0)) {
      const bool ok = wait_or_abort(o_done, (nstage - 1) & 1, abort);
      if (__all_sync(kFull, ok)) {
        tc_fence_after();
        if (rv) write_record(m_used, l, -1, nullptr);
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float o[32];
          tmem_ld32(tmem + lane_base + C::kColO + 32 * ch, o);
          if (rv) write_record(0.f, 0.f, ch, o);
        }
      } else if (!*abort) {
        fail();
      }
    }
  }

  // ======================================================================== teardown
  // every role is done: the issuer saw its MMAs complete, the producer its loads land
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

namespace {

// Shared-memory size set once per device and kernel, and the CTAs an SM holds, counted from
// the SM's resources: shared memory (each CTA also takes the per-block reserve), registers
// (allocated per warp in units of 256) and warps; then checked against the SM's 512
// tensor-memory columns (an allocation that cannot be met would wait for a CTA that cannot
// finish first).  The runtime's occupancy query was seen to report one CTA where the
// profiler's limits and the runs show two.  0 on failure, with the error in *err.
template <int D, bool FP8>
int prefix_tc_configure(int device, cudaError_t* err) {
  using C = TcPrefixCfg<D, FP8>;
  // per device, set once; concurrent first calls may both compute it (the same value)
  static std::atomic<int> per_sm_of[64] = {};
  *err = cudaSuccess;
  if (device < 0 || device >= 64) {
    *err = cudaErrorInvalidDevice;
    return 0;
  }
  const int known = per_sm_of[device].load(std::memory_order_acquire);
  if (known > 0) return known;
  auto kern = cascade_prefix_tc_kernel<D, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
  // the largest shared-memory carveout, so that every CTA the shared memory can hold fits
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
  const long long smem_cta = static_cast<long long>(C::kBytes) + fa.sharedSizeBytes + reserve;
  const long long regs_warp = (static_cast<long long>(fa.numRegs) * 32 + 255) / 256 * 256;
  const int warps = C::kThreads / 32;
  long long per_sm = smem_sm / smem_cta;
  per_sm = std::min(per_sm, regs_sm / (regs_warp * warps));
  per_sm = std::min(per_sm, static_cast<long long>(threads_sm / 32 / warps));
  if (per_sm < 1 || per_sm * C::kTmemCols > 512) {
    *err = cudaErrorInvalidConfiguration;
    return 0;
  }
  per_sm_of[device].store(static_cast<int>(per_sm), std::memory_order_release);
  return static_cast<int>(per_sm);
}

}  // namespace

template <int D, bool FP8>
int cascade_prefix_tc_ctas_per_sm(int device) {
  cudaError_t e;
  return prefix_tc_configure<D, FP8>(device, &e);
}

template <int D, bool FP8>
cudaError_t launch_cascade_prefix_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixParams& p, dim3 grid,
                                     cudaStream_t stream, int device) {
  using C = TcPrefixCfg<D, FP8>;
  cudaError_t e;
  if (prefix_tc_configure<D, FP8>(device, &e) == 0) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cascade_prefix_tc_kernel<D, FP8>, tk, tv, p);
}

#define PKV_DEFINE_PREFIX_TC(D, FP8)                                                                              \
  template int cascade_prefix_tc_ctas_per_sm<D, FP8>(int);                                                       \
  template cudaError_t launch_cascade_prefix_tc<D, FP8>(const CUtensorMap&, const CUtensorMap&, const PrefixParams&, \
                                                        dim3, cudaStream_t, int);
PKV_DEFINE_PREFIX_TC(64, false)
PKV_DEFINE_PREFIX_TC(128, false)
PKV_DEFINE_PREFIX_TC(64, true)
PKV_DEFINE_PREFIX_TC(128, true)
#undef PKV_DEFINE_PREFIX_TC

}  // namespace pkv
