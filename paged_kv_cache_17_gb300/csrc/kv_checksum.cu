// kv_checksum.cu -- a read-only pass over the cached K/V of every (sequence, kv head),
// gathered through the block tables exactly as the decode gathers them.
//
// The pages describe no such operation.  It serves two purposes: an integrity check of a
// pool (a checksum of what a sequence's table points at, to compare after a block copy or
// a migration), and the practical ceiling of the decode's reads on this GPU: the same
// grid (one CTA per kv head, sequence and context partition, the decode's partition
// rule), the same producer warp reading block ids 32 at a time and issuing one TMA tensor
// load per K tile and per V tile into a 32 KiB ring with full/empty mbarriers, and
// consumer warps that do nothing with a tile but fold it into a 32-bit word.
//
// Checksum of kv head h of sequence b with n tokens, for K (and likewise V):
//   x_t = XOR of the 32-bit little-endian words of row t (D elements of kv head h),
//   sum = XOR over t < n of rotl32(x_t, t mod 32),
// so equal rows at different positions do not cancel.  XOR is order-free, so the
// partitions and warps combine with atomicXor and the result is deterministic.
#include <cuda_runtime.h>

#include <atomic>

#include "decode_launch.cuh"

namespace pkv {

template <int RB, int NWC>
struct ChecksumCfg {
  static constexpr int kTile = kBlockSize * RB;           // one K or V tile of one kv head
  static constexpr int kStages = 32768 / (2 * kTile);     // a 32 KiB ring of K + V tiles
  static constexpr int kThreads = (NWC + 1) * 32;
  static constexpr int kBarOffset = 2 * kStages * kTile;
  static constexpr int kSmemBytes = 128 + kBarOffset + 2 * kStages * 8;  // 128: alignment slack
  static constexpr int kChunksPerRow = RB / 16;           // 16-byte chunks of one row
  static constexpr int kChunksPerLane = kTile / 16 / 32;  // of one tile, per lane
  static_assert(RB == 64 || RB == 128 || RB == 256, "row bytes");
  static_assert(kStages % NWC == 0, "each stage is always consumed by the same warp");
};

__device__ __forceinline__ uint32_t rotl32(uint32_t x, int r) { return (x << r) | (x >> ((32 - r) & 31)); }

template <int RB, int NWC>
__global__ void __launch_bounds__((NWC + 1) * 32)
    kv_checksum_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const ChecksumParams p) {
  using C = ChecksumCfg<RB, NWC>;
  constexpr int STAGES = C::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* k_tiles = smem;
  uint8_t* v_tiles = smem + STAGES * C::kTile;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;

  const int h = blockIdx.x, b = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int len = p.context_lens[b];
  const int cap = min(p.max_context_len, p.max_blocks * kBlockSize);
  if (len < 0 || len > cap) {
    if (threadIdx.x == 0 && s == 0) set_flag(p.status, PKV_DEVFLAG_BAD_CONTEXT_LEN);
    len = len < 0 ? 0 : cap;
  }
  const int nblk = (len + kBlockSize - 1) / kBlockSize;
  const int blk0 = s * p.split_blocks;
  if (blk0 >= nblk) return;
  const int nloc = min(nblk, blk0 + p.split_blocks) - blk0;
  const int32_t* row = p.block_tables + static_cast<size_t>(b) * p.max_blocks + blk0;
  int ids = (warp == NWC && lane < nloc) ? row[lane] : 0;

  if (threadIdx.x == NWC * 32) tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v);
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NWC) {
    // ---------------------------------------------------------------- producer warp
    bool timed_out = false;
    int issued = 0;
    for (int base = 0; base < nloc && !timed_out; base += 32) {
      const int next = (base + 32 + lane < nloc) ? row[base + 32 + lane] : 0;
      if ((ids < 0 || ids >= p.num_blocks) && base + lane < nloc) set_flag(p.status, PKV_DEVFLAG_BAD_BLOCK_ID);
      const int cnt = min(32, nloc - base);
      for (int k = 0; k < cnt; ++k) {
        const int pb = __shfl_sync(kFull, ids, k);
        const int it = base + k, st = it % STAGES;
        if (lane == 0) {
          if (it >= STAGES && !mbar_wait(&empty_bar[st], ((it / STAGES) - 1) & 1)) {
            set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
            timed_out = true;
          }
          if (!timed_out) {
            // an id outside the pool reads a box entirely outside the tensor: zeros
            const int row0 = (pb >= 0 && pb < p.num_blocks) ? pb * kBlockSize : -kBlockSize;
            mbar_arrive_expect_tx(&full_bar[st], 2 * C::kTile);
            tma_load_3d(k_tiles + st * C::kTile, &tm_k, 0, h, row0, &full_bar[st]);
            tma_load_3d(v_tiles + st * C::kTile, &tm_v, 0, h, row0, &full_bar[st]);
          }
        }
        timed_out = __shfl_sync(kFull, timed_out, 0);
        if (timed_out) break;
        issued = it + 1;
      }
      ids = next;
    }
    if (lane == 0) {  // every issued copy lands before the CTA exits
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        if (!mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1)) {
          set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
          break;
        }
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  // Lane l folds chunks l, l + 32, ... of a tile: each load instruction of the warp reads
  // 512 contiguous bytes (no bank conflicts).  rotl distributes over XOR, so every chunk
  // enters the sum rotated by its row's position, with no per-row reduction.
  uint32_t kacc = 0, vacc = 0;
  for (int it = warp; it < nloc; it += NWC) {
    const int sg = it % STAGES;
    if (!mbar_wait(&full_bar[sg], (it / STAGES) & 1)) {
      if (lane == 0) set_flag(p.status, PKV_DEVFLAG_WAIT_TIMEOUT);
      break;
    }
    const uint4* kt = reinterpret_cast<const uint4*>(k_tiles + sg * C::kTile);
    const uint4* vt = reinterpret_cast<const uint4*>(v_tiles + sg * C::kTile);
    const int tok0 = (blk0 + it) * kBlockSize;
#pragma unroll
    for (int i = 0; i < C::kChunksPerLane; ++i) {
      const int j = i * 32 + lane;
      const int t = tok0 + j / C::kChunksPerRow;
      const uint4 a = kt[j], v = vt[j];
      const uint32_t xk = t < len ? (a.x ^ a.y ^ a.z ^ a.w) : 0u;  // rows past the context: 0
      const uint32_t xv = t < len ? (v.x ^ v.y ^ v.z ^ v.w) : 0u;
      kacc ^= rotl32(xk, t & 31);
      vacc ^= rotl32(xv, t & 31);
    }
    // The stage goes back to the producer only once its reads are ordered before the next
    // TMA load into it: they went through the generic proxy, the refill goes through the
    // async proxy, so a proxy fence is needed (without it the refill could land under a read
    // still pending and the sums came out wrong when stages were reused).
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[sg]);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    kacc ^= __shfl_xor_sync(kFull, kacc, m);
    vacc ^= __shfl_xor_sync(kFull, vacc, m);
  }
  if (lane == 0) {
    uint32_t* o = p.out + (static_cast<size_t>(b) * p.hkv + h) * 2;
    atomicXor(o, kacc);
    atomicXor(o + 1, vacc);
  }
}

template <int RB>
static cudaError_t launch_rb(const CUtensorMap& tk, const CUtensorMap& tv, const ChecksumParams& p, dim3 grid,
                             cudaStream_t stream) {
  constexpr int NWC = 2;
  using C = ChecksumCfg<RB, NWC>;
  static_assert(C::kSmemBytes <= 48 * 1024, "no opt-in shared memory needed");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kv_checksum_kernel<RB, NWC>, tk, tv, p);
}

cudaError_t launch_kv_checksum(int row_bytes, const CUtensorMap& tk, const CUtensorMap& tv, const ChecksumParams& p,
                               dim3 grid, cudaStream_t stream) {
  switch (row_bytes) {
    case 64: return launch_rb<64>(tk, tv, p, grid, stream);
    case 128: return launch_rb<128>(tk, tv, p, grid, stream);
    case 256: return launch_rb<256>(tk, tv, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
