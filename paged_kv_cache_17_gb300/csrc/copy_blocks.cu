// copy_blocks.cu -- copy whole pool blocks (copy-on-write).
//
// habr.com/ru/articles/1021832, section 4 "Copy-on-Write для parallel sampling": sequences
// forked from one prompt share its blocks through reference counts; before one of them
// writes into a shared block, that block is copied and the writer's table points at the
// copy, the original staying untouched.  The host decides which blocks to copy; this kernel
// moves the bytes: for every (src, dst) pair, block dst of the K pool and of the V pool
// becomes a copy of block src (all 16 slots, every kv head).
//
// Work item = one chunk of up to 2048 16-byte units (32 KiB) of the K or the V block of one
// pair; a CTA of 256 threads loads its eight units per thread before storing any, so each
// SM keeps tens of KiB of reads in flight, and every warp touches 512 contiguous bytes per
// access (coalesced).  Pairs with an id outside the pool are skipped and flagged; nothing
// is read or written through them.  A pair whose dst is another pair's src gets no ordering
// guarantee (the host never issues such a list: a copy target is a freshly allocated block).
#include <cuda_runtime.h>

#include "decode_launch.cuh"

namespace pkv {

namespace {
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;
constexpr int kCopyChunk = kCopyThreads * kCopyUnroll;  // 16-byte units per work item
}  // namespace

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const int64_t* __restrict__ pairs,
                                                                   int64_t num_pairs, int64_t units_per_block,
                                                                   int chunks_per_block, uint4* k_cache,
                                                                   uint4* v_cache, int64_t num_blocks,
                                                                   uint32_t* status) {
  const int64_t per_pair = 2 * static_cast<int64_t>(chunks_per_block);
  const int64_t items = num_pairs * per_pair;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int64_t pr = it / per_pair;
    const int rem = static_cast<int>(it - pr * per_pair);
    const int is_v = rem >= chunks_per_block;
    const int chunk = rem - is_v * chunks_per_block;
    const int64_t src = pairs[2 * pr], dst = pairs[2 * pr + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (rem == 0 && threadIdx.x == 0) set_flag(status, PKV_DEVFLAG_BAD_BLOCK_ID);
      continue;
    }
    if (src == dst) continue;
    uint4* pool = is_v ? v_cache : k_cache;
    const int64_t base = static_cast<int64_t>(chunk) * kCopyChunk;
    const uint4* from = pool + src * units_per_block + base;
    uint4* to = pool + dst * units_per_block + base;
    const int64_t left = units_per_block - base;
    const int lim = left < kCopyChunk ? static_cast<int>(left) : kCopyChunk;
    uint4 r[kCopyUnroll];
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const int i = static_cast<int>(threadIdx.x) + j * kCopyThreads;
      if (i < lim) r[j] = from[i];
    }
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const int i = static_cast<int>(threadIdx.x) + j * kCopyThreads;
      if (i < lim) to[i] = r[j];
    }
  }
}

cudaError_t launch_copy_blocks(const int64_t* pairs, int64_t num_pairs, int64_t block_bytes, void* k_cache,
                               void* v_cache, int64_t num_blocks, uint32_t* status, int sm_count,
                               cudaStream_t stream) {
  const int64_t units = block_bytes / 16;
  if (num_pairs == 0 || units == 0) return cudaSuccess;
  const int chunks = static_cast<int>((units + kCopyChunk - 1) / kCopyChunk);
  const int64_t items = num_pairs * 2 * chunks;
  const int64_t cap = static_cast<int64_t>(sm_count) * 64;  // beyond this the CTAs loop over items
  const int64_t grid = items < cap ? items : cap;
  copy_blocks_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, stream>>>(
      pairs, num_pairs, units, chunks, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks,
      status);
  return cudaGetLastError();
}

}  // namespace pkv
