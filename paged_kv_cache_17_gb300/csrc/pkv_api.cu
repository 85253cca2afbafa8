// pkv_api.cu -- the C ABI (include/pkv.h): argument checks, the context-partition choice,
// TMA tensor maps over the caller's pool, the device status word and kernel dispatch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/pkv.h"
#include "cascade.cuh"
#include "decode_launch.cuh"

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;
constexpr int kMinSplitBlocks = 32;   // a context partition covers at least 512 tokens ...
constexpr int kMaxSplitBlocks = 128;  // ... and at most 2048 (unless forced)
constexpr int kMaxPrefixSlots = pkv::kMaxPrefixRecords;  // prefix-pass splits per prefix

__device__ uint32_t g_pkv_status;  // PKV_DEVFLAG_* bits, one word per device

thread_local std::string t_last_error;

pkv_status fail(pkv_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pkv_status fail(pkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

pkv_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device index %d out of range", dev);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!d.ready) {
      if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
      cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
      cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_pkv_status)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(status)");
      d.status = static_cast<uint32_t*>(p);
      if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
          return fail(PKV_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
      d.ready = true;
    }
  }
  if (d.cc_major != 10 || d.cc_minor != 3)
    return fail(PKV_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", d.cc_major, d.cc_minor);
  *out = &d;
  return PKV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_cache(const pkv_cache_desc* c) {
  if (!c) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
  if (!c->k_cache || !c->v_cache) return fail(PKV_ERR_INVALID_ARG, "k_cache / v_cache is NULL");
  if (!aligned(c->k_cache, 16) || !aligned(c->v_cache, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_cache / v_cache must be 16-byte aligned");
  if (c->block_size != 16) return fail(PKV_ERR_UNSUPPORTED, "block_size must be 16 (got %d)", c->block_size);
  if (c->num_kv_heads <= 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads must be positive");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", c->head_dim);
  if (c->num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "num_blocks must be positive");
  if (c->num_blocks * 16 > 0x7fffffffLL) return fail(PKV_ERR_INVALID_ARG, "num_blocks * 16 must fit in int32");
  if (c->kv_dtype != PKV_KV_BF16 && c->kv_dtype != PKV_KV_FP8_E4M3)
    return fail(PKV_ERR_INVALID_ARG, "unknown kv_dtype %d", static_cast<int>(c->kv_dtype));
  if (c->kv_dtype == PKV_KV_FP8_E4M3 && !c->scales)
    return fail(PKV_ERR_INVALID_ARG, "an E4M3 pool needs scales [2][num_kv_heads]");
  if (c->kv_dtype == PKV_KV_BF16 && c->scales) return fail(PKV_ERR_INVALID_ARG, "a bf16 pool takes no scales");
  if (c->scales && !aligned(c->scales, 4)) return fail(PKV_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  return PKV_OK;
}

// ---------------------------------------------------------------- context partitions

struct Split {
  int split_blocks;
  int max_splits;
};

// Partitions of equal logical length (a multiple of 16 tokens), sized so that a batch at its
// maximal length spreads over about three waves of CTAs (three resident per SM), clamped to
// 512..2048 tokens: shorter partitions cost more merging and CTA start-up, longer ones leave
// a long tail of lone CTAs (measured optimum of the tensor-core decode on the 8B-, 70B- and
// shared-prefix-shaped steps).  PKV_SPLIT_TOKENS (a positive multiple of 16) overrides the
// choice, for tuning and tests.
Split choose_split(int batch, int hkv, int max_context_len, int sm_count) {
  const int max_nblk = (max_context_len + 15) / 16;
  Split r{1, 1};
  if (max_nblk <= 0) return r;
  int sb = 0;
  if (const char* env = std::getenv("PKV_SPLIT_TOKENS")) {
    const long v = std::strtol(env, nullptr, 10);
    if (v >= 16) sb = static_cast<int>(v / 16);
  }
  if (sb == 0) {
    const long long units = static_cast<long long>(batch) * hkv;
    const long long slots = 3LL * sm_count * 3;
    long long want = (static_cast<long long>(max_nblk) * units + slots - 1) / slots;
    if (want < kMinSplitBlocks) want = kMinSplitBlocks;
    if (want > kMaxSplitBlocks) want = kMaxSplitBlocks;
    sb = static_cast<int>((want + 3) / 4 * 4);
  }
  if (sb > max_nblk) sb = max_nblk;
  r.split_blocks = sb;
  r.max_splits = (max_nblk + sb - 1) / sb;
  return r;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t ml, acc, total;
};

// Partial records per (sequence, kv head): pre_slots from a shared-prefix pass, then one per
// context partition.  A plain decode with one partition needs no workspace.
WsLayout ws_layout(int batch, int hkv, int g, int d, const Split& sp, int pre_slots) {
  WsLayout w{0, 0, 0};
  if (sp.max_splits <= 1 && pre_slots == 0) return w;
  const size_t units = static_cast<size_t>(batch) * hkv;
  const size_t slots = static_cast<size_t>(pre_slots) + sp.max_splits;
  w.ml = round256(units * slots * g * 2 * sizeof(float));
  w.acc = round256(units * slots * g * d * sizeof(float));
  w.total = w.ml + w.acc;
  return w;
}

// Merge weights of one (b, h) use G * (records + 1) floats of the tile area.
Split fit_split(Split sp, int g, int max_context_len, int tile_area_bytes, int pre_slots) {
  const int max_nblk = (max_context_len + 15) / 16;
  while (sp.max_splits > 1 && static_cast<long long>(g) * (pre_slots + sp.max_splits + 1) * 4 > tile_area_bytes) {
    sp.split_blocks *= 2;
    if (sp.split_blocks > max_nblk) sp.split_blocks = max_nblk;
    sp.max_splits = (max_nblk + sp.split_blocks - 1) / sp.split_blocks;
  }
  return sp;
}

bool encode_kv_map(CUtensorMap* tm, void* base, int64_t num_blocks, int hkv, int d, bool fp8) {
  const cuuint64_t esz = fp8 ? 1 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv),
                              static_cast<cuuint64_t>(num_blocks) * 16};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esz, static_cast<cuuint64_t>(hkv) * d * esz};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same pool view with 64-element (128-byte) boxes of 16 rows, 128-byte swizzled: the
// tile layout the tensor-core prefix pass reads with ldmatrix (bf16 pools only).
bool encode_kv_map_sw128(CUtensorMap* tm, void* base, int64_t num_blocks, int hkv, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv),
                              static_cast<cuuint64_t>(num_blocks) * 16};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hkv) * d * 2};
  const cuuint32_t box[3] = {64, 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The pool's E4M3 codes as boxes of 16 rows x D codes, swizzled so that the tensor-core
// E4M3 decode reads its per-lane runs of codes without bank conflicts: the 128-byte swizzle
// for 128-byte rows (D = 128), the 64-byte swizzle for 64-byte rows (D = 64).
bool encode_kv_map_e4m3_swz(CUtensorMap* tm, void* base, int64_t num_blocks, int hkv, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv),
                              static_cast<cuuint64_t>(num_blocks) * 16};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv) * d};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Splits of the prefix pass: each split is a run of whole 64-key stages (a multiple of four
// blocks), at least two stages long, at most kMaxPrefixRecords per prefix; the count
// minimises (waves of CTAs, `slots` = SMs x CTAs resident per SM at a time) x (blocks per
// split + 8), the 8 blocks standing for a CTA's start-up and the merge work every extra
// record adds; the fewest splits on a tie.  PKV_PREFIX_SPLIT_BLOCKS (>= 4) fixes the blocks
// per split, for tuning and tests.
struct PrefixPlan {
  int tiles;         // 128-row query tiles per prefix
  int pre_slots;     // splits per prefix
  int split_blocks;  // prefix blocks per split
};

PrefixPlan plan_prefix(int num_prefixes, int max_members, int max_prefix_len, int g, int hkv, long long slots) {
  PrefixPlan pp{0, 0, 0};
  const int pblocks = (max_prefix_len + 15) / 16;
  if (num_prefixes <= 0 || max_members <= 0 || pblocks <= 0) return pp;
  pp.tiles = static_cast<int>((static_cast<long long>(max_members) * g + 127) / 128);
  const long long per_split = static_cast<long long>(pp.tiles) * hkv * num_prefixes;
  if (const char* env = std::getenv("PKV_PREFIX_SPLIT_BLOCKS")) {  // tuning and tests: blocks per split
    const long v = std::strtol(env, nullptr, 10);
    if (v >= 4) {
      long want = v < pblocks ? v : pblocks;
      if (want * kMaxPrefixSlots < pblocks) want = (pblocks + kMaxPrefixSlots - 1) / kMaxPrefixSlots;
      const int sb = static_cast<int>((want + 3) / 4 * 4);
      pp.split_blocks = sb;
      pp.pre_slots = (pblocks + sb - 1) / sb;
      return pp;
    }
  }
  const int max_splits = pblocks / 8 > 1 ? (pblocks / 8 < kMaxPrefixSlots ? pblocks / 8 : kMaxPrefixSlots) : 1;
  long long best_cost = -1;
  for (int n = 1; n <= max_splits; ++n) {
    const int sb = ((pblocks + n - 1) / n + 3) / 4 * 4;
    const int nsplit = (pblocks + sb - 1) / sb;
    if (nsplit != n) continue;  // the same split as a smaller count
    const long long waves = (per_split * n + slots - 1) / slots;
    const long long cost = waves * (sb + 8);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      pp.split_blocks = sb;
      pp.pre_slots = n;
    }
  }
  return pp;
}

using LaunchFn = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const pkv::DecodeParams&, dim3, cudaStream_t,
                                 int);
using InfoFn = pkv::DecodeLaunchInfo (*)();

struct Variant {
  LaunchFn launch;
  InfoFn info;
  bool swizzled = false;     // the tensor-core form reads 128-byte-swizzled 64-column boxes (bf16)
  bool tensor_core = false;  // the tensor-core form (either pool type)
};

template <int D, bool FP8, bool CAS>
Variant pick_g(int g) {
  switch (g) {
    case 1: return {pkv::launch_decode<D, 1, FP8, CAS>, pkv::decode_launch_info<D, 1, FP8, CAS>};
    case 2: return {pkv::launch_decode<D, 2, FP8, CAS>, pkv::decode_launch_info<D, 2, FP8, CAS>};
    case 4: return {pkv::launch_decode<D, 4, FP8, CAS>, pkv::decode_launch_info<D, 4, FP8, CAS>};
    case 8: return {pkv::launch_decode<D, 8, FP8, CAS>, pkv::decode_launch_info<D, 8, FP8, CAS>};
    default: return {nullptr, nullptr};
  }
}

template <int D, bool FP8, bool CAS>
Variant pick_mma(int g) {
  switch (g) {
    case 1: return {pkv::launch_decode_mma<D, 1, FP8, CAS>, pkv::decode_mma_launch_info<D, 1, FP8, CAS>, !FP8, true};
    case 2: return {pkv::launch_decode_mma<D, 2, FP8, CAS>, pkv::decode_mma_launch_info<D, 2, FP8, CAS>, !FP8, true};
    case 4: return {pkv::launch_decode_mma<D, 4, FP8, CAS>, pkv::decode_mma_launch_info<D, 4, FP8, CAS>, !FP8, true};
    case 8: return {pkv::launch_decode_mma<D, 8, FP8, CAS>, pkv::decode_mma_launch_info<D, 8, FP8, CAS>, !FP8, true};
    default: return {nullptr, nullptr, false, false};
  }
}

// The tensor-core form unless PKV_DECODE_CUDA_CORES=1 asks for the CUDA-core kernel (kept
// for comparison and tested).
bool use_mma() {
  const char* env = std::getenv("PKV_DECODE_CUDA_CORES");
  return !(env && env[0] == '1');
}

// The plain decode, or the cascade variant that merges shared-prefix records.
Variant pick_variant(int d, bool fp8, int g, bool cas) {
  if (use_mma()) {
    if (fp8) {
      if (cas) return d == 64 ? pick_mma<64, true, true>(g) : pick_mma<128, true, true>(g);
      return d == 64 ? pick_mma<64, true, false>(g) : pick_mma<128, true, false>(g);
    }
    if (cas) return d == 64 ? pick_mma<64, false, true>(g) : pick_mma<128, false, true>(g);
    return d == 64 ? pick_mma<64, false, false>(g) : pick_mma<128, false, false>(g);
  }
  if (cas) {
    if (d == 64) return fp8 ? pick_g<64, true, true>(g) : pick_g<64, false, true>(g);
    return fp8 ? pick_g<128, true, true>(g) : pick_g<128, false, true>(g);
  }
  if (d == 64) return fp8 ? pick_g<64, true, false>(g) : pick_g<64, false, false>(g);
  return fp8 ? pick_g<128, true, false>(g) : pick_g<128, false, false>(g);
}

}  // namespace

// ==================================================================== C ABI

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

const char* pkv_last_error(void) { return t_last_error.c_str(); }

__attribute__((visibility("hidden"))) void pkv_internal_set_error(const char* msg) { t_last_error = msg; }

int32_t pkv_version(void) { return kVersion; }

pkv_status pkv_paged_kv_append(const pkv_cache_desc* cache, const void* k, const void* v,
                               const int64_t* slot_mapping, int64_t num_tokens, pkv_stream_t stream) {
  t_last_error.clear();
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "k, v and slot_mapping must be non-NULL");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(PKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  if (!aligned(slot_mapping, 8)) return fail(PKV_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  cudaError_t e = pkv::launch_append(k, v, slot_mapping, num_tokens, cache->num_kv_heads, cache->head_dim,
                                     cache->kv_dtype == PKV_KV_FP8_E4M3, cache->k_cache, cache->v_cache,
                                     cache->num_blocks * 16, cache->scales, dev->status,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PKV_OK;
}

pkv_status pkv_copy_blocks(const pkv_cache_desc* cache, const int64_t* block_pairs, int64_t num_pairs,
                           pkv_stream_t stream) {
  t_last_error.clear();
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "num_pairs must be >= 0");
  if (num_pairs == 0) return PKV_OK;
  if (!block_pairs) return fail(PKV_ERR_INVALID_ARG, "block_pairs must be non-NULL");
  if (!aligned(block_pairs, 8)) return fail(PKV_ERR_INVALID_ARG, "block_pairs must be 8-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  const int64_t block_bytes = static_cast<int64_t>(cache->block_size) * cache->num_kv_heads * cache->head_dim *
                              (cache->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2);
  cudaError_t e = pkv::launch_copy_blocks(block_pairs, num_pairs, block_bytes, cache->k_cache, cache->v_cache,
                                          cache->num_blocks, dev->status, dev->sm_count,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy-blocks launch");
  return PKV_OK;
}

int32_t pkv_decode_partition_tokens(int32_t batch, int32_t num_kv_heads, int32_t max_context_len) {
  t_last_error.clear();
  if (batch <= 0 || num_kv_heads <= 0 || max_context_len < 0) {
    fail(PKV_ERR_INVALID_ARG, "batch, num_kv_heads must be positive and max_context_len >= 0");
    return 0;
  }
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != PKV_OK) return 0;
  return choose_split(batch, num_kv_heads, max_context_len, dev->sm_count).split_blocks * 16;
}


static pkv_status plan(int32_t batch, int32_t hq, int32_t hkv, int32_t d, int32_t max_len, bool fp8, Split* sp,
                       WsLayout* ws, Variant* var, DeviceInfo** devp, int pre_slots = 0) {
  if (batch < 0 || batch > 65535) return fail(PKV_ERR_INVALID_ARG, "batch must be in [0, 65535]");
  if (hkv <= 0 || hq <= 0 || hq % hkv != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", hq, hkv);
  const int g = hq / hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(PKV_ERR_UNSUPPORTED, "query-group size %d not in {1, 2, 4, 8}", g);
  if (d != 64 && d != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", d);
  if (max_len < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len must be >= 0");
  DeviceInfo* dev = nullptr;
  pkv_status st = device_info(&dev);
  if (st != PKV_OK) return st;
  *var = pick_variant(d, fp8, g, pre_slots > 0);
  const pkv::DecodeLaunchInfo li = var->info();
  *sp = fit_split(choose_split(batch, hkv, max_len, dev->sm_count), g, max_len, li.tile_area_bytes, pre_slots);
  if (sp->max_splits > 65535) return fail(PKV_ERR_UNSUPPORTED, "context too long for the partition grid");
  if (static_cast<long long>(g) * (pre_slots + sp->max_splits + 1) * 4 > li.tile_area_bytes)
    return fail(PKV_ERR_UNSUPPORTED, "too many partial records per sequence to merge");
  *ws = ws_layout(batch, hkv, g, d, *sp, pre_slots);
  *devp = dev;
  return PKV_OK;
}

size_t pkv_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t max_context_len, int32_t num_prefixes, int32_t max_members,
                                  int32_t max_prefix_len) {
  t_last_error.clear();
  if (num_prefixes < 0 || max_members < 0 || max_prefix_len < 0 || num_kv_heads <= 0 || num_q_heads <= 0) {
    fail(PKV_ERR_INVALID_ARG, "negative prefix sizes or non-positive head counts");
    return 0;
  }
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != PKV_OK) return 0;
  // the most prefix records either pool type plans for (its CTAs per SM set the splits)
  int device = 0;
  cudaGetDevice(&device);
  // (the tcgen05 pass for either pool type, and the mma.sync pass for small E4M3 groups)
  const bool small = static_cast<long long>(max_members) * (num_q_heads / num_kv_heads) <= 32;
  const bool mt1 = static_cast<long long>(max_members) * (num_q_heads / num_kv_heads) <= 16;
  int per_sm[4] = {head_dim == 64 ? pkv::cascade_prefix_tc_ctas_per_sm<64, false>(device)
                                        : pkv::cascade_prefix_tc_ctas_per_sm<128, false>(device),
                         head_dim == 64 ? pkv::cascade_prefix_tc_ctas_per_sm<64, true>(device)
                                        : pkv::cascade_prefix_tc_ctas_per_sm<128, true>(device),
                         !small ? 1
                         : head_dim == 64
                             ? (mt1 ? pkv::cascade_prefix_mma_ctas_per_sm<64, 1>(device)
                                    : pkv::cascade_prefix_mma_ctas_per_sm<64, 2>(device))
                             : (mt1 ? pkv::cascade_prefix_mma_ctas_per_sm<128, 1>(device)
                                    : pkv::cascade_prefix_mma_ctas_per_sm<128, 2>(device)),
                         1};
  per_sm[3] = std::min(per_sm[2], 2);  // the mma.sync pass as the cascade call plans it
  int max_per_sm = 1;
  for (int k = 0; k < 4; ++k) {
    if (per_sm[k] <= 0) {
      fail(PKV_ERR_CUDA, "the prefix pass does not fit on an SM of this device");
      return 0;
    }
    max_per_sm = std::max(max_per_sm, per_sm[k]);
  }
  // every slot count the call can plan with: a whole number of CTAs per SM up to what any
  // pass fits (the plan or PKV_PREFIX_CTAS_PER_SM), and half of it (bf16 passes small next to
  // their decode); the split count is not monotonic in the slots, so all of them are tried
  PrefixPlan pp{0, 0, 0};
  for (int v = 1; v <= max_per_sm; ++v)
    for (int half = 0; half < 2; ++half) {
      long long slots = static_cast<long long>(dev->sm_count) * v;
      if (half) slots = std::max(1LL, slots / 2);
      const PrefixPlan pk = plan_prefix(num_prefixes, max_members, max_prefix_len, num_q_heads / num_kv_heads,
                                        num_kv_heads, slots);
      if (pk.pre_slots > pp.pre_slots) pp = pk;
    }
  Split sp;
  WsLayout ws;
  Variant var;
  if (plan(batch, num_q_heads, num_kv_heads, head_dim, max_context_len, false, &sp, &ws, &var, &dev,
           pp.pre_slots) != PKV_OK)
    return 0;
  return ws.total;
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_context_len) {
  t_last_error.clear();
  Split sp;
  WsLayout ws;
  Variant var;
  DeviceInfo* dev;
  // the workspace does not depend on the element type of the pool
  if (plan(batch, num_q_heads, num_kv_heads, head_dim, max_context_len, false, &sp, &ws, &var, &dev) != PKV_OK)
    return 0;
  return ws.total;
}

}  // extern "C"

namespace {

// The step's new tokens for the fused append of the decode (one per sequence).
struct FusedAppend {
  const void* k;
  const void* v;
  const int64_t* slots;
};

// Validation and launch shared by the plain and the cascade decode: the decode kernel over
// each sequence's own blocks, merging pre_slots shared-prefix records per (b, h) for the
// sequences that seq_prefix marks (none when seq_prefix is NULL); with `fused`, the decode
// kernel also appends each sequence's new token (tensor-core form, plain decode only).
pkv_status decode_common(const pkv_cache_desc* cache, const void* q, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                         int32_t max_context_len, float softmax_scale, void* out, pkv_out_dtype out_dtype,
                         void* workspace, size_t workspace_bytes, pkv_stream_t stream, const int32_t* seq_prefix,
                         int pre_slots, const FusedAppend* fused = nullptr) {
  if (!q || !block_tables || !context_lens || !out)
    return fail(PKV_ERR_INVALID_ARG, "q, block_tables, context_lens and out must be non-NULL");
  if (!aligned(q, 16)) return fail(PKV_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (!aligned(out, 16)) return fail(PKV_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PKV_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_FP32)
    return fail(PKV_ERR_INVALID_ARG, "unknown out_dtype %d", static_cast<int>(out_dtype));
  if (max_blocks_per_seq <= 0) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * 16)
    return fail(PKV_ERR_INVALID_ARG, "max_context_len %d exceeds max_blocks_per_seq * 16 = %lld", max_context_len,
                static_cast<long long>(max_blocks_per_seq) * 16);
  if (!std::isfinite(softmax_scale)) return fail(PKV_ERR_INVALID_ARG, "softmax_scale must be finite");
  const bool fp8 = cache->kv_dtype == PKV_KV_FP8_E4M3;
  Split sp;
  WsLayout ws;
  Variant var;
  DeviceInfo* dev = nullptr;
  pkv_status st =
      plan(batch, num_q_heads, cache->num_kv_heads, cache->head_dim, max_context_len, fp8, &sp, &ws, &var, &dev,
           pre_slots);
  if (st != PKV_OK) return st;
  if (ws.total > 0) {
    if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required", ws.total);
    if (!aligned(workspace, 256)) return fail(PKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (workspace_bytes < ws.total)
      return fail(PKV_ERR_WORKSPACE, "workspace has %zu bytes, %zu required", workspace_bytes, ws.total);
  }
  // the tensor-core form reads swizzled boxes (bf16: 64-column halves; E4M3: whole rows of
  // codes), the CUDA-core form plain ones
  CUtensorMap tk, tv;
  const bool maps_ok =
      var.swizzled ? encode_kv_map_sw128(&tk, cache->k_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim) &&
                         encode_kv_map_sw128(&tv, cache->v_cache, cache->num_blocks, cache->num_kv_heads,
                                             cache->head_dim)
      : (fp8 && var.tensor_core)
          ? encode_kv_map_e4m3_swz(&tk, cache->k_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim) &&
                encode_kv_map_e4m3_swz(&tv, cache->v_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim)
          : encode_kv_map(&tk, cache->k_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim, fp8) &&
                encode_kv_map(&tv, cache->v_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim, fp8);
  if (!maps_ok) return fail(PKV_ERR_INVALID_ARG, "cannot describe the KV pool as a TMA tensor map");

  pkv::DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.scales = cache->scales;
  p.out = out;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  p.part_ml = ws.total ? reinterpret_cast<float*>(wsb) : nullptr;
  p.part_acc = ws.total ? reinterpret_cast<float*>(wsb + ws.ml) : nullptr;
  p.seq_prefix = pre_slots > 0 ? seq_prefix : nullptr;
  p.status = dev->status;
  p.max_blocks = max_blocks_per_seq;
  p.hq = num_q_heads;
  p.hkv = cache->num_kv_heads;
  p.num_blocks = static_cast<int>(cache->num_blocks);
  p.max_context_len = max_context_len;
  p.split_blocks = sp.split_blocks;
  p.max_splits = sp.max_splits;
  p.pre_slots = pre_slots;
  p.rec_slots = pre_slots + sp.max_splits;
  p.score_scale = softmax_scale * 1.4426950408889634f;  // log2(e)
  p.out_fp32 = out_dtype == PKV_OUT_FP32;
  // Where the tensor-core decode merges the prefix records: in the merge kernel after it, so
  // that no decode CTA waits for the prefix pass (for bf16 pools the pass runs beside the
  // decode, one prefix CTA per SM; see the cascade call).  E4M3 fork step 56.3 us against
  // 56.7 us with the merge in the decode CTA.  PKV_CASCADE_DEFER=0 merges in the decode CTA
  // (tuning and tests).
  if (pre_slots > 0 && var.tensor_core) {
    bool defer = true;
    if (const char* env = std::getenv("PKV_CASCADE_DEFER")) defer = env[0] == '1';
    p.defer_prefix = defer ? 1 : 0;
  }
  if (fused) {
    p.fused = 1;
    p.k_new = static_cast<const uint16_t*>(fused->k);
    p.v_new = static_cast<const uint16_t*>(fused->v);
    p.new_slots = fused->slots;
    p.k_pool = cache->k_cache;
    p.v_pool = cache->v_cache;
  }
  // failure-detection tests: a short consumer wait and a late producer (tensor-core form)
  if (const char* env = std::getenv("PKV_TEST_CONSUMER_WAIT_CYCLES")) {
    const long long v = std::strtoll(env, nullptr, 10);
    p.test_consumer_wait_cycles = v > 0 ? v : 0;
  }
  if (const char* env = std::getenv("PKV_TEST_PRODUCER_DELAY_CYCLES")) {
    const long long v = std::strtoll(env, nullptr, 10);
    p.test_producer_delay_cycles = v > 0 ? std::min(v, 100000000LL) : 0;  // at most about 50 ms
  }
  int device = 0;
  cudaGetDevice(&device);
  const dim3 grid(static_cast<unsigned>(cache->num_kv_heads), static_cast<unsigned>(batch),
                  static_cast<unsigned>(sp.max_splits));
  cudaError_t e = var.launch(tk, tv, p, grid, reinterpret_cast<cudaStream_t>(stream), device);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (sp.max_splits > 1 || p.defer_prefix) {  // records to merge: split sequences, deferred prefixes
    e = pkv::launch_merge_partitions(cache->head_dim, num_q_heads / cache->num_kv_heads, fp8, p,
                                     dim3(static_cast<unsigned>(cache->num_kv_heads), static_cast<unsigned>(batch)),
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode_attention(const pkv_cache_desc* cache, const void* q, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                      int32_t num_q_heads, int32_t max_context_len, float softmax_scale, void* out,
                                      pkv_out_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                      pkv_stream_t stream) {
  t_last_error.clear();
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (batch == 0) return PKV_OK;
  return decode_common(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, max_context_len,
                       softmax_scale, out, out_dtype, workspace, workspace_bytes, stream, nullptr, 0);
}

pkv_status pkv_paged_append_decode(const pkv_cache_desc* cache, const void* k, const void* v,
                                   const int64_t* slot_mapping, const void* q, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                   int32_t num_q_heads, int32_t max_context_len, float softmax_scale, void* out,
                                   pkv_out_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                   pkv_stream_t stream) {
  t_last_error.clear();
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "batch must be >= 0");
  if (batch == 0) return PKV_OK;
  if (!k || !v || !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "k, v and slot_mapping must be non-NULL");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(PKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  if (!aligned(slot_mapping, 8)) return fail(PKV_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  // The CUDA-core form has no fused append: the two calls, in order, compute the same.
  if (!use_mma()) {
    st = pkv_paged_kv_append(cache, k, v, slot_mapping, batch, stream);
    if (st != PKV_OK) return st;
    return pkv_paged_decode_attention(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                                      max_context_len, softmax_scale, out, out_dtype, workspace, workspace_bytes,
                                      stream);
  }
  const FusedAppend fa{k, v, slot_mapping};
  return decode_common(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, max_context_len,
                       softmax_scale, out, out_dtype, workspace, workspace_bytes, stream, nullptr, 0, &fa);
}

pkv_status pkv_cascade_decode_attention(const pkv_cache_desc* cache, const void* q, const pkv_prefix_desc* px,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                        int32_t max_context_len, float softmax_scale, void* out,
                                        pkv_out_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                        pkv_stream_t stream) {
  t_last_error.clear();
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (!px) return fail(PKV_ERR_INVALID_ARG, "prefixes must be non-NULL");
  if (px->num_prefixes < 0 || px->max_members < 0 || px->max_prefix_len < 0 || px->max_prefix_blocks < 0)
    return fail(PKV_ERR_INVALID_ARG, "prefix sizes must be non-negative");
  if (batch == 0) return PKV_OK;
  if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "batch must be >= 0");
  const bool any_prefix = px->num_prefixes > 0 && px->max_members > 0 && px->max_prefix_len > 0;
  if (!any_prefix)
    return decode_common(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                         max_context_len, softmax_scale, out, out_dtype, workspace, workspace_bytes, stream, nullptr,
                         0);
  if (!px->prefix_tables || !px->prefix_lens || !px->member_indptr || !px->member_seqs || !px->seq_prefix)
    return fail(PKV_ERR_INVALID_ARG, "prefix tables, lengths, member lists and seq_prefix must be non-NULL");
  if (!aligned(px->prefix_tables, 4) || !aligned(px->prefix_lens, 4) || !aligned(px->member_indptr, 4) ||
      !aligned(px->member_seqs, 4) || !aligned(px->seq_prefix, 4))
    return fail(PKV_ERR_INVALID_ARG, "prefix arrays must be 4-byte aligned");
  if (px->max_prefix_len % 16 != 0) return fail(PKV_ERR_INVALID_ARG, "max_prefix_len must be a multiple of 16");
  if (static_cast<int64_t>(px->max_prefix_blocks) * 16 < px->max_prefix_len)
    return fail(PKV_ERR_INVALID_ARG, "max_prefix_len exceeds max_prefix_blocks * 16");
  const int hkv = cache->num_kv_heads;
  if (num_q_heads <= 0 || num_q_heads % hkv != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  const int g = num_q_heads / hkv;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  const bool fp8 = cache->kv_dtype == PKV_KV_FP8_E4M3;
  int device = 0;
  cudaGetDevice(&device);
  // Small member groups of an E4M3 pool (at most 32 query rows per prefix and kv head, such
  // as a best-of-8 fork with G = 4) take the mma.sync pass, which reads the codes straight
  // into its MMA fragments; the rest the tcgen05 pass with its 128-row tiles.
  // PKV_PREFIX_PASS=tc | mma picks one where both apply (tuning and tests).
  const long long group_rows = static_cast<long long>(px->max_members) * g;
  bool mma_pass = fp8 && group_rows <= 32;
  if (const char* env = std::getenv("PKV_PREFIX_PASS")) {
    if (std::strcmp(env, "tc") == 0) mma_pass = false;
    else if (std::strcmp(env, "mma") == 0) mma_pass = fp8 && group_rows <= 32;
  }
  const int mma_mt = group_rows <= 16 ? 1 : 2;
  const int per_sm = mma_pass ? (cache->head_dim == 64
                                     ? (mma_mt == 1 ? pkv::cascade_prefix_mma_ctas_per_sm<64, 1>(device)
                                                    : pkv::cascade_prefix_mma_ctas_per_sm<64, 2>(device))
                                     : (mma_mt == 1 ? pkv::cascade_prefix_mma_ctas_per_sm<128, 1>(device)
                                                    : pkv::cascade_prefix_mma_ctas_per_sm<128, 2>(device)))
                   : cache->head_dim == 64
                         ? (fp8 ? pkv::cascade_prefix_tc_ctas_per_sm<64, true>(device)
                                : pkv::cascade_prefix_tc_ctas_per_sm<64, false>(device))
                         : (fp8 ? pkv::cascade_prefix_tc_ctas_per_sm<128, true>(device)
                                : pkv::cascade_prefix_tc_ctas_per_sm<128, false>(device));
  if (per_sm <= 0) return fail(PKV_ERR_CUDA, "the prefix pass does not fit on an SM of this device");
  // bf16 pools: one prefix CTA per SM, so that three decode CTAs share each SM with it and
  // stream the sequences' own blocks while the prefix pass runs (shared-prefix step 82.7 ->
  // 75.4 us); E4M3 pools: every CTA an SM holds (the prefix pass is the longer part there,
  // fork step 64.4 -> 56.3 us).  PKV_PREFIX_CTAS_PER_SM overrides this, for tuning and tests.
  // The mma.sync pass (four per SM fit): two per SM, so that decode CTAs stream the sequences'
  // own blocks beside it (fork step 55.7 -> 53.8 us).
  int plan_per_sm = mma_pass ? std::min(per_sm, 2) : (fp8 ? per_sm : 1);
  long long plan_slots = static_cast<long long>(dev->sm_count) * plan_per_sm;
  if (const char* env = std::getenv("PKV_PREFIX_CTAS_PER_SM")) {
    const long v = std::strtol(env, nullptr, 10);
    if (v >= 1 && v <= per_sm) plan_slots = static_cast<long long>(dev->sm_count) * v;
  } else if (!fp8) {
    // bf16 pools, where the pass runs beside the decode: when the pass's work (128-row tiles
    // x prefix blocks) is under half the decode's (sequences x kv heads x half the longest
    // context, in blocks), it is planned for half the SMs, so its splits are fewer and longer
    // and the decode keeps more of the GPU (shared-prefix step 75.9-76.8 -> 72.7 us); a
    // prefix-heavy call keeps every SM for the pass, which is then the longer part
    const long long tiles = (static_cast<long long>(px->max_members) * g + 127) / 128;
    const long long pass_work = static_cast<long long>(px->num_prefixes) * tiles * hkv *
                                ((static_cast<long long>(px->max_prefix_len) + 15) / 16);
    const long long dec_work = static_cast<long long>(batch) * hkv * ((static_cast<long long>(max_context_len) + 15) / 16) / 2;
    if (2 * pass_work < dec_work) plan_slots = std::max(1LL, plan_slots / 2);
  }
  PrefixPlan pp = plan_prefix(px->num_prefixes, px->max_members, px->max_prefix_len, g, hkv, plan_slots);
  if (mma_pass) pp.tiles = 1;
  if (static_cast<long long>(px->num_prefixes) * pp.pre_slots > 65535 || pp.tiles > 0x7fffffff / 2)
    return fail(PKV_ERR_UNSUPPORTED, "too many prefixes for the prefix-pass grid");
  Split sp;
  WsLayout ws;
  Variant var;
  if ((st = plan(batch, num_q_heads, hkv, cache->head_dim, max_context_len, false, &sp, &ws, &var, &dev,
                 pp.pre_slots)) != PKV_OK)
    return st;
  if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required", ws.total);
  if (!aligned(workspace, 256)) return fail(PKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (workspace_bytes < ws.total)
    return fail(PKV_ERR_WORKSPACE, "workspace has %zu bytes, %zu required", workspace_bytes, ws.total);
  if (!q || !aligned(q, 16)) return fail(PKV_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
  if (!std::isfinite(softmax_scale)) return fail(PKV_ERR_INVALID_ARG, "softmax_scale must be finite");

  CUtensorMap tk, tv;
  const bool maps_ok =
      mma_pass ? true  // the mma.sync pass copies the codes without tensor maps
      : fp8    ? encode_kv_map(&tk, cache->k_cache, cache->num_blocks, hkv, cache->head_dim, true) &&
                  encode_kv_map(&tv, cache->v_cache, cache->num_blocks, hkv, cache->head_dim, true)
               : encode_kv_map_sw128(&tk, cache->k_cache, cache->num_blocks, hkv, cache->head_dim) &&
                  encode_kv_map_sw128(&tv, cache->v_cache, cache->num_blocks, hkv, cache->head_dim);
  if (!maps_ok) return fail(PKV_ERR_INVALID_ARG, "cannot describe the KV pool as a TMA tensor map");
  pkv::PrefixParams pr{};
  pr.q = static_cast<const uint16_t*>(q);
  pr.prefix_tables = px->prefix_tables;
  pr.prefix_lens = px->prefix_lens;
  pr.indptr = px->member_indptr;
  pr.seqs = px->member_seqs;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  pr.part_ml = reinterpret_cast<float*>(wsb);
  pr.part_acc = reinterpret_cast<float*>(wsb + ws.ml);
  pr.status = dev->status;
  pr.max_prefix_blocks = px->max_prefix_blocks;
  pr.max_members = px->max_members;
  pr.batch = batch;
  pr.hq = num_q_heads;
  pr.hkv = hkv;
  pr.group = g;
  pr.num_blocks = static_cast<int>(cache->num_blocks);
  pr.split_blocks = pp.split_blocks;
  pr.pre_slots = pp.pre_slots;
  pr.rec_slots = pp.pre_slots + sp.max_splits;
  pr.score_scale = softmax_scale * 1.4426950408889634f;  // log2(e)
  pr.scales = cache->scales;
  pr.k_codes = static_cast<const uint8_t*>(cache->k_cache);
  pr.v_codes = static_cast<const uint8_t*>(cache->v_cache);
  const dim3 pgrid(static_cast<unsigned>(pp.tiles), static_cast<unsigned>(hkv),
                   static_cast<unsigned>(px->num_prefixes * pp.pre_slots));
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (mma_pass) {
    if (cache->head_dim == 64)
      e = mma_mt == 1 ? pkv::launch_cascade_prefix_mma<64, 1>(pr, pgrid, cs, device)
                      : pkv::launch_cascade_prefix_mma<64, 2>(pr, pgrid, cs, device);
    else
      e = mma_mt == 1 ? pkv::launch_cascade_prefix_mma<128, 1>(pr, pgrid, cs, device)
                      : pkv::launch_cascade_prefix_mma<128, 2>(pr, pgrid, cs, device);
  } else if (cache->head_dim == 64)
    e = fp8 ? pkv::launch_cascade_prefix_tc<64, true>(tk, tv, pr, pgrid, cs, device)
            : pkv::launch_cascade_prefix_tc<64, false>(tk, tv, pr, pgrid, cs, device);
  else
    e = fp8 ? pkv::launch_cascade_prefix_tc<128, true>(tk, tv, pr, pgrid, cs, device)
            : pkv::launch_cascade_prefix_tc<128, false>(tk, tv, pr, pgrid, cs, device);
  if (e != cudaSuccess) return cuda_fail(e, "prefix-pass launch");
  return decode_common(cache, q, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, max_context_len,
                       softmax_scale, out, out_dtype, workspace, workspace_bytes, stream, px->seq_prefix,
                       pp.pre_slots);
}

pkv_status pkv_stage_copy(void* dst, const void* src, size_t bytes, pkv_stream_t stream) {
  t_last_error.clear();
  if (bytes == 0) return PKV_OK;
  if (!dst || !src) return fail(PKV_ERR_INVALID_ARG, "dst and src must be non-NULL");
  if (!aligned(dst, 16) || !aligned(src, 16)) return fail(PKV_ERR_INVALID_ARG, "dst and src must be 16-byte aligned");
  if (bytes % 16 != 0) return fail(PKV_ERR_INVALID_ARG, "bytes (%zu) must be a multiple of 16", bytes);
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
  if (d < s + bytes && s < d + bytes) return fail(PKV_ERR_INVALID_ARG, "dst and src overlap");
  DeviceInfo* dev = nullptr;
  pkv_status st = device_info(&dev);
  if (st != PKV_OK) return st;
  // both sides must be memory the device addresses: device, page-locked host or managed
  // memory (ordinary host memory is refused here rather than faulting in the kernel)
  for (const void* ptr : {static_cast<const void*>(dst), src}) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
      cudaGetLastError();
      return fail(PKV_ERR_INVALID_ARG, "cannot query the memory behind %p", ptr);
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged)
      return fail(PKV_ERR_INVALID_ARG, "%p is neither device nor page-locked host memory", ptr);
  }
  const cudaError_t e = pkv::launch_stage_copy(dst, src, bytes, dev->sm_count, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stage copy launch");
  return PKV_OK;
}

pkv_status pkv_paged_kv_checksum(const pkv_cache_desc* cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                 int32_t max_context_len, uint32_t* checksums, pkv_stream_t stream) {
  t_last_error.clear();
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (batch < 0 || batch > 65535) return fail(PKV_ERR_INVALID_ARG, "batch must be in [0, 65535]");
  if (batch == 0) return PKV_OK;
  if (!block_tables || !context_lens || !checksums)
    return fail(PKV_ERR_INVALID_ARG, "block_tables, context_lens and checksums must be non-NULL");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(checksums, 4))
    return fail(PKV_ERR_INVALID_ARG, "block_tables, context_lens and checksums must be 4-byte aligned");
  if (max_blocks_per_seq <= 0) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
  if (max_context_len < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len must be >= 0");
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * 16)
    return fail(PKV_ERR_INVALID_ARG, "max_context_len %d exceeds max_blocks_per_seq * 16 = %lld", max_context_len,
                static_cast<long long>(max_blocks_per_seq) * 16);
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  const bool fp8 = cache->kv_dtype == PKV_KV_FP8_E4M3;
  const Split sp = choose_split(batch, cache->num_kv_heads, max_context_len, dev->sm_count);
  if (sp.max_splits > 65535) return fail(PKV_ERR_UNSUPPORTED, "context too long for the partition grid");
  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, cache->k_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim, fp8) ||
      !encode_kv_map(&tv, cache->v_cache, cache->num_blocks, cache->num_kv_heads, cache->head_dim, fp8))
    return fail(PKV_ERR_INVALID_ARG, "cannot describe the KV pool as a TMA tensor map");
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t out_bytes = static_cast<size_t>(batch) * cache->num_kv_heads * 2 * sizeof(uint32_t);
  cudaError_t e = cudaMemsetAsync(checksums, 0, out_bytes, cs);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the checksums");
  pkv::ChecksumParams p{};
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = checksums;
  p.status = dev->status;
  p.max_blocks = max_blocks_per_seq;
  p.hkv = cache->num_kv_heads;
  p.num_blocks = static_cast<int>(cache->num_blocks);
  p.max_context_len = max_context_len;
  p.split_blocks = sp.split_blocks;
  const dim3 grid(static_cast<unsigned>(cache->num_kv_heads), static_cast<unsigned>(batch),
                  static_cast<unsigned>(sp.max_splits));
  e = pkv::launch_kv_checksum(cache->head_dim * (fp8 ? 1 : 2), tk, tv, p, grid, cs);
  if (e != cudaSuccess) return cuda_fail(e, "checksum launch");
  return PKV_OK;
}

pkv_status pkv_check_device_status(pkv_stream_t stream, uint32_t* flags) {
  t_last_error.clear();
  DeviceInfo* dev = nullptr;
  pkv_status st = device_info(&dev);
  if (st != PKV_OK) return st;
  uint32_t host = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&host, dev->status, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (flags) *flags = host;
  if (host) {
    e = cudaMemsetAsync(dev->status, 0, sizeof host, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    return fail(PKV_ERR_DEVICE_CHECK, "device-side check failed (flags 0x%x)", host);
  }
  return PKV_OK;
}

}  // extern "C"
