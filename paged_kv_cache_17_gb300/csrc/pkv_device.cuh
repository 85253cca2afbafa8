// pkv_device.cuh -- device primitives for the paged decode kernels (sm_103a).
//
// Inline PTX for mbarriers and TMA tensor loads, exact bf16 / E4M3 -> fp32 widening,
// packed fp32x2 FMA, bounded waits.  No waits without an iteration limit: a wait that
// runs out sets a bit in the device status word and returns false.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#define PKV_DEVFLAG_BAD_SLOT 0x1u
#define PKV_DEVFLAG_BAD_CONTEXT_LEN 0x2u
#define PKV_DEVFLAG_BAD_BLOCK_ID 0x4u
#define PKV_DEVFLAG_WAIT_TIMEOUT 0x8u

namespace pkv {

constexpr int kBlockSize = 16;  // tokens per physical block
constexpr unsigned kFull = 0xffffffffu;
// A pipeline wait gives up after this many SM cycles (about a second at GB300 clocks).
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_flag(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - start > limit) return false;
  }
}

// Spin for about `cycles` SM cycles (bounded by its argument).
__device__ __forceinline__ void spin_cycles(long long cycles) {
  const long long start = clock64();
  while (clock64() - start < cycles) __nanosleep(256);
}

// ------------------------------------------------------------------ TMA

// 3-D tiled tensor load global -> shared, completing on an mbarrier (transaction bytes).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy accesses of shared memory before later
// async-proxy (TMA) accesses, e.g. before a stage that was just read is refilled.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// ------------------------------------------------------------------ element widening

// bf16 pair packed in a 32-bit word (element i in the low half, i+1 in the high half);
// widening a bf16 to fp32 appends 16 zero bits, so both are exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(__byte_perm(w, 0u, 0x1044u)); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// OCP E4M3 byte `B` of w (0 = lowest), as an fp32 equal to its value times 2^-120:
// sign to bit 31, the 7 magnitude bits to bits 26..20.  For normal codes this is the
// fp32 with exponent field E and mantissa M (value 2^(E-127) (1 + M/8) = 2^-120 value);
// for subnormal codes (E == 0) it is the fp32 denormal M * 2^-129 = 2^-120 * M * 2^-9.
// Exact for every non-NaN code (the kernels never apply flush-to-zero).
template <int B>
__device__ __forceinline__ float e4m3_x2m120(uint32_t w) {
  const uint32_t top = __byte_perm(w, 0u, (B << 12) | 0x444);  // byte B -> bits 31..24, rest 0
  const int32_t sh = static_cast<int32_t>(top) >> 4;           // sign copies over bits 31..27
  return __uint_as_float(static_cast<uint32_t>(sh) & 0x87f00000u);
}

// ------------------------------------------------------------------ E4M3 quantisation

// Eight bf16 values (16 bytes) -> eight OCP E4M3 codes (8 bytes): each value divided by the
// scale as an IEEE binary32 division, then rounded to nearest-even E4M3 with saturation to
// +-448 (the append's encoding; the fused append of the decode uses the same function).
__device__ __forceinline__ uint2 e4m3_quant8(uint4 w, float sc) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float a0 = __fdiv_rn(bf16_lo(in[2 * j]), sc), a1 = __fdiv_rn(bf16_hi(in[2 * j]), sc);
    const float a2 = __fdiv_rn(bf16_lo(in[2 * j + 1]), sc), a3 = __fdiv_rn(bf16_hi(in[2 * j + 1]), sc);
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a2, a3), __NV_SATFINITE, __NV_E4M3);
    out[j] = (lo & 0xffffu) | (hi << 16);
  }
  return make_uint2(out[0], out[1]);
}

// ------------------------------------------------------------------ math

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// 2^x through the hardware approximation (ex2.approx); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float shfl_xor(float v, int m) { return __shfl_xor_sync(kFull, v, m); }

// Programmatic dependent launch: wait for the preceding kernel's results / let the next
// kernel start its prologue.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace pkv
