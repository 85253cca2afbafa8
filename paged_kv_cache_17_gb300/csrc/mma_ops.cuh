// mma_ops.cuh -- warp-level tensor-core building blocks (hand-written PTX) shared by the
// decode kernel's MMA form and the cascade prefix pass: ldmatrix, movmatrix, mma.sync
// m16n8k16 with bf16 or fp16 inputs and fp32 accumulation, and the 128-byte-swizzled tile
// addressing that TMA writes and ldmatrix reads without bank conflicts.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace pkv {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transpose of an 8x8 16-bit matrix held in the ldmatrix fragment layout (thread t: row
// t/4, elements 2(t%4), 2(t%4)+1), returned in the same layout.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// D (16x8, f32) += A (16x16, row) * B (16x8, col); inputs bf16 (F16 false) or fp16
template <bool F16>
__device__ __forceinline__ void mma16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// a pair of fp32 values as 16-bit pairs hi + lo with lo = rn(x - hi): about 16 significant
// bits in all, so products with hi and lo summed in fp32 are accurate to fp32 rounding level
template <bool F16>
__device__ __forceinline__ void split16(float a, float b, uint32_t& hi, uint32_t& lo) {
  if constexpr (F16) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_f16(a - hf.x, b - hf.y);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_bf16(a - hf.x, b - hf.y);
  }
}

// sum of the two 16-bit values (bf16, or fp16 when F16) packed in w, in fp32 (exact widening)
template <bool F16>
__device__ __forceinline__ float sum16(uint32_t w) {
  if constexpr (F16) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    return f.x + f.y;
  } else {
    return __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
  }
}

// two E4M3 codes (low byte = first element) -> two fp16 values, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// Byte offset of 16-byte chunk c of row r in a tile of 16 rows x D one-byte (E4M3) codes, as
// the swizzled TMA load writes it: the 128-byte swizzle for 128-byte rows (D = 128: the chunk
// index xor-ed with r mod 8), the 64-byte swizzle for 64-byte rows (D = 64: xor-ed with
// (r / 2) mod 4).  Under it, 16-byte loads of one chunk per row from 8 consecutive rows, or
// of 8 chunks of one row, meet no bank conflicts.
template <int D>
__device__ __forceinline__ int e4m3_off(int r, int c) {
  static_assert(D == 64 || D == 128, "head_dim");
  if constexpr (D == 128) return r * 128 + ((c ^ (r & 7)) << 4);
  else return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

// codes 0, 1 (e4m3_lo) or 2, 3 (e4m3_hi) of a 32-bit word of four E4M3 codes as an fp16 pair
__device__ __forceinline__ uint32_t e4m3_lo(uint32_t w) { return e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xffffu)); }
__device__ __forceinline__ uint32_t e4m3_hi(uint32_t w) { return e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16)); }

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Shared address of row r (0..15 within a 16-row box group) and 16-byte chunk c of a tile
// stored as boxes of 16 rows x 128 bytes (64 16-bit elements), one box per 64 columns,
// 128-byte swizzled: the chunk index within a row is xor-ed with the row index mod 8.
// rows_per_box_group: 16 rows per box; a tile of R rows (R a multiple of 16) holds
// (R / 16) x (D / 64) boxes, box (R / 16 index, column half) at (ri * halves + half).
template <int D>
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, int row, int c) {
  constexpr int kHalves = D / 64;
  const int box = (row >> 4) * kHalves + (c >> 3);
  const int r = row & 15;
  return base + box * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

}  // namespace pkv
