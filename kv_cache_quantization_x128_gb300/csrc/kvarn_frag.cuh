// Register-fragment helpers shared by the attention kernels (mma.sync m16n8k16
// with fp16 operands and fp32 accumulators; fp16 code conversion; quad reductions).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace kvarn {

// fp32 pair -> (hi, lo) fp16 pairs with hi + lo ~ x to ~22 bits.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The same split of an fp32 pair; the residual x - hi is one packed fma (exact).
__device__ __forceinline__ void split2p(float2 x, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x.x, x.y);
  const float2 r = __ffma2_rn(__half22float2(h), make_float2(-1.f, -1.f), x);
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Products of two fp16 pairs in fp32 (exact: 11 x 11 significant bits), from the
// packed halves without converting them first.
__device__ __forceinline__ float2 mul_h2(uint32_t a, uint32_t b) {
  float2 r;
  asm("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
      " fma.rn.f32.f16 %0, a0, b0, 0f00000000;\n fma.rn.f32.f16 %1, a1, b1, 0f00000000;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t h2raw(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ float2 h2pair(const uint16_t* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}

template <uint32_t kMask>
__device__ __forceinline__ uint32_t lop_magic(uint32_t w) {
  // (w & kMask) | 0x64006400: the selected bits become the low mantissa bits of two
  // fp16 values 1024 + field
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(w), "n"(kMask), "n"(0x64006400u));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// fp16x2 constants: field = (1024 + scale * code) * (1/scale) - 1024/scale, exact
constexpr uint32_t kH_One = 0x3C003C00u;       // 1
constexpr uint32_t kH_M1024 = 0xE400E400u;     // -1024
constexpr uint32_t kH_Sixteenth = 0x2C002C00u; // 1/16
constexpr uint32_t kH_M64 = 0xD400D400u;       // -64
constexpr uint32_t kH_Quarter = 0x34003400u;   // 1/4
constexpr uint32_t kH_M256 = 0xDC00DC00u;      // -256
constexpr uint32_t kH_64th = 0x24002400u;      // 1/64
constexpr uint32_t kH_M16 = 0xCC00CC00u;       // -16

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}
__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
  return x;
}

}  // namespace kvarn
