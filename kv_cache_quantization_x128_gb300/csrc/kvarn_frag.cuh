// Register-fragment helpers shared by the attention kernels (mma.sync m16n8k16
// with fp16 operands and fp32 accumulators; code conversion by the fp6 / fp4
// conversion instructions; quad reductions).
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

// The same split of an fp32 pair; each residual x - hi is one mixed-precision fma
// of the fp16 half with -1 (exact).
__device__ __forceinline__ void split2p(float2 x, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x.x, x.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  float r0, r1;
  asm("{\n .reg .f16 h0, h1, m;\n mov.b32 {h0, h1}, %2;\n mov.b16 m, 0xBC00;\n"
      " fma.rn.f32.f16 %0, h0, m, %3;\n fma.rn.f32.f16 %1, h1, m, %4;\n}"
      : "=f"(r0), "=f"(r1)
      : "r"(hi), "f"(x.x), "f"(x.y));
  const __half2 l = __floats2half2_rn(r0, r1);
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

// Four 4-bit codes in the low nibbles of the bytes of m -> two fp16 pairs (code / 8):
// bytes 0, 1 -> lo, bytes 2, 3 -> hi (fp6 e2m3 patterns 0..15 are the values c / 8).
__device__ __forceinline__ void cvt4(uint32_t m, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e2m3x2 %0, l;\n cvt.rn.f16x2.e2m3x2 %1, h;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(m));
}
// Eight 2-bit codes at bits 8b and 8b + 4 of m -> four fp16 pairs (code / 2), one per
// byte b (fp4 e2m1 patterns 0..3 are the values c / 2).
__device__ __forceinline__ void cvt2(uint32_t m, uint32_t (&r)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(m));
}

constexpr uint32_t kH_One = 0x3C003C00u;       // fp16x2 (1, 1)

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
