// Per-group quantization of one 128 x 128 tensor tile from its two Hadamard
// products in TMEM (KVarN README, "How KVarN works", stages 3-4): the log-space
// column/row variance normalisation, fp16 scales, group extremes, RTN and packing
// into a shared-memory stage laid out as the record's part for that tensor. A
// group is 256 threads (8 warps) synchronised by one named barrier; the kernels
// that use it (tile quantization, the fused serving step) own the TMA/MMA side.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvarn_common.cuh"
#include "kvarn_tc.cuh"

namespace kvarn {
namespace {

constexpr int kGroupThreads = 256;
constexpr int kVec = 136;                         // parity-split vector (even at 0, odd at 68)
constexpr int kNumVec = 6;                        // a, b, g (2^-3.5/r), hc (1/c), w, c0

enum { kVA = 0, kVB = 1, kVG = 2, kVHc = 3, kVW = 4, kVC0 = 5 };

// position of entry e in a parity-split vector
__device__ __forceinline__ int ps(int e) { return (e & 1) * 68 + (e >> 1); }

constexpr float kVarScale = 1.0f / 128.0f;

__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}   // (2^-3.5)^2: statistics of the +-1 transform

// A thread's whole half line (64 values, two x32 loads) from TMEM; the registers
// are valid after tmem_wait_line.
__device__ __forceinline__ void tmem_ld_line(uint32_t taddr, float (&x)[64]) {
  tmem_ld_16x64b_x32_nowait(taddr, x);
  tmem_ld_16x64b_x32_nowait(taddr + 64, x + 32);
}
__device__ __forceinline__ void tmem_wait_line(float (&x)[64]) {
  tmem_wait_x32(x);
  tmem_wait_x32(x + 32);
}

// Population variance and mean over the pair's 128 values of w_e * x_e, where the
// thread's line in TMEM is at `taddr` (entries e = p + 2k, k < 64, streamed in two
// halves of 32) and w is a parity-split vector. One sweep accumulates the first
// two moments about a shift close to the mean (the line's mean from the previous
// iteration); if the shift was far from the mean (mean square more than twice the
// variance, or a non-positive variance), a second sweep recomputes the moments
// about the exact mean, so the result keeps the accuracy of a centred two-pass
// variance.
__device__ __forceinline__ float pair_moments(float (&x)[64], uint32_t taddr, const float* wv, int p, float shift,
                                             float& mean, uint32_t next_taddr) {
  const float2 nsh = make_float2(-shift, -shift);
  float2 s0 = make_float2(0.f, 0.f), s1 = s0, s2 = s0, s3 = s0, q0 = s0, q1 = s0, q2 = s0, q3 = s0;
  tmem_wait_line(x);   // the whole sweep was started at the end of the one before
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float* xh = x + 32 * hh;
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
      const float4 w = reinterpret_cast<const float4*>(wv + p * 68)[8 * hh + q];
      const float4 v = reinterpret_cast<const float4*>(wv + p * 68)[8 * hh + q + 1];
      const float2 d0 = __ffma2_rn(make_float2(w.x, w.y), make_float2(xh[4 * q], xh[4 * q + 1]), nsh);
      const float2 d1 = __ffma2_rn(make_float2(w.z, w.w), make_float2(xh[4 * q + 2], xh[4 * q + 3]), nsh);
      const float2 d2 = __ffma2_rn(make_float2(v.x, v.y), make_float2(xh[4 * q + 4], xh[4 * q + 5]), nsh);
      const float2 d3 = __ffma2_rn(make_float2(v.z, v.w), make_float2(xh[4 * q + 6], xh[4 * q + 7]), nsh);
      s0 = __fadd2_rn(s0, d0);
      s1 = __fadd2_rn(s1, d1);
      s2 = __fadd2_rn(s2, d2);
      s3 = __fadd2_rn(s3, d3);
      q0 = __ffma2_rn(d0, d0, q0);
      q1 = __ffma2_rn(d1, d1, q1);
      q2 = __ffma2_rn(d2, d2, q2);
      q3 = __ffma2_rn(d3, d3, q3);
    }
  }
  s0 = __fadd2_rn(s0, s2);
  s1 = __fadd2_rn(s1, s3);
  q0 = __fadd2_rn(q0, q2);
  q1 = __fadd2_rn(q1, q3);
  float s = (s0.x + s0.y) + (s1.x + s1.y), m2 = (q0.x + q0.y) + (q1.x + q1.y);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  m2 += __shfl_xor_sync(0xffffffffu, m2, 2);
  float d = s * (1.0f / 128.0f);
  const float msq = m2 * (1.0f / 128.0f);
  float var = msq - d * d;
  const bool recentre = !(msq <= 2.0f * var);   // shift far from the mean, or var <= 0
  // The second sweep holds warp-collective instructions (tcgen05.ld, shuffles), so
  // the whole warp runs it when any pair needs it; other pairs keep their result.
  if (__any_sync(0xffffffffu, recentre)) {
    const float c = shift + d;
    const float2 nc = make_float2(-c, -c);
    float2 r0 = make_float2(0.f, 0.f), r1 = r0;
    tmem_ld_line(taddr, x);
    tmem_wait_line(x);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float* xh = x + 32 * hh;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 w = reinterpret_cast<const float4*>(wv + p * 68)[8 * hh + q];
        const float2 e0 = __ffma2_rn(make_float2(w.x, w.y), make_float2(xh[4 * q], xh[4 * q + 1]), nc);
        const float2 e1 = __ffma2_rn(make_float2(w.z, w.w), make_float2(xh[4 * q + 2], xh[4 * q + 3]), nc);
        r0 = __ffma2_rn(e0, e0, r0);
        r1 = __ffma2_rn(e1, e1, r1);
      }
    }
    float r = (r0.x + r0.y) + (r1.x + r1.y);
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    if (recentre) {
      var = r * (1.0f / 128.0f);
      shift = c;
      d = 0.f;
    }
  }
  tmem_ld_line(next_taddr, x);   // the next sweep, waited there
  mean = shift + d;
  return fmaxf(var, 0.0f);
}

// v / sqrt(u): reciprocal square root refined by one Newton-Raphson step
// (y1 = y0 + y0 (1 - u y0^2) / 2), then one multiply.
__device__ __forceinline__ float div_sqrt(float v, float u) {
  const float y0 = rsqrtf(u);
  const float e = fmaf(-u * y0, y0, 1.0f);
  const float y1 = fmaf(0.5f * y0, e, y0);
  return v * y1;
}

// Keys, after the last column pass: the fp16 scale c of token `line` (b its final
// normaliser) into the metadata, and 1/c into the vector the extremes and codes use.
// Returns 1/c; `store` selects the thread that writes.
template <bool kLean>
__device__ __forceinline__ float key_token_scale(uint16_t* meta, float* vh, int line, int pl, float b, bool store) {
  const uint16_t cb = f2h_bits(clampf(1.0f / b, kFp16MinNormal, kFp16Max));
  const float hc = 1.0f / h2f_bits(cb);
  if (store) {
    meta[(kLean ? 0 : 1) * 128 + line] = cb;
    vh[pl] = hc;
  }
  return hc;
}

// Zero point and scale of group `line` from its extremes mn, mx of y, in fp16, and
// the code-pass coefficients: v = (x * own) * w + c0 = ((y - z) / s + 1/2) / levels,
// where `lf` is the group's own factor of y (the part of 1/(r c) and 2^-3.5 that is
// constant along the group).
template <int kBits, bool kLean>
__device__ __forceinline__ void group_zero_scale(uint16_t* meta, float* vw, float* vc0, int line, int pl, float mn,
                                                 float mx, float lf) {
  constexpr float kLevels = static_cast<float>((1 << kBits) - 1);
  const uint16_t zb = f2h_bits(clampf(mn, -kFp16Max, kFp16Max));
  const float z = h2f_bits(zb);
  const uint16_t sbits = f2h_bits(clampf(fmaxf(mx - z, 0.0f) / kLevels, kFp16MinNormal, kFp16Max));
  const float inv_s = 1.0f / h2f_bits(sbits);
  meta[(kLean ? 1 : 2) * 128 + line] = sbits;
  meta[(kLean ? 2 : 3) * 128 + line] = zb;
  vw[pl] = lf * inv_s * (1.0f / kLevels);
  vc0[pl] = fmaf(-z, inv_s, 0.5f) * (1.0f / kLevels);
}

// A hook that quantize_group runs, after a group barrier, once the item's last TMEM
// data is in registers (when kActive and go): the caller may then reuse the group's
// TMEM. NoHook: none.
struct NoHook {
  static constexpr bool kActive = false;
  bool go = false;
  __device__ void operator()() const {}
};

// Quantize the tensor of group g (0 = K, 1 = V) of the current item from TMEM;
// writes the group's stage (codes + metadata). `tile` is the item's fp16 operand
// (canonical layout), `line`/`p` locate the thread's half line, `ta1`/`ta2` are
// its TMEM addresses of D1 and D2.
template <int kKind, int kBits, bool kLean, class Hook = NoHook>
__device__ __forceinline__ bool quantize_group(float* vec, uint8_t* stage, const uint8_t* tile, uint32_t ta1,
                                               uint32_t ta2, int line, int p, int n_iters, float eps, int bar_id,
                                               bool ok, const Hook& hook = Hook()) {
  float* va = vec + kVA * kVec;
  float* vb = vec + kVB * kVec;
  float* vg = vec + kVG * kVec;
  float* vh = vec + kVHc * kVec;
  float* vw = vec + kVW * kVec;
  float* vc0 = vec + kVC0 * kVec;
  uint16_t* meta = reinterpret_cast<uint16_t*>(stage + kD * kB * kBits / 8);   // after the codes
  const int pl = ps(line);

  if (p == 0) {
    va[pl] = 1.0f;
    vb[pl] = 1.0f;
  }
  // The thread pair of a line keeps that line's scale and mean in registers (both
  // threads compute them; thread p = 0 publishes the scale for the other lines).
  float a_own = 1.0f, b_own = 1.0f, mean_r = 0.0f;
  // the first column shift is exact: with a = 1 the mean of a +-1 Hadamard column
  // is the token's channel-0 input value
  float mean_c = __half2float(*reinterpret_cast<const __half*>(tile + sw_offset(line, 0)));
  // every thread saw its copies and the tensor core finish, or the group stops
  if (!named_bar_and(bar_id, kGroupThreads, ok)) return false;
  // TMEM sweeps: every sweep is loaded at the end of the one before
  float x[64];
  tmem_ld_line(ta2, x);

  float own = 0.0f;   // the line's own factor in the codes pass (keys: 1/c, values: g)
  for (int it = 0; it < n_iters; ++it) {
    // column pass: token j = line, channels e = p + 2k (D2), weights a
    {
      float mean;
      const float var = pair_moments(x, ta2, va, p, mean_c, mean, ta1) * kVarScale;
      b_own = div_sqrt(b_own, fmaf(b_own * b_own, var, eps));
      mean_c = mean;
      if (p == 0) vb[pl] = b_own;
      if (kKind == 0 && it + 1 == n_iters) own = key_token_scale<kLean>(meta, vh, line, pl, b_own, p == 0);
    }
    named_bar(bar_id, kGroupThreads);
    // row pass: channel i = line, tokens e = p + 2k (D1), weights b; after the keys'
    // last one their extremes sweep D1 again (the key groups are its lines)
    {
      float mean;
      const uint32_t next = kKind == 0 && it + 1 == n_iters ? ta1 : ta2;
      const float var = pair_moments(x, ta1, vb, p, mean_r, mean, next) * kVarScale;
      a_own = div_sqrt(a_own, fmaf(a_own * a_own, var, eps));
      mean_r = mean;
      if (p == 0) va[pl] = a_own;
    }
    named_bar(bar_id, kGroupThreads);
  }

  if (kKind == 0) {
    // keys: r of the channel (the line) and the channel's extremes of
    // y = (x * hc_j) * g_i over D1 (hc published after the last column pass); the
    // factor g_i constant along the line is positive, so it multiplies the extremes
    const uint16_t rb = f2h_bits(clampf(1.0f / a_own, kFp16MinNormal, kFp16Max));
    const float g = kLean ? kInvSqrt128 : kInvSqrt128 / h2f_bits(rb);
    if (p == 0 && !kLean) meta[0 * 128 + line] = rb;
    float mn = INFINITY, mx = -INFINITY;
    tmem_wait_line(x);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float* xh = x + 32 * hh;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 w = reinterpret_cast<const float4*>(vh + p * 68)[8 * hh + q];
        const float2 y0 = __fmul2_rn(make_float2(xh[4 * q], xh[4 * q + 1]), make_float2(w.x, w.y));
        const float2 y1 = __fmul2_rn(make_float2(xh[4 * q + 2], xh[4 * q + 3]), make_float2(w.z, w.w));
        mn = fmin3(fmin3(mn, y0.x, y0.y), y1.x, y1.y);
        mx = fmax3(fmax3(mx, y0.x, y0.y), y1.x, y1.y);
      }
    }
    tmem_ld_line(ta2, x);   // the codes sweep
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (p == 0) group_zero_scale<kBits, kLean>(meta, vw, vc0, line, pl, mn * g, mx * g, g);
    named_bar(bar_id, kGroupThreads);
  }
  if (kKind == 1) {
    // fp16 scales of the values: r per channel (line as channel), c per token (line
    // as token); the +-1 transform's 2^-3.5 is folded into g; lean metadata keeps r,
    // and c (constant in each token's group) is folded into s, z
    const uint16_t rb = f2h_bits(clampf(1.0f / a_own, kFp16MinNormal, kFp16Max));
    const uint16_t cb = f2h_bits(clampf(1.0f / b_own, kFp16MinNormal, kFp16Max));
    own = kInvSqrt128 / h2f_bits(rb);
    const float hc = kLean ? 1.0f : 1.0f / h2f_bits(cb);
    if (p == 0) {
      if (!kLean) {
        meta[0 * 128 + line] = rb;
        meta[1 * 128 + line] = cb;
      } else {
        meta[line] = rb;
      }
      vg[pl] = own;
    }
    named_bar(bar_id, kGroupThreads);

    // extremes of y = (x * g_i) * hc_j per token (D2 rows); two halves of 64 columns
    // (registers k = 32 hh + kl); the factor that is constant along the thread's line
    // is positive, so it multiplies the extremes afterwards (same rounding as per element)
    float mn = INFINITY, mx = -INFINITY;
    tmem_wait_line(x);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float* xh = x + 32 * hh;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 w = reinterpret_cast<const float4*>(vg + p * 68)[8 * hh + q];
        const float2 y0 = __fmul2_rn(make_float2(xh[4 * q], xh[4 * q + 1]), make_float2(w.x, w.y));
        const float2 y1 = __fmul2_rn(make_float2(xh[4 * q + 2], xh[4 * q + 3]), make_float2(w.z, w.w));
        mn = fmin3(fmin3(mn, y0.x, y0.y), y1.x, y1.y);
        mx = fmax3(fmax3(mx, y0.x, y0.y), y1.x, y1.y);
      }
    }
    tmem_ld_line(ta1, x);   // the codes sweep
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (p == 0) group_zero_scale<kBits, kLean>(meta, vw, vc0, line, pl, mn * hc, mx * hc, hc);
    named_bar(bar_id, kGroupThreads);
  }

  // codes: keys token-major (D2 rows: token = line, channels e = p + 2k), values
  // channel-major (D1 rows: channel = line, tokens e = p + 2k); half hh holds
  // k = 32 hh + kl. 4-bit codes (keys or values) fill line rows of 64 bytes, words
  // w = 2hh, 2hh + 1 of each 16-byte group; 2-bit codes fill word u = hh
  constexpr float kLevels = static_cast<float>((1 << kBits) - 1);
  const float2 own2 = make_float2(own, own);
  tmem_wait_line(x);
  if (Hook::kActive && hook.go) {   // the group has read its TMEM for this item: the hook may reuse it
    tc_fence_before();
    named_bar(bar_id, kGroupThreads);
    tc_fence_after();
    hook();
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float* xh = x + 32 * hh;
    // v = (x * own) * w_e + c0_e = (y - z) / s + 1/2, clamped to [0, levels]; the
    // round-down add of 2^23 leaves 0x4B000000 + floor(v) in the bits, and each
    // word accumulates (bits << shift) with the 0x4B000000 terms removed at the end.
    // The shifts are constants (the thread's offset, 8p for nibbles and 4p for
    // crumbs, is applied once after the bias is removed): a runtime shift per code
    // cost 5 % of the kernel.
    uint32_t part[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 w = reinterpret_cast<const float4*>(vw + p * 68)[8 * hh + q];
      const float4 c = reinterpret_cast<const float4*>(vc0 + p * 68)[8 * hh + q];
      const float2 t0 = __fmul2_rn(make_float2(xh[4 * q], xh[4 * q + 1]), own2);
      const float2 t1 = __fmul2_rn(make_float2(xh[4 * q + 2], xh[4 * q + 3]), own2);
      // u = clamp(v / levels, 0, 1); floor(u * levels) is the clamped code
      const float2 u0 = make_float2(fma_sat(t0.x, w.x, c.x), fma_sat(t0.y, w.y, c.y));
      const float2 u1 = make_float2(fma_sat(t1.x, w.z, c.z), fma_sat(t1.y, w.w, c.w));
      const float2 lv = make_float2(kLevels, kLevels), mg = make_float2(8388608.0f, 8388608.0f);
      const float2 f0 = __ffma2_rd(u0, lv, mg);
      const float2 f1 = __ffma2_rd(u1, lv, mg);
      const uint32_t bits[4] = {__float_as_uint(f0.x), __float_as_uint(f0.y), __float_as_uint(f1.x),
                                __float_as_uint(f1.y)};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kl = 4 * q + u;
        if (kBits == 4) {
          // element e = 32w + 16a + 8b + 2g4 + p -> k = 16w + 8a + 4b + g4, nibble 4b + 2p + a of word w
          const int wl = kl >> 4, a = (kl >> 3) & 1, b = (kl >> 2) & 1, g4 = kl & 3;
          part[wl][g4] += bits[u] << (16 * b + 4 * a);
        } else {
          // element e = 64u + 16k2 + 8b + 2g4 + p -> k = 32u + 8k2 + 4b + g4, crumb 4k2 + 2p + b of word u
          const int k2 = (kl >> 3) & 3, b = (kl >> 2) & 1, g4 = kl & 3;
          part[0][g4] += bits[u] << (8 * k2 + 2 * b);
        }
      }
    }
    if (kBits == 4) {
      // each word got 4 nibbles (a, b) from this thread: remove their 0x4B000000 terms
      const uint32_t bias = 0x4B000000u * (1u + (1u << 4) + (1u << 16) + (1u << 20));
      uint8_t* row = stage + line * 64;
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const uint32_t m0 = (part[0][g4] - bias) << (8 * p), m1 = (part[1][g4] - bias) << (8 * p);
        const uint32_t f0 = m0 | __shfl_xor_sync(0xffffffffu, m0, 2);
        const uint32_t f1 = m1 | __shfl_xor_sync(0xffffffffu, m1, 2);
        if (p == hh) *reinterpret_cast<uint2*>(row + g4 * 16 + hh * 8) = make_uint2(f0, f1);
      }
    } else {
      // each word got 8 crumbs (k2, b) from this thread, at bits 8k2 + 2b
      const uint32_t bias = 0x4B000000u * 0x05050505u;
      const int i = line;
      // keys: token row of 32 bytes, 8-byte group g4, word hh; values: 512-byte
      // panel of 16 channels, 16-byte cell of the channel pair, word hh
      uint8_t* base = kKind == 0 ? stage + i * 32 + hh * 4 : stage + (i >> 4) * 512 + ((i >> 3) & 1) * 8 + hh * 4;
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const uint32_t m = (part[0][g4] - bias) << (4 * p);
        const uint32_t f = m | __shfl_xor_sync(0xffffffffu, m, 2);
        const int off = kKind == 0 ? g4 * 8 : ((i & 7) * 4 + g4) * 16;
        if (p == hh) *reinterpret_cast<uint32_t*>(base + off) = f;
      }
    }
  }
  return true;
}

}  // namespace
}  // namespace kvarn
