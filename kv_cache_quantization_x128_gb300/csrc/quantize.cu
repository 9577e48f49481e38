// KVarN tile quantization (KVarN README, "How KVarN works", stages 2-4):
// Hadamard rotation along channels, log-space column/row variance normalisation,
// asymmetric round-to-nearest (4-bit keys per channel, 2-bit values per token) and
// packing into the 14336-byte record documented in kvarn.h.
//
// One persistent CTA per SM, 512 threads in two independent 8-warp groups: group 0
// quantizes the K tile and group 1 the V tile of each (block, kv-head) work item.
// Per item and group:
//   1. one thread starts two 2-D TMA copies (64 channels x 128 tokens each) of the
//      next item's tile into the group's spare buffer, in the 128-byte swizzled
//      K-major layout, completing on an mbarrier;
//   2. the same thread issues tcgen05.mma twice over K = 128: D1 = H X^T (TMEM
//      lanes = channels, columns = tokens) and D2 = X H (lanes = tokens, columns =
//      channels), with H the +-1 Sylvester matrix (exact in fp16) and fp32
//      accumulation; the 1/sqrt(128) factor is folded into the statistics;
//   3. each column pass reads D2 and each row pass reads D1 straight from TMEM
//      (tcgen05.ld 16x64b: two threads per line, 64 values each), so both passes
//      are thread-local loops plus one shuffle with the partner thread; every
//      sweep (the thread's 64 values) is loaded at the end of the sweep before it,
//      so its latency overlaps the reduction, the scale update and the barrier;
//   4. fp16 scales, group extremes (for keys taken in the last row pass, whose
//      lines are the key groups), RTN, packing into a shared-memory stage, and two
//      bulk stores of the group's part of the record.
// The groups share only the Hadamard operand and the TMEM allocation (256 columns
// each), so one group's MMA latency and barriers overlap the other's arithmetic.
// The slot check of an item is agreed on at the barrier that ends the previous one.
#include <cuda.h>

#include <mutex>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_tc.cuh"

namespace kvarn {
namespace {

constexpr int kGroupThreads = 256;
constexpr int kThreads = 2 * kGroupThreads;
constexpr int kTileOp = kB * kD * 2;              // 32768 B: one fp16 128x128 operand
constexpr int kVec = 136;                         // parity-split vector (even at 0, odd at 68)
constexpr int kNumVec = 6;                        // a, b, g (2^-3.5/r), hc (1/c), w, c0

constexpr int kOffH = 0;
constexpr int kOffIn = kOffH + kTileOp;                        // [group][buf] operands
static_assert(kOffIn % 1024 == 0, "align");

// Shared-memory layout after the operands, per preset: a stage (codes + metadata)
// of each tensor sized to its bit width, double buffered. Sizing the stages to the
// preset, not to the widest one, was measured 1.5 % faster for k4v2.
template <int KB, int VB>
struct QSmem {
  static constexpr int kStageK = kD * kB * KB / 8 + 1024;
  static constexpr int kStageV = kD * kB * VB / 8 + 1024;
  static constexpr int kOffStageK = kOffIn + 4 * kTileOp;              // [buf]
  static constexpr int kOffStageV = kOffStageK + 2 * kStageK;           // [buf]
  static constexpr int kOffVec = kOffStageV + 2 * kStageV;              // [group][vector][kVec] fp32
  static constexpr int kOffBar = kOffVec + 2 * kNumVec * kVec * 4;      // mma [group], load [group][buf]
  static constexpr int kOffTmem = kOffBar + 48;
  static constexpr int kBytes = kOffTmem + 16;
  static_assert(kBytes <= 232448, "quantize shared memory");
  static_assert(kOffStageV % 16 == 0 && kOffVec % 16 == 0, "align");
};

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

// ------------------------------------------------------------------ work sources
// A work item w is a (tile, kv-head) pair; both sources keep w below 2^31.
struct PrefillSource {
  CUtensorMap map[2];   // K, V as [n_tokens rows][hkv * 128 channels] fp16
  const int64_t* slot;
  int64_t n_items;      // (n_tokens / 128) * hkv
  int hkv;
  int64_t num_blocks;

  __device__ bool needs_load(int64_t) const { return true; }
  __device__ void scatter(int64_t, int, int) const {}
  // TMA coordinates (channel, token) of the item's 128 x 128 tile of tensor g
  __device__ void coords(int64_t w, int, int& x, int& y) const {
    const uint32_t chunk = static_cast<uint32_t>(w) / static_cast<uint32_t>(hkv);
    x = static_cast<int>(static_cast<uint32_t>(w) - chunk * hkv) * kD;
    y = static_cast<int>(chunk) * kB;
  }
  struct Check {
    int64_t base = -1, mine = -1;
  };
  // Slot entries this thread checks for item w, loaded one item ahead of use.
  __device__ Check prepare(int64_t w, int gt) const {
    const int64_t t0 = static_cast<int64_t>(static_cast<uint32_t>(w) / static_cast<uint32_t>(hkv)) * kB;
    Check c;
    c.base = slot[t0];
    c.mine = slot[t0 + (gt & (kB - 1))];
    return c;
  }
  __device__ bool check_ok(const Check& c, int gt) const {
    return c.base >= 0 && (c.base % kB) == 0 && c.base / kB < num_blocks && c.mine == c.base + (gt & (kB - 1));
  }
  // Record index of item w once the group agreed its slots are valid.
  __device__ int64_t target(int64_t w, const Check& c, int, unsigned*) const {
    const uint32_t chunk = static_cast<uint32_t>(w) / static_cast<uint32_t>(hkv);
    return (c.base / kB) * hkv + (static_cast<uint32_t>(w) - chunk * hkv);
  }
};

struct AppendSource {
  CUtensorMap map;              // workspace as [n_seqs * hkv * 2 * 128 rows][128 channels] fp16
  const uint16_t* k_new;        // [n_seqs][hkv][128] fp16: the token appended to each sequence
  const uint16_t* v_new;
  uint16_t* ws;                 // the workspace the map describes
  int32_t* seq_lens_out;        // lengths after the append (may be NULL)
  const int32_t* seq_lens;      // lengths before the append
  const int32_t* block_tables;  // [n_seqs][max_blocks]
  int64_t n_items;              // n_seqs * hkv
  int hkv;
  int max_blocks;
  int64_t num_blocks;

  __device__ bool needs_load(int64_t w) const {
    const int L = seq_lens[static_cast<uint32_t>(w) / static_cast<uint32_t>(hkv)];
    return L >= 0 && (L % kB) == kB - 1;
  }
  __device__ void coords(int64_t w, int g, int& x, int& y) const {
    x = 0;
    y = (static_cast<int>(w) * 2 + g) * kB;
  }
  // Threads t < 16 of group g copy 16 bytes each of item w's new token (tensor g)
  // into its workspace row L % 128; thread 0 of the key group also writes the new
  // length of the item's sequence (kv-head 0). The writers fence the global writes
  // against the async proxy; a group barrier then orders them before the TMA copy
  // of the tile.
  __device__ void scatter(int64_t w, int g, int t) const {
    if (t < 0 || t >= 16) return;
    const uint32_t s = static_cast<uint32_t>(w) / static_cast<uint32_t>(hkv);
    const uint32_t h = static_cast<uint32_t>(w) - s * hkv;
    const int L = seq_lens[s];
    if (L < 0) return;
    const uint16_t* src = (g ? v_new : k_new) + static_cast<int64_t>(w) * kD + t * 8;
    uint16_t* dst = ws + ((static_cast<int64_t>(w) * 2 + g) * kB + L % kB) * kD + t * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    if (g == 0 && h == 0 && t == 0 && seq_lens_out != nullptr) seq_lens_out[s] = L + 1;
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  struct Check {};
  __device__ Check prepare(int64_t, int) const { return Check{}; }
  __device__ bool check_ok(const Check&, int) const { return true; }
  __device__ int64_t target(int64_t w, const Check&, int gt, unsigned* flags) const {
    if (!needs_load(w)) return -1;
    const uint32_t s = static_cast<uint32_t>(w) / static_cast<uint32_t>(hkv);
    const uint32_t h = static_cast<uint32_t>(w) - s * hkv;
    const int bi = seq_lens[s] / kB;
    if (bi >= max_blocks) {
      if (gt == 0) raise_flag(flags, KVARN_FLAG_BAD_LENGTH);
      return -1;
    }
    const int64_t blk = block_tables[static_cast<int64_t>(s) * max_blocks + bi];
    if (blk < 0 || blk >= num_blocks) {
      if (gt == 0) raise_flag(flags, KVARN_FLAG_BAD_BLOCK);
      return -1;
    }
    return blk * hkv + h;
  }
};

__device__ __forceinline__ const CUtensorMap* tensor_map(const PrefillSource& s, int g) { return &s.map[g]; }
__device__ __forceinline__ const CUtensorMap* tensor_map(const AppendSource& s, int) { return &s.map; }

// Thread gt == 0 of group g starts the two TMA copies (64 channels each) of item
// w's tile into `dst`, completing on `bar`.
template <class Src>
__device__ __forceinline__ void issue_tile(const Src& src, int64_t w, int g, uint8_t* dst, uint64_t* bar) {
  int x, y;
  src.coords(w, g, x, y);
  const CUtensorMap* map = tensor_map(src, g);
  mbar_arrive_expect_tx(bar, kTileOp);
  tma_load_2d(dst, map, x, y, bar);
  tma_load_2d(dst + kTileOp / 2, map, x + 64, y, bar);
}

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
//
// With kExt, the same sweep also takes the extremes over the pair's values of
// x_e * h_e (h a second parity-split vector), returned in mn, mx for both threads.
template <bool kExt = false>
__device__ __forceinline__ float pair_moments(float (&x)[64], uint32_t taddr, const float* wv, int p, float shift,
                                             float& mean, uint32_t next_taddr, const float* hv = nullptr,
                                             float* mn_out = nullptr, float* mx_out = nullptr) {
  const float2 nsh = make_float2(-shift, -shift);
  float2 s0 = make_float2(0.f, 0.f), s1 = s0, s2 = s0, s3 = s0, q0 = s0, q1 = s0, q2 = s0, q3 = s0;
  float mn = INFINITY, mx = -INFINITY;
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
      if (kExt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float4 h = reinterpret_cast<const float4*>(hv + p * 68)[8 * hh + q + r];
          const float2 y0 = __fmul2_rn(make_float2(xh[4 * (q + r)], xh[4 * (q + r) + 1]), make_float2(h.x, h.y));
          const float2 y1 = __fmul2_rn(make_float2(xh[4 * (q + r) + 2], xh[4 * (q + r) + 3]), make_float2(h.z, h.w));
          mn = fmin3(fmin3(mn, y0.x, y0.y), y1.x, y1.y);
          mx = fmax3(fmax3(mx, y0.x, y0.y), y1.x, y1.y);
        }
      }
    }
  }
  if (kExt) {
    *mn_out = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
    *mx_out = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
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

// Quantize the tensor of group g (0 = K, 1 = V) of the current item from TMEM;
// writes the group's stage (codes + metadata). `tile` is the item's fp16 operand
// (canonical layout), `line`/`p` locate the thread's half line, `ta1`/`ta2` are
// its TMEM addresses of D1 and D2.
template <int kKind, int kBits, bool kLean>
__device__ __forceinline__ bool quantize_group(float* vec, uint8_t* stage, const uint8_t* tile, uint32_t ta1,
                                               uint32_t ta2, int line, int p, int n_iters, float eps, int bar_id,
                                               bool ok) {
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
    // row pass: channel i = line, tokens e = p + 2k (D1), weights b
    if (kKind == 1 || it + 1 < n_iters) {
      float mean;
      const float var = pair_moments(x, ta1, vb, p, mean_r, mean, ta2) * kVarScale;
      a_own = div_sqrt(a_own, fmaf(a_own * a_own, var, eps));
      mean_r = mean;
      if (p == 0) va[pl] = a_own;
    } else {
      // last row pass of the keys: the same sweep takes each channel's extremes of
      // x_ij / c_j, so r, s and z of the channel follow without another sweep
      float mean, mn, mx;
      const float var = pair_moments<true>(x, ta1, vb, p, mean_r, mean, ta2, vh, &mn, &mx) * kVarScale;
      if (p == 0) {
        const float an = div_sqrt(a_own, fmaf(a_own * a_own, var, eps));
        const uint16_t rb = f2h_bits(clampf(1.0f / an, kFp16MinNormal, kFp16Max));
        if (!kLean) meta[0 * 128 + line] = rb;
        const float g = kLean ? kInvSqrt128 : kInvSqrt128 / h2f_bits(rb);
        group_zero_scale<kBits, kLean>(meta, vw, vc0, line, pl, mn * g, mx * g, g);
      }
    }
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

// 128 registers a thread (all that 512 threads can hold): a whole sweep in flight
// needs 64 of them; 112 spilled and measured 5 % slower.
template <class Src, int KB, int VB, bool kLean>
__global__ void __maxnreg__(128)
    quantize_kernel(const __grid_constant__ Src src, uint8_t* __restrict__ cache, int n_iters, float eps,
                    unsigned* flags) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int grp = tid / kGroupThreads;     // 0 = K, 1 = V
  const int gt = tid % kGroupThreads;
  const int bar_id = 1 + grp;
  using S = QSmem<KB, VB>;
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* load_bar = mma_bar + 2 + 2 * grp;   // this group's [buf]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffTmem);
  if (static_cast<int64_t>(blockIdx.x) >= src.n_items) return;

  // Sylvester +-1 Hadamard operand (H[i][k] = (-1)^popcount(i & k)), swizzled layout
  for (int e = tid; e < kD * kD; e += kThreads) {
    const int i = e >> 7, kk = e & 127;
    *reinterpret_cast<uint16_t*>(smem + kOffH + sw_offset(i, kk)) = (__popc(i & kk) & 1) ? 0xBC00u : 0x3C00u;
  }
  if (tid == 0) {
    for (int b = 0; b < 6; ++b) mbar_init(&mma_bar[b], 1);
    fence_mbar_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // this thread's half line in TMEM
  const int gw = gt >> 5, t = gt & 31;
  const uint32_t lane0 = 32 * (gw & 3) + 16 * (gw >> 2);
  const int line = static_cast<int>(lane0) + (t >> 2) + 8 * (t & 1);
  const int p = (t >> 1) & 1;
  const uint32_t d1 = tmem_addr(tmem, 0, 256 * grp);
  const uint32_t d2 = d1 + 128;
  const uint32_t ta1 = tmem_addr(tmem, lane0, 256 * grp);
  const uint32_t ta2 = ta1 + 128;
  float* vec = reinterpret_cast<float*>(smem + S::kOffVec) + grp * kNumVec * kVec;
  const uint32_t sh = smem_u32(smem + kOffH);
  uint8_t* tiles = smem + kOffIn + grp * 2 * kTileOp;   // this group's [buf]
  constexpr uint32_t kIdesc = idesc_f16_f32(128, 128);

  // The copy of item w's tile is started one item ahead; the slot check of the
  // next item is agreed on at the barrier that ends the current one.
  int64_t item = blockIdx.x;
  uint32_t pend = 0;               // bit b: a copy into buffer b has not been waited for
  uint32_t load_parity = 0;        // bit b: phase parity of buffer b's barrier
  // appended tokens go into the workspace two items ahead of their tile's copy
  src.scatter(item, grp, gt);
  if (item + gridDim.x < src.n_items) src.scatter(item + gridDim.x, grp, gt - 16);
  typename Src::Check check = src.prepare(item, gt);
  int64_t dst = -1;
  if (named_bar_and(bar_id, kGroupThreads, src.check_ok(check, gt)))
    dst = src.target(item, check, gt, flags);
  else if (gt == 0)
    raise_flag(flags, KVARN_FLAG_BAD_SLOTS);
  if (src.needs_load(item)) {
    if (gt == 0) issue_tile(src, item, grp, tiles, &load_bar[0]);
    pend = 1;
  }
  uint32_t mma_parity = 0;
  bool mma_inflight = false;       // thread gt == 0: an issued MMA not yet seen complete
  for (int k = 0; item < src.n_items; ++k, item += gridDim.x) {
    const int buf = k & 1;
    const int64_t next = item + gridDim.x;
    const bool has_next = next < src.n_items;
    typename Src::Check check_next{};
    if (has_next) {
      if (src.needs_load(next)) {   // buffer buf ^ 1 was last read by the previous item
        if (gt == 0) issue_tile(src, next, grp, tiles + (buf ^ 1) * kTileOp, &load_bar[buf ^ 1]);
        pend |= 2u >> buf;
      }
      check_next = src.prepare(next, gt);
      if (next + gridDim.x < src.n_items) src.scatter(next + gridDim.x, grp, gt);   // before this item's end barrier
    }
    bool ok = true;
    if ((pend >> buf) & 1u) {
      ok = mbar_wait(&load_bar[buf], (load_parity >> buf) & 1u, flags);
      if (ok) {
        load_parity ^= 1u << buf;
        pend &= ~(1u << buf);
      }
    }
    if (dst >= 0) {
      uint8_t* stage = smem + (grp == 0 ? S::kOffStageK + buf * S::kStageK : S::kOffStageV + buf * S::kStageV);
      if (gt == 0) {
        if (ok) {
          const uint32_t sx = smem_u32(tiles + buf * kTileOp);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint64_t dh = smem_desc_sw128(sw_kstep(sh, s));
            const uint64_t dx = smem_desc_sw128(sw_kstep(sx, s));
            umma_f16(d1, dh, dx, kIdesc, s > 0);   // D1[i][j] = sum_k H[i][k] X[j][k]
            umma_f16(d2, dx, dh, kIdesc, s > 0);   // D2[j][i] = sum_k X[j][k] H[i][k]
          }
          umma_commit(&mma_bar[grp]);
          mma_inflight = true;
        }
        bulk_wait_read<1>();              // the stage written two items ago has been stored
      }
      if (ok) {
        ok = mbar_wait(&mma_bar[grp], mma_parity, flags);
        if (ok) {
          mma_parity ^= 1;
          mma_inflight = false;
        }
      }
      tc_fence_after();
      const uint8_t* tile = tiles + buf * kTileOp;
      if (grp == 0)
        ok = quantize_group<0, KB, kLean>(vec, stage, tile, ta1, ta2, line, p, n_iters, eps, bar_id, ok);
      else
        ok = quantize_group<1, VB, kLean>(vec, stage, tile, ta1, ta2, line, p, n_iters, eps, bar_id, ok);
      if (!ok) break;                     // a copy or the tensor core never signalled (flag raised)
      fence_proxy_async_smem();
      tc_fence_before();
    }
    // end of the item: its stage is complete, and the group agrees on the next item's slots
    const bool next_ok = named_bar_and(bar_id, kGroupThreads, !has_next || src.check_ok(check_next, gt));
    tc_fence_after();
    if (dst >= 0 && gt == 0) {
      using L = RecordLayout<KB, VB, kLean>;
      uint8_t* stage = smem + (grp == 0 ? S::kOffStageK + buf * S::kStageK : S::kOffStageV + buf * S::kStageV);
      uint8_t* rec = cache + dst * static_cast<int64_t>(L::kBytes);
      if (grp == 0) {
        bulk_s2g(rec + L::kKCodeOff, stage, L::kKCodeBytes);
        bulk_s2g(rec + L::kKMetaOff, stage + L::kKCodeBytes, L::kMetaBytes);
      } else {
        bulk_s2g(rec + L::kVCodeOff, stage, L::kVCodeBytes);
        bulk_s2g(rec + L::kVMetaOff, stage + L::kVCodeBytes, L::kMetaBytes);
      }
      bulk_commit();
    }
    if (has_next) {
      dst = -1;
      if (next_ok)
        dst = src.target(next, check_next, gt, flags);
      else if (gt == 0)
        raise_flag(flags, KVARN_FLAG_BAD_SLOTS);
    }
  }
  if (gt == 0) {
    // after a timeout: let copies and MMAs still in flight finish (bounded) before
    // the shared memory and TMEM are released
    for (int b = 0; b < 2; ++b)
      if ((pend >> b) & 1u) mbar_wait(&load_bar[b], (load_parity >> b) & 1u, flags);
    if (mma_inflight) mbar_wait(&mma_bar[grp], mma_parity, flags);
    bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid < 32) tmem_dealloc(tmem, 512);
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <class Src, int KB, int VB, bool kLean>
cudaError_t launch_quantize_bits(const Src& src, uint8_t* cache, int n_iters, float eps, unsigned* flags,
                            cudaStream_t stream, int max_ctas) {
  if (src.n_items <= 0) return cudaSuccess;
  if (src.n_items > INT32_MAX) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(quantize_kernel<Src, KB, VB, kLean>, QSmem<KB, VB>::kBytes, smem_set);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count();
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > src.n_items) grid = src.n_items;
  quantize_kernel<Src, KB, VB, kLean><<<static_cast<unsigned>(grid), kThreads, QSmem<KB, VB>::kBytes, stream>>>(src, cache, n_iters, eps,
                                                                                             flags);
  return cudaGetLastError();
}

// The kernel instance of a preset (k4v2, k4v4, k2v2; k4v2 with lean metadata).
template <class Src>
cudaError_t launch_quantize(const Src& src, uint8_t* cache, int k_bits, int v_bits, bool lean, int n_iters, float eps,
                            unsigned* flags, cudaStream_t stream, int max_ctas) {
  if (k_bits == 4 && v_bits == 2 && !lean)
    return launch_quantize_bits<Src, 4, 2, false>(src, cache, n_iters, eps, flags, stream, max_ctas);
  if (k_bits == 4 && v_bits == 2 && lean)
    return launch_quantize_bits<Src, 4, 2, true>(src, cache, n_iters, eps, flags, stream, max_ctas);
  if (k_bits == 4 && v_bits == 4 && !lean)
    return launch_quantize_bits<Src, 4, 4, false>(src, cache, n_iters, eps, flags, stream, max_ctas);
  if (k_bits == 2 && v_bits == 2 && !lean)
    return launch_quantize_bits<Src, 2, 2, false>(src, cache, n_iters, eps, flags, stream, max_ctas);
  return cudaErrorInvalidValue;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// TMA map of an fp16 matrix [rows][row_elems] read in boxes of 64 channels x 128
// rows with the 128-byte swizzle (row_elems a multiple of 64, base 16-byte aligned).
cudaError_t tile_map(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  if (rows > (1ull << 32) || row_elems > (1ull << 32)) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {row_elems * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                        elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quantize_prefill(const uint16_t* k, const uint16_t* v, const int64_t* slot, int64_t n_tokens,
                                    int hkv, int64_t num_blocks, uint8_t* cache, int k_bits, int v_bits, bool lean,
                                    int n_iters, float eps, unsigned* flags, cudaStream_t stream, int max_ctas) {
  PrefillSource src{};
  cudaError_t err = tile_map(&src.map[0], k, static_cast<uint64_t>(hkv) * kD, static_cast<uint64_t>(n_tokens));
  if (err == cudaSuccess)
    err = tile_map(&src.map[1], v, static_cast<uint64_t>(hkv) * kD, static_cast<uint64_t>(n_tokens));
  if (err != cudaSuccess) return err;
  src.slot = slot;
  src.n_items = (n_tokens / kB) * hkv;
  src.hkv = hkv;
  src.num_blocks = num_blocks;
  return launch_quantize(src, cache, k_bits, v_bits, lean, n_iters, eps, flags, stream, max_ctas);
}

cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, const int32_t* seq_lens,
                          int32_t* seq_lens_out, const int32_t* block_tables, int n_seqs, int hkv, int max_blocks,
                          int64_t num_blocks, uint16_t* ws, uint8_t* cache, int k_bits, int v_bits, bool lean,
                          int n_iters, float eps, unsigned* flags, cudaStream_t stream) {
  if (n_seqs <= 0) return cudaSuccess;
  if (static_cast<int64_t>(n_seqs) * hkv * 2 * kB > INT32_MAX) return cudaErrorInvalidValue;
  AppendSource src{};
  const cudaError_t err = tile_map(&src.map, ws, kD, static_cast<uint64_t>(n_seqs) * hkv * 2 * kB);
  if (err != cudaSuccess) return err;
  src.k_new = k_new;
  src.v_new = v_new;
  src.ws = ws;
  src.seq_lens_out = seq_lens_out;
  src.seq_lens = seq_lens;
  src.block_tables = block_tables;
  src.n_items = static_cast<int64_t>(n_seqs) * hkv;
  src.hkv = hkv;
  src.max_blocks = max_blocks;
  src.num_blocks = num_blocks;
  return launch_quantize(src, cache, k_bits, v_bits, lean, n_iters, eps, flags, stream, 0);
}

}  // namespace kvarn
