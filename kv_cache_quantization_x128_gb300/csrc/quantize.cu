// KVarN tile quantization kernels (stages 2-4 of "How KVarN works", KVarN README):
// Hadamard rotation along channels, log-space column/row variance normalisation,
// asymmetric round-to-nearest (4-bit keys per channel, 2-bit values per token) and
// packing into the 14336-byte record documented in kvarn.h.
//
// One persistent CTA per SM (256 threads) walks (tile, kv-head) work items. The
// next item's 2 x 128 token rows are fetched by 1-D bulk copies (TMA) into a
// second shared-memory buffer while the current one is processed; the finished
// record is staged in shared memory and written by one 14336-byte bulk store.
//
// Thread roles. Thread t pairs with t^1 (adjacent lanes): e = 16*warp + lane/2,
// half = lane & 1.
//   column role: token j = e, channels [64*half, 64*half+64)  -> registers xc[64]
//   row role   : channel i = e, tokens [64*half, 64*half+64) -> registers xr[64]
// Both copies of the rotated tile live in registers, so every column pass and
// every row pass is a thread-local loop plus one shuffle with the partner lane.
#include "kvarn_common.cuh"
#include "kvarn_launch.h"

namespace kvarn {
namespace {

constexpr int kThreads = 256;
constexpr int kRowPitch = 272;                     // padded smem row of 256 B of fp16
constexpr int kInTile = kB * kRowPitch;            // 34816 B per (tensor, tile)
constexpr int kVecPad = 132;                       // 128 floats + 4 words of padding

// dynamic shared memory layout (bytes)
constexpr int kOffIn = 0;                                  // [2 bufs][K,V][kInTile]
constexpr int kOffT = kOffIn + 4 * kInTile;                // fp32 [128][128] transpose
constexpr int kOffStage = kOffT + kD * kB * 4;             // packed record
constexpr int kOffA = kOffStage + kRec;                    // a_i (inverse row scales)
constexpr int kOffB = kOffA + kVecPad * 4;                 // b_j (inverse column scales)
constexpr int kOffG = kOffB + kVecPad * 4;                 // 1 / r_i (fp16 r)
constexpr int kOffHc = kOffG + kVecPad * 4;                // 1 / c_j (fp16 c)
constexpr int kOffW = kOffHc + kVecPad * 4;                // per group: G*inv_s or inv_s
constexpr int kOffC0 = kOffW + kVecPad * 4;                // per group: 0.5 - z*inv_s
constexpr int kOffBar = kOffC0 + kVecPad * 4;              // 2 mbarriers
constexpr int kOffDst = kOffBar + 16;                      // int64 dst record per buffer
constexpr int kSmemBytes = kOffDst + 16;

static_assert(kSmemBytes <= 232448, "quantize smem");
static_assert(kOffT % 16 == 0 && kOffStage % 16 == 0 && kOffBar % 8 == 0, "align");

__device__ __forceinline__ int vpad(int i) { return i + ((i >> 6) << 2); }

// Swizzled float index of element (token j, channel i) in the transpose buffer.
__device__ __forceinline__ int tidx(int j, int i) {
  const int c = i >> 2;
  const int x = (((j & 3) << 1) | ((c >> 4) & 1)) ^ (((j >> 6) & 1) << 2);
  return j * kD + ((c ^ x) << 2) + (i & 3);
}

// ------------------------------------------------------------------ work sources
struct PrefillSource {
  const uint16_t* k;
  const uint16_t* v;
  const int64_t* slot;
  int64_t n_items;      // (n_tokens / 128) * hkv
  int hkv;
  int64_t num_blocks;

  // Warp-wide: validates item `w` and returns its record index (block*hkv + head)
  // or -1 (skip); sets the K/V row base pointers and row stride in elements.
  __device__ int64_t resolve(int64_t w, const uint16_t*& kb, const uint16_t*& vb, int64_t& stride,
                             unsigned* flags) const {
    const int lane = threadIdx.x & 31;
    const int64_t chunk = w / hkv;
    const int h = static_cast<int>(w - chunk * hkv);
    const int64_t t0 = chunk * kB;
    const int64_t base = slot[t0];
    bool ok = base >= 0 && (base % kB) == 0 && base / kB < num_blocks;
    for (int m = 0; m < 4; ++m) {
      const int r = lane + 32 * m;
      ok = ok && slot[t0 + r] == base + r;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) raise_flag(flags, KVARN_FLAG_BAD_SLOTS);
      return -1;
    }
    stride = static_cast<int64_t>(hkv) * kD;
    kb = k + t0 * stride + static_cast<int64_t>(h) * kD;
    vb = v + t0 * stride + static_cast<int64_t>(h) * kD;
    return (base / kB) * hkv + h;
  }
};

struct AppendSource {
  const uint16_t* ws;           // [n_seqs][hkv][2][128][128]
  const int32_t* seq_lens;      // lengths before the append
  const int32_t* block_tables;  // [n_seqs][max_blocks]
  int64_t n_items;              // n_seqs * hkv
  int hkv;
  int max_blocks;
  int64_t num_blocks;

  __device__ int64_t resolve(int64_t w, const uint16_t*& kb, const uint16_t*& vb, int64_t& stride,
                             unsigned* flags) const {
    const int lane = threadIdx.x & 31;
    const int64_t s = w / hkv;
    const int h = static_cast<int>(w - s * hkv);
    const int L = seq_lens[s];
    if (L < 0 || (L % kB) != kB - 1) return -1;  // this token does not complete a tile
    const int bi = L / kB;
    if (bi >= max_blocks) {
      if (lane == 0) raise_flag(flags, KVARN_FLAG_BAD_LENGTH);
      return -1;
    }
    const int64_t blk = block_tables[s * max_blocks + bi];
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) raise_flag(flags, KVARN_FLAG_BAD_BLOCK);
      return -1;
    }
    stride = kD;
    kb = ws + ((s * hkv + h) * 2 + 0) * static_cast<int64_t>(kB * kD);
    vb = ws + ((s * hkv + h) * 2 + 1) * static_cast<int64_t>(kB * kD);
    return blk * hkv + h;
  }
};

// Warp 0: resolve item `w` into buffer `buf` and start its copies.
template <class Src>
__device__ void prefetch(const Src& src, int64_t w, int buf, uint8_t* smem, unsigned* flags) {
  const int lane = threadIdx.x & 31;
  const uint16_t* kb = nullptr;
  const uint16_t* vb = nullptr;
  int64_t stride = 0;
  const int64_t dst = src.resolve(w, kb, vb, stride, flags);
  int64_t* s_dst = reinterpret_cast<int64_t*>(smem + kOffDst);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  if (lane == 0) s_dst[buf] = dst;
  if (dst < 0) return;
  if (lane == 0) mbar_arrive_expect_tx(&bars[buf], 2u * kB * kD * 2u);
  __syncwarp();
  uint8_t* in_k = smem + kOffIn + (buf * 2 + 0) * kInTile;
  uint8_t* in_v = smem + kOffIn + (buf * 2 + 1) * kInTile;
  for (int m = 0; m < 4; ++m) {
    const int r = lane + 32 * m;
    bulk_g2s(in_k + r * kRowPitch, kb + r * stride, kD * 2, &bars[buf]);
    bulk_g2s(in_v + r * kRowPitch, vb + r * stride, kD * 2, &bars[buf]);
  }
}

__device__ __forceinline__ void h8_to_f(const uint4& u, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 t = __half22float2(h[q]);
    f[2 * q] = t.x;
    f[2 * q + 1] = t.y;
  }
}

// Column pass (col role, data xc over channels, weights w = a) or row pass (row
// role, data xr over tokens, weights w = b): returns the population variance of
// w_k * x_k over the 128 entries of this thread's line (both halves).
__device__ __forceinline__ float line_variance(const float* x, const float* wvec, int half) {
  const float4* w4 = reinterpret_cast<const float4*>(wvec + vpad(64 * half));
  float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float4 w = w4[q];
    p0 = fmaf(w.x, x[4 * q + 0], p0);
    p1 = fmaf(w.y, x[4 * q + 1], p1);
    p2 = fmaf(w.z, x[4 * q + 2], p2);
    p3 = fmaf(w.w, x[4 * q + 3], p3);
  }
  float s1 = (p0 + p1) + (p2 + p3);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
  const float mean = s1 * (1.0f / 128.0f);
  p0 = p1 = p2 = p3 = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float4 w = w4[q];
    const float t0 = fmaf(w.x, x[4 * q + 0], -mean);
    const float t1 = fmaf(w.y, x[4 * q + 1], -mean);
    const float t2 = fmaf(w.z, x[4 * q + 2], -mean);
    const float t3 = fmaf(w.w, x[4 * q + 3], -mean);
    p0 = fmaf(t0, t0, p0);
    p1 = fmaf(t1, t1, p1);
    p2 = fmaf(t2, t2, p2);
    p3 = fmaf(t3, t3, p3);
  }
  float s2 = (p0 + p1) + (p2 + p3);
  s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
  return s2 * (1.0f / 128.0f);
}

__device__ __forceinline__ uint32_t code_bits(float v, float top) {
  // floor(v) of clamp(v, 0, top) through a round-down add of 2^23; the low bits of
  // the sum are the integer code (exact for 0 <= v < 2^22).
  const float c = fminf(fmaxf(v, 0.0f), top);
  return __float_as_uint(__fadd_rd(c, 8388608.0f)) - 0x4B000000u;
}

// Stages 2-4 for one tensor (kind 0 = K, 1 = V) of the current item.
template <int kKind>
__device__ __forceinline__ void quantize_tensor(const uint8_t* tin, uint8_t* smem, float eps, int n_iters) {
  const int tid = threadIdx.x;
  const int e = ((tid >> 5) << 4) + ((tid & 31) >> 1);
  const int half = tid & 1;
  float* T = reinterpret_cast<float*>(smem + kOffT);
  float* sa = reinterpret_cast<float*>(smem + kOffA);
  float* sb = reinterpret_cast<float*>(smem + kOffB);
  float* sG = reinterpret_cast<float*>(smem + kOffG);
  float* sHc = reinterpret_cast<float*>(smem + kOffHc);
  float* sW = reinterpret_cast<float*>(smem + kOffW);
  float* sC0 = reinterpret_cast<float*>(smem + kOffC0);
  uint8_t* stage = smem + kOffStage;
  uint16_t* meta = reinterpret_cast<uint16_t*>(stage + (kKind == 0 ? kKMetaOff : kVMetaOff));

  // ---- stage 2: Hadamard rotation of token j = e along channels (col role)
  float xc[64];
  {
    const uint8_t* row = tin + e * kRowPitch;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float fo[8], fp[8];
      h8_to_f(*reinterpret_cast<const uint4*>(row + half * 128 + q * 16), fo);
      h8_to_f(*reinterpret_cast<const uint4*>(row + (half ^ 1) * 128 + q * 16), fp);
#pragma unroll
      for (int u = 0; u < 8; ++u) xc[8 * q + u] = half ? (fp[u] - fo[u]) : (fo[u] + fp[u]);
    }
#pragma unroll
    for (int s = 32; s >= 1; s >>= 1) {
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        if ((i & s) == 0) {
          const float u = xc[i], w = xc[i + s];
          xc[i] = u + w;
          xc[i + s] = u - w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) xc[i] *= kInvSqrt128;
  }
  // transpose through shared memory into the row role
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4) {
    const int i0 = 64 * half + 4 * c4;
    *reinterpret_cast<float4*>(T + tidx(e, i0)) = make_float4(xc[4 * c4], xc[4 * c4 + 1], xc[4 * c4 + 2], xc[4 * c4 + 3]);
  }
  if (half == 0) {
    sa[vpad(e)] = 1.0f;
    sb[vpad(e)] = 1.0f;
  }
  __syncthreads();
  float xr[64];
#pragma unroll
  for (int s = 0; s < 64; ++s) xr[s] = T[tidx(64 * half + s, e)];

  // ---- stage 3: n_iters x (column pass, row pass), product form of the log scales
  for (int it = 0; it < n_iters; ++it) {
    {
      const float var = line_variance(xc, sa, half);       // var_i(a_i x_ij), token j = e
      if (half == 0) {
        const float b = sb[vpad(e)];
        sb[vpad(e)] = b / sqrtf(fmaf(b * b, var, eps));
      }
    }
    __syncthreads();
    {
      const float var = line_variance(xr, sb, half);       // var_j(b_j x_ij), channel i = e
      if (half == 0) {
        const float a = sa[vpad(e)];
        sa[vpad(e)] = a / sqrtf(fmaf(a * a, var, eps));
      }
    }
    __syncthreads();
  }

  // ---- fp16 scales r (per channel) and c (per token)
  if (half == 0) {
    const uint16_t rb = f2h_bits(clampf(1.0f / sa[vpad(e)], kFp16MinNormal, kFp16Max));
    const uint16_t cb = f2h_bits(clampf(1.0f / sb[vpad(e)], kFp16MinNormal, kFp16Max));
    meta[0 * 128 + e] = rb;
    meta[1 * 128 + e] = cb;
    sG[vpad(e)] = 1.0f / h2f_bits(rb);
    sHc[vpad(e)] = 1.0f / h2f_bits(cb);
  }
  __syncthreads();

  // ---- stage 4: RTN. y_ij = (x_ij * (1/c_j)) * (1/r_i).
  constexpr float kLevels = kKind == 0 ? 15.0f : 3.0f;
  if (kKind == 0) {
    // key groups: channel i = e over tokens (row role)
    const float g = sG[vpad(e)];
    float mn = INFINITY, mx = -INFINITY;
    {
      const float4* h4 = reinterpret_cast<const float4*>(sHc + vpad(64 * half));
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 w = h4[q];
        const float y0 = (xr[4 * q + 0] * w.x) * g, y1 = (xr[4 * q + 1] * w.y) * g;
        const float y2 = (xr[4 * q + 2] * w.z) * g, y3 = (xr[4 * q + 3] * w.w) * g;
        mn = fminf(fminf(mn, y0), fminf(y1, fminf(y2, y3)));
        mx = fmaxf(fmaxf(mx, y0), fmaxf(y1, fmaxf(y2, y3)));
      }
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    }
    if (half == 0) {
      const uint16_t zb = f2h_bits(clampf(mn, -kFp16Max, kFp16Max));
      const float z = h2f_bits(zb);
      const uint16_t sbits = f2h_bits(clampf(fmaxf(mx - z, 0.0f) / kLevels, kFp16MinNormal, kFp16Max));
      const float inv_s = 1.0f / h2f_bits(sbits);
      meta[2 * 128 + e] = sbits;
      meta[3 * 128 + e] = zb;
      sW[vpad(e)] = g * inv_s;
      sC0[vpad(e)] = fmaf(-z, inv_s, 0.5f);
    }
    __syncthreads();
    // codes in the col role: token j = e, channels 64*half + k
    const float hc = sHc[vpad(e)];
    const float4* w4 = reinterpret_cast<const float4*>(sW + vpad(64 * half));
    const float4* c4 = reinterpret_cast<const float4*>(sC0 + vpad(64 * half));
    uint32_t code[64];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 w = w4[q], c = c4[q];
      code[4 * q + 0] = code_bits(fmaf(xc[4 * q + 0] * hc, w.x, c.x), kLevels);
      code[4 * q + 1] = code_bits(fmaf(xc[4 * q + 1] * hc, w.y, c.y), kLevels);
      code[4 * q + 2] = code_bits(fmaf(xc[4 * q + 2] * hc, w.z, c.z), kLevels);
      code[4 * q + 3] = code_bits(fmaf(xc[4 * q + 3] * hc, w.w, c.w), kLevels);
    }
    // pack: channel i = 32w + 16a + 8b + 2g + h, nibble p = 4h + 2a + b of word w
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
      uint32_t words[2];
#pragma unroll
      for (int wl = 0; wl < 2; ++wl) {
        uint32_t word = 0;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int h = p >> 2, a = (p >> 1) & 1, b = p & 1;
          const int k = 32 * wl + 16 * a + 8 * b + 2 * g4 + h;   // channel - 64*half
          word |= code[k] << (4 * p);
        }
        words[wl] = word;
      }
      *reinterpret_cast<uint2*>(stage + kKCodeOff + e * 64 + g4 * 16 + half * 8) = make_uint2(words[0], words[1]);
    }
  } else {
    // value groups: token j = e over channels (col role)
    const float hc = sHc[vpad(e)];
    float mn = INFINITY, mx = -INFINITY;
    {
      const float4* g4v = reinterpret_cast<const float4*>(sG + vpad(64 * half));
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 w = g4v[q];
        const float y0 = (xc[4 * q + 0] * hc) * w.x, y1 = (xc[4 * q + 1] * hc) * w.y;
        const float y2 = (xc[4 * q + 2] * hc) * w.z, y3 = (xc[4 * q + 3] * hc) * w.w;
        mn = fminf(fminf(mn, y0), fminf(y1, fminf(y2, y3)));
        mx = fmaxf(fmaxf(mx, y0), fmaxf(y1, fmaxf(y2, y3)));
      }
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    }
    if (half == 0) {
      const uint16_t zb = f2h_bits(clampf(mn, -kFp16Max, kFp16Max));
      const float z = h2f_bits(zb);
      const uint16_t sbits = f2h_bits(clampf(fmaxf(mx - z, 0.0f) / kLevels, kFp16MinNormal, kFp16Max));
      const float inv_s = 1.0f / h2f_bits(sbits);
      meta[2 * 128 + e] = sbits;
      meta[3 * 128 + e] = zb;
      sW[vpad(e)] = hc * inv_s;
      sC0[vpad(e)] = fmaf(-z, inv_s, 0.5f);
    }
    __syncthreads();
    // codes in the row role: channel i = e, tokens j = 64*half + s
    const float g = sG[vpad(e)];
    const float4* w4 = reinterpret_cast<const float4*>(sW + vpad(64 * half));
    const float4* c4 = reinterpret_cast<const float4*>(sC0 + vpad(64 * half));
    uint32_t code[64];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 w = w4[q], c = c4[q];
      code[4 * q + 0] = code_bits(fmaf(xr[4 * q + 0] * g, w.x, c.x), kLevels);
      code[4 * q + 1] = code_bits(fmaf(xr[4 * q + 1] * g, w.y, c.y), kLevels);
      code[4 * q + 2] = code_bits(fmaf(xr[4 * q + 2] * g, w.z, c.z), kLevels);
      code[4 * q + 3] = code_bits(fmaf(xr[4 * q + 3] * g, w.w, c.w), kLevels);
    }
    // pack: token t = 64*half + s, crumb p = 8(t&1) + 2((t>>4)&3) + ((t>>3)&1) of
    // word u = half in cell (i&7)*4 + ((t>>1)&3) of panel i>>4, slot (i>>3)&1.
    const int i = e;
    uint8_t* panel = stage + kVCodeOff + (i >> 4) * 512 + ((i >> 3) & 1) * 8 + half * 4;
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
      uint32_t word = 0;
#pragma unroll
      for (int s = 0; s < 64; ++s) {
        if (((s >> 1) & 3) == g4) {
          const int p = 8 * (s & 1) + 2 * ((s >> 4) & 3) + ((s >> 3) & 1);
          word |= code[s] << (2 * p);
        }
      }
      *reinterpret_cast<uint32_t*>(panel + ((i & 7) * 4 + g4) * 16) = word;
    }
  }
}

template <class Src>
__global__ void __launch_bounds__(kThreads, 1)
    quantize_kernel(Src src, uint8_t* __restrict__ cache, int n_iters, float eps, unsigned* flags) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const int64_t* s_dst = reinterpret_cast<const int64_t*>(smem + kOffDst);
  int64_t item = blockIdx.x;
  if (item >= src.n_items) return;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid < 32) prefetch(src, item, 0, smem, flags);
  __syncthreads();
  uint32_t parity = 0;
  for (int k = 0;; ++k) {
    const int cur = k & 1;
    const int64_t next = item + gridDim.x;
    if (tid < 32 && next < src.n_items) prefetch(src, next, cur ^ 1, smem, flags);
    const int64_t dst = s_dst[cur];
    if (dst >= 0) {
      const bool ok = mbar_wait(&bars[cur], (parity >> cur) & 1u, flags);
      parity ^= 1u << cur;
      if (__syncthreads_and(ok)) {
        if (tid == 0) bulk_wait_read_all();  // previous record has left the stage
        quantize_tensor<0>(smem + kOffIn + (cur * 2 + 0) * kInTile, smem, eps, n_iters);
        __syncthreads();
        quantize_tensor<1>(smem + kOffIn + (cur * 2 + 1) * kInTile, smem, eps, n_iters);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
          bulk_s2g(cache + dst * static_cast<int64_t>(kRec), smem + kOffStage, kRec);
          bulk_commit();
        }
      } else {
        break;
      }
    }
    __syncthreads();
    item = next;
    if (item >= src.n_items) break;
  }
  if (tid == 0) bulk_wait_all();
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <class Src>
cudaError_t launch_quantize(const Src& src, uint8_t* cache, int n_iters, float eps, unsigned* flags,
                            cudaStream_t stream, int max_ctas) {
  if (src.n_items <= 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(quantize_kernel<Src>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count();
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > src.n_items) grid = src.n_items;
  quantize_kernel<Src><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(src, cache, n_iters, eps, flags);
  return cudaGetLastError();
}

// New token of each (sequence, kv-head) into its workspace slot; h == 0 also
// writes the new length.
__global__ void append_scatter_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                                      const int32_t* __restrict__ seq_lens, int32_t* __restrict__ seq_lens_out,
                                      uint16_t* __restrict__ ws, int n_seqs, int hkv) {
  const int64_t pair = blockIdx.x;  // s * hkv + h
  const int64_t s = pair / hkv;
  const int h = static_cast<int>(pair - s * hkv);
  const int L = seq_lens[s];
  if (L < 0) return;
  const int pos = L % kB;
  const int t = threadIdx.x;  // 0..31: 16-byte pieces of K (0..15) and V (16..31)
  const int which = t >> 4, piece = t & 15;
  const uint16_t* src = (which ? v_new : k_new) + pair * kD + piece * 8;
  uint16_t* dst = ws + (((s * hkv + h) * 2 + which) * kB + pos) * static_cast<int64_t>(kD) + piece * 8;
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  if (h == 0 && t == 0 && seq_lens_out != nullptr) seq_lens_out[s] = L + 1;
}

}  // namespace

cudaError_t launch_quantize_prefill(const uint16_t* k, const uint16_t* v, const int64_t* slot, int64_t n_tokens,
                                    int hkv, int64_t num_blocks, uint8_t* cache, int n_iters, float eps,
                                    unsigned* flags, cudaStream_t stream, int max_ctas) {
  PrefillSource src{k, v, slot, (n_tokens / kB) * hkv, hkv, num_blocks};
  return launch_quantize(src, cache, n_iters, eps, flags, stream, max_ctas);
}

cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, const int32_t* seq_lens,
                          int32_t* seq_lens_out, const int32_t* block_tables, int n_seqs, int hkv, int max_blocks,
                          int64_t num_blocks, uint16_t* ws, uint8_t* cache, int n_iters, float eps,
                          unsigned* flags, cudaStream_t stream) {
  if (n_seqs <= 0) return cudaSuccess;
  append_scatter_kernel<<<static_cast<unsigned>(static_cast<int64_t>(n_seqs) * hkv), 32, 0, stream>>>(
      k_new, v_new, seq_lens, seq_lens_out, ws, n_seqs, hkv);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  AppendSource src{ws, seq_lens, block_tables, static_cast<int64_t>(n_seqs) * hkv, hkv, max_blocks, num_blocks};
  return launch_quantize(src, cache, n_iters, eps, flags, stream, 0);
}

}  // namespace kvarn
