// Chunked-prefill attention over the packed KVarN cache plus the fresh fp16 chunk
// (KVarN README, "How KVarN works": scales are re-applied on read and the
// orthonormal rotation keeps attention scores). Chunk token p of a sequence with
// L0 cached tokens attends the L0 cached tokens (floor(L0/128) packed tiles, then
// the L0 % 128 fp16 workspace tokens) and chunk tokens 0..p.
//
// One CTA per (8 chunk tokens, kv-head, sequence), 8 warps; warp w runs chunk
// token 8 * blockIdx.x + w with its GQA group of q-heads as the rows of m16n8k16
// MMAs (fp16 hi part in rows 0-7, lo part in rows 8-15, as in decode). Per packed
// tile the CTA bulk-copies the record once, turns the codes into fp16 in shared
// memory (keys [token][channel], values [channel][token]) and the scales into
// fp32 vectors, and every warp reads its B operands with ldmatrix:
//   QK^T: A = q_r * r^K s^K, B = key codes; score_j = c^K_j (D + beta);
//   PV:   A = p * c^V s^V,   B = value codes; acc_i += r^V_i (D + gamma).
// The packed pass runs in the rotated domain (q_r = H q); the accumulator is then
// rotated back once (H is its own inverse), and the fresh pass (workspace tail and
// chunk, causal) continues in the input domain with unrotated q and plain fp16
// K/V, under the same online softmax (log2 domain).
#include "kvarn_common.cuh"
#include "kvarn_frag.cuh"
#include "kvarn_launch.h"

namespace kvarn {
namespace {

constexpr int kPWarps = 8;                        // chunk tokens per CTA, one per warp
constexpr int kPThreads = kPWarps * 32;
constexpr int kPitch = 136;                       // fp16 per shared row: 128 + 8 (rows 272 B apart)
constexpr int kTileBytes = 128 * kPitch * 2;
constexpr int kMaxRec = 18432;                    // largest record (k4v4)
constexpr int kOffK = 0;                          // fp16 [128][kPitch]
constexpr int kOffV = kOffK + kTileBytes;         // fp16 [128][kPitch]
constexpr int kOffRec = kOffV + kTileBytes;       // packed records [2] (the next one in flight)
constexpr int kOffScale = kOffRec + 2 * kMaxRec;  // fp32 [6][128]
constexpr int kOffCtl = kOffScale + 6 * 128 * 4;  // mbarriers [2]
constexpr int kPSmem = kOffCtl + 16;
constexpr float kLog2eP = 1.4426950408889634f;

struct PrefillArgs {
  const uint16_t* q;           // [n_tokens][hq][128]
  const uint16_t* k_new;       // [n_tokens][hkv][128]
  const uint16_t* v_new;
  const int32_t* cu;           // [n_seqs + 1]
  const int32_t* seq_lens;     // cached tokens before each chunk
  const int32_t* block_tables; // [n_seqs][max_blocks]
  const uint8_t* cache;
  const uint16_t* ws;          // [n_seqs][hkv][2][128][128] or NULL
  uint16_t* out;               // [n_tokens][hq][128]
  unsigned* flags;
  int64_t num_blocks;
  int hkv, group, max_blocks;
};

__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

// Unnormalised FWHT over the 128 channels of the q fragment layout (thread (g, c)
// holds channels 16ks + 2c + {0, 1, 8, 9} in qv[ks][0..3]).
__device__ __forceinline__ void fwht_q(float (&qv)[8][4], int c) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const float u0 = qv[ks][0] + qv[ks][1], u1 = qv[ks][0] - qv[ks][1];
    const float u2 = qv[ks][2] + qv[ks][3], u3 = qv[ks][2] - qv[ks][3];
    qv[ks][0] = u0 + u2; qv[ks][2] = u0 - u2; qv[ks][1] = u1 + u3; qv[ks][3] = u1 - u3;
  }
#pragma unroll
  for (int bit = 1; bit <= 2; bit <<= 1) {
    const bool upper = (c & bit) != 0;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float o = __shfl_xor_sync(0xffffffffu, qv[ks][t], bit);
        qv[ks][t] = upper ? (o - qv[ks][t]) : (qv[ks][t] + o);
      }
  }
#pragma unroll
  for (int bit = 1; bit < 8; bit <<= 1)
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      if ((ks & bit) == 0)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float u = qv[ks][t], w = qv[ks | bit][t];
          qv[ks][t] = u + w;
          qv[ks | bit][t] = u - w;
        }
}

// Unnormalised FWHT over the 128 channels of the accumulator layout (thread (g, c)
// holds channels 8n + 2c + {0, 1} in acc[n][0..1]).
__device__ __forceinline__ void fwht_acc(float (&acc)[16][2], int c) {
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const float u = acc[n][0], w = acc[n][1];
    acc[n][0] = u + w;
    acc[n][1] = u - w;
  }
#pragma unroll
  for (int bit = 1; bit <= 2; bit <<= 1) {
    const bool upper = (c & bit) != 0;
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float o = __shfl_xor_sync(0xffffffffu, acc[n][t], bit);
        acc[n][t] = upper ? (o - acc[n][t]) : (acc[n][t] + o);
      }
  }
#pragma unroll
  for (int bit = 1; bit < 16; bit <<= 1)
#pragma unroll
    for (int n = 0; n < 16; ++n)
      if ((n & bit) == 0)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float u = acc[n][t], w = acc[n | bit][t];
          acc[n][t] = u + w;
          acc[n | bit][t] = u - w;
        }
}

// A pair of fp16 code values stored at `dst`.
__device__ __forceinline__ void put_pair(uint16_t* dst, uint32_t v) { *reinterpret_cast<uint32_t*>(dst) = v; }

// 4-bit word (codes of indices i0 + {0, 1, 8, 9} of two 16-index steps, low nibbles
// for the first step, high nibbles for the second): pairs code / 8 at index offsets
// 0, 8, 16, 24 from i0 along a shared row.
__device__ __forceinline__ void nibble_word(uint32_t w, uint16_t* row, int i0) {
  uint32_t lo, hi;
  cvt4(w & 0x0F0F0F0Fu, lo, hi);
  put_pair(row + i0, lo);
  put_pair(row + i0 + 8, hi);
  cvt4((w >> 4) & 0x0F0F0F0Fu, lo, hi);
  put_pair(row + i0 + 16, lo);
  put_pair(row + i0 + 24, hi);
}
// 2-bit word (four 16-index steps, one per byte): pairs code / 2 at index offsets
// 16k + 8r from i0 (k the byte, r = 0 for bits {0, 4} and 1 for bits {2, 6}).
__device__ __forceinline__ void crumb_word(uint32_t w, uint16_t* row, int i0) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    uint32_t v[4];
    cvt2((w >> (2 * r)) & 0x33333333u, v);
#pragma unroll
    for (int k = 0; k < 4; ++k) put_pair(row + i0 + 16 * k + 8 * r, v[k]);
  }
}

// The CTA turns the record in shared memory into fp16 key codes [token][channel],
// fp16 value codes [channel][token] and the six scale vectors (record layouts as
// in kvarn.h).
template <int KB, int VB, bool kLean>
__device__ __forceinline__ void unpack_tile(const uint8_t* rec, uint16_t* ks, uint16_t* vs, float* sc, int tid) {
  using L = RecordLayout<KB, VB, kLean>;
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(rec + L::kKCodeOff);
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(rec + L::kVCodeOff);
  if (KB == 4) {
    for (int wi = tid; wi < 2048; wi += kPThreads) {     // token t: 16 words, group (wi>>2)&3, word wi&3
      const int t = wi >> 4;
      nibble_word(kw[wi], ks + t * kPitch, 32 * (wi & 3) + 2 * ((wi >> 2) & 3));
    }
  } else {
    for (int wi = tid; wi < 1024; wi += kPThreads) {     // token t: 8 words, group (wi>>1)&3, word wi&1
      const int t = wi >> 3;
      crumb_word(kw[wi], ks + t * kPitch, 64 * (wi & 1) + 2 * ((wi >> 1) & 3));
    }
  }
  if (VB == 4) {
    for (int wi = tid; wi < 2048; wi += kPThreads) {     // channel i: 16 words
      const int i = wi >> 4;
      nibble_word(vw[wi], vs + i * kPitch, 32 * (wi & 3) + 2 * ((wi >> 2) & 3));
    }
  } else {
    for (int wi = tid; wi < 1024; wi += kPThreads) {     // panel m, cell, partner `which`, word u
      const int m = wi >> 7, cell = (wi >> 2) & 31, which = (wi >> 1) & 1, u = wi & 1;
      const int i = 16 * m + 8 * which + (cell >> 2);
      crumb_word(vw[wi], vs + i * kPitch, 64 * u + 2 * (cell & 3));
    }
  }
  if (tid < 128) {
    const uint16_t* km = reinterpret_cast<const uint16_t*>(rec + L::kKMetaOff);
    const uint16_t* vm = reinterpret_cast<const uint16_t*>(rec + L::kVMetaOff);
    const float kr = kLean ? 1.0f : h2f_bits(km[L::kKr + tid]);
    const float vc = kLean ? 1.0f : h2f_bits(vm[L::kVc + tid]);
    // the fp16 codes in shared memory are code / 8 (4-bit) or code / 2 (2-bit): the
    // step vectors carry the factor back (a power of two: exact)
    constexpr float kKf = KB == 4 ? 8.0f : 2.0f, kVf = VB == 4 ? 8.0f : 2.0f;
    sc[0 * 128 + tid] = kKf * kr * h2f_bits(km[L::kKs + tid]);   // per channel: r s (keys)
    sc[1 * 128 + tid] = kr * h2f_bits(km[L::kKz + tid]);   // per channel: r z
    sc[2 * 128 + tid] = h2f_bits(km[L::kKc + tid]);        // per token: c
    sc[3 * 128 + tid] = kVf * vc * h2f_bits(vm[L::kVs + tid]);   // per token: c s (values)
    sc[4 * 128 + tid] = vc * h2f_bits(vm[L::kVz + tid]);   // per token: c z
    sc[5 * 128 + tid] = h2f_bits(vm[L::kVr + tid]);        // per channel: r
  }
}

// One 128-token block for warp (g, c): keys ks [token][channel] fp16, values vs
// ([channel][token] if kPacked, else [token][channel]), scales sc (packed only),
// tokens with index > limit masked (fresh only).
template <bool kPacked>
__device__ __forceinline__ void attend_block(const uint16_t* ks, const uint16_t* vs, const float* sc,
                                             const float (&qv)[8][4], int g, int c, int lane, int limit,
                                             float& m_run, float& l_run, float (&acc)[16][2]) {
  uint32_t A[8][4];
  float beta = 0.f;
#pragma unroll
  for (int ks8 = 0; ks8 < 8; ++ks8) {
    const int ch0 = 16 * ks8 + 2 * c;
    float s0 = 1.f, s1 = 1.f, s2 = 1.f, s3 = 1.f;
    if (kPacked) {
      s0 = sc[ch0]; s1 = sc[ch0 + 1]; s2 = sc[ch0 + 8]; s3 = sc[ch0 + 9];
      beta = fmaf(qv[ks8][0], sc[128 + ch0], beta);
      beta = fmaf(qv[ks8][1], sc[128 + ch0 + 1], beta);
      beta = fmaf(qv[ks8][2], sc[128 + ch0 + 8], beta);
      beta = fmaf(qv[ks8][3], sc[128 + ch0 + 9], beta);
    }
    split2(qv[ks8][0] * s0, qv[ks8][1] * s1, A[ks8][0], A[ks8][1]);
    split2(qv[ks8][2] * s2, qv[ks8][3] * s3, A[ks8][2], A[ks8][3]);
  }
  if (kPacked) beta = quad_sum(beta);

  // scores of tokens 8nt + 2c + {0, 1}; ldmatrix x4 gives the B fragments of two k-steps
  float sc2[16][2];
#pragma unroll
  for (int ntg = 0; ntg < 4; ++ntg) {
    float d[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int nt = 4 * ntg + j;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks + (8 * nt + (lane & 7)) * kPitch + 32 * kp + 8 * (lane >> 3), b0, b1, b2, b3);
        mma16816(d[j], A[2 * kp], b0, b1);
        mma16816(d[j], A[2 * kp + 1], b2, b3);
      }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int nt = 4 * ntg + j;
      const int t0 = 8 * nt + 2 * c;
      float v0 = d[j][0] + d[j][2], v1 = d[j][1] + d[j][3];
      if (kPacked) {
        v0 = sc[256 + t0] * (v0 + beta);
        v1 = sc[256 + t0 + 1] * (v1 + beta);
      } else {
        if (t0 > limit) v0 = -INFINITY;
        if (t0 + 1 > limit) v1 = -INFINITY;
      }
      sc2[nt][0] = v0;
      sc2[nt][1] = v1;
    }
  }

  // online softmax (log2 domain)
  float tmax = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) tmax = fmaxf(tmax, fmaxf(sc2[nt][0], sc2[nt][1]));
  tmax = quad_max(tmax);
  const float m_new = fmaxf(m_run, tmax);
  if (m_new == -INFINITY) return;           // every token of the block masked
  const float corr = ex2(m_run - m_new);
  m_run = m_new;
  float lsum = 0.f;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    sc2[nt][0] = ex2(sc2[nt][0] - m_new);
    sc2[nt][1] = ex2(sc2[nt][1] - m_new);
    lsum += sc2[nt][0] + sc2[nt][1];
  }
  l_run = fmaf(l_run, corr, lsum);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    acc[n][0] *= corr;
    acc[n][1] *= corr;
  }

  // p' fragments and gamma; tokens 16ks + 2c + {0, 1} (nt = 2ks) and + {8, 9}
  float gamma = 0.f;
#pragma unroll
  for (int ks8 = 0; ks8 < 8; ++ks8) {
    const int t0 = 16 * ks8 + 2 * c;
    const float p0 = sc2[2 * ks8][0], p1 = sc2[2 * ks8][1], p2 = sc2[2 * ks8 + 1][0], p3 = sc2[2 * ks8 + 1][1];
    float s0 = 1.f, s1 = 1.f, s2 = 1.f, s3 = 1.f;
    if (kPacked) {
      s0 = sc[384 + t0]; s1 = sc[384 + t0 + 1]; s2 = sc[384 + t0 + 8]; s3 = sc[384 + t0 + 9];
      gamma = fmaf(p0, sc[512 + t0], gamma);
      gamma = fmaf(p1, sc[512 + t0 + 1], gamma);
      gamma = fmaf(p2, sc[512 + t0 + 8], gamma);
      gamma = fmaf(p3, sc[512 + t0 + 9], gamma);
    }
    split2(p0 * s0, p1 * s1, A[ks8][0], A[ks8][1]);
    split2(p2 * s2, p3 * s3, A[ks8][2], A[ks8][3]);
  }
  if (kPacked) gamma = quad_sum(gamma);

  // PV: channel n-tiles n2 = 4 n2g + j
#pragma unroll
  for (int n2g = 0; n2g < 4; ++n2g) {
    float d[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n2 = 4 * n2g + j;
        uint32_t b0, b1, b2, b3;
        if (kPacked)    // values [channel][token]
          ldsm_x4(vs + (8 * n2 + (lane & 7)) * kPitch + 32 * kp + 8 * (lane >> 3), b0, b1, b2, b3);
        else            // values [token][channel]
          ldsm_x4_t(vs + (32 * kp + 8 * (lane >> 3) + (lane & 7)) * kPitch + 8 * n2, b0, b1, b2, b3);
        mma16816(d[j], A[2 * kp], b0, b1);
        mma16816(d[j], A[2 * kp + 1], b2, b3);
      }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n2 = 4 * n2g + j;
      const int ch = 8 * n2 + 2 * c;
      const float v0 = d[j][0] + d[j][2], v1 = d[j][1] + d[j][3];
      if (kPacked) {
        acc[n2][0] = fmaf(sc[640 + ch], v0 + gamma, acc[n2][0]);
        acc[n2][1] = fmaf(sc[640 + ch + 1], v1 + gamma, acc[n2][1]);
      } else {
        acc[n2][0] += v0;
        acc[n2][1] += v1;
      }
    }
  }
}

// q of head g (< group) of chunk token `tok`, channels of the fragment layout,
// times `scale`; zeros for rows beyond the group.
__device__ __forceinline__ void load_q_frag(const PrefillArgs& a, int64_t tok, int h, int g, int c, float scale,
                                            float (&qv)[8][4]) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) qv[ks][0] = qv[ks][1] = qv[ks][2] = qv[ks][3] = 0.f;
  if (g >= a.group) return;
  const uint16_t* row = a.q + (tok * a.hkv * a.group + static_cast<int64_t>(h) * a.group + g) * kD;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const float2 p0 = h2pair(row + 16 * ks + 2 * c), p1 = h2pair(row + 16 * ks + 2 * c + 8);
    qv[ks][0] = p0.x * scale; qv[ks][1] = p0.y * scale; qv[ks][2] = p1.x * scale; qv[ks][3] = p1.y * scale;
  }
}

template <int KB, int VB, bool kLean>
__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using L = RecordLayout<KB, VB, kLean>;
  uint16_t* ks = reinterpret_cast<uint16_t*>(smem + kOffK);
  uint16_t* vs = reinterpret_cast<uint16_t*>(smem + kOffV);
  uint8_t* rec = smem + kOffRec;
  float* sc = reinterpret_cast<float*>(smem + kOffScale);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffCtl);      // [2]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int h = blockIdx.y, s = blockIdx.z;
  const int t0 = a.cu[s], chunk = a.cu[s + 1] - t0;
  if (static_cast<int>(blockIdx.x) * kPWarps >= chunk) return;        // whole CTA: nothing to do
  const int p = blockIdx.x * kPWarps + warp;                           // this warp's chunk token
  const bool active = p < chunk;
  const int L0 = max(a.seq_lens[s], 0);
  int n_full = L0 / kB;
  if (n_full > a.max_blocks) {
    n_full = a.max_blocks;
    if (tid == 0 && blockIdx.x == 0 && h == 0) raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
  }
  int n_ws = L0 % kB;
  if (n_ws > 0 && a.ws == nullptr) {
    n_ws = 0;
    if (tid == 0 && blockIdx.x == 0 && h == 0) raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
  }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  float acc[16][2];
#pragma unroll
  for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  float qv[8][4];
  const int64_t tok = static_cast<int64_t>(t0) + (active ? p : 0);

  // packed tiles, rotated domain: q_r = H q * log2(e) / sqrt(128), as FWHT(q) * log2(e) / 128
  load_q_frag(a, tok, h, g, c, kLog2eP / 128.0f, qv);
  fwht_q(qv, c);
  // thread 0 starts the copy of packed tile ti into record buffer b; false (and the
  // flag) for a block index outside the cache. Same answer in every thread.
  auto prefetch = [&](int ti, int b) {
    const int64_t blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + ti];
    const bool valid = blk >= 0 && blk < a.num_blocks;
    if (tid == 0) {
      if (valid) {
        mbar_arrive_expect_tx(&bar[b], L::kBytes);
        bulk_g2s(rec + b * kMaxRec, a.cache + (blk * a.hkv + h) * static_cast<int64_t>(L::kBytes), L::kBytes,
                 &bar[b]);
      } else {
        raise_flag(a.flags, KVARN_FLAG_BAD_BLOCK);
      }
    }
    return valid;
  };
  uint32_t phase = 0;                     // bit b: parity of record buffer b's barrier
  uint32_t pending = 0;                   // bit b: a copy into buffer b not yet waited for
  bool alive = true;
  bool cur = n_full > 0 && prefetch(0, 0);
  if (cur) pending |= 1u;
  for (int ti = 0; ti < n_full; ++ti) {
    const int b = ti & 1;
    // the next tile's copy overlaps this one's work (buffer b ^ 1 was last read by
    // the unpack of tile ti - 1, before the barrier that followed it)
    const bool next = ti + 1 < n_full && prefetch(ti + 1, b ^ 1);
    if (next) pending |= 2u >> b;
    if (cur) {
      const bool ok = mbar_wait(&bar[b], (phase >> b) & 1u, a.flags);
      if (ok) {
        phase ^= 1u << b;
        pending &= ~(1u << b);
      }
      if (!__syncthreads_and(ok)) {       // the copy never arrived (flag raised): stop
        alive = false;
        break;
      }
      unpack_tile<KB, VB, kLean>(rec + b * kMaxRec, ks, vs, sc, tid);
      __syncthreads();
      if (active) attend_block<true>(ks, vs, sc, qv, g, c, lane, 0, m_run, l_run, acc);
      __syncthreads();                    // shared tiles and record buffer b are rewritten next
    }
    cur = next;
  }
  if (!alive) {
    if (tid == 0)                         // let copies still in flight land before the CTA exits
      for (int b = 0; b < 2; ++b)
        if ((pending >> b) & 1u) mbar_wait(&bar[b], (phase >> b) & 1u, a.flags);
    return;
  }

  // back to the input domain: acc_u = H acc_r (orthonormal H), then the fresh tokens
  fwht_acc(acc, c);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    acc[n][0] *= kInvSqrt128;
    acc[n][1] *= kInvSqrt128;
  }
  load_q_frag(a, tok, h, g, c, kLog2eP * kInvSqrt128, qv);
  // fresh token f: workspace token f (f < n_ws) or chunk token f - n_ws; this CTA's
  // last token attends f <= n_ws + p_last
  const int p_last = min(chunk - 1, static_cast<int>(blockIdx.x) * kPWarps + kPWarps - 1);
  const int n_fresh = n_ws + p_last + 1;
  for (int fb = 0; fb * kB < n_fresh; ++fb) {
    // rows f = 128 fb + r; 16-byte pieces: K and V, 128 rows x 16 pieces each
    for (int e = tid; e < 2 * 128 * 16; e += kPThreads) {
      const int which = e >> 11, r = (e >> 4) & 127, piece = e & 15;
      const int f = fb * kB + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (f < n_fresh) {
        const uint16_t* src;
        if (f < n_ws)
          src = a.ws + (((static_cast<int64_t>(s) * a.hkv + h) * 2 + which) * kB + f) * kD;
        else
          src = (which ? a.v_new : a.k_new) + ((static_cast<int64_t>(t0) + f - n_ws) * a.hkv + h) * kD;
        v = *reinterpret_cast<const uint4*>(src + piece * 8);
      }
      *reinterpret_cast<uint4*>((which ? vs : ks) + r * kPitch + piece * 8) = v;
    }
    __syncthreads();
    if (active) attend_block<false>(ks, vs, nullptr, qv, g, c, lane, n_ws + p - fb * kB, m_run, l_run, acc);
    __syncthreads();
  }

  if (!active || g >= a.group) return;
  const float l = quad_sum(l_run);
  const float inv_l = l > 0.f ? 1.0f / l : 0.f;
  uint16_t* orow = a.out + (tok * a.hkv * a.group + static_cast<int64_t>(h) * a.group + g) * kD;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const uint32_t lo = f2h_bits(acc[n][0] * inv_l), hi = f2h_bits(acc[n][1] * inv_l);
    *reinterpret_cast<uint32_t*>(orow + 8 * n + 2 * c) = lo | (hi << 16);
  }
}

template <int KB, int VB, bool kLean>
cudaError_t launch_prefill_kernel(const PrefillArgs& a, int n_seqs, int max_chunk, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(prefill_kernel<KB, VB, kLean>, kPSmem, smem_set);
  if (err != cudaSuccess) return err;
  const dim3 grid((max_chunk + kPWarps - 1) / kPWarps, a.hkv, n_seqs);
  prefill_kernel<KB, VB, kLean><<<grid, kPThreads, kPSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, const int32_t* cu_tokens,
                           const int32_t* seq_lens, const int32_t* block_tables, const uint8_t* cache,
                           const uint16_t* ws, int n_seqs, int max_chunk, int hkv, int group, int max_blocks,
                           int64_t num_blocks, int k_bits, int v_bits, bool lean, uint16_t* out, unsigned* flags,
                           cudaStream_t stream) {
  if (n_seqs <= 0 || max_chunk <= 0) return cudaSuccess;
  PrefillArgs a{q, k_new, v_new, cu_tokens, seq_lens, block_tables, cache, ws, out, flags, num_blocks,
                hkv, group, max_blocks};
  if (k_bits == 4 && v_bits == 2) return lean ? launch_prefill_kernel<4, 2, true>(a, n_seqs, max_chunk, stream)
                                              : launch_prefill_kernel<4, 2, false>(a, n_seqs, max_chunk, stream);
  if (k_bits == 4 && v_bits == 4 && !lean) return launch_prefill_kernel<4, 4, false>(a, n_seqs, max_chunk, stream);
  if (k_bits == 2 && v_bits == 2 && !lean) return launch_prefill_kernel<2, 2, false>(a, n_seqs, max_chunk, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvarn
