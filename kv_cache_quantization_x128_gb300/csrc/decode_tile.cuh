// Device code of paged decode attention over the packed cache (KVarN README,
// "How KVarN works": the scales are re-applied on read; the orthonormal rotation
// keeps attention scores): the split phase (stream-K over tiles, tensor-core tile
// attention, partial records) and the merge of partial records with the fp16
// workspace tokens, as device functions that the decode kernels and the fused
// serving step call.
#pragma once
#include <stdint.h>

#include "kvarn_common.cuh"
#include "kvarn_frag.cuh"

namespace kvarn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWarps = 12;                   // split warps per CTA (at most)
constexpr int kMaxCtas = 1024;                  // upper bound used to size scratch
constexpr int kPartStride = 132;                // floats per q-head: acc[128], max, sum, pad
constexpr int kRecFloats = 8 * kPartStride;     // one partial record (8 q-head slots)

// Split-phase shapes for KB-bit keys and VB-bit values.
// SplitCfg: up to 12 warps (3 per scheduler), each with one record stage, q_r in
// shared memory so that 168 registers hold the rest, and the tile after the next one
// prefetched into L2: 12 warps for the 10-14 KB records, 10 for k4v4's 18 KB. The
// split kernel's shape for batches of many (sequence, kv-head) units.
template <int KB, int VB, bool kLean = false>
struct SplitCfg {
  using L = RecordLayout<KB, VB, kLean>;
  static constexpr int fits(int w) { return w * (L::kBytes + 8 + 4096) <= 232448; }
  static constexpr int kWarps = fits(12) ? 12 : fits(10) ? 10 : 8;
  static constexpr int kStages = 1;
  static constexpr bool kQSmem = true;
  static constexpr int kQOff = kWarps * kStages * (L::kBytes + 8);   // q_r: [warp][ks][lane] float4
  static constexpr int kSmem = kQOff + kWarps * 4096;
  static_assert(kSmem <= 232448 && kQOff % 16 == 0 && kWarps <= kMaxWarps, "decode stages");
};
// SplitCfg2: the most warps (8 down to 6) whose two record stages each fit in shared
// memory, q_r in registers. The split kernel's shape for a few long units (a third
// fewer warps, so a third fewer partial records to merge per unit), and the serving
// step's (its blocks have 8 warps).
template <int KB, int VB, bool kLean = false>
struct SplitCfg2 {
  using L = RecordLayout<KB, VB, kLean>;
  static constexpr int fits(int w) { return w * 2 * (L::kBytes + 8) <= 232448; }
  static constexpr int kWarps = fits(8) ? 8 : fits(7) ? 7 : 6;
  static constexpr int kStages = 2;
  static constexpr bool kQSmem = false;
  static constexpr int kQOff = 0;
  static constexpr int kSmem = kWarps * kStages * (L::kBytes + 8);
  static_assert(kSmem <= 232448, "decode stages");
};

struct DecodeArgs {
  const uint16_t* q;
  const uint8_t* cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int64_t* prefix;      // [n_seqs + 1] exclusive prefix of full tiles
  int64_t* ranges;      // [n_ctas * kWarps][2] tile range of each split-kernel warp
  float* part;          // [records][8][132]
  int32_t* cover;       // [n_seqs * hkv][2]: first and last split warp of each unit (-1: none)
  unsigned* flags;
  int64_t num_blocks;
  int n_seqs;
  int hkv;
  int group;            // q-heads per kv-head (1..8)
  int max_blocks;
  int n_ctas;           // CTAs of the split kernel
  int warps;            // warps per CTA of the split kernel
};

__device__ __forceinline__ int full_tiles(const DecodeArgs& a, int s) {
  const int L = max(a.seq_lens[s], 0);
  return min(L / kB, a.max_blocks);
}

// Range [beg, end) of global tiles owned by warp `wg` of the split kernel.
template <int kWarps>
__device__ __forceinline__ void warp_range(int64_t total, int n_ctas, int64_t wg, int64_t& beg, int64_t& end) {
  const int64_t b = wg / kWarps, w = wg % kWarps;
  const int64_t c0 = b * total / n_ctas, c1 = (b + 1) * total / n_ctas;
  beg = c0 + w * (c1 - c0) / kWarps;
  end = c0 + (w + 1) * (c1 - c0) / kWarps;
}

// ------------------------------------------------------------------ tile cursor
struct Cursor {
  int s, h, ti, nf;
};

// sequence s holding global tile g (prefix[s]*hkv <= g < prefix[s+1]*hkv)
__device__ __forceinline__ Cursor locate(const DecodeArgs& a, int64_t g) {
  int lo = 0, hi = a.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.prefix[mid] * a.hkv <= g) lo = mid; else hi = mid - 1;
  }
  Cursor c;
  c.s = lo;
  c.nf = static_cast<int>(a.prefix[lo + 1] - a.prefix[lo]);
  const int64_t off = g - a.prefix[lo] * a.hkv;
  c.h = static_cast<int>(off / c.nf);
  c.ti = static_cast<int>(off - static_cast<int64_t>(c.h) * c.nf);
  return c;
}

__device__ __forceinline__ void advance(const DecodeArgs& a, Cursor& c) {
  if (++c.ti < c.nf) return;
  c.ti = 0;
  if (++c.h < a.hkv) return;
  c.h = 0;
  do {
    ++c.s;
    c.nf = c.s < a.n_seqs ? static_cast<int>(a.prefix[c.s + 1] - a.prefix[c.s]) : 1;
  } while (c.nf == 0);
}

// Lane 0: start the copy of the tile at cursor `c` into `stage`; a block index
// outside [0, num_blocks) completes the barrier phase without data and returns false.
template <int kRecBytes>
__device__ __forceinline__ bool issue_tile(const DecodeArgs& a, const Cursor& c, uint8_t* stage, uint64_t* bar) {
  const int64_t blk = a.block_tables[static_cast<int64_t>(c.s) * a.max_blocks + c.ti];
  if (blk < 0 || blk >= a.num_blocks) {
    raise_flag(a.flags, KVARN_FLAG_BAD_BLOCK);
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
    return false;
  }
  mbar_arrive_expect_tx(bar, kRecBytes);
  bulk_g2s(stage, a.cache + (blk * a.hkv + c.h) * static_cast<int64_t>(kRecBytes), kRecBytes, bar);
  return true;
}

// Lane 0: prefetch the record of the tile at cursor `c` into L2 (nothing for a block
// index outside [0, num_blocks); its copy will raise the flag).
template <int kRecBytes>
__device__ __forceinline__ void prefetch_tile(const DecodeArgs& a, const Cursor& c) {
  const int64_t blk = a.block_tables[static_cast<int64_t>(c.s) * a.max_blocks + c.ti];
  if (blk < 0 || blk >= a.num_blocks) return;
  const uint8_t* src = a.cache + (blk * a.hkv + c.h) * static_cast<int64_t>(kRecBytes);
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(static_cast<uint32_t>(kRecBytes))
               : "memory");
}

// q_r2 of this thread's 32 channels for (sequence s, kv-head h): H q * log2(e)/sqrt(128),
// computed as FWHT(q) * log2(e) / 128. Thread (g, c) holds head g, channels
// 16ks + 2c + {0, 1, 8, 9}; channel bits 1-2 live across the quad (lanes ^1, ^2).
__device__ __forceinline__ void load_q(const DecodeArgs& a, int s, int h, int g, int c, float (&qv)[8][4]) {
  const int hq = a.hkv * a.group;
  if (g < a.group) {
    const uint16_t* row = a.q + (static_cast<int64_t>(s) * hq + static_cast<int64_t>(h) * a.group + g) * kD;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const float2 p0 = h2pair(row + 16 * ks + 2 * c), p1 = h2pair(row + 16 * ks + 2 * c + 8);
      qv[ks][0] = p0.x; qv[ks][1] = p0.y; qv[ks][2] = p1.x; qv[ks][3] = p1.y;
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) qv[ks][0] = qv[ks][1] = qv[ks][2] = qv[ks][3] = 0.f;
  }
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {       // channel bits 0 and 3: inside the thread
    const float u0 = qv[ks][0] + qv[ks][1], u1 = qv[ks][0] - qv[ks][1];
    const float u2 = qv[ks][2] + qv[ks][3], u3 = qv[ks][2] - qv[ks][3];
    qv[ks][0] = u0 + u2; qv[ks][2] = u0 - u2; qv[ks][1] = u1 + u3; qv[ks][3] = u1 - u3;
  }
#pragma unroll
  for (int bit = 1; bit <= 2; bit <<= 1) {   // channel bits 1 and 2: across the quad
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
  for (int bit = 1; bit < 8; bit <<= 1)      // channel bits 4-6: the ks index
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      if ((ks & bit) == 0)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float u = qv[ks][t], w = qv[ks | bit][t];
          qv[ks][t] = u + w;
          qv[ks | bit][t] = u - w;
        }
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int t = 0; t < 4; ++t) qv[ks][t] *= kLog2e / 128.0f;
}

// One packed tile: update the running (max, sum, acc) of head g.
// q_r comes from qv, or from shared memory (qsm[32 ks], this thread's float4 of k-step
// ks) when kQSmem.
template <int KB, int VB, bool kLean, bool kQSmem>
__device__ __forceinline__ void attend_tile(const uint8_t* rec, const float (&qv)[8][4], const float4* qsm, int g,
                                            int c, float& m_run, float& l_run, float (&acc)[16][2]) {
  using L = RecordLayout<KB, VB, kLean>;
  const uint16_t* km = reinterpret_cast<const uint16_t*>(rec + L::kKMetaOff);
  const uint16_t* vm = reinterpret_cast<const uint16_t*>(rec + L::kVMetaOff);

  // q' fragments (hi rows g, lo rows g + 8) and beta (fp32 pairs)
  uint32_t A[8][4];
  float2 beta2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int ch0 = 16 * ks + 2 * c;
    // r s and r z in fp32 straight from the fp16 pairs (lean records fold r into s, z)
    const uint32_t s0 = h2raw(km + L::kKs + ch0), s1 = h2raw(km + L::kKs + ch0 + 8);
    const uint32_t z0 = h2raw(km + L::kKz + ch0), z1 = h2raw(km + L::kKz + ch0 + 8);
    const uint32_t r0 = kLean ? kH_One : h2raw(km + L::kKr + ch0);
    const uint32_t r1 = kLean ? kH_One : h2raw(km + L::kKr + ch0 + 8);
    const float2 rs0 = mul_h2(r0, s0), rs1 = mul_h2(r1, s1);
    const float2 rz0 = mul_h2(r0, z0), rz1 = mul_h2(r1, z1);
    const float4 qq = kQSmem ? qsm[32 * ks] : make_float4(qv[ks][0], qv[ks][1], qv[ks][2], qv[ks][3]);
    const float2 qa = make_float2(qq.x, qq.y), qb = make_float2(qq.z, qq.w);
    split2p(__fmul2_rn(qa, rs0), A[ks][0], A[ks][1]);
    split2p(__fmul2_rn(qb, rs1), A[ks][2], A[ks][3]);
    beta2 = __ffma2_rn(qa, rz0, beta2);
    beta2 = __ffma2_rn(qb, rz1, beta2);
  }
  const float beta = quad_sum(beta2.x + beta2.y);
  const float2 beta_2 = make_float2(beta, beta);
  const float2 kf2 = make_float2(KB == 4 ? 8.f : 2.f, KB == 4 ? 8.f : 2.f);   // codes were converted to c / 8 or c / 2

  // scores of tokens 8nt + 2c + {0, 1}, four n-tiles at a time (independent chains)
  float2 sc[16];
#pragma unroll
  for (int ntg = 0; ntg < 4; ++ntg) {
    float d[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
    if (KB == 4) {
      // token row of 64 bytes, this thread's 16: word m holds k-steps 2m (low byte
      // of each half) and 2m + 1 (high byte)
      uint32_t kw[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(rec + L::kKCodeOff + (8 * (4 * ntg + j) + g) * 64 + c * 16);
        kw[j][0] = v.x; kw[j][1] = v.y; kw[j][2] = v.z; kw[j][3] = v.w;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b00, b01, b10, b11;
          cvt4(kw[j][m] & 0x0F0F0F0Fu, b00, b01);
          cvt4((kw[j][m] >> 4) & 0x0F0F0F0Fu, b10, b11);
          mma16816(d[j], A[2 * m], b00, b01);
          mma16816(d[j], A[2 * m + 1], b10, b11);
        }
    } else {
      // token row of 32 bytes, this thread's 8: word u holds k-steps 4u + 2sg + {0, 1}
      // in byte sg of each half (crumbs 0-1 and 2-3 of the byte)
      uint32_t kw[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint2 v = *reinterpret_cast<const uint2*>(rec + L::kKCodeOff + (8 * (4 * ntg + j) + g) * 32 + c * 8);
        kw[j][0] = v.x; kw[j][1] = v.y;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b0[4], b1[4];
          cvt2(kw[j][u] & 0x33333333u, b0);
          cvt2((kw[j][u] >> 2) & 0x33333333u, b1);
#pragma unroll
          for (int b = 0; b < 4; ++b) mma16816(d[j], A[4 * u + b], b0[b], b1[b]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int nt = 4 * ntg + j;
      const float2 ck = h2pair(km + L::kKc + 8 * nt + 2 * c);
      sc[nt] = __fmul2_rn(ck, __ffma2_rn(__fadd2_rn(make_float2(d[j][0], d[j][1]), make_float2(d[j][2], d[j][3])),
                                         kf2, beta_2));
    }
  }

  // online softmax (log2 domain)
  float tmax = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) tmax = fmax3f(tmax, sc[nt].x, sc[nt].y);
  tmax = quad_max(tmax);
  const float m_new = fmaxf(m_run, tmax);
  const float corr = ex2(m_run - m_new);
  m_run = m_new;
  const float2 mneg = make_float2(-m_new, -m_new);
  float2 lsum2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const float2 e = __fadd2_rn(sc[nt], mneg);
    sc[nt] = make_float2(ex2(e.x), ex2(e.y));
    lsum2 = __fadd2_rn(lsum2, sc[nt]);
  }
  l_run = fmaf(l_run, corr, lsum2.x + lsum2.y);
  const float2 corr2 = make_float2(corr, corr);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const float2 v = __fmul2_rn(make_float2(acc[n][0], acc[n][1]), corr2);
    acc[n][0] = v.x;
    acc[n][1] = v.y;
  }

  // p' fragments and gamma; tokens 16ks + 2c + {0,1} (nt = 2ks) and + {8,9} (nt = 2ks+1)
  float2 gamma2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int t0 = 16 * ks + 2 * c;
    // c s and c z in fp32 straight from the fp16 pairs (lean records fold c into s, z)
    const uint32_t s0 = h2raw(vm + L::kVs + t0), s1 = h2raw(vm + L::kVs + t0 + 8);
    const uint32_t z0 = h2raw(vm + L::kVz + t0), z1 = h2raw(vm + L::kVz + t0 + 8);
    const uint32_t c0 = kLean ? kH_One : h2raw(vm + L::kVc + t0);
    const uint32_t c1 = kLean ? kH_One : h2raw(vm + L::kVc + t0 + 8);
    const float2 cs0 = mul_h2(c0, s0), cs1 = mul_h2(c1, s1);
    const float2 cz0 = mul_h2(c0, z0), cz1 = mul_h2(c1, z1);
    split2p(__fmul2_rn(sc[2 * ks], cs0), A[ks][0], A[ks][1]);
    split2p(__fmul2_rn(sc[2 * ks + 1], cs1), A[ks][2], A[ks][3]);
    gamma2 = __ffma2_rn(sc[2 * ks], cz0, gamma2);
    gamma2 = __ffma2_rn(sc[2 * ks + 1], cz1, gamma2);
  }
  const float gamma = quad_sum(gamma2.x + gamma2.y);
  const float2 gamma_2 = make_float2(gamma, gamma);
  const float2 vf2 = make_float2(VB == 4 ? 8.f : 2.f, VB == 4 ? 8.f : 2.f);

  if (VB == 2) {
    // PV with 2-bit values: channel n-tile nt2 = 2np + which; cell (g, c) of panel np serves both `which`;
    // two panels at a time -> four independent chains
  #pragma unroll
    for (int npg = 0; npg < 4; ++npg) {
      uint32_t vw[2][4];
  #pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(rec + L::kVCodeOff + (2 * npg + i) * 512 + (g * 4 + c) * 16);
        vw[i][0] = v.x; vw[i][1] = v.y; vw[i][2] = v.z; vw[i][3] = v.w;   // [which*2 + u]
      }
      float d[4][4];
  #pragma unroll
      for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
  #pragma unroll
      for (int u = 0; u < 2; ++u)
  #pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = j >> 1, which = j & 1;
          const uint32_t w = vw[i][which * 2 + u];
          uint32_t b0[4], b1[4];
          cvt2(w & 0x33333333u, b0);
          cvt2((w >> 2) & 0x33333333u, b1);
  #pragma unroll
          for (int b = 0; b < 4; ++b) mma16816(d[j], A[4 * u + b], b0[b], b1[b]);
        }
  #pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int nt2 = 2 * (2 * npg + (j >> 1)) + (j & 1);
        const float2 rv = h2pair(vm + L::kVr + 8 * nt2 + 2 * c);
        const float2 v = __ffma2_rn(
            rv, __ffma2_rn(__fadd2_rn(make_float2(d[j][0], d[j][1]), make_float2(d[j][2], d[j][3])), vf2, gamma_2),
            make_float2(acc[nt2][0], acc[nt2][1]));
        acc[nt2][0] = v.x;
        acc[nt2][1] = v.y;
      }
    }
  } else {
    // PV with 4-bit values: channel row of 64 bytes, this thread's 16; word m holds
    // token k-steps 2m and 2m + 1 (low and high byte of each half); four channel
    // n-tiles at a time -> four independent chains
#pragma unroll
    for (int npg = 0; npg < 4; ++npg) {
      uint32_t vw[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(rec + L::kVCodeOff + (8 * (4 * npg + j) + g) * 64 + c * 16);
        vw[j][0] = v.x; vw[j][1] = v.y; vw[j][2] = v.z; vw[j][3] = v.w;
      }
      float d[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b00, b01, b10, b11;
          cvt4(vw[j][m] & 0x0F0F0F0Fu, b00, b01);
          cvt4((vw[j][m] >> 4) & 0x0F0F0F0Fu, b10, b11);
          mma16816(d[j], A[2 * m], b00, b01);
          mma16816(d[j], A[2 * m + 1], b10, b11);
        }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int nt2 = 4 * npg + j;
        const float2 rv = h2pair(vm + L::kVr + 8 * nt2 + 2 * c);
        const float2 v = __ffma2_rn(
            rv, __ffma2_rn(__fadd2_rn(make_float2(d[j][0], d[j][1]), make_float2(d[j][2], d[j][3])), vf2, gamma_2),
            make_float2(acc[nt2][0], acc[nt2][1]));
        acc[nt2][0] = v.x;
        acc[nt2][1] = v.y;
      }
    }
  }
}

// Partial record of one (sequence, kv-head) over the tiles this warp attended.
__device__ __forceinline__ void flush_record(const DecodeArgs& a, int64_t rec_idx, int g, int c, float m_run,
                                             float l_run, const float (&acc)[16][2]) {
  const float l = quad_sum(l_run);
  if (g >= a.group) return;
  float* out = a.part + rec_idx * kRecFloats + g * kPartStride;
#pragma unroll
  for (int n = 0; n < 16; ++n) *reinterpret_cast<float2*>(out + 8 * n + 2 * c) = make_float2(acc[n][0], acc[n][1]);
  if (c == 0) *reinterpret_cast<float2*>(out + 128) = make_float2(m_run, l);
}

// The split phase of CTA `cta` in shape Cfg: warp w < kWarps attends its range of
// tiles (warps beyond kWarps, in a larger block, have none); `smem` holds the stages
// (and q_r when Cfg::kQSmem).
template <int KB, int VB, bool kLean, class Cfg = SplitCfg<KB, VB, kLean>>
__device__ __forceinline__ void split_body(const DecodeArgs& a, uint8_t* smem, int cta) {
  constexpr int kWarps = Cfg::kWarps, kStages = Cfg::kStages;
  constexpr int kRecBytes = RecordLayout<KB, VB, kLean>::kBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kWarps) return;
  const int g = lane >> 2, c = lane & 3;
  const int64_t wg = static_cast<int64_t>(cta) * kWarps + warp;
  const int64_t total = a.prefix[a.n_seqs] * a.hkv;
  int64_t gb, ge;
  warp_range<kWarps>(total, a.n_ctas, wg, gb, ge);
  if (lane == 0) {
    a.ranges[2 * wg] = gb;
    a.ranges[2 * wg + 1] = ge;
  }
  if (gb >= ge) return;   // warps are independent: no CTA-wide barrier below

  float4* qsm = reinterpret_cast<float4*>(smem + Cfg::kQOff) + warp * 256 + lane;   // used when Cfg::kQSmem
  uint8_t* stages = smem + warp * kStages * kRecBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * kRecBytes) + warp * kStages;
  if (lane == 0) {
    for (int k = 0; k < kStages; ++k) mbar_init(&bars[k], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // load cursor (tiles being copied) runs kStages tiles ahead of the compute cursor
  Cursor lc = locate(a, gb);
  Cursor cc = lc;
  uint32_t valid = 0;
  for (int k = 0; k < kStages && gb + k < ge; ++k) {
    if (k > 0) advance(a, lc);
    bool ok = false;
    if (lane == 0) ok = issue_tile<kRecBytes>(a, lc, stages + k * kRecBytes, &bars[k]);
    if (__shfl_sync(0xffffffffu, ok, 0)) valid |= 1u << k;
  }

  Cursor pc = lc;   // one stage: the tile after the one being copied, prefetched into L2
  if (kStages == 1 && gb + 1 < ge) {
    advance(a, pc);
    if (lane == 0) prefetch_tile<kRecBytes>(a, pc);
  }
  float qv[8][4];
  float acc[16][2];
  float m_run = -INFINITY, l_run = 0.f;
  int64_t unit = -1;
  uint32_t phase = 0;
  bool clean = true;   // every issued copy was waited for
  for (int64_t k = 0; gb + k < ge; ++k) {
    const int stg = static_cast<int>(k % kStages);
    const int64_t u = static_cast<int64_t>(cc.s) * a.hkv + cc.h;
    if (u != unit) {
      if (unit >= 0) flush_record(a, wg + unit, g, c, m_run, l_run, acc);
      unit = u;
      if (lane == 0 && cc.ti == 0) a.cover[2 * u] = static_cast<int32_t>(wg);   // the unit's first split warp
      load_q(a, cc.s, cc.h, g, c, qv);
      if (Cfg::kQSmem) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) qsm[32 * ks] = make_float4(qv[ks][0], qv[ks][1], qv[ks][2], qv[ks][3]);
      }
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = 0.f;
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stg], (phase >> stg) & 1u, a.flags));
    phase ^= 1u << stg;
    if (!ok) {        // a copy never arrived (flag raised): stop this warp
      clean = false;
      break;
    }
    if (lane == 0 && cc.ti == cc.nf - 1) a.cover[2 * u + 1] = static_cast<int32_t>(wg);   // and its last
    if ((valid >> stg) & 1u)
      attend_tile<KB, VB, kLean, Cfg::kQSmem>(stages + stg * kRecBytes, qv, qsm, g, c, m_run, l_run, acc);
    __syncwarp();
    if (gb + k + kStages < ge) {     // refill this stage with the tile kStages ahead
      advance(a, lc);
      bool issued = false;
      if (lane == 0) issued = issue_tile<kRecBytes>(a, lc, stages + stg * kRecBytes, &bars[stg]);
      if (__shfl_sync(0xffffffffu, issued, 0)) valid |= 1u << stg; else valid &= ~(1u << stg);
      if (kStages == 1 && gb + k + 2 < ge) {
        advance(a, pc);
        if (lane == 0) prefetch_tile<kRecBytes>(a, pc);
      }
    }
    advance(a, cc);
  }
  if (unit >= 0) flush_record(a, wg + unit, g, c, m_run, l_run, acc);
  __syncwarp();
  if (lane == 0 && clean)   // the stages' shared memory may be reused after this phase
    for (int k = 0; k < kStages; ++k) mbar_inval(&bars[k]);
}

// ------------------------------------------------------------------ merge
// The fp16 workspace tokens of a unit (exact, unrotated K and V rows of its partial
// last tile) are attended by the unit's 8 warps together, warp w taking tokens
// 16w .. 16w + 15 for all q-heads of the group at once with m16n8k16 MMAs; each
// warp leaves per head its running max, sum and 128-channel output in shared
// memory, and the records' merge then folds them in.
struct WsPart {
  float o[8][8][128];   // [warp][q-head][channel]
  float m[8][8];        // [warp][q-head] max of the warp's scores (log2 domain)
  float l[8][8];        // [warp][q-head] sum of 2^(score - max)
};

// Workspace tokens of sequence s: L % 128, or none (flag raised) without a workspace.
__device__ __forceinline__ int ws_tokens(const DecodeArgs& a, const uint16_t* ws, int s, bool report) {
  const int n_ws = max(a.seq_lens[s], 0) % kB;
  if (n_ws > 0 && ws == nullptr) {   // tail tokens without a workspace: attend the tiles only
    if (report) raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
    return 0;
  }
  return n_ws;
}

// Warp w's share of the workspace tokens of unit (kv-head h, sequence s). Thread
// (g, c) = (lane / 4, lane % 4). The MMAs' K index is permuted the same way in both
// operands so that every load is 16 bytes: in k-step ks the fragment's positions
// 2c, 2c+1 carry channels 32c + 4ks + {0, 1} and 2c+8, 2c+9 channels 32c + 4ks + {2, 3}.
// S = q K^T: A = q (rows 0-7 the group's heads, exact fp16; rows 8-15 zero), B = the
// K rows of tokens 16w + 8nt + g. PV: A = p as fp16 hi (rows 0-7) and lo (rows 8-15),
// K index = the warp's 16 tokens in the S accumulators' order; B = the V rows, n-tile
// j's column g being channel 16g + j, so each thread loads 32 contiguous bytes of
// each of its four tokens.
__device__ __forceinline__ void merge_ws_part(const DecodeArgs& a, const uint16_t* __restrict__ ws, int h, int s,
                                              int n_ws, int w, WsPart& sm) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int t0 = 16 * w;
  if (t0 >= n_ws) return;
  const int64_t wbase = (static_cast<int64_t>(s) * a.hkv + h) * 2 * static_cast<int64_t>(kB * kD);
  const uint16_t* wk = ws + wbase;
  const uint16_t* wv = ws + wbase + kB * kD;

  // q fragments of head g (zero for heads past the group)
  uint32_t qa[8][2];
  if (g < a.group) {
    const uint4* qr = reinterpret_cast<const uint4*>(
        a.q + ((static_cast<int64_t>(s) * a.hkv + h) * a.group + g) * kD + 32 * c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = qr[j];
      qa[2 * j][0] = v.x; qa[2 * j][1] = v.y; qa[2 * j + 1][0] = v.z; qa[2 * j + 1][1] = v.w;
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) qa[ks][0] = qa[ks][1] = 0u;
  }
  // scores: tokens t0 + 8nt + 2c + {0, 1} of head g (rows past n_ws, still inside the
  // unit's 128 workspace rows, are read and masked out)
  float d[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint4* kr = reinterpret_cast<const uint4*>(wk + (t0 + 8 * nt + g) * kD + 32 * c);
    uint4 kv4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) kv4[j] = kr[j];
    d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t a0[4] = {qa[2 * j][0], 0u, qa[2 * j][1], 0u};
      const uint32_t a1[4] = {qa[2 * j + 1][0], 0u, qa[2 * j + 1][1], 0u};
      mma16816(d[nt], a0, kv4[j].x, kv4[j].y);
      mma16816(d[nt], a1, kv4[j].z, kv4[j].w);
    }
  }
  constexpr float kScale = kLog2e * kInvSqrt128;
  float sc[2][2];
  float mx = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      sc[nt][e] = (t0 + 8 * nt + 2 * c + e < n_ws) ? d[nt][e] * kScale : -INFINITY;
      mx = fmaxf(mx, sc[nt][e]);
    }
  mx = quad_max(mx);   // finite: token t0 is valid
  float lsum = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      sc[nt][e] = exp2f(sc[nt][e] - mx);   // 0 for the masked tokens
      lsum += sc[nt][e];
    }
  lsum = quad_sum(lsum);
  uint32_t pa[4];
  split2p(make_float2(sc[0][0], sc[0][1]), pa[0], pa[1]);
  split2p(make_float2(sc[1][0], sc[1][1]), pa[2], pa[3]);

  // PV in two halves of eight n-tiles (channels 16g + 8hf .. 16g + 8hf + 7)
  const int tk[4] = {t0 + 2 * c, t0 + 2 * c + 1, t0 + 2 * c + 8, t0 + 2 * c + 9};
  float* orow = &sm.o[w][g][0];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint4 vr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)   // masked tokens contribute zero (their rows are never multiplied)
      vr[i] = tk[i] < n_ws ? *reinterpret_cast<const uint4*>(wv + tk[i] * kD + 16 * g + 8 * hf)
                           : make_uint4(0u, 0u, 0u, 0u);
    float o[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w01 = (&vr[0].x)[j >> 1], w1 = (&vr[1].x)[j >> 1];
      const uint32_t w8 = (&vr[2].x)[j >> 1], w9 = (&vr[3].x)[j >> 1];
      const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;   // high or low halves of both words
      const uint32_t b0 = __byte_perm(w01, w1, sel), b1 = __byte_perm(w8, w9, sel);
      o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      mma16816(o[j], pa, b0, b1);
    }
    // column 2c of n-tile j is channel 16(2c) + 8hf + j, column 2c + 1 channel 16(2c+1) + 8hf + j;
    // rows g (hi) and g + 8 (lo) add up to head g
    float4* o0 = reinterpret_cast<float4*>(orow + 32 * c + 8 * hf);
    float4* o1 = reinterpret_cast<float4*>(orow + 32 * c + 16 + 8 * hf);
    o0[0] = make_float4(o[0][0] + o[0][2], o[1][0] + o[1][2], o[2][0] + o[2][2], o[3][0] + o[3][2]);
    o0[1] = make_float4(o[4][0] + o[4][2], o[5][0] + o[5][2], o[6][0] + o[6][2], o[7][0] + o[7][2]);
    o1[0] = make_float4(o[0][1] + o[0][3], o[1][1] + o[1][3], o[2][1] + o[2][3], o[3][1] + o[3][3]);
    o1[1] = make_float4(o[4][1] + o[4][3], o[5][1] + o[5][3], o[6][1] + o[6][3], o[7][1] + o[7][3]);
  }
  if (c == 0) {
    sm.m[w][g] = mx;
    sm.l[w][g] = lsum;
  }
}

// The split warps whose ranges cover unit u's tiles, [wlo, whi): from the warp that
// took its first tile to the one that took its last, as the split phase marked them
// (ranges are contiguous and ordered; an empty range in between left no record; a
// unit without both marks, after a timed-out split warp, merges no records).
// `cv` is the unit's pair of marks, loaded by the caller with the sequence's length.
__device__ __forceinline__ void covering_warps(const DecodeArgs& a, int s, int2 cv, int64_t& wlo, int64_t& whi) {
  wlo = whi = 0;
  if (full_tiles(a, s) > 0) {
    if (cv.x >= 0 && cv.y >= cv.x && cv.y < static_cast<int64_t>(a.n_ctas) * a.warps) {
      wlo = cv.x;
      whi = static_cast<int64_t>(cv.y) + 1;
    }
  }
}

// Q-head gg's partial records w = wlo + first, wlo + first + kStride, ... below whi,
// merged online kBatch at a time into (M, l, acc): all of a batch's loads (each
// record's range check, max and sum, and the lane's 4 channels, 4l..4l+3) are in
// flight together; the running max then moves to the batch's and the sums are
// rescaled. Every lane reads the same maxima, so M, l and the rescale are
// warp-uniform. A record without data (an empty split range, or an index past whi,
// which reads the unit's last record again) gets weight 0 and is selected away,
// never multiplied.
template <int kBatch, int kStride>
__device__ __forceinline__ void merge_records(const DecodeArgs& a, const int64_t* rg, int64_t u, int gg, int64_t wlo,
                                              int64_t whi, int first, float& M, float& l, float (&acc)[4]) {
  const int lane = threadIdx.x & 31;
  for (int64_t w0 = wlo + first; w0 < whi; w0 += kBatch * kStride) {
    float4 v[kBatch];
    float2 ml[kBatch];
    bool ok[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t wj = w0 + j * kStride;
      const int64_t wr = min(wj, whi - 1);
      const longlong2 r = *reinterpret_cast<const longlong2*>(rg + 2 * wr);
      const float* pp = a.part + (wr + u) * kRecFloats + gg * kPartStride;
      ml[j] = *reinterpret_cast<const float2*>(pp + 128);
      v[j] = *reinterpret_cast<const float4*>(pp + 4 * lane);
      ok[j] = wj < whi && r.x < r.y;
    }
    float mb = M;
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (ok[j]) mb = fmaxf(mb, ml[j].x);
    if (mb > M) {
      const float sc = exp2f(M - mb);   // 0 while M is -inf (nothing summed yet)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] *= sc;
      l *= sc;
      M = mb;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const bool use = ok[j] && ml[j].x != -INFINITY;
      const float f = use ? exp2f(ml[j].x - M) : 0.f;
      acc[0] = fmaf(use ? v[j].x : 0.f, f, acc[0]);
      acc[1] = fmaf(use ? v[j].y : 0.f, f, acc[1]);
      acc[2] = fmaf(use ? v[j].z : 0.f, f, acc[2]);
      acc[3] = fmaf(use ? v[j].w : 0.f, f, acc[3]);
      l = fmaf(use ? ml[j].y : 0.f, f, l);
    }
  }
}

// Partial records' state of the warps that merged a share of a unit's records for
// q-head g: [share - 1][g] = acc[128], max, sum (kPartStride floats).
template <int kParts>
struct RecShares {
  float v[kParts > 1 ? kParts - 1 : 1][8][kPartStride];
};

// Q-head gg of unit (kv-head h, sequence s), one warp: the records' state (M, l, acc:
// lane l owns channels 4l..4l+3, rotated domain) is combined with the other shares'
// (`shares` of them in rs) and with the workspace warps' outputs (sm), un-rotated by
// a 128-point FWHT, normalised and stored as fp16.
template <int kParts>
__device__ __forceinline__ void merge_finish(const DecodeArgs& a, uint16_t* __restrict__ out, int h, int s, int gg,
                                             int n_ws, const WsPart& sm, const RecShares<kParts>* rs, float M,
                                             float l, float (&acc)[4]) {
  const int lane = threadIdx.x & 31;
  const int64_t qrow = (static_cast<int64_t>(s) * a.hkv * a.group + static_cast<int64_t>(h) * a.group + gg) * kD;
  // the other shares of the records, then the workspace warps, against the common max
  const int n_wsw = (n_ws + 15) >> 4;
  float Mt = M;
#pragma unroll
  for (int p = 0; p < kParts - 1; ++p) Mt = fmaxf(Mt, rs->v[p][gg][128]);
  for (int w = 0; w < n_wsw; ++w) Mt = fmaxf(Mt, sm.m[w][gg]);
  {
    const float sc = M == -INFINITY ? 0.f : exp2f(M - Mt);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] *= sc;
    l *= sc;
  }
#pragma unroll
  for (int p = 0; p < kParts - 1; ++p) {
    const float mp = rs->v[p][gg][128];
    const float f = mp == -INFINITY ? 0.f : exp2f(mp - Mt);
    const float4 v = *reinterpret_cast<const float4*>(&rs->v[p][gg][4 * lane]);
    acc[0] = fmaf(f != 0.f ? v.x : 0.f, f, acc[0]);
    acc[1] = fmaf(f != 0.f ? v.y : 0.f, f, acc[1]);
    acc[2] = fmaf(f != 0.f ? v.z : 0.f, f, acc[2]);
    acc[3] = fmaf(f != 0.f ? v.w : 0.f, f, acc[3]);
    l = fmaf(f != 0.f ? rs->v[p][gg][129] : 0.f, f, l);
  }
  float wacc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int w = 0; w < n_wsw; ++w) {
    const float f = exp2f(sm.m[w][gg] - Mt);
    const float4 v = *reinterpret_cast<const float4*>(&sm.o[w][gg][4 * lane]);
    wacc[0] = fmaf(v.x, f, wacc[0]);
    wacc[1] = fmaf(v.y, f, wacc[1]);
    wacc[2] = fmaf(v.z, f, wacc[2]);
    wacc[3] = fmaf(v.w, f, wacc[3]);
    l = fmaf(sm.l[w][gg], f, l);
  }
  // un-rotate: FWHT over the 128 channels (4 per lane), then scale by 1/sqrt(128)
  {
    const float a0 = acc[0] + acc[1], a1 = acc[0] - acc[1], a2 = acc[2] + acc[3], a3 = acc[2] - acc[3];
    acc[0] = a0 + a2;
    acc[1] = a1 + a3;
    acc[2] = a0 - a2;
    acc[3] = a1 - a3;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float other = __shfl_xor_sync(0xffffffffu, acc[k], o);
        acc[k] = upper ? (other - acc[k]) : (acc[k] + other);
      }
    }
  }
  const float inv_l = (l > 0.f) ? 1.0f / l : 0.f;
  uint16_t res[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) res[k] = f2h_bits(fmaf(acc[k], kInvSqrt128, wacc[k]) * inv_l);
  *reinterpret_cast<uint2*>(out + qrow + 4 * lane) =
      make_uint2(res[0] | (static_cast<uint32_t>(res[1]) << 16), res[2] | (static_cast<uint32_t>(res[3]) << 16));
}

// The split phase's outputs (marks, ranges, records) are ready when merge_body starts.
struct SplitDone {
  static constexpr bool kReady = true;
  __device__ void operator()() const {}
};

// Unit (kv-head h, sequence s) with the block's 8 kParts warps: warps 0-7 attend the
// workspace tokens (merge_ws_part); warp w takes share w / 8 of the partial records
// for q-head w % 8 (every kParts-th record); after one block barrier the warps of
// share 0 combine the shares with the workspace part and finish their q-heads. sm and
// rs are the block's shared memory (rs unused when kParts is 1). The workspace part
// reads only the call's inputs; unless Wait::kReady, wait() runs after it, before
// anything the split phase wrote is read.
template <int kBatch = 8, int kParts = 1, class Wait = SplitDone>
__device__ __forceinline__ void merge_body(const DecodeArgs& a, const uint16_t* __restrict__ ws,
                                           uint16_t* __restrict__ out, int h, int s, WsPart& sm,
                                           RecShares<kParts>* rs, const int64_t* rg, const Wait& wait = Wait()) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gg = warp & 7, share = warp >> 3;
  const int64_t u = static_cast<int64_t>(s) * a.hkv + h;
  int2 cv = make_int2(-1, -1);
  if (Wait::kReady) cv = *reinterpret_cast<const int2*>(a.cover + 2 * u);   // in flight with the length
  const int n_ws = ws_tokens(a, ws, s, threadIdx.x == 0);
  if (warp < 8) merge_ws_part(a, ws, h, s, n_ws, warp, sm);
  if (!Wait::kReady) {
    wait();
    cv = *reinterpret_cast<const int2*>(a.cover + 2 * u);
  }
  float M = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (gg < a.group) {
    int64_t wlo, whi;
    covering_warps(a, s, cv, wlo, whi);
    merge_records<kBatch, kParts>(a, rg, u, gg, wlo, whi, share, M, l, acc);
    if (kParts > 1 && share > 0) {
      float* dst = rs->v[share - 1][gg];
      *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      if (lane == 0) *reinterpret_cast<float2*>(dst + 128) = make_float2(M, l);
    }
  }
  __syncthreads();
  if (share == 0 && gg < a.group) merge_finish<kParts>(a, out, h, s, gg, n_ws, sm, rs, M, l, acc);
}

size_t prefix_bytes(int n_seqs) { return ((static_cast<size_t>(n_seqs) + 1) * sizeof(int64_t) + 255) & ~size_t(255); }
constexpr size_t kRangeBytes = static_cast<size_t>(kMaxCtas) * kMaxWarps * 2 * sizeof(int64_t);
// The units' first and last split warps, after the records of n_ctas CTAs.
size_t cover_bytes(int n_seqs, int hkv) { return (static_cast<size_t>(n_seqs) * hkv * 2 * sizeof(int32_t) + 255) & ~size_t(255); }
int32_t* cover_ptr(float* part, int n_seqs, int hkv, int n_ctas) {
  const size_t records = static_cast<size_t>(n_ctas) * kMaxWarps + static_cast<size_t>(n_seqs) * hkv;
  return reinterpret_cast<int32_t*>(part + records * kRecFloats);
}

}  // namespace
}  // namespace kvarn
