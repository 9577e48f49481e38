// Split phase of paged decode attention on the 5th-generation tensor core
// (tcgen05), for 4-bit keys and 2-bit values (KVarN README, "How KVarN works":
// the scales are re-applied on read; the orthonormal rotation keeps attention
// scores). It writes the same partial records as the warp-level split kernel,
// so the same merge kernel finishes the job.
//
// One persistent CTA per SM: kTcTeams teams of 4 warps and one issuing warp.
// A team owns a contiguous range of the flattened (sequence, kv-head, tile)
// space (stream-K over teams) and takes one tile at a time; its 128 threads are
// the 128 TMEM lanes of its columns:
//   keys:   thread t turns token t's 4-bit codes into fp16 (code / 8) and stores
//           them in TMEM lane t (A of QK^T, channels in natural order);
//           thread (head hh, channels 8jj..8jj+7) writes q' = q_r r^K s^K as an
//           fp16 hi and lo row (B, 16 rows x 128 channels, shared memory) and
//           sums beta = sum_i q_r,i r^K_i z^K_i over its 16 threads;
//   QK^T:   S[t][n] = A_K[t] . B_q[n] (M = 128 tokens, N = 16, fp32 in TMEM);
//           score_t,h = c^K_t ((S[t][h] + S[t][8 + h]) * 8 * 2^-e_h + beta_h), log2
//           domain (q' carried as q' 2^e_h);
//   values: thread c stores channel c's 2-bit codes as fp16 (code / 2) in TMEM
//           lane c (A of PV, tokens in natural order);
//   PV:     B_p rows = p' = p c^V s^V 2^e (hi, lo), O[c][n] = A_V[c] . B_p[n];
//           acc_c,h += r^V_c ((O[c][h] + O[c][8 + h]) * 2 * 2^-e + gamma_h),
//           gamma_h = sum_t p_t,h c^V_t z^V_t.
// The running max is lazy: a tile rescales only when one of its scores exceeds
// the running max by more than kTcTau (always on a unit's first tile), so most
// tiles need no reduction over tokens, and p stays <= 2^kTcTau. The running sum is
// kept per token slot and reduced when the team leaves a (sequence, kv-head).
// The tensor core drops subnormal fp16 operands (measured: q' carried as is, its
// lo parts subnormal, moved outputs by up to 4.5e-3), so q' (per head) and p' (per
// tile) are scaled by powers of two that bring their largest element near 2^13
// and the scale is taken out again in fp32.
// The issuing warp's lane 0 issues every team's UMMAs (a thread issuing UMMAs
// stalls while the tensor core is busy, so no team thread does) in the order the
// teams become ready, polling their mbarriers.
#pragma once
#include <stdint.h>

#include "decode_tile.cuh"
#include "kvarn_tc.cuh"

namespace kvarn {
namespace {

constexpr int kTcTeams = 3;                       // 4-warp teams per CTA
constexpr int kTcStages = 2;                      // record stages per team
constexpr int kTcThreads = kTcTeams * 128 + 32;   // + the issuing warp
constexpr uint32_t kTcTeamCols = 160;             // TMEM columns per team
constexpr uint32_t kTcAK = 0, kTcAV = 64, kTcS = 128, kTcO = 144;
constexpr uint32_t kTcBHalf = 2048;               // K-half stride of the 16-row B operands
constexpr float kTcTau = 4.0f;                    // lazy running max threshold (log2 units)
// per-team shared memory: B_q, B_p (1024-aligned), pz [8][128] f32, small f32 slots
// (beta[8], gamma[8], tile max[8], score factors[8], per-warp max of c s[4]),
// mbarriers (records[2], qk ready / done, pv ready / done), then the record stages
constexpr int kTcOffBq = 0, kTcOffBp = 4096, kTcOffPz = 8192, kTcOffX = 12288, kTcOffBar = 12544;
constexpr int kTcOffRec = 12608;
constexpr int kTcBarRec = 0, kTcBarQkReady = 2, kTcBarQkDone = 3, kTcBarPvReady = 4, kTcBarPvDone = 5;

template <bool kLean>
struct TcCfg {
  using L = RecordLayout<4, 2, kLean>;
  static constexpr int kTeamBytes = (kTcOffRec + kTcStages * L::kBytes + 1023) / 1024 * 1024;
  static constexpr int kOffFin = kTcTeams * kTeamBytes;     // the issuer's final mbarrier
  static constexpr int kOffSlot = kOffFin + 8;              // TMEM base address
  static constexpr int kSmem = kOffSlot + 8;
  static_assert(kSmem <= 232448, "decode tc shared memory");
};
static_assert(kTcTeams * kTcTeamCols <= 512, "TMEM columns");
static_assert(kTcOffRec % 16 == 0, "record stage alignment");

// Byte offset of element (row r, K index k) of a 16-row fp16 B operand in the
// 128-byte swizzled K-major layout (8-row groups 1024 B apart, K halves 2048 B).
__device__ __forceinline__ uint32_t tc_swo(int r, int k) {
  return static_cast<uint32_t>((k >> 6) * kTcBHalf + (r >> 3) * 1024 + (r & 7) * 128 +
                               ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// Thread t of the warp: 16 consecutive fp32 columns of TMEM lane (base lane + t).
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]));
}
// Thread t of the warp: 32 consecutive columns of TMEM lane (base lane + t) from r.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T (kind::f16): A's row m in TMEM lane m, its K
// elements two per 32-bit column.
__device__ __forceinline__ void tc_umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool tc_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool tc_bar_or(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " barrier.red.or.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}
// Operand writes of this thread (shared memory, TMEM) visible to the tensor core.
__device__ __forceinline__ void tc_operands_written() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  fence_proxy_async_smem();
  tc_fence_before();
}
__device__ __forceinline__ float tc_sum16(float x) {   // over the 16 lanes of a half warp
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float tc_max16(float x) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
// Power of two 2^k with k = top - floor(log2 m) (m >= 0; k clamped so that 2^k and
// 2^-k are normal floats), and 2^-k.
__device__ __forceinline__ float2 tc_pow2_scale(float m, int top) {
  const int ef = (__float_as_int(m) >> 23) & 0xff;       // biased exponent of m (0 for 0)
  const int se = min(max(127 + top + 127 - ef, 2), 252);  // biased exponent of 2^k
  return make_float2(__int_as_float(se << 23), __int_as_float((254 - se) << 23));
}

// q_r2 of head hh, channels 8jj..8jj+7: FWHT(q) * log2(e) / 128 (channel bits 0-2
// inside the thread, bits 3-6 across the 16 threads of the head).
__device__ __forceinline__ void tc_load_q(const DecodeArgs& a, int s, int h, int hh, int jj, float (&qr)[8]) {
  if (hh < a.group) {
    const uint16_t* row =
        a.q + (static_cast<int64_t>(s) * a.hkv * a.group + static_cast<int64_t>(h) * a.group + hh) * kD + 8 * jj;
    const uint4 w = *reinterpret_cast<const uint4*>(row);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = h2pair(reinterpret_cast<const uint16_t*>(&ws[e]));
      qr[2 * e] = f.x;
      qr[2 * e + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) qr[i] = 0.f;
  }
#pragma unroll
  for (int bit = 1; bit < 8; bit <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & bit) == 0) {
        const float u = qr[i], v = qr[i | bit];
        qr[i] = u + v;
        qr[i | bit] = u - v;
      }
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const bool upper = (jj & o) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, qr[i], o);
      qr[i] = upper ? (other - qr[i]) : (qr[i] + other);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) qr[i] *= kLog2e / 128.0f;
}

// Token t's 4-bit key codes -> fp16 (code / 8) in 64 TMEM columns of its lane:
// column 16m + 8nib + 4half + c holds channels 16(2m + nib) + 2c + 8half + {0, 1}
// (the record's token row: 16-byte part c, word m, nibble nib, bytes 2half, 2half + 1).
template <bool kLean>
__device__ __forceinline__ void tc_keys(const uint8_t* rec, int t, uint32_t taddr) {
  using L = RecordLayout<4, 2, kLean>;
  const uint4* row = reinterpret_cast<const uint4*>(rec + L::kKCodeOff + t * 64);
  uint4 part[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) part[c] = row[c];
#pragma unroll
  for (int mh = 0; mh < 2; ++mh) {
    uint32_t r[32];
#pragma unroll
    for (int mm = 0; mm < 2; ++mm)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int m = 2 * mh + mm;
        const uint32_t w = m == 0 ? part[c].x : m == 1 ? part[c].y : m == 2 ? part[c].z : part[c].w;
        cvt4(w & 0x0F0F0F0Fu, r[16 * mm + c], r[16 * mm + 4 + c]);
        cvt4((w >> 4) & 0x0F0F0F0Fu, r[16 * mm + 8 + c], r[16 * mm + 12 + c]);
      }
    tc_st32(taddr + 32 * mh, r);
  }
}

// Channel t's 2-bit value codes -> fp16 (code / 2) in 64 TMEM columns of its lane:
// column 8(4u + b) + 4half + c holds tokens 16(4u + b) + 2c + 8half + {0, 1} (the
// record's panel t / 16, cell (t % 8, c), half (t / 8) % 2, word u, byte b).
template <bool kLean>
__device__ __forceinline__ void tc_values(const uint8_t* rec, int t, uint32_t taddr) {
  using L = RecordLayout<4, 2, kLean>;
  const uint8_t* base = rec + L::kVCodeOff + (t >> 4) * 512 + (t & 7) * 64 + ((t >> 3) & 1) * 8;
  uint2 w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint2*>(base + c * 16);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t x = u ? w[c].y : w[c].x;
      uint32_t v0[4], v1[4];
      cvt2(x & 0x33333333u, v0);
      cvt2((x >> 2) & 0x33333333u, v1);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        r[8 * b + c] = v0[b];
        r[8 * b + 4 + c] = v1[b];
      }
    }
    tc_st32(taddr + 32 * u, r);
  }
}

// Thread (hh, jj): q' 2^e hi / lo of head hh, channels 8jj..8jj+7 into B_q rows hh
// and 8 + hh (2^e brings the head's largest |q'| into [2^13, 2^14)); returns beta of
// head hh (summed over the head's 16 threads) and 2^-e.
template <bool kLean>
__device__ __forceinline__ float2 tc_qprime(const uint8_t* rec, const float (&qr)[8], int hh, int jj, uint8_t* bq) {
  using L = RecordLayout<4, 2, kLean>;
  const uint16_t* km = reinterpret_cast<const uint16_t*>(rec + L::kKMetaOff);
  const uint4 sv = *reinterpret_cast<const uint4*>(km + L::kKs + 8 * jj);
  const uint4 zv = *reinterpret_cast<const uint4*>(km + L::kKz + 8 * jj);
  uint4 rv = make_uint4(kH_One, kH_One, kH_One, kH_One);
  if (!kLean) rv = *reinterpret_cast<const uint4*>(km + L::kKr + 8 * jj);
  const uint32_t s4[4] = {sv.x, sv.y, sv.z, sv.w}, z4[4] = {zv.x, zv.y, zv.z, zv.w};
  const uint32_t r4[4] = {rv.x, rv.y, rv.z, rv.w};
  float2 x[4];
  float2 beta2 = make_float2(0.f, 0.f);
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 qa = make_float2(qr[2 * e], qr[2 * e + 1]);
    x[e] = __fmul2_rn(qa, mul_h2(r4[e], s4[e]));
    beta2 = __ffma2_rn(qa, mul_h2(r4[e], z4[e]), beta2);
    m = fmax3f(m, fabsf(x[e].x), fabsf(x[e].y));
  }
  const float2 sc = tc_pow2_scale(tc_max16(m), 13);
  const float2 sc2 = make_float2(sc.x, sc.x);
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split2p(__fmul2_rn(x[e], sc2), hi[e], lo[e]);
  *reinterpret_cast<uint4*>(bq + tc_swo(hh, 8 * jj)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(bq + tc_swo(8 + hh, 8 * jj)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  return make_float2(tc_sum16(beta2.x + beta2.y), sc.y);
}

// Partial record of the unit the team leaves: acc (thread = channel), running max
// and the token slots' sums reduced over the team.
__device__ __forceinline__ void tc_flush(const DecodeArgs& a, int64_t rec_idx, int t, int hh, int jj, int bar_id,
                                         float* pz, const float (&acc)[8], const float (&lsum)[8],
                                         const float (&mrun)[8]) {
#pragma unroll
  for (int h = 0; h < 8; ++h) pz[h * 128 + t] = lsum[h];
  named_bar(bar_id, 128);
  const float4 x0 = *reinterpret_cast<const float4*>(pz + hh * 128 + 8 * jj);
  const float4 x1 = *reinterpret_cast<const float4*>(pz + hh * 128 + 8 * jj + 4);
  const float l = tc_sum16(((x0.x + x0.y) + (x0.z + x0.w)) + ((x1.x + x1.y) + (x1.z + x1.w)));
  float* out = a.part + rec_idx * kRecFloats;
#pragma unroll
  for (int h = 0; h < 8; ++h)
    if (h < a.group) out[h * kPartStride + t] = acc[h];
  if (jj == 0 && hh < a.group) *reinterpret_cast<float2*>(out + hh * kPartStride + 128) = make_float2(mrun[hh], l);
}

// The 128 threads of team `team` over global tiles [gb, ge).
template <bool kLean>
__device__ __forceinline__ void tc_team(const DecodeArgs& a, uint8_t* tsm, uint32_t tm, int team, int64_t gb,
                                        int64_t ge, int64_t wg) {
  using L = RecordLayout<4, 2, kLean>;
  const int t = static_cast<int>(threadIdx.x) - team * 128;
  const int wq = t >> 5;                    // warp of the team = TMEM lane quarter
  const int hh = t >> 4, jj = t & 15;       // (head, channel group) role
  const int bar_id = 1 + team;
  uint8_t* bq = tsm + kTcOffBq;
  uint8_t* bp = tsm + kTcOffBp;
  float* pz = reinterpret_cast<float*>(tsm + kTcOffPz);
  float* xs = reinterpret_cast<float*>(tsm + kTcOffX);      // beta, gamma, tile max, factors, c s max
  uint64_t* bars = reinterpret_cast<uint64_t*>(tsm + kTcOffBar);
  uint8_t* stages = tsm + kTcOffRec;
  const uint32_t trow = tm + (static_cast<uint32_t>(32 * wq) << 16);
  if (t == 0) {
    a.ranges[2 * wg] = gb;
    a.ranges[2 * wg + 1] = ge;
  }
  if (gb >= ge) return;

  Cursor lc = locate(a, gb);
  Cursor cc = lc;
  if (t == 0)
    for (int k = 0; k < kTcStages && gb + k < ge; ++k) {
      if (k > 0) advance(a, lc);
      issue_tile<L::kBytes>(a, lc, stages + k * L::kBytes, &bars[kTcBarRec + k]);
    }

  float qr[8], acc[8], lsum[8], mrun[8];
  int64_t unit = -1;
  uint32_t rph = 0, qph = 0, pph = 0;
  bool ok = true;
  for (int64_t k = 0; gb + k < ge; ++k) {
    const int stg = static_cast<int>(k % kTcStages);
    const uint8_t* rec = stages + stg * L::kBytes;
    const uint16_t* km = reinterpret_cast<const uint16_t*>(rec + L::kKMetaOff);
    const uint16_t* vm = reinterpret_cast<const uint16_t*>(rec + L::kVMetaOff);
    const int64_t u = static_cast<int64_t>(cc.s) * a.hkv + cc.h;
    if (u != unit) {
      if (unit >= 0) tc_flush(a, wg + unit, t, hh, jj, bar_id, pz, acc, lsum, mrun);
      unit = u;
      if (t == 0 && cc.ti == 0) a.cover[2 * u] = static_cast<int32_t>(wg);   // the unit's first split team
      tc_load_q(a, cc.s, cc.h, hh, jj, qr);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        acc[h] = 0.f;
        lsum[h] = 0.f;
        mrun[h] = -INFINITY;
      }
    }
    if (t == 0 && cc.ti == cc.nf - 1) a.cover[2 * u + 1] = static_cast<int32_t>(wg);   // and its last
    const int64_t blk = a.block_tables[static_cast<int64_t>(cc.s) * a.max_blocks + cc.ti];
    const bool valid = blk >= 0 && blk < a.num_blocks;
    ok = mbar_wait(&bars[kTcBarRec + stg], (rph >> stg) & 1u, a.flags) && ok;
    rph ^= 1u << stg;
    const bool go = __all_sync(0xffffffffu, ok) && valid;   // warp-uniform: TMEM stores are warp-wide

    // keys -> A_K, q' -> B_q, beta; then the tensor core may start QK^T
    if (go) {
      tc_keys<kLean>(rec, t, trow + kTcAK);
      const float2 bf = tc_qprime<kLean>(rec, qr, hh, jj, bq);
      if (jj == 0) {
        xs[hh] = bf.x;
        xs[24 + hh] = 8.f * bf.y;     // codes were converted to c / 8
      }
    }
    tc_operands_written();
    tc_arrive(&bars[kTcBarQkReady]);
    // values -> A_V (under QK^T) and this thread's token and channel scales
    float ck = 0.f, cs = 0.f, cz = 0.f, rv = 0.f;
    if (go) {
      tc_values<kLean>(rec, t, trow + kTcAV);
      ck = h2f_bits(km[L::kKc + t]);
      const float cv = kLean ? 1.f : h2f_bits(vm[L::kVc + t]);
      cs = cv * h2f_bits(vm[L::kVs + t]);
      cz = cv * h2f_bits(vm[L::kVz + t]);
      rv = h2f_bits(vm[L::kVr + t]);
    }
    {
      float cm = cs;                          // the tile's largest c s, per warp
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      if ((t & 31) == 0) xs[32 + wq] = cm;
    }
    tc_operands_written();
    ok = named_bar_and(bar_id, 128, ok);      // beta visible; every wait so far succeeded
    if (!ok) break;
    if (t == 0 && gb + k + kTcStages < ge) {  // the record is read: refill its stage kTcStages ahead
      advance(a, lc);
      issue_tile<L::kBytes>(a, lc, stages + stg * L::kBytes, &bars[kTcBarRec + stg]);
    }

    // scores of token t
    ok = mbar_wait(&bars[kTcBarQkDone], qph, a.flags);
    qph ^= 1u;
    tc_fence_after();
    float sv[16];
    tc_ld16(trow + kTcS, sv);
    float sc[8];
    bool need = false;
    float2 psc = make_float2(1.f, 1.f);      // p' scale 2^e and 2^-e
    if (valid) {
      const float4 b0 = *reinterpret_cast<const float4*>(xs), b1 = *reinterpret_cast<const float4*>(xs + 4);
      const float4 f0 = *reinterpret_cast<const float4*>(xs + 24), f1 = *reinterpret_cast<const float4*>(xs + 28);
      const float4 c4 = *reinterpret_cast<const float4*>(xs + 32);
      const float beta[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      const float fq[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        sc[h] = ck * fmaf(sv[h] + sv[8 + h], fq[h], beta[h]);
        need |= sc[h] > mrun[h] + kTcTau;
      }
      // p' = p c s 2^e <= 2^kTcTau max(c s) 2^e < 2^14
      psc = tc_pow2_scale(fmaxf(fmaxf(c4.x, c4.y), fmaxf(c4.z, c4.w)), 13 - static_cast<int>(kTcTau));
    }
    if (tc_bar_or(bar_id, 128, need || !ok)) {
      // a score above the lazy threshold (or a failed wait): exact tile max, rescale
      ok = named_bar_and(bar_id, 128, ok);
      if (!ok) break;
#pragma unroll
      for (int h = 0; h < 8; ++h) pz[h * 128 + t] = sc[h];
      named_bar(bar_id, 128);
      const float4 x0 = *reinterpret_cast<const float4*>(pz + hh * 128 + 8 * jj);
      const float4 x1 = *reinterpret_cast<const float4*>(pz + hh * 128 + 8 * jj + 4);
      const float m = tc_max16(fmaxf(fmaxf(fmax3f(x0.x, x0.y, x0.z), fmax3f(x0.w, x1.x, x1.y)), fmaxf(x1.z, x1.w)));
      if (jj == 0) xs[16 + hh] = m;
      named_bar(bar_id, 128);
      const float4 m0 = *reinterpret_cast<const float4*>(xs + 16), m1 = *reinterpret_cast<const float4*>(xs + 20);
      const float tmax[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float mn = fmaxf(mrun[h], tmax[h]);
        const float corr = ex2(mrun[h] - mn);
        acc[h] *= corr;
        lsum[h] *= corr;
        mrun[h] = mn;
      }
    }

    // p, its running sums, p' -> B_p (hi, lo), p c z -> pz
    if (valid) {
      const float csq = cs * psc.x;
      float pp[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float p = ex2(sc[h] - mrun[h]);
        lsum[h] += p;
        pp[h] = p * csq;
        pz[h * 128 + t] = p * cz;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t hi, lo;
        split2p(make_float2(pp[2 * e], pp[2 * e + 1]), hi, lo);
        *reinterpret_cast<uint16_t*>(bp + tc_swo(2 * e, t)) = static_cast<uint16_t>(hi);
        *reinterpret_cast<uint16_t*>(bp + tc_swo(2 * e + 1, t)) = static_cast<uint16_t>(hi >> 16);
        *reinterpret_cast<uint16_t*>(bp + tc_swo(8 + 2 * e, t)) = static_cast<uint16_t>(lo);
        *reinterpret_cast<uint16_t*>(bp + tc_swo(9 + 2 * e, t)) = static_cast<uint16_t>(lo >> 16);
      }
    }
    tc_operands_written();
    tc_arrive(&bars[kTcBarPvReady]);
    named_bar(bar_id, 128);                   // pz complete
    {
      const float4 x0 = *reinterpret_cast<const float4*>(pz + hh * 128 + 8 * jj);
      const float4 x1 = *reinterpret_cast<const float4*>(pz + hh * 128 + 8 * jj + 4);
      const float gsum = tc_sum16(((x0.x + x0.y) + (x0.z + x0.w)) + ((x1.x + x1.y) + (x1.z + x1.w)));
      if (jj == 0) xs[8 + hh] = gsum;
    }
    named_bar(bar_id, 128);                   // gamma visible

    // PV into the accumulators (thread = channel t)
    ok = mbar_wait(&bars[kTcBarPvDone], pph, a.flags) && ok;
    pph ^= 1u;
    tc_fence_after();
    float ov[16];
    tc_ld16(trow + kTcO, ov);
    if (valid) {
      const float4 g0 = *reinterpret_cast<const float4*>(xs + 8), g1 = *reinterpret_cast<const float4*>(xs + 12);
      const float gamma[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float vf = 2.f * psc.y;           // codes were converted to c / 2
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[h] = fmaf(rv, fmaf(ov[h] + ov[8 + h], vf, gamma[h]), acc[h]);
    }
    advance(a, cc);
  }
  ok = named_bar_and(bar_id, 128, ok);
  if (unit >= 0 && ok) tc_flush(a, wg + unit, t, hh, jj, bar_id, pz, acc, lsum, mrun);
}

// Lane 0 of the issuing warp: every team's UMMAs, in the order the teams get ready.
template <bool kLean>
__device__ __forceinline__ void tc_issue(const DecodeArgs& a, uint8_t* smem, uint32_t tmem, int64_t total) {
  using C = TcCfg<kLean>;
  constexpr uint32_t kId = idesc_f16_f32(128, 16);
  int64_t rem[kTcTeams];
  uint32_t ph_qk = 0, ph_pv = 0, next_pv = 0;   // per-team bits
  for (int j = 0; j < kTcTeams; ++j) {
    int64_t gb, ge;
    warp_range<kTcTeams>(total, a.n_ctas, static_cast<int64_t>(blockIdx.x) * kTcTeams + j, gb, ge);
    rem[j] = ge > gb ? 2 * (ge - gb) : 0;
  }
  unsigned long long t_last = global_ns();
  for (unsigned n = 0;; ++n) {
    bool any = false, prog = false;
#pragma unroll
    for (int j = 0; j < kTcTeams; ++j) {
      if (rem[j] == 0) continue;
      any = true;
      uint8_t* tsm = smem + j * C::kTeamBytes;
      uint64_t* bars = reinterpret_cast<uint64_t*>(tsm + kTcOffBar);
      const bool pv = (next_pv >> j) & 1u;
      if (!tc_test(&bars[pv ? kTcBarPvReady : kTcBarQkReady], ((pv ? ph_pv : ph_qk) >> j) & 1u)) continue;
      tc_fence_after();
      const uint32_t tt = tmem + j * kTcTeamCols;
      const uint32_t b = smem_u32(tsm + (pv ? kTcOffBp : kTcOffBq));
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t desc = smem_desc_sw128(b + (s >> 2) * kTcBHalf + (s & 3) * 32);
        tc_umma_ts(tt + (pv ? kTcO : kTcS), tt + (pv ? kTcAV : kTcAK) + 8 * s, desc, kId, s > 0);
      }
      umma_commit(&bars[pv ? kTcBarPvDone : kTcBarQkDone]);
      if (pv) ph_pv ^= 1u << j; else ph_qk ^= 1u << j;
      next_pv ^= 1u << j;
      --rem[j];
      prog = true;
    }
    if (!any) break;
    if (!prog) __nanosleep(32);
    if (prog) {
      t_last = global_ns();
    } else if ((n & 63) == 0 && global_ns() - t_last > kWaitNs) {
      raise_flag(a.flags, KVARN_FLAG_WAIT_TIMEOUT);
      break;
    }
  }
  // every issued product complete before TMEM is released
  uint64_t* fin = reinterpret_cast<uint64_t*>(smem + C::kOffFin);
  umma_commit(fin);
  mbar_wait(fin, 0, a.flags);
}

// The kernel body (one CTA per SM, kTcThreads threads, TcCfg<kLean>::kSmem bytes of
// dynamic shared memory).
template <bool kLean>
__device__ __forceinline__ void decode_tc_body(const DecodeArgs& a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using C = TcCfg<kLean>;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::kOffSlot);
  const int warp = threadIdx.x >> 5;
  const int64_t total = a.prefix[a.n_seqs] * a.hkv;
  if (threadIdx.x == 0) {
    for (int j = 0; j < kTcTeams; ++j) {
      uint64_t* bars = reinterpret_cast<uint64_t*>(smem + j * C::kTeamBytes + kTcOffBar);
      mbar_init(&bars[kTcBarRec], 1);
      mbar_init(&bars[kTcBarRec + 1], 1);
      mbar_init(&bars[kTcBarQkReady], 128);
      mbar_init(&bars[kTcBarQkDone], 1);
      mbar_init(&bars[kTcBarPvReady], 128);
      mbar_init(&bars[kTcBarPvDone], 1);
    }
    mbar_init(reinterpret_cast<uint64_t*>(smem + C::kOffFin), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (warp < kTcTeams * 4) {
    const int team = warp >> 2;
    const int64_t wg = static_cast<int64_t>(blockIdx.x) * kTcTeams + team;
    int64_t gb, ge;
    warp_range<kTcTeams>(total, a.n_ctas, wg, gb, ge);
    tc_team<kLean>(a, smem + team * C::kTeamBytes, tmem + team * kTcTeamCols, team, gb, ge, wg);
  } else if (threadIdx.x == kTcTeams * 128) {
    tc_issue<kLean>(a, smem, tmem, total);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace
}  // namespace kvarn
