// KVarN paged decode attention over the packed cache (KVarN README, "How KVarN
// works": scales are re-applied on read; the orthonormal rotation keeps
// attention scores, so q is rotated by the same H and the output un-rotated).
//
// decode_split_kernel: grid (split, kv-head, sequence). Each CTA streams up to
// kTilesPerSplit packed tiles of one (sequence, kv-head) through 1-D bulk copies
// (one 14336-byte record per tile) and runs the GQA group (up to 8 q-heads) on
// m16n8k16 tensor-core MMAs with an online softmax in the log2 domain:
//   QK^T: A = q' = q_r * r^K * s^K per channel (fp16 hi part in rows 0-7, fp16 lo
//         part in rows 8-15, so the product carries ~22 bits of q'), B = 4-bit key
//         codes converted to fp16 in registers; score_j = c^K_j (D_hi + D_lo + beta),
//         beta = sum_i q_r,i r^K_i z^K_i.
//   PV:   A = p' = p_j c^V_j s^V_j (hi / lo rows), B = 2-bit value codes;
//         acc_i += r^V_i (D_hi + D_lo + gamma), gamma = sum_j p_j c^V_j z^V_j.
// Partial (max, sum, acc) per split go to scratch; decode_merge_kernel merges the
// splits with the fp16 workspace tokens of the partial last tile, un-rotates the
// accumulator by H^T and normalises.
#include "kvarn_common.cuh"
#include "kvarn_launch.h"

namespace kvarn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// fp32 pair -> (hi, lo) fp16 pairs with hi + lo ~ x to ~22 bits.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float2 h2pair(const uint16_t* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}

template <uint32_t kMask>
__device__ __forceinline__ uint32_t lop_magic(uint32_t w) {
  // (w & kMask) | 0x64006400: places the selected bits in the mantissa of two fp16
  // values 1024 + field.
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(w), "n"(kMask), "n"(0x64006400u));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// fp16x2 constants
constexpr uint32_t kH_One = 0x3C003C00u;       // 1.0
constexpr uint32_t kH_M1024 = 0xE400E400u;     // -1024
constexpr uint32_t kH_Sixteenth = 0x2C002C00u; // 1/16
constexpr uint32_t kH_M64 = 0xD400D400u;       // -64
constexpr uint32_t kH_Quarter = 0x34003400u;   // 1/4
constexpr uint32_t kH_M256 = 0xDC00DC00u;      // -256
constexpr uint32_t kH_M16 = 0xCC00CC00u;       // -16

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

struct DecodeArgs {
  const uint16_t* q;
  const uint8_t* cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* part;          // [n_seqs][hkv][n_split][8][132]
  unsigned* flags;
  int64_t num_blocks;
  int hkv;
  int group;            // q-heads per kv-head (1..8)
  int max_blocks;
  int n_split;
  int tiles_per_split;
};

constexpr int kPartStride = 132;  // floats per (split, q-head) partial: acc[128], max, sum, 2 pad (16-byte rows)

template <int kWarps, int kStages>
struct SplitSmem {
  static constexpr int kOffStage = 0;
  static constexpr int kOffQ = kWarps * kStages * kRec;          // fp32 [8][128]
  static constexpr int kOffBar = kOffQ + 8 * 128 * 4;            // [kWarps][kStages] mbarriers
  static constexpr int kBytes = kOffBar + kWarps * kStages * 8;
  static_assert(kWarps * 8 * kPartStride * 4 <= kWarps * kStages * kRec, "merge area fits in stages");
};

template <int kWarps, int kStages>
__global__ void __launch_bounds__(kWarps * 32)
    decode_split_kernel(DecodeArgs args) {
  using S = SplitSmem<kWarps, kStages>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int sp = blockIdx.x, h = blockIdx.y;
  const int64_t s = blockIdx.z;

  int L = args.seq_lens[s];
  if (L < 0) L = 0;
  int n_full = L / kB;
  if (n_full > args.max_blocks) n_full = args.max_blocks;
  const int t_begin = sp * args.tiles_per_split;
  const int t_end = min(t_begin + args.tiles_per_split, n_full);
  if (t_begin >= t_end) return;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  float* qs = reinterpret_cast<float*>(smem + S::kOffQ);
  const int32_t* btab = args.block_tables + s * args.max_blocks;

  if (tid < kWarps * kStages) mbar_init(&bars[tid], 1);
  fence_mbar_init();
  __syncthreads();

  // ---- issue the first kStages loads of this warp's tiles
  // warp `warp` takes tiles t_begin + warp + kWarps * k, k = 0, 1, ...
  uint32_t valid_mask = 0;  // bit k%kStages: stage holds a valid tile
  if (lane == 0) {
    for (int k = 0; k < kStages; ++k) {
      const int t = t_begin + warp + kWarps * k;
      if (t >= t_end) break;
      const int64_t blk = btab[t];
      if (blk < 0 || blk >= args.num_blocks) {
        raise_flag(args.flags, KVARN_FLAG_BAD_BLOCK);
        continue;
      }
      uint64_t* bar = &bars[warp * kStages + k];
      mbar_arrive_expect_tx(bar, kRec);
      bulk_g2s(smem + S::kOffStage + (warp * kStages + k) * kRec,
               args.cache + (blk * args.hkv + h) * static_cast<int64_t>(kRec), kRec, bar);
      valid_mask |= 1u << k;
    }
  }
  valid_mask = __shfl_sync(0xffffffffu, valid_mask, 0);

  // ---- q of the group, rotated: q_r2 = FWHT(q) * log2(e) / 128 (= H q * log2(e)/sqrt(128))
  for (int idx = tid; idx < 8 * 128; idx += kWarps * 32) {
    const int gg = idx >> 7, ch = idx & 127;
    float v = 0.f;
    if (gg < args.group)
      v = h2f_bits(args.q[(s * args.hkv * args.group + static_cast<int64_t>(h) * args.group + gg) * kD + ch]);
    qs[idx] = v;
  }
  __syncthreads();
  for (int st = 1; st < 128; st <<= 1) {
    for (int idx = tid; idx < 8 * 64; idx += kWarps * 32) {
      const int gg = idx >> 6, pr = idx & 63;
      const int lo = ((pr / st) * 2 * st) + (pr % st);
      const float u = qs[gg * 128 + lo], w = qs[gg * 128 + lo + st];
      qs[gg * 128 + lo] = u + w;
      qs[gg * 128 + lo + st] = u - w;
    }
    __syncthreads();
  }
  float qv[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int ch0 = 16 * ks + 2 * c;
    qv[ks][0] = qs[g * 128 + ch0] * (kLog2e / 128.0f);
    qv[ks][1] = qs[g * 128 + ch0 + 1] * (kLog2e / 128.0f);
    qv[ks][2] = qs[g * 128 + ch0 + 8] * (kLog2e / 128.0f);
    qv[ks][3] = qs[g * 128 + ch0 + 9] * (kLog2e / 128.0f);
  }

  float m_run = -INFINITY, l_run = 0.f;
  float acc[16][2];
#pragma unroll
  for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = 0.f;

  int k = 0;
  uint32_t phase_bits = 0;  // per stage: parity of the next phase to wait for
  for (int t = t_begin + warp; t < t_end; t += kWarps, ++k) {
    const int stg = k % kStages;
    if ((valid_mask >> stg) & 1u) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[warp * kStages + stg], (phase_bits >> stg) & 1u,
                                                        args.flags));
      phase_bits ^= 1u << stg;
      if (!ok) break;  // a copy never arrived: stop this warp (flag raised)
      {
        const uint8_t* rec = smem + S::kOffStage + (warp * kStages + stg) * kRec;
        const uint16_t* km = reinterpret_cast<const uint16_t*>(rec + kKMetaOff);
        const uint16_t* vm = reinterpret_cast<const uint16_t*>(rec + kVMetaOff);

        // -- q' fragments (hi/lo rows) and beta
        uint32_t A[8][4];
        float beta = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int ch0 = 16 * ks + 2 * c;
          const float2 r0 = h2pair(km + ch0), r1 = h2pair(km + ch0 + 8);
          const float2 s0 = h2pair(km + 256 + ch0), s1 = h2pair(km + 256 + ch0 + 8);
          const float2 z0 = h2pair(km + 384 + ch0), z1 = h2pair(km + 384 + ch0 + 8);
          split2(qv[ks][0] * (r0.x * s0.x), qv[ks][1] * (r0.y * s0.y), A[ks][0], A[ks][1]);
          split2(qv[ks][2] * (r1.x * s1.x), qv[ks][3] * (r1.y * s1.y), A[ks][2], A[ks][3]);
          beta = fmaf(qv[ks][0], r0.x * z0.x, beta);
          beta = fmaf(qv[ks][1], r0.y * z0.y, beta);
          beta = fmaf(qv[ks][2], r1.x * z1.x, beta);
          beta = fmaf(qv[ks][3], r1.y * z1.y, beta);
        }
        beta = quad_sum(beta);

        // -- scores for tokens 8nt + 2c + {0,1}
        float sc[16][2];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          const uint4 kw = *reinterpret_cast<const uint4*>(rec + kKCodeOff + (8 * nt + g) * 64 + c * 16);
          const uint32_t words[4] = {kw.x, kw.y, kw.z, kw.w};
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t w0 = words[m], w8 = words[m] >> 8;
            const uint32_t b00 = hfma2_u(lop_magic<0x000F000Fu>(w0), kH_One, kH_M1024);
            const uint32_t b01 = hfma2_u(lop_magic<0x00F000F0u>(w0), kH_Sixteenth, kH_M64);
            mma16816(d, A[2 * m], b00, b01);
            const uint32_t b10 = hfma2_u(lop_magic<0x000F000Fu>(w8), kH_One, kH_M1024);
            const uint32_t b11 = hfma2_u(lop_magic<0x00F000F0u>(w8), kH_Sixteenth, kH_M64);
            mma16816(d, A[2 * m + 1], b10, b11);
          }
          const float2 ck = h2pair(km + 128 + 8 * nt + 2 * c);
          sc[nt][0] = ck.x * ((d[0] + d[2]) + beta);
          sc[nt][1] = ck.y * ((d[1] + d[3]) + beta);
        }

        // -- online softmax (log2 domain), head g
        float tmax = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) tmax = fmaxf(tmax, fmaxf(sc[nt][0], sc[nt][1]));
        tmax = quad_max(tmax);
        const float m_new = fmaxf(m_run, tmax);
        const float corr = exp2f(m_run - m_new);
        m_run = m_new;
        float lsum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          sc[nt][0] = exp2f(sc[nt][0] - m_new);
          sc[nt][1] = exp2f(sc[nt][1] - m_new);
          lsum += sc[nt][0] + sc[nt][1];
        }
        l_run = fmaf(l_run, corr, lsum);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          acc[n][0] *= corr;
          acc[n][1] *= corr;
        }

        // -- p' fragments and gamma; tokens 16ks + 2c + {0,1} (nt = 2ks), +8 (nt = 2ks+1)
        float gamma = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int t0 = 16 * ks + 2 * c;
          const float2 c0 = h2pair(vm + 128 + t0), c1 = h2pair(vm + 128 + t0 + 8);
          const float2 s0 = h2pair(vm + 256 + t0), s1 = h2pair(vm + 256 + t0 + 8);
          const float2 z0 = h2pair(vm + 384 + t0), z1 = h2pair(vm + 384 + t0 + 8);
          const float p0 = sc[2 * ks][0], p1 = sc[2 * ks][1], p2 = sc[2 * ks + 1][0], p3 = sc[2 * ks + 1][1];
          split2(p0 * (c0.x * s0.x), p1 * (c0.y * s0.y), A[ks][0], A[ks][1]);
          split2(p2 * (c1.x * s1.x), p3 * (c1.y * s1.y), A[ks][2], A[ks][3]);
          gamma = fmaf(p0, c0.x * z0.x, gamma);
          gamma = fmaf(p1, c0.y * z0.y, gamma);
          gamma = fmaf(p2, c1.x * z1.x, gamma);
          gamma = fmaf(p3, c1.y * z1.y, gamma);
        }
        gamma = quad_sum(gamma);

        // -- PV over channel n-tiles 8*nt2 + {0..7}; one 16-byte cell serves nt2 = 2np, 2np+1
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          const uint4 vw = *reinterpret_cast<const uint4*>(rec + kVCodeOff + np * 512 + (g * 4 + c) * 16);
          const uint32_t words[2][2] = {{vw.x, vw.y}, {vw.z, vw.w}};
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
#pragma unroll
              for (int sg = 0; sg < 2; ++sg) {
                const uint32_t w = sg ? (words[which][u] >> 8) : words[which][u];
                // crumb q = 2*(ks&1) + type at shift sg; ks = 4u + 2sg + (q>>1)
                const uint32_t q0 = hfma2_u(lop_magic<0x00030003u>(w), kH_One, kH_M1024);
                const uint32_t q1 = hfma2_u(lop_magic<0x000C000Cu>(w), kH_Quarter, kH_M256);
                const uint32_t q2 = hfma2_u(lop_magic<0x00300030u>(w), kH_Sixteenth, kH_M64);
                const uint32_t q3 = hfma2_u(lop_magic<0x00C000C0u>(w), 0x24002400u /*1/64*/, kH_M16);
                mma16816(d, A[4 * u + 2 * sg + 0], q0, q1);
                mma16816(d, A[4 * u + 2 * sg + 1], q2, q3);
              }
            }
            const int nt2 = 2 * np + which;
            const float2 rv = h2pair(vm + 8 * nt2 + 2 * c);
            acc[nt2][0] = fmaf(rv.x, (d[0] + d[2]) + gamma, acc[nt2][0]);
            acc[nt2][1] = fmaf(rv.y, (d[1] + d[3]) + gamma, acc[nt2][1]);
          }
        }
      }
    }
    __syncwarp();
    // refill this stage with the warp's tile k + kStages
    const int tn = t + kWarps * kStages;
    if (tn < t_end) {
      bool issued = false;
      if (lane == 0) {
        const int64_t blk = btab[tn];
        if (blk < 0 || blk >= args.num_blocks) {
          raise_flag(args.flags, KVARN_FLAG_BAD_BLOCK);
        } else {
          uint64_t* bar = &bars[warp * kStages + stg];
          mbar_arrive_expect_tx(bar, kRec);
          bulk_g2s(smem + S::kOffStage + (warp * kStages + stg) * kRec,
                   args.cache + (blk * args.hkv + h) * static_cast<int64_t>(kRec), kRec, bar);
          issued = true;
        }
      }
      issued = __shfl_sync(0xffffffffu, issued, 0);
      if (issued) valid_mask |= 1u << stg; else valid_mask &= ~(1u << stg);
    }
  }

  // ---- merge the warps of this CTA through shared memory, write the split partial
  l_run = quad_sum(l_run);
  __syncthreads();  // every warp has consumed all of its stages
  float* mrg = reinterpret_cast<float*>(smem + S::kOffStage);
  {
    float* mw = mrg + (warp * 8 + g) * kPartStride;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      mw[8 * n + 2 * c] = acc[n][0];
      mw[8 * n + 2 * c + 1] = acc[n][1];
    }
    if (c == 0) {
      mw[128] = m_run;
      mw[129] = l_run;
    }
  }
  __syncthreads();
  float* out = args.part + ((s * args.hkv + h) * args.n_split + sp) * (8 * kPartStride);
  for (int idx = tid; idx < args.group * 128; idx += kWarps * 32) {
    const int gg = idx >> 7, ch = idx & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg[(w * 8 + gg) * kPartStride + 128]);
    float a = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = mrg[(w * 8 + gg) * kPartStride + 128];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      a = fmaf(mrg[(w * 8 + gg) * kPartStride + ch], f, a);
      l = fmaf(mrg[(w * 8 + gg) * kPartStride + 129], f, l);
    }
    out[gg * kPartStride + ch] = a;
    if (ch == 0) {
      out[gg * kPartStride + 128] = M;
      out[gg * kPartStride + 129] = l;
    }
  }
}

// One CTA per (kv-head, sequence), one warp per q-head of the group; lane l owns
// channels 4l..4l+3.
__global__ void __launch_bounds__(256) decode_merge_kernel(DecodeArgs args, const uint16_t* __restrict__ ws,
                                                           uint16_t* __restrict__ out) {
  __shared__ float sc[8][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int64_t s = blockIdx.y;
  const int gg = warp;
  int L = args.seq_lens[s];
  if (L < 0) L = 0;
  int n_full = L / kB;
  if (n_full > args.max_blocks) {
    n_full = args.max_blocks;
    if (threadIdx.x == 0 && h == 0) raise_flag(args.flags, KVARN_FLAG_BAD_LENGTH);
  }
  int n_ws = L % kB;
  if (n_ws > 0 && ws == nullptr) {  // tail tokens without a workspace: attend the tiles only
    n_ws = 0;
    if (threadIdx.x == 0) raise_flag(args.flags, KVARN_FLAG_BAD_LENGTH);
  }
  const int n_sp = (n_full + args.tiles_per_split - 1) / args.tiles_per_split;
  if (gg >= args.group) return;
  const int64_t qrow = (s * args.hkv * args.group + static_cast<int64_t>(h) * args.group + gg) * kD;

  const float* part = args.part + ((s * args.hkv + h) * args.n_split) * (8 * kPartStride) + gg * kPartStride;
  float M = -INFINITY;
  for (int p = 0; p < n_sp; ++p) M = fmaxf(M, part[p * 8 * kPartStride + 128]);

  // workspace tokens: exact fp16 K/V, unrotated
  const uint16_t* wk = ws ? ws + ((s * args.hkv + h) * 2 + 0) * static_cast<int64_t>(kB * kD) : nullptr;
  const uint16_t* wv = ws ? ws + ((s * args.hkv + h) * 2 + 1) * static_cast<int64_t>(kB * kD) : nullptr;
  float qf[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) qf[u] = h2f_bits(args.q[qrow + 4 * lane + u]) * (kLog2e * kInvSqrt128);
  for (int t = 0; t < n_ws; ++t) {
    float d = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) d = fmaf(qf[u], h2f_bits(wk[t * kD + 4 * lane + u]), d);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) sc[gg][t] = d;
    M = fmaxf(M, d);
  }
  __syncwarp();

  float acc[4] = {0.f, 0.f, 0.f, 0.f}, wacc[4] = {0.f, 0.f, 0.f, 0.f};
  float l = 0.f;
  for (int p = 0; p < n_sp; ++p) {
    const float* pp = part + p * 8 * kPartStride;
    const float mp = pp[128];
    const float f = (mp == -INFINITY) ? 0.f : exp2f(mp - M);
    l = fmaf(pp[129], f, l);
    const float4 a = *reinterpret_cast<const float4*>(pp + 4 * lane);
    acc[0] = fmaf(a.x, f, acc[0]);
    acc[1] = fmaf(a.y, f, acc[1]);
    acc[2] = fmaf(a.z, f, acc[2]);
    acc[3] = fmaf(a.w, f, acc[3]);
  }
  for (int t = 0; t < n_ws; ++t) {
    const float pw = exp2f(sc[gg][t] - M);
    l += pw;
#pragma unroll
    for (int u = 0; u < 4; ++u) wacc[u] = fmaf(pw, h2f_bits(wv[t * kD + 4 * lane + u]), wacc[u]);
  }
  // un-rotate: FWHT over the 128 channels (4 per lane), then scale by 1/sqrt(128)
  {
    float a0 = acc[0] + acc[1], a1 = acc[0] - acc[1], a2 = acc[2] + acc[3], a3 = acc[2] - acc[3];
    acc[0] = a0 + a2;
    acc[1] = a1 + a3;
    acc[2] = a0 - a2;
    acc[3] = a1 - a3;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float other = __shfl_xor_sync(0xffffffffu, acc[u], o);
        acc[u] = upper ? (other - acc[u]) : (acc[u] + other);
      }
    }
  }
  const float inv_l = (l > 0.f) ? 1.0f / l : 0.f;
  uint16_t res[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) res[u] = f2h_bits(fmaf(acc[u], kInvSqrt128, wacc[u]) * inv_l);
  *reinterpret_cast<uint2*>(out + qrow + 4 * lane) =
      make_uint2(res[0] | (static_cast<uint32_t>(res[1]) << 16), res[2] | (static_cast<uint32_t>(res[3]) << 16));
}

}  // namespace

int decode_tiles_per_split(int max_blocks) {
  (void)max_blocks;
  return 16;
}

int decode_num_splits(int max_blocks) {
  const int c = decode_tiles_per_split(max_blocks);
  return max_blocks <= 0 ? 1 : (max_blocks + c - 1) / c;
}

size_t decode_part_bytes(int n_seqs, int hkv, int max_blocks) {
  return static_cast<size_t>(n_seqs) * hkv * decode_num_splits(max_blocks) * 8 * kPartStride * sizeof(float);
}

cudaError_t launch_decode(const uint16_t* q, const uint8_t* cache, const uint16_t* ws, const int32_t* block_tables,
                          const int32_t* seq_lens, int n_seqs, int hkv, int group, int max_blocks, int64_t num_blocks,
                          uint16_t* out, void* scratch, unsigned* flags, cudaStream_t stream) {
  if (n_seqs <= 0) return cudaSuccess;
  constexpr int kW = 4, kS = 1;
  using S = SplitSmem<kW, kS>;
  DecodeArgs a;
  a.q = q;
  a.cache = cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.part = static_cast<float*>(scratch);
  a.flags = flags;
  a.num_blocks = num_blocks;
  a.hkv = hkv;
  a.group = group;
  a.max_blocks = max_blocks;
  a.n_split = decode_num_splits(max_blocks);
  a.tiles_per_split = decode_tiles_per_split(max_blocks);
  cudaError_t err =
      cudaFuncSetAttribute(decode_split_kernel<kW, kS>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  if (err != cudaSuccess) return err;
  if (max_blocks > 0) {
    dim3 grid(a.n_split, hkv, n_seqs);
    decode_split_kernel<kW, kS><<<grid, kW * 32, S::kBytes, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  dim3 mgrid(hkv, n_seqs);
  decode_merge_kernel<<<mgrid, 256, 0, stream>>>(a, ws, out);
  return cudaGetLastError();
}

}  // namespace kvarn
