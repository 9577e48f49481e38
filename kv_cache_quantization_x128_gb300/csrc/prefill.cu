// Chunked-prefill attention over the packed KVarN cache plus the fresh fp16 chunk
// (KVarN README, "How KVarN works": scales are re-applied on read and the
// orthonormal rotation keeps attention scores). Chunk token p of a sequence with
// L0 cached tokens attends the L0 cached tokens (floor(L0/128) packed tiles, then
// the L0 % 128 fp16 workspace tokens) and chunk tokens 0..p.
//
// One CTA per (16 chunk tokens, kv-head, sequence): its 128 rows are the 16 tokens
// times 8 GQA head slots (row 8t + g), the M of 128 x N x 16 tcgen05 MMAs with
// fp32 accumulators in TMEM. B operands are fp16 in shared memory in the 128-byte
// swizzled K-major layout; every fp32 operand is carried as an fp16 hi + lo pair
// (three products, hi*hi + hi*lo + lo*hi, keep ~22 bits: fp16 alone moves outputs
// of keys with outlier channels by up to 3e-2). Per packed tile:
//   QK^T: A = q_r (hi, lo; shared memory), B = k~ (hi, lo) with k~[j][i] = code *
//         r^K_i s^K_i and a 129th row r^K z^K, so S[:, 128] = beta;
//         score_j = c^K_j (S_j + beta);
//   PV:   A = p' (hi, lo; TMEM, two values per column) with p'_j = p_j c^V_j s^V_j,
//         B = value codes (exact); acc_i += r^V_i (D_i + gamma),
//         gamma = sum_j p_j c^V_j z^V_j.
// Two threads own a row (channels 0-63 and 64-127 of S and of the accumulator,
// which lives in registers). Warps 0-7 do all the per-tile thread work (code
// unpacking, softmax, accumulator); the first warp of a third warpgroup only issues
// the UMMAs and starts the record copies, so no row warp waits in an issue (a thread
// issuing a tile's UMMAs was measured to stay there for most of their run). setmaxnreg
// moves the registers to the row warps (232 each, 40 for the issuing warpgroup).
// Per tile t the row warps take S(t), the softmax and p'(t), then unpack tile t + 1's
// keys while PV(t) runs, so its QK^T is queued as soon as they are ready.
// The packed pass runs in the rotated domain (q_r = H q);
// the accumulator is then rotated back once (H is its own inverse) and the fresh
// pass (workspace tail and chunk, causal) continues in the input domain with
// unrotated q and plain fp16 K/V under the same online softmax (log2 domain).
#include "kvarn_common.cuh"
#include "kvarn_frag.cuh"
#include "kvarn_launch.h"
#include "kvarn_tc.cuh"

namespace kvarn {
namespace {

constexpr int kRowThreads = 256;                  // 8 row warps: two threads per row in the row phases
constexpr int kPThreads = kRowThreads + 128;      // + one warpgroup whose first warp issues the UMMAs
// Registers after the split (setmaxnreg): 2 x 128 x 232 + 128 x 40 = 384 x 168, the
// launch's allocation at 168 a thread.
constexpr int kRowRegs = 232, kIssueRegs = 40;
constexpr int kPTokens = 16;                      // chunk tokens per CTA (x 8 head slots = 128 rows)
constexpr uint32_t kHalfB = 18432;                // K-half stride of the keys operand (144 rows)
constexpr uint32_t kHalfQ = 16384;                // K-half stride of the 128-row operands
constexpr int kMaxRec = 18432;                    // largest record (k4v4)
constexpr int kOffQ = 0;                          // A of QK^T: q hi, q lo (32 KB each)
constexpr int kOffB = 65536;                      // B of QK^T: k~ hi, lo (36 KB each)
constexpr int kOffV = kOffB + 4 * kHalfB;         // B of PV: values [channel][token] (32 KB)
constexpr int kOffRec = kOffV + 2 * kHalfQ;       // packed records [2] (the next one in flight)
constexpr int kScN = 5 * 128;                     // scale floats of one tile
constexpr int kOffSc = kOffRec + 2 * kMaxRec;     // fp32 [2][5][128]: c^K, c s^V, c z^V, r^V, r s^K
constexpr int kOffX = kOffSc + 2 * kScN * 4;      // fp32 [3][2][128]: row max, gamma and sum of each half
constexpr int kOffBar = kOffX + 3 * 1024;         // mbarriers: records [2], QK^T, PV
constexpr int kOffSlot = kOffBar + 32;            // TMEM base address
constexpr int kPSmem = kOffSlot + 8;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;   // TMEM columns: S (144), PV product (128), p' hi, lo (64 + 64)
constexpr float kLog2eP = 1.4426950408889634f;
static_assert(kOffV % 1024 == 0 && kOffRec % 16 == 0 && kPSmem <= 232448, "prefill shared memory");

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

// Byte offset of element (row r, K index k) in a 128-byte swizzled K-major operand
// whose two 64-wide K halves are `half` bytes apart.
__device__ __forceinline__ uint32_t swo(int r, int k, uint32_t half) {
  return static_cast<uint32_t>(k >> 6) * half + static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 +
                                                                      ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}
__device__ __forceinline__ uint64_t op_desc(uint32_t base, int s, uint32_t half) {
  return smem_desc_sw128(base + static_cast<uint32_t>(s >> 2) * half + static_cast<uint32_t>(s & 3) * 32);
}

// Thread t of the warp: TMEM lane (base lane + t), 32 consecutive columns.
__device__ __forceinline__ void tld_x32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tld_x1(uint32_t taddr, float& v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(*reinterpret_cast<uint32_t*>(&v)) : "r"(taddr));
}
__device__ __forceinline__ void tld_wait1(float& v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(*reinterpret_cast<uint32_t*>(&v)));
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A's row m in TMEM lane m, its K elements two per
// 32-bit column (K step k of 16 at column a_tmem + 8 k); issued by one thread.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Thread t of the warp: 32 consecutive columns of TMEM lane (base lane + t) from v.
__device__ __forceinline__ void tst_x32(uint32_t taddr, const uint32_t* r) {
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

// 64 fp32 values as fp16 (hi, lo) pairs into 32 TMEM columns each (hi at taddr, lo at
// taddr + 64), two values per column.
__device__ __forceinline__ void tmem_split_store(const float (&x)[64], uint32_t taddr) {
  uint32_t h[32], l[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) split2p(make_float2(x[2 * e], x[2 * e + 1]), h[e], l[e]);
  tst_x32(taddr, h);
  tst_x32(taddr + 64, l);
}

// Unnormalised FWHT over 64 values (the butterflies of index bits 0-5).
__device__ __forceinline__ void fwht64(float (&x)[64]) {
#pragma unroll
  for (int bit = 1; bit < 64; bit <<= 1)
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if ((i & bit) == 0) {
        const float u = x[i], w = x[i | bit];
        x[i] = u + w;
        x[i | bit] = u - w;
      }
}

// Last butterfly (index bit 6) between the two threads of a row through shared
// memory `xb` ([2][64][128] fp32, column-major so a warp's lanes hit distinct banks):
// the lower half becomes own + partner, the upper half partner - own.
__device__ __forceinline__ void fwht_pair(float (&x)[64], float* xb, int row, int hf) {
#pragma unroll
  for (int i = 0; i < 64; ++i) xb[(hf * 64 + i) * 128 + row] = x[i];
  named_bar(2, kRowThreads);
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float o = xb[((hf ^ 1) * 64 + i) * 128 + row];
    x[i] = hf == 0 ? x[i] + o : o - x[i];
  }
  named_bar(2, kRowThreads);
}

// 64 fp32 values of a row (K indices k0 .. k0 + 63) as fp16 hi and lo parts into two
// swizzled operands, 16 bytes at a time.
__device__ __forceinline__ void store_split(const float (&x)[64], uint8_t* hi, uint8_t* lo, int row, int k0,
                                            uint32_t half) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split2p(make_float2(x[8 * q + 2 * e], x[8 * q + 2 * e + 1]), h[e], l[e]);
    const uint32_t off = swo(row, k0 + 8 * q, half);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// A pair of key code values (fp16 pair v) times r s^K of their two channels (rsp),
// as fp16 hi and lo parts at byte offset `off` of the two key operands.
__device__ __forceinline__ void put_key_pair(uint8_t* bh, uint8_t* bl, uint32_t off, uint32_t v, float2 rsp) {
  uint32_t h, l;
  split2p(__fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&v)), rsp), h, l);
  *reinterpret_cast<uint32_t*>(bh + off) = h;
  *reinterpret_cast<uint32_t*>(bl + off) = l;
}

// Scale vectors of the record (threads 0-127: index tid) and the 129th key row
// r^K z^K (hi, lo). Codes in the operands are code / 8 (4-bit) or code / 2 (2-bit);
// r s^K and c s^V carry the factor back (a power of two: exact).
template <int KB, int VB, bool kLean>
__device__ __forceinline__ void unpack_scales(const uint8_t* rec, float* sc, uint8_t* bh, uint8_t* bl, int tid) {
  using L = RecordLayout<KB, VB, kLean>;
  const uint16_t* km = reinterpret_cast<const uint16_t*>(rec + L::kKMetaOff);
  const uint16_t* vm = reinterpret_cast<const uint16_t*>(rec + L::kVMetaOff);
  constexpr float kKf = KB == 4 ? 8.0f : 2.0f, kVf = VB == 4 ? 8.0f : 2.0f;
  const float kr = kLean ? 1.0f : h2f_bits(km[L::kKr + tid]);
  const float vc = kLean ? 1.0f : h2f_bits(vm[L::kVc + tid]);
  sc[0 * 128 + tid] = h2f_bits(km[L::kKc + tid]);                 // per token: c^K
  sc[1 * 128 + tid] = kVf * vc * h2f_bits(vm[L::kVs + tid]);      // per token: c s^V
  sc[2 * 128 + tid] = vc * h2f_bits(vm[L::kVz + tid]);            // per token: c z^V
  sc[3 * 128 + tid] = h2f_bits(vm[L::kVr + tid]);                 // per channel: r^V
  sc[4 * 128 + tid] = kKf * kr * h2f_bits(km[L::kKs + tid]);      // per channel: r s^K
  const float rz = kr * h2f_bits(km[L::kKz + tid]);
  const uint16_t hz = f2h_bits(rz);
  const uint32_t off = swo(128, tid, kHalfB);
  *reinterpret_cast<uint16_t*>(bh + off) = hz;
  *reinterpret_cast<uint16_t*>(bl + off) = f2h_bits(rz - h2f_bits(hz));
}

// Code words of a record, as the decode fragments lay them out (kvarn.h), go to
// operand rows and K indices as follows; thread tid handles words tid + 256 k.
//  * 4-bit (keys [token][channel], values [channel][token]): word wi of row wi >> 4
//    holds the pairs at K indices c0 + {0, 8} (low nibbles) and c0 + {16, 24} (high
//    nibbles), c0 = 32 (wi & 3) + 2 ((wi >> 2) & 3).
//  * 2-bit keys: word wi of token wi >> 3 holds, in bits 2r of byte m, the pair at
//    channel c0 + 16 m + 8 r, c0 = 64 (wi & 1) + 2 ((wi >> 1) & 3).
//  * 2-bit values: word wi (panel wi >> 7, cell (wi >> 2) & 31, partner (wi >> 1) & 1,
//    word wi & 1) of channel 16 panel + 8 partner + cell / 4 holds, like the keys,
//    the pairs at tokens c0 + 16 m + 8 r, c0 = 64 (wi & 1) + 2 (cell & 3).
// Per k the row moves by 16 (4-bit) or 32 (2-bit) rows, a whole number of 8-row
// swizzle groups, so each thread's byte offsets are computed once and advance by
// 2048 or 4096 bytes.
template <int KB, int VB, bool kLean>
__device__ __forceinline__ void unpack_values(const uint8_t* rec, uint8_t* vb, int tid) {
  using L = RecordLayout<KB, VB, kLean>;
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(rec + L::kVCodeOff);
  if (VB == 4) {
    const int r0 = tid >> 4, c0 = 32 * (tid & 3) + 2 * ((tid >> 2) & 3);
    uint32_t off[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) off[q] = swo(r0, c0 + 8 * q, kHalfQ);
#pragma unroll 2
    for (int k = 0; k < 8; ++k) {
      const uint32_t w = vw[tid + 256 * k];
      uint32_t v[4];
      cvt4(w & 0x0F0F0F0Fu, v[0], v[1]);
      cvt4((w >> 4) & 0x0F0F0F0Fu, v[2], v[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint32_t*>(vb + off[q] + 2048 * k) = v[q];
    }
  } else {
    const int r0 = 16 * (tid >> 7) + 8 * ((tid >> 1) & 1) + ((tid >> 4) & 7);
    const int c0 = 64 * (tid & 1) + 2 * ((tid >> 2) & 3);
    uint32_t off[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int m = 0; m < 4; ++m) off[r][m] = swo(r0, c0 + 16 * m + 8 * r, kHalfQ);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = vw[tid + 256 * k];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t v[4];
        cvt2((w >> (2 * r)) & 0x33333333u, v);
#pragma unroll
        for (int m = 0; m < 4; ++m) *reinterpret_cast<uint32_t*>(vb + off[r][m] + 4096 * k) = v[m];
      }
    }
  }
}

// Key codes of the record, times r s^K per channel, into the QK^T operand
// [token][channel] (hi, lo).
template <int KB, int VB, bool kLean>
__device__ __forceinline__ void unpack_keys(const uint8_t* rec, const float* rs, uint8_t* bh, uint8_t* bl, int tid) {
  using L = RecordLayout<KB, VB, kLean>;
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(rec + L::kKCodeOff);
  if (KB == 4) {
    const int r0 = tid >> 4, c0 = 32 * (tid & 3) + 2 * ((tid >> 2) & 3);
    uint32_t off[4];
    float2 f[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      off[q] = swo(r0, c0 + 8 * q, kHalfB);
      f[q] = *reinterpret_cast<const float2*>(rs + c0 + 8 * q);
    }
#pragma unroll 2
    for (int k = 0; k < 8; ++k) {
      const uint32_t w = kw[tid + 256 * k];
      uint32_t v[4];
      cvt4(w & 0x0F0F0F0Fu, v[0], v[1]);
      cvt4((w >> 4) & 0x0F0F0F0Fu, v[2], v[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) put_key_pair(bh, bl, off[q] + 2048 * k, v[q], f[q]);
    }
  } else {
    const int r0 = tid >> 3, c0 = 64 * (tid & 1) + 2 * ((tid >> 1) & 3);
    uint32_t off[2][4];
    float2 f[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        off[r][m] = swo(r0, c0 + 16 * m + 8 * r, kHalfB);
        f[r][m] = *reinterpret_cast<const float2*>(rs + c0 + 16 * m + 8 * r);
      }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = kw[tid + 256 * k];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t v[4];
        cvt2((w >> (2 * r)) & 0x33333333u, v);
#pragma unroll
        for (int m = 0; m < 4; ++m) put_key_pair(bh, bl, off[r][m] + 4096 * k, v[m], f[r][m]);
      }
    }
  }
}

// Named barriers: 0 (__syncthreads) at the start and the end only; 1 the row max
// exchange and 2 the other row-only points (256 threads); 3 "p' (and the tile's values)
// ready" and 4 "keys ready": the row threads arrive, the issuing warp waits (288).
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
// A row thread's operand writes (shared memory, TMEM) visible to the tensor core,
// then its arrival on producer barrier `id`.
__device__ __forceinline__ void rows_ready(int id) {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  fence_proxy_async_smem();
  tc_fence_before();
  bar_arrive(id, kRowThreads + 32);
}

template <int KB, int VB, bool kLean>
__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using L = RecordLayout<KB, VB, kLean>;
  uint8_t* opq = smem + kOffQ;                    // q hi at +0, lo at +32 KB
  uint8_t* opb = smem + kOffB;                    // k~ hi at +0, lo at +2 * kHalfB
  uint8_t* opv = smem + kOffV;
  uint8_t* rec = smem + kOffRec;
  float* scb = reinterpret_cast<float*>(smem + kOffSc);   // [2][kScN]
  float* xch = reinterpret_cast<float*>(smem + kOffX);
  float* xb = reinterpret_cast<float*>(smem + kOffB);     // FWHT exchange ([2][64][128] fp32) when opb is free
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);   // records [2], QK^T, PV
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, s = blockIdx.z;
  const int t0 = a.cu[s], chunk = a.cu[s + 1] - t0;
  // a chunk longer than the grid covers (max_chunk too small): its tail tokens get
  // no CTA and their output rows are not written, so the last CTA of the row says so
  if (tid == 0 && h == 0 && blockIdx.x == gridDim.x - 1 && chunk > static_cast<int>(gridDim.x) * kPTokens)
    raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
  if (static_cast<int>(blockIdx.x) * kPTokens >= chunk) return;      // whole CTA: nothing to do
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
  // fresh token f: workspace token f (f < n_ws) or chunk token f - n_ws; this CTA's
  // last token attends f < n_fresh
  const int p_last = min(chunk - 1, static_cast<int>(blockIdx.x) * kPTokens + kPTokens - 1);
  const int n_fresh = n_ws + p_last + 1;
  const int n_fb = (n_fresh + kB - 1) / kB;
  // tile ti's block index is inside the cache (same answer in every thread); a tile
  // outside attends nothing
  auto valid_tile = [&](int ti) {
    const int64_t blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + ti];
    return blk >= 0 && blk < a.num_blocks;
  };

  if (tid == 0) {
    for (int b = 0; b < 4; ++b) mbar_init(&bar[b], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const uint32_t s_tm = tmem + kColS, o_tm = tmem + kColO;
  const uint32_t q_hi = smem_u32(opq), q_lo = q_hi + 2 * kHalfQ;
  const uint32_t b_hi = smem_u32(opb), b_lo = b_hi + 2 * kHalfB;
  const uint32_t v_op = smem_u32(opv);
  constexpr uint32_t kId144 = idesc_f16_f32(128, 144), kId128 = idesc_f16_f32(128, 128);

  const bool rower = warp < kRowThreads / 32;
  const int sub = warp & 3, hf = (warp >> 2) & 1;
  const int row = 32 * sub + lane;
  const int p = static_cast<int>(blockIdx.x) * kPTokens + (row >> 3), gh = row & 7;
  const bool active = rower && p < chunk && gh < a.group;
  const int64_t qrow = (static_cast<int64_t>(t0) + p) * a.hkv * a.group + static_cast<int64_t>(h) * a.group + gh;

  if (!rower) {
    // ------------------------------------------------------------ issuing warpgroup
    regs_dec<kIssueRegs>();
    if (warp == kRowThreads / 32) {
      const bool leader = lane == 0;
      uint32_t n_qk = 0, n_pv = 0;        // commits on the QK^T and PV barriers
      auto prefetch = [&](int ti) {       // record of tile ti into buffer ti & 1
        if (ti >= n_full) return;
        const int64_t blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + ti];
        const int b = ti & 1;
        if (blk >= 0 && blk < a.num_blocks) {
          mbar_arrive_expect_tx(&bar[b], L::kBytes);
          bulk_g2s(rec + b * kMaxRec, a.cache + (blk * a.hkv + h) * static_cast<int64_t>(L::kBytes), L::kBytes,
                   &bar[b]);
        } else {
          raise_flag(a.flags, KVARN_FLAG_BAD_BLOCK);
        }
      };
      auto issue_qk = [&](bool packed) {  // S = q (hi, lo) x keys (hi, lo: three products, or hi)
#pragma unroll 1
        for (int k = 0; k < 8; ++k) {
          const uint64_t ah = op_desc(q_hi, k, kHalfQ), al = op_desc(q_lo, k, kHalfQ);
          const uint64_t bh = op_desc(b_hi, k, kHalfB);
          if (packed) {
            umma_f16(s_tm, ah, bh, kId144, k > 0);
            umma_f16(s_tm, ah, op_desc(b_lo, k, kHalfB), kId144, 1);
            umma_f16(s_tm, al, bh, kId144, 1);
          } else {
            umma_f16(s_tm, ah, bh, kId128, k > 0);
            umma_f16(s_tm, al, bh, kId128, 1);
          }
        }
        umma_commit(&bar[2]);
        ++n_qk;
      };
      auto issue_pv = [&]() {             // D = p' (TMEM, hi and lo) x values
#pragma unroll 1
        for (int k = 0; k < 8; ++k) {
          const uint64_t bv = op_desc(v_op, k, kHalfQ);
          umma_f16_ts(o_tm, tmem + kColP + 8 * k, bv, kId128, k > 0);
          umma_f16_ts(o_tm, tmem + kColP + 64 + 8 * k, bv, kId128, 1);
        }
        umma_commit(&bar[3]);
        ++n_pv;
      };
      if (n_full > 0) {
        if (leader) {
          prefetch(0);
          prefetch(1);
        }
        named_bar(4, kRowThreads + 32);   // keys and values of tile 0
        tc_fence_after();
        if (leader) issue_qk(true);
        for (int t = 0; t < n_full; ++t) {
          named_bar(3, kRowThreads + 32); // p'(t); record t + 2's buffer is free
          tc_fence_after();
          if (leader) {
            prefetch(t + 2);
            issue_pv();
          }
          if (t + 1 < n_full) {
            named_bar(4, kRowThreads + 32);   // keys of tile t + 1
            tc_fence_after();
            if (leader) issue_qk(true);
          }
        }
      }
      for (int fb = 0; fb < n_fb; ++fb) {
        named_bar(4, kRowThreads + 32);
        tc_fence_after();
        if (leader) issue_qk(false);
        named_bar(3, kRowThreads + 32);
        tc_fence_after();
        if (leader) issue_pv();
      }
      // the last products are done before TMEM is released (bounded waits)
      if (leader) {
        if (n_qk) mbar_wait(&bar[2], (n_qk - 1) & 1u, a.flags);
        if (n_pv) mbar_wait(&bar[3], (n_pv - 1) & 1u, a.flags);
      }
    }
  } else {
    // ------------------------------------------------------------ row warpgroups
    regs_inc<kRowRegs>();
    const uint32_t trow = tmem_addr(tmem, 32 * sub, 0);          // this warp's lanes
    bool ok = true;
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t qk_par = 0, pv_par = 0, rpar = 0;
    auto wait_qk = [&]() {
      const bool r = mbar_wait(&bar[2], qk_par, a.flags);
      if (r) qk_par ^= 1u;
      tc_fence_after();
      return r;
    };
    auto wait_pv = [&]() {
      const bool r = mbar_wait(&bar[3], pv_par, a.flags);
      if (r) pv_par ^= 1u;
      tc_fence_after();
      return r;
    };
    // softmax of this thread's 64 scores x (log2 domain, -inf = masked) against the
    // row max over both halves; x becomes p, the accumulator is rescaled
    auto softmax = [&](float (&x)[64]) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; j += 2) mx = fmax3f(mx, x[j], x[j + 1]);
      xch[hf * 128 + row] = mx;
      named_bar(1, kRowThreads);
      mx = fmaxf(mx, xch[(hf ^ 1) * 128 + row]);
      const float m_new = fmaxf(m_run, mx);
      float corr = 1.f;
      if (m_new == -INFINITY) {                   // every token so far masked
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = 0.f;
      } else {
        corr = ex2(m_run - m_new);
        m_run = m_new;
        const float2 nm = make_float2(-m_new, -m_new);
        float2 ls = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          const float2 e = __fadd2_rn(make_float2(x[j], x[j + 1]), nm);
          x[j] = ex2(e.x);
          x[j + 1] = ex2(e.y);
          ls = __fadd2_rn(ls, make_float2(x[j], x[j + 1]));
        }
        l_run = fmaf(l_run, corr, ls.x + ls.y);
      }
      const float2 c2 = make_float2(corr, corr);
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 v = __fmul2_rn(make_float2(acc[i], acc[i + 1]), c2);
        acc[i] = v.x;
        acc[i + 1] = v.y;
      }
    };

    // -------------------------------------------------------------- packed tiles
    if (n_full > 0) {
      // q_r = H q * log2(e) / sqrt(128), as FWHT(q) * log2(e) / 128, into the A operand
      {
        float x[64];
        const uint16_t* qp = a.q + qrow * kD + 64 * hf;
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 f = active ? h2pair(qp + i) : make_float2(0.f, 0.f);
          x[i] = f.x;
          x[i + 1] = f.y;
        }
        fwht64(x);
        fwht_pair(x, xb, row, hf);
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] *= kLog2eP / 128.0f;
        store_split(x, opq, opq + 2 * kHalfQ, row, 64 * hf, kHalfQ);
      }
      // rows 129-143 of the keys operand stay zero (row 128 is rewritten per tile; the
      // exchange above used this space)
      for (int e = tid; e < 2 * 2 * 15 * 8; e += kRowThreads) {   // [hi/lo][K half][row 129..143][chunk]
        const int part = e / 240, rem = e % 240, k0 = 64 * (rem / 120), r = 129 + (rem % 120) / 8, c = rem % 8;
        *reinterpret_cast<uint4*>(opb + part * 2 * kHalfB + swo(r, k0 + 8 * c, kHalfB)) = make_uint4(0, 0, 0, 0);
      }
      auto wait_rec = [&](int ti) {
        if (!valid_tile(ti)) return true;
        const int b = ti & 1;
        const bool r = mbar_wait(&bar[b], (rpar >> b) & 1u, a.flags);
        if (r) rpar ^= 1u << b;
        return r;
      };
      // tile ti's scales (buffer ti & 1) and keys; a masked tile gets zero scales, which
      // keep its PV term zero
      auto stage_keys = [&](int ti) {
        float* sct = scb + (ti & 1) * kScN;
        if (valid_tile(ti)) {
          const uint8_t* r = rec + (ti & 1) * kMaxRec;
          if (tid < 128) unpack_scales<KB, VB, kLean>(r, sct, opb, opb + 2 * kHalfB, tid);
          named_bar(2, kRowThreads);
          unpack_keys<KB, VB, kLean>(r, sct + 4 * 128, opb, opb + 2 * kHalfB, tid);
        } else {
          for (int e = tid; e < kScN; e += kRowThreads) sct[e] = 0.f;
          named_bar(2, kRowThreads);
        }
      };
      auto stage_values = [&](int ti) {
        if (valid_tile(ti)) {
          unpack_values<KB, VB, kLean>(rec + (ti & 1) * kMaxRec, opv, tid);
        } else {
          for (int e = tid; e < static_cast<int>(2 * kHalfQ / 16); e += kRowThreads)
            reinterpret_cast<uint4*>(opv)[e] = make_uint4(0, 0, 0, 0);
        }
      };

      ok = wait_rec(0) && ok;
      stage_keys(0);
      stage_values(0);
      rows_ready(4);
      for (int t = 0; t < n_full; ++t) {
        const float* sct = scb + (t & 1) * kScN;
        ok = wait_qk() && ok;
        float x[64], beta;
        tld_x32(trow + kColS + 64 * hf, x);
        tld_x32(trow + kColS + 64 * hf + 32, x + 32);
        tld_x1(trow + kColS + 128, beta);
        tmem_wait_x32(x);
        tmem_wait_x32(x + 32);
        tld_wait1(beta);
        if (valid_tile(t)) {
          const float2 b2 = make_float2(beta, beta);
          const float4* ck = reinterpret_cast<const float4*>(sct + 64 * hf);
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 c = ck[j >> 2];
            const float2 u = __fmul2_rn(__fadd2_rn(make_float2(x[j], x[j + 1]), b2), make_float2(c.x, c.y));
            const float2 w = __fmul2_rn(__fadd2_rn(make_float2(x[j + 2], x[j + 3]), b2), make_float2(c.z, c.w));
            x[j] = u.x; x[j + 1] = u.y; x[j + 2] = w.x; x[j + 3] = w.y;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = -INFINITY;
        }
        softmax(x);
        float gam;
        {
          float2 g2 = make_float2(0.f, 0.f);
          const float4* cs = reinterpret_cast<const float4*>(sct + 1 * 128 + 64 * hf);
          const float4* cz = reinterpret_cast<const float4*>(sct + 2 * 128 + 64 * hf);
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 z = cz[j >> 2], c = cs[j >> 2];
            const float2 p0 = make_float2(x[j], x[j + 1]), p1 = make_float2(x[j + 2], x[j + 3]);
            g2 = __ffma2_rn(p0, make_float2(z.x, z.y), g2);
            g2 = __ffma2_rn(p1, make_float2(z.z, z.w), g2);
            const float2 u = __fmul2_rn(p0, make_float2(c.x, c.y)), w = __fmul2_rn(p1, make_float2(c.z, c.w));
            x[j] = u.x; x[j + 1] = u.y; x[j + 2] = w.x; x[j + 3] = w.y;
          }
          gam = g2.x + g2.y;
        }
        tmem_split_store(x, trow + kColP + 32 * hf);
        xch[256 + hf * 128 + row] = gam;
        rows_ready(3);                    // p'(t): the issuer starts PV(t)
        if (t + 1 < n_full) {             // keys of tile t + 1 while PV(t) runs
          ok = wait_rec(t + 1) && ok;
          stage_keys(t + 1);
          rows_ready(4);
        } else {
          named_bar(2, kRowThreads);      // gamma's other half is written
        }
        gam += xch[256 + (hf ^ 1) * 128 + row];
        ok = wait_pv() && ok;
        tld_x32(trow + kColO + 64 * hf, x);
        tld_x32(trow + kColO + 64 * hf + 32, x + 32);
        tmem_wait_x32(x);
        tmem_wait_x32(x + 32);
        {
          const float2 g2 = make_float2(gam, gam);
          const float4* rv = reinterpret_cast<const float4*>(sct + 3 * 128 + 64 * hf);
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            const float4 v = rv[i >> 2];
            const float2 u = __ffma2_rn(make_float2(v.x, v.y), __fadd2_rn(make_float2(x[i], x[i + 1]), g2),
                                        make_float2(acc[i], acc[i + 1]));
            const float2 w = __ffma2_rn(make_float2(v.z, v.w), __fadd2_rn(make_float2(x[i + 2], x[i + 3]), g2),
                                        make_float2(acc[i + 2], acc[i + 3]));
            acc[i] = u.x; acc[i + 1] = u.y; acc[i + 2] = w.x; acc[i + 3] = w.y;
          }
        }
        if (t + 1 < n_full) stage_values(t + 1);   // PV(t) has read the values operand
        named_bar(2, kRowThreads);        // gamma, scales and operands are rewritten next
      }
      // back to the input domain: acc_u = H acc_r = FWHT(acc_r) / sqrt(128)
      fwht64(acc);
      fwht_pair(acc, xb, row, hf);
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] *= kInvSqrt128;
    }

    // -------------------------------------------------------------- fresh tokens
    // q * log2(e) / sqrt(128), unrotated, into the A operand (the packed pass is done)
    {
      float x[64];
      const uint16_t* qp = a.q + qrow * kD + 64 * hf;
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 f = active ? h2pair(qp + i) : make_float2(0.f, 0.f);
        x[i] = f.x * (kLog2eP * kInvSqrt128);
        x[i + 1] = f.y * (kLog2eP * kInvSqrt128);
      }
      store_split(x, opq, opq + 2 * kHalfQ, row, 64 * hf, kHalfQ);
    }
    // row `row` attends f <= n_ws + p
    const int lim = min(n_ws + p, n_fresh - 1);
    auto fresh_src = [&](int f, int which) -> const uint16_t* {
      if (f < n_ws) return a.ws + (((static_cast<int64_t>(s) * a.hkv + h) * 2 + which) * kB + f) * kD;
      return (which ? a.v_new : a.k_new) + ((static_cast<int64_t>(t0) + f - n_ws) * a.hkv + h) * kD;
    };
    for (int fb = 0; fb < n_fb; ++fb) {
      // keys [token][channel] into the B operand of QK^T (hi part only: fp16 exact)
      for (int e = tid; e < 128 * 16; e += kRowThreads) {
        const int jj = e >> 4, c8 = e & 15, f = fb * kB + jj;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (f < n_fresh) v = *reinterpret_cast<const uint4*>(fresh_src(f, 0) + 8 * c8);
        *reinterpret_cast<uint4*>(opb + swo(jj, 8 * c8, kHalfB)) = v;
      }
      // values transposed to [channel][token]: lane = token, so each 2-byte store of a
      // warp fills 64 contiguous bytes of one channel row
      for (int e = tid; e < 128 * 16; e += kRowThreads) {
        const int c8 = e >> 7, jj = e & 127, f = fb * kB + jj;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (f < n_fresh) v = *reinterpret_cast<const uint4*>(fresh_src(f, 1) + 8 * c8);
        const uint16_t* u = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) *reinterpret_cast<uint16_t*>(opv + swo(8 * c8 + e2, jj, kHalfQ)) = u[e2];
      }
      rows_ready(4);
      ok = wait_qk() && ok;
      float x[64];
      tld_x32(trow + kColS + 64 * hf, x);
      tld_x32(trow + kColS + 64 * hf + 32, x + 32);
      tmem_wait_x32(x);
      tmem_wait_x32(x + 32);
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (fb * kB + 64 * hf + j > lim) x[j] = -INFINITY;
      softmax(x);
      tmem_split_store(x, trow + kColP + 32 * hf);
      rows_ready(3);
      ok = wait_pv() && ok;
      tld_x32(trow + kColO + 64 * hf, x);
      tld_x32(trow + kColO + 64 * hf + 32, x + 32);
      tmem_wait_x32(x);
      tmem_wait_x32(x + 32);
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 u = __fadd2_rn(make_float2(acc[i], acc[i + 1]), make_float2(x[i], x[i + 1]));
        acc[i] = u.x;
        acc[i + 1] = u.y;
      }
      named_bar(2, kRowThreads);          // the operands are rewritten next
    }
    // output: acc / l over both halves (nothing is written after a timeout)
    xch[512 + hf * 128 + row] = l_run;
    ok = named_bar_and(2, kRowThreads, ok);
    if (ok && active) {
      const float l = xch[512 + row] + xch[512 + 128 + row];
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      uint16_t* orow = a.out + qrow * kD + 64 * hf;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = static_cast<uint32_t>(f2h_bits(acc[8 * q + 2 * e] * inv_l)) |
                 (static_cast<uint32_t>(f2h_bits(acc[8 * q + 2 * e + 1] * inv_l)) << 16);
        *reinterpret_cast<uint4*>(orow + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }

  // ---------------------------------------------------------------- end (all warps)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int KB, int VB, bool kLean>
cudaError_t launch_prefill_kernel(const PrefillArgs& a, int n_seqs, int max_chunk, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(prefill_kernel<KB, VB, kLean>, kPSmem, smem_set);
  if (err != cudaSuccess) return err;
  const dim3 grid((max_chunk + kPTokens - 1) / kPTokens, a.hkv, n_seqs);
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
