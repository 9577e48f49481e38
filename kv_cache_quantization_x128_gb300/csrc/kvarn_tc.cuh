// tcgen05 (5th-generation tensor core) and TMEM helpers for sm_103a.
#pragma once
#include <stdint.h>

#include "kvarn_common.cuh"

namespace kvarn {

// TMEM address: bits [31:16] lane, [15:0] column.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// Warp-wide: allocate `ncols` TMEM columns, address written to *dst (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Operands of 128 rows x 128 fp16 along K are stored as two K-major halves of 64
// (16 KB each) in the 128-byte swizzled layout that a 2-D TMA box of 64 x 128
// fp16 writes: row r at (r/8)*1024 + (r%8)*128, its 16-byte chunk c at chunk
// position c ^ (r%8). The halves must be 1024-byte aligned.
__host__ __device__ constexpr uint32_t sw_offset(int r, int k) {
  return static_cast<uint32_t>((k >> 6) * 16384 + (r >> 3) * 1024 + (r & 7) * 128 +
                               ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}
// The Sylvester +-1 Hadamard operand H[r][k] = (-1)^popcount(r & k) (fp16) in that
// layout, written by threads tid = 0 .. nthreads - 1 one 16-byte chunk (k = 8m .. 8m + 7
// of row r) at a time: popcount(r & (8m + j)) = popcount(r & 8m) + popcount(r & j)
// for j < 8, so a chunk is row r's pattern over j, negated when r & 8m has odd parity.
__device__ __forceinline__ void fill_hadamard_sw128(uint8_t* dst, int tid, int nthreads) {
  for (int e = tid; e < 128 * 16; e += nthreads) {
    const int r = e >> 4, m = e & 15;
    const uint32_t flip = (__popc(r & (8 * m)) & 1) ? 0x80008000u : 0u;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = (__popc(r & (2 * j)) & 1) ? 0xBC00u : 0x3C00u;
      const uint32_t hi = (__popc(r & (2 * j + 1)) & 1) ? 0xBC00u : 0x3C00u;
      w[j] = (lo | (hi << 16)) ^ flip;
    }
    *reinterpret_cast<uint4*>(dst + sw_offset(r, 8 * m)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
// Shared-memory matrix descriptor of that layout: 8-row groups 1024 B apart
// (stride byte offset), 128-byte swizzle (mode 2 in bits [61, 64)); the leading
// byte offset is unused when the K extent of one MMA lies inside the swizzle row.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;   // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version for sm_100 family
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}
// Start address of K step s (16 elements) of such an operand at `base`: 32 B
// further along the swizzle row, the second half 16 KB on.
__device__ __forceinline__ uint32_t sw_kstep(uint32_t base, int s) {
  return base + (s >> 2) * 16384 + (s & 3) * 32;
}
// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t m, uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 16 lanes x 64 fp32 columns per warp: thread t gets lane base + (t>>2) + 8(t&1),
// columns ((t>>1)&1) + 2k for k = 0..31 (register k). The registers are valid
// only after tmem_wait_x32 on the same array: the wait names them as operands,
// so no use of them moves above it, while independent loads and arithmetic can
// move across both.
__device__ __forceinline__ void tmem_ld_16x64b_x32_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.16x64b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_x32(float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]),"+r"(r[16]),"+r"(r[17]),"+r"(r[18]),"+r"(r[19]),"+r"(r[20]),"+r"(r[21]),"+r"(r[22]),"+r"(r[23]),"+r"(r[24]),"+r"(r[25]),"+r"(r[26]),"+r"(r[27]),"+r"(r[28]),"+r"(r[29]),"+r"(r[30]),"+r"(r[31]));
}

// ---------------------------------------------------------------- TMA (2-D tiles)
// Box of the tensor map at coordinates (x, y) into shared memory, completion
// counted on `bar`; x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tensor_map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- named barriers
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " barrier.red.and.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

}  // namespace kvarn
