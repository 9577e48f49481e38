// Device-side helpers shared by the libkvarn kernels (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int kD = 128;            // channels per head
constexpr int kB = 128;            // tokens per tile
constexpr int kRec = KVARN_RECORD_BYTES;
constexpr int kKCodeOff = 0;
constexpr int kVCodeOff = 8192;
constexpr int kKMetaOff = 12288;
constexpr int kVMetaOff = 13312;
constexpr float kFp16MinNormal = 6.103515625e-05f;   // 2^-14
constexpr float kFp16Max = 65504.0f;
constexpr float kInvSqrt128 = 0.088388347648318440f; // 2^-3.5

// Record of one (block, kv-head) for KB-bit keys and VB-bit values: key codes,
// value codes, key metadata, value metadata. Full metadata is fp16 (r, c, s, z) x
// 128 per tensor; lean metadata keeps (c, s, z) for keys and (r, s, z) for values
// (the scale constant inside a quantization group is folded into its s and z).
template <int KB, int VB, bool kLean = false>
struct RecordLayout {
  static constexpr int kKBits = KB, kVBits = VB;
  static constexpr int kMetaBytes = kLean ? 768 : 1024;   // per tensor
  static constexpr int kKCodeBytes = kD * kB * KB / 8;
  static constexpr int kVCodeBytes = kD * kB * VB / 8;
  static constexpr int kKCodeOff = 0;
  static constexpr int kVCodeOff = kKCodeBytes;
  static constexpr int kKMetaOff = kKCodeBytes + kVCodeBytes;
  static constexpr int kVMetaOff = kKMetaOff + kMetaBytes;
  static constexpr int kBytes = kVMetaOff + kMetaBytes;
  // fp16 offsets of the vectors inside a tensor's metadata (-1: not stored)
  static constexpr int kKr = kLean ? -1 : 0, kKc = kLean ? 0 : 128, kKs = kLean ? 128 : 256, kKz = kLean ? 256 : 384;
  static constexpr int kVr = 0, kVc = kLean ? -1 : 128, kVs = kLean ? 128 : 256, kVz = kLean ? 256 : 384;
};
static_assert(RecordLayout<4, 2>::kBytes == kRec && RecordLayout<4, 2>::kVMetaOff == kVMetaOff, "k4v2 record");
static_assert(RecordLayout<4, 2, true>::kBytes == 13824, "k4v2 lean record");

// Kernels report data errors by OR-ing KVARN_FLAG_* bits into a device flag word
// whose address the host passes in.
__device__ __forceinline__ void raise_flag(unsigned int* flags, unsigned int bit) { atomicOr(flags, bit); }

// A wait on a copy gives up after kWaitNs nanoseconds of the global timer (far
// above any copy time) and reports KVARN_FLAG_WAIT_TIMEOUT instead of hanging.
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Bounded wait for the phase with parity `parity` to complete. Returns false (and
// raises KVARN_FLAG_WAIT_TIMEOUT) if it did not complete within `limit_ns` of the
// global timer (kWaitNs unless a self-test asks for less).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* flags,
                                          unsigned long long limit_ns = kWaitNs) {
  const uint32_t addr = smem_u32(bar);
  unsigned long long t0 = 0;
  for (unsigned int n = 0;; ++n) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if (n == 0) {
      t0 = global_ns();
    } else if ((n & 63) == 0 && global_ns() - t0 > limit_ns) {
      raise_flag(flags, KVARN_FLAG_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- bulk copies (TMA, 1-D)
// global -> shared, completion counted on `bar` (bytes multiple of 16, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// shared -> global, tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* dst_gmem, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// At most N of this thread's bulk groups may still be reading their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Make generic-proxy shared-memory writes visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- fp16 helpers
__device__ __forceinline__ uint16_t f2h_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }
__device__ __forceinline__ float h2f_bits(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ float clampf(float x, float lo, float hi) { return fminf(fmaxf(x, lo), hi); }

}  // namespace kvarn
