// Internal launchers shared between the libkvarn translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/kvarn.h"

namespace kvarn {

// Sets a kernel's dynamic shared-memory limit once per device (bit d of `done`);
// later launches, e.g. inside a CUDA-graph capture, make no runtime call for it.
template <class Kernel>
inline cudaError_t set_smem_once(Kernel* kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const bool cacheable = dev >= 0 && dev < 64;
  if (cacheable && ((done.load(std::memory_order_acquire) >> dev) & 1ull)) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess && cacheable) done.fetch_or(1ull << dev, std::memory_order_acq_rel);
  return err;
}

// k_bits / v_bits / lean: a preset of kvarn.h (4/2, 4/4, 2/2; lean with 4/2 only),
// checked by the caller.
cudaError_t launch_quantize_prefill(const uint16_t* k, const uint16_t* v, const int64_t* slot, int64_t n_tokens,
                                    int hkv, int64_t num_blocks, uint8_t* cache, int k_bits, int v_bits, bool lean,
                                    int n_iters, float eps, unsigned* flags, cudaStream_t stream, int max_ctas);

cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, const int32_t* seq_lens,
                          int32_t* seq_lens_out, const int32_t* block_tables, int n_seqs, int hkv, int max_blocks,
                          int64_t num_blocks, uint16_t* ws, uint8_t* cache, int k_bits, int v_bits, bool lean,
                          int n_iters, float eps, unsigned* flags, cudaStream_t stream);

cudaError_t launch_decode(const uint16_t* q, const uint8_t* cache, const uint16_t* ws, const int32_t* block_tables,
                          const int32_t* seq_lens, int n_seqs, int hkv, int group, int max_blocks, int64_t num_blocks,
                          int k_bits, int v_bits, bool lean, uint16_t* out, void* scratch, unsigned* flags,
                          cudaStream_t stream);

cudaError_t launch_prefill(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, const int32_t* cu_tokens,
                           const int32_t* seq_lens, const int32_t* block_tables, const uint8_t* cache,
                           const uint16_t* ws, int n_seqs, int max_chunk, int hkv, int group, int max_blocks,
                           int64_t num_blocks, int k_bits, int v_bits, bool lean, uint16_t* out, unsigned* flags,
                           cudaStream_t stream);

cudaError_t launch_serve_step(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* seq_lens, int32_t* seq_lens_out, const int32_t* block_tables,
                              uint16_t* ws, uint8_t* cache, int n_seqs, int hkv, int group, int max_blocks,
                              int64_t num_blocks, int k_bits, int v_bits, bool lean, int n_iters, float eps,
                              uint16_t* out, void* scratch, unsigned* flags, cudaStream_t stream);
// Device scratch of launch_decode: tile prefix per sequence + partial records, and
// at its end kServeBarrierBytes for the serving step's grid barrier words.
constexpr size_t kServeBarrierBytes = 256;
size_t decode_part_bytes(int n_seqs, int hkv, int max_blocks);
size_t serve_barrier_offset(int n_seqs, int hkv, int max_blocks);
unsigned* serve_barrier_words(void* scratch, int n_seqs, int hkv, int max_blocks);
// Bounded-wait self-test (serve.cu): which = 0 mbarrier wait, 1 grid barrier.
cudaError_t launch_wait_selftest(int which, unsigned long long limit_ns, void* barrier_words, unsigned* flags,
                                 cudaStream_t stream);
// Scratch launch_decode touches when the split kernel runs `n_ctas` CTAs (the
// device's SM count, at most 1024).
size_t decode_scratch_bytes_for_ctas(int n_seqs, int hkv, int n_ctas);
int decode_num_ctas();

// api.cu: device flag word, per-thread error message
cudaError_t flags_device_ptr(unsigned** out);
kvarn_status set_error(kvarn_status st, const char* msg);
void clear_error();
// The entry points' shared argument checks: a kvarn_meta that names a preset and
// valid sizes (KVARN_EINVAL / KVARN_EUNSUPPORTED), and a device pointer that is
// non-NULL (KVARN_EINVAL) and 16-byte aligned (KVARN_EALIGN). Both set the
// thread's error message.
kvarn_status check_meta_status(const kvarn_meta* meta);
kvarn_status check_device_ptr(const void* p, const char* name);

}  // namespace kvarn
