// C ABI of libkvarn (declared in include/kvarn.h): host-side argument checks,
// then kernel launches on the caller's stream. Nothing here allocates memory.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <cstring>
#include <mutex>

#include "../../include/kvarn.h"
#include "kvarn_launch.h"

namespace {

thread_local char g_err[512] = "";

// One flag word per device that loads the library.
__device__ unsigned int g_device_flags;

__attribute__((format(printf, 2, 3))) kvarn_status fail(kvarn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvarn_status check_meta(const kvarn_meta* m) {
  if (m == nullptr) return fail(KVARN_EINVAL, "meta is NULL");
  if (m->head_dim != KVARN_HEAD_DIM) return fail(KVARN_EUNSUPPORTED, "head_dim must be 128 (got %lld)", (long long)m->head_dim);
  if (m->block_size != KVARN_BLOCK_SIZE)
    return fail(KVARN_EUNSUPPORTED, "block_size must be 128 (got %lld)", (long long)m->block_size);
  if (!((m->k_bits == 4 && (m->v_bits == 2 || m->v_bits == 4)) || (m->k_bits == 2 && m->v_bits == 2)))
    return fail(KVARN_EUNSUPPORTED, "bit widths must be a preset: k4v2, k4v4 or k2v2 (got k%lldv%lld)",
                (long long)m->k_bits, (long long)m->v_bits);
  if (m->num_kv_heads < 1) return fail(KVARN_EINVAL, "num_kv_heads must be >= 1 (got %lld)", (long long)m->num_kv_heads);
  if (m->num_q_heads < m->num_kv_heads || m->num_q_heads % m->num_kv_heads != 0)
    return fail(KVARN_EINVAL, "num_q_heads must be a positive multiple of num_kv_heads (got %lld)",
                (long long)m->num_q_heads);
  if (m->num_q_heads / m->num_kv_heads > KVARN_MAX_GQA_GROUP)
    return fail(KVARN_EUNSUPPORTED, "GQA group (Hq/Hkv) must be <= 8 (got %lld)",
                (long long)(m->num_q_heads / m->num_kv_heads));
  if (m->n_iters < 1 || m->n_iters > 16) return fail(KVARN_EINVAL, "n_iters must be in 1..16 (got %lld)", (long long)m->n_iters);
  if (!(m->eps > 0.0f) || !(m->eps < 1.0f)) return fail(KVARN_EINVAL, "eps must be in (0, 1)");
  if (m->num_blocks < 0) return fail(KVARN_EINVAL, "num_blocks must be >= 0 (got %lld)", (long long)m->num_blocks);
  if (m->max_blocks_per_seq < 0)
    return fail(KVARN_EINVAL, "max_blocks_per_seq must be >= 0 (got %lld)", (long long)m->max_blocks_per_seq);
  if (m->layout != 0 && m->layout != KVARN_LAYOUT_LEAN)
    return fail(KVARN_EINVAL, "layout must be 0 or KVARN_LAYOUT_LEAN (got %lld)", (long long)m->layout);
  if (m->layout == KVARN_LAYOUT_LEAN && !(m->k_bits == 4 && m->v_bits == 2))
    return fail(KVARN_EUNSUPPORTED, "lean metadata is offered with k4v2 only");
  return KVARN_OK;
}

kvarn_status need_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(KVARN_EINVAL, "%s is NULL", name);
  if (!aligned16(p)) return fail(KVARN_EALIGN, "%s is not 16-byte aligned", name);
  return KVARN_OK;
}

kvarn_status flags_ptr(unsigned** out) {
  const cudaError_t e = kvarn::flags_device_ptr(out);
  if (e != cudaSuccess) return fail(KVARN_ECUDA, "device flag word: %s", cudaGetErrorString(e));
  return KVARN_OK;
}

kvarn_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVARN_OK;
  return fail(KVARN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define KV_TRY(x)                         \
  do {                                    \
    kvarn_status st_ = (x);               \
    if (st_ != KVARN_OK) return st_;      \
  } while (0)

}  // namespace

extern "C" {

size_t kvarn_record_bytes(void) { return KVARN_RECORD_BYTES; }

size_t kvarn_meta_record_bytes(const kvarn_meta* meta) {
  if (check_meta(meta) != KVARN_OK) return 0;
  return static_cast<size_t>(KVARN_HEAD_DIM) * KVARN_BLOCK_SIZE * (meta->k_bits + meta->v_bits) / 8 +
         (meta->layout == KVARN_LAYOUT_LEAN ? 1536 : 2048);
}

size_t kvarn_cache_bytes(const kvarn_meta* meta) {
  if (check_meta(meta) != KVARN_OK) return 0;
  return static_cast<size_t>(meta->num_blocks) * meta->num_kv_heads * kvarn_meta_record_bytes(meta);
}

size_t kvarn_workspace_bytes(const kvarn_meta* meta, int32_t max_seqs) {
  if (check_meta(meta) != KVARN_OK || max_seqs < 0) return 0;
  return static_cast<size_t>(max_seqs) * meta->num_kv_heads * 2 * KVARN_BLOCK_SIZE * KVARN_HEAD_DIM * 2;
}

size_t kvarn_decode_scratch_bytes(const kvarn_meta* meta, int32_t n_seqs) {
  if (check_meta(meta) != KVARN_OK || n_seqs < 0) return 0;
  return kvarn::decode_part_bytes(n_seqs, meta->num_kv_heads, meta->max_blocks_per_seq);
}

kvarn_status kvarn_quantize_tiles(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                                  int64_t n_tokens, uint8_t* cache, const kvarn_meta* meta, void* stream) {
  g_err[0] = 0;
  KV_TRY(check_meta(meta));
  if (n_tokens < 0 || n_tokens % KVARN_BLOCK_SIZE != 0)
    return fail(KVARN_EINVAL, "n_tokens must be a non-negative multiple of 128 (got %lld)", (long long)n_tokens);
  if (n_tokens == 0) return KVARN_OK;
  if (n_tokens > INT32_MAX || (n_tokens / KVARN_BLOCK_SIZE) * meta->num_kv_heads > INT32_MAX)
    return fail(KVARN_EINVAL, "n_tokens and (n_tokens / 128) * num_kv_heads must be below 2^31 (got %lld)",
                (long long)n_tokens);
  KV_TRY(need_ptr(k, "k"));
  KV_TRY(need_ptr(v, "v"));
  KV_TRY(need_ptr(slot_mapping, "slot_mapping"));
  KV_TRY(need_ptr(cache, "cache"));
  if (meta->num_blocks == 0) return fail(KVARN_EINVAL, "num_blocks is 0");
  unsigned* fl = nullptr;
  KV_TRY(flags_ptr(&fl));
  return cuda_status(kvarn::launch_quantize_prefill(k, v, slot_mapping, n_tokens, meta->num_kv_heads,
                                                    meta->num_blocks, cache, meta->k_bits, meta->v_bits,
                                                    meta->layout == KVARN_LAYOUT_LEAN, meta->n_iters, meta->eps, fl,
                                                    static_cast<cudaStream_t>(stream), 0),
                     "kvarn_quantize_tiles");
}

kvarn_status kvarn_append_decode(const uint16_t* k_new, const uint16_t* v_new, const int32_t* seq_lens,
                                 int32_t* seq_lens_out, const int32_t* block_tables, int32_t n_seqs,
                                 uint16_t* workspace, uint8_t* cache, const kvarn_meta* meta, void* stream) {
  g_err[0] = 0;
  KV_TRY(check_meta(meta));
  if (n_seqs < 0) return fail(KVARN_EINVAL, "n_seqs must be >= 0 (got %lld)", (long long)n_seqs);
  if (n_seqs == 0) return KVARN_OK;
  KV_TRY(need_ptr(k_new, "k_new"));
  KV_TRY(need_ptr(v_new, "v_new"));
  KV_TRY(need_ptr(seq_lens, "seq_lens"));
  if (seq_lens_out != nullptr) KV_TRY(need_ptr(seq_lens_out, "seq_lens_out"));
  if (seq_lens_out == seq_lens) return fail(KVARN_EINVAL, "seq_lens_out must not alias seq_lens");
  KV_TRY(need_ptr(block_tables, "block_tables"));
  KV_TRY(need_ptr(workspace, "workspace"));
  KV_TRY(need_ptr(cache, "cache"));
  if (meta->max_blocks_per_seq < 1) return fail(KVARN_EINVAL, "max_blocks_per_seq must be >= 1");
  unsigned* fl = nullptr;
  KV_TRY(flags_ptr(&fl));
  return cuda_status(kvarn::launch_append(k_new, v_new, seq_lens, seq_lens_out, block_tables, n_seqs,
                                          meta->num_kv_heads, meta->max_blocks_per_seq, meta->num_blocks,
                                          workspace, cache, meta->k_bits, meta->v_bits,
                                          meta->layout == KVARN_LAYOUT_LEAN, meta->n_iters, meta->eps, fl,
                                          static_cast<cudaStream_t>(stream)),
                     "kvarn_append_decode");
}

kvarn_status kvarn_decode_attention(const uint16_t* q, const uint8_t* cache, const uint16_t* workspace,
                                    const int32_t* block_tables, const int32_t* seq_lens, int32_t n_seqs,
                                    uint16_t* out, void* scratch, size_t scratch_bytes, const kvarn_meta* meta,
                                    void* stream) {
  g_err[0] = 0;
  KV_TRY(check_meta(meta));
  if (n_seqs < 0) return fail(KVARN_EINVAL, "n_seqs must be >= 0 (got %lld)", (long long)n_seqs);
  if (n_seqs == 0) return KVARN_OK;
  if (n_seqs > 65535) return fail(KVARN_EINVAL, "n_seqs must be <= 65535 (got %lld)", (long long)n_seqs);
  KV_TRY(need_ptr(q, "q"));
  KV_TRY(need_ptr(seq_lens, "seq_lens"));
  KV_TRY(need_ptr(out, "out"));
  if (meta->max_blocks_per_seq > 0) {
    KV_TRY(need_ptr(cache, "cache"));
    KV_TRY(need_ptr(block_tables, "block_tables"));
  }
  if (workspace != nullptr) KV_TRY(need_ptr(workspace, "workspace"));
  const size_t need = kvarn::decode_part_bytes(n_seqs, meta->num_kv_heads, meta->max_blocks_per_seq);
  if (need > 0) {
    KV_TRY(need_ptr(scratch, "scratch"));
    if (scratch_bytes < need)
      return fail(KVARN_ESCRATCH, "scratch too small: need %lld bytes", static_cast<long long>(need));
  }
  unsigned* fl = nullptr;
  KV_TRY(flags_ptr(&fl));
  return cuda_status(kvarn::launch_decode(q, cache, workspace, block_tables, seq_lens, n_seqs, meta->num_kv_heads,
                                          meta->num_q_heads / meta->num_kv_heads, meta->max_blocks_per_seq,
                                          meta->num_blocks, meta->k_bits, meta->v_bits,
                                          meta->layout == KVARN_LAYOUT_LEAN, out, scratch, fl,
                                          static_cast<cudaStream_t>(stream)),
                     "kvarn_decode_attention");
}

kvarn_status kvarn_serve_step(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* seq_lens, int32_t* seq_lens_out, const int32_t* block_tables,
                              int32_t n_seqs, uint16_t* workspace, uint8_t* cache, uint16_t* out, void* scratch,
                              size_t scratch_bytes, const kvarn_meta* meta, void* stream) {
  g_err[0] = 0;
  KV_TRY(check_meta(meta));
  if (n_seqs < 0 || n_seqs > 65535) return fail(KVARN_EINVAL, "n_seqs must be in 0..65535 (got %lld)", (long long)n_seqs);
  if (n_seqs == 0) return KVARN_OK;
  KV_TRY(need_ptr(q, "q"));
  KV_TRY(need_ptr(k_new, "k_new"));
  KV_TRY(need_ptr(v_new, "v_new"));
  KV_TRY(need_ptr(seq_lens, "seq_lens"));
  KV_TRY(need_ptr(seq_lens_out, "seq_lens_out"));
  if (seq_lens_out == seq_lens) return fail(KVARN_EINVAL, "seq_lens_out must not alias seq_lens");
  KV_TRY(need_ptr(block_tables, "block_tables"));
  KV_TRY(need_ptr(workspace, "workspace"));
  KV_TRY(need_ptr(cache, "cache"));
  KV_TRY(need_ptr(out, "out"));
  if (meta->max_blocks_per_seq < 1) return fail(KVARN_EINVAL, "max_blocks_per_seq must be >= 1");
  const size_t need = kvarn::decode_part_bytes(n_seqs, meta->num_kv_heads, meta->max_blocks_per_seq);
  KV_TRY(need_ptr(scratch, "scratch"));
  if (scratch_bytes < need)
    return fail(KVARN_ESCRATCH, "scratch too small: need %lld bytes", static_cast<long long>(need));
  unsigned* fl = nullptr;
  KV_TRY(flags_ptr(&fl));
  return cuda_status(kvarn::launch_serve_step(q, k_new, v_new, seq_lens, seq_lens_out, block_tables, workspace,
                                              cache, n_seqs, meta->num_kv_heads,
                                              meta->num_q_heads / meta->num_kv_heads, meta->max_blocks_per_seq,
                                              meta->num_blocks, meta->k_bits, meta->v_bits,
                                              meta->layout == KVARN_LAYOUT_LEAN, meta->n_iters, meta->eps, out,
                                              scratch, fl, static_cast<cudaStream_t>(stream)),
                     "kvarn_serve_step");
}

kvarn_status kvarn_prefill_attention(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                     const int32_t* cu_tokens, const int32_t* seq_lens, int32_t n_seqs,
                                     int32_t max_chunk, const int32_t* block_tables, const uint8_t* cache,
                                     const uint16_t* workspace, uint16_t* out, const kvarn_meta* meta,
                                     void* stream) {
  g_err[0] = 0;
  KV_TRY(check_meta(meta));
  if (n_seqs < 0 || n_seqs > 65535) return fail(KVARN_EINVAL, "n_seqs must be in 0..65535 (got %lld)", (long long)n_seqs);
  if (max_chunk < 0) return fail(KVARN_EINVAL, "max_chunk must be >= 0 (got %lld)", (long long)max_chunk);
  if (n_seqs == 0 || max_chunk == 0) return KVARN_OK;
  KV_TRY(need_ptr(q, "q"));
  KV_TRY(need_ptr(k_new, "k_new"));
  KV_TRY(need_ptr(v_new, "v_new"));
  KV_TRY(need_ptr(cu_tokens, "cu_tokens"));
  KV_TRY(need_ptr(seq_lens, "seq_lens"));
  KV_TRY(need_ptr(out, "out"));
  if (meta->max_blocks_per_seq > 0) {
    KV_TRY(need_ptr(cache, "cache"));
    KV_TRY(need_ptr(block_tables, "block_tables"));
  }
  if (workspace != nullptr) KV_TRY(need_ptr(workspace, "workspace"));
  unsigned* fl = nullptr;
  KV_TRY(flags_ptr(&fl));
  return cuda_status(kvarn::launch_prefill(q, k_new, v_new, cu_tokens, seq_lens, block_tables, cache, workspace,
                                           n_seqs, max_chunk, meta->num_kv_heads,
                                           meta->num_q_heads / meta->num_kv_heads, meta->max_blocks_per_seq,
                                           meta->num_blocks, meta->k_bits, meta->v_bits,
                                           meta->layout == KVARN_LAYOUT_LEAN, out, fl,
                                           static_cast<cudaStream_t>(stream)),
                     "kvarn_prefill_attention");
}

kvarn_status kvarn_check_bounded_waits(int32_t which, uint32_t limit_us, void* scratch, size_t scratch_bytes,
                                       void* stream) {
  g_err[0] = 0;
  if (which != KVARN_WAIT_MBARRIER && which != KVARN_WAIT_GRID)
    return fail(KVARN_EINVAL, "which must be KVARN_WAIT_MBARRIER or KVARN_WAIT_GRID (got %lld)", (long long)which);
  if (limit_us < 1 || limit_us > 1000000)
    return fail(KVARN_EINVAL, "limit_us must be in 1..1000000 (got %llu)", (unsigned long long)limit_us);
  if (which == KVARN_WAIT_GRID) {
    KV_TRY(need_ptr(scratch, "scratch"));
    if (scratch_bytes < 8) return fail(KVARN_ESCRATCH, "scratch too small: need 8 bytes");
  }
  unsigned* fl = nullptr;
  KV_TRY(flags_ptr(&fl));
  return cuda_status(kvarn::launch_wait_selftest(which, 1000ull * limit_us, scratch, fl,
                                                 static_cast<cudaStream_t>(stream)),
                     "kvarn_check_bounded_waits");
}

kvarn_status kvarn_device_flags(uint32_t* flags, void* stream) {
  g_err[0] = 0;
  if (flags == nullptr) return fail(KVARN_EINVAL, "flags is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e, "kvarn_device_flags: synchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_flags, sizeof(v));
  if (e != cudaSuccess) return cuda_status(e, "kvarn_device_flags: read");
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_device_flags, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_status(e, "kvarn_device_flags: clear");
  *flags = v;
  return KVARN_OK;
}

const char* kvarn_last_error(void) { return g_err; }

}  // extern "C"

// ---------------------------------------------------------------- internal accessors
// Used by other translation units of the library (not part of the C ABI).
namespace kvarn {

// The flag word's address on the current device, looked up on the first call per
// device and kept (later calls, e.g. inside a CUDA-graph capture, make no lookup).
cudaError_t flags_device_ptr(unsigned** out) {
  static std::mutex mu;
  static void* known[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cacheable = dev >= 0 && dev < 64;
  std::lock_guard<std::mutex> lock(mu);
  if (cacheable && known[dev] != nullptr) {
    *out = static_cast<unsigned*>(known[dev]);
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_flags);
  if (e != cudaSuccess) return e;
  if (cacheable) known[dev] = p;
  *out = static_cast<unsigned*>(p);
  return cudaSuccess;
}

kvarn_status set_error(kvarn_status st, const char* msg) {
  snprintf(g_err, sizeof(g_err), "%s", msg);
  return st;
}

void clear_error() { g_err[0] = 0; }

kvarn_status check_meta_status(const kvarn_meta* meta) { return check_meta(meta); }

kvarn_status check_device_ptr(const void* p, const char* name) { return need_ptr(p, name); }

}  // namespace kvarn
