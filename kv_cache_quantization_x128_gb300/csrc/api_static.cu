// kvarn_decode_attention_static: decode attention for callers that cannot
// allocate device memory. kvarn_decode_attention needs a scratch buffer from the
// caller; some callers have no way to get one: a serving engine that has handed
// all of its free device memory to a pre-reserved KV-cache pool and routes every
// other request through its own allocator, or a plain-C host with no device
// allocator of its own. This variant takes its scratch from a fixed array of
// device memory inside the library instead, and allocates nothing.
//
// The array is a file-scope __device__ variable of kStaticScratchBytes, so every
// GPU that loads the library holds it until the process exits. All calls on a
// device share it: two calls whose work overlaps on the GPU (e.g. on different
// streams without ordering) race on it and must not be issued. Nothing in it has
// to start at zero: within a call the kernels write every scratch word before
// they read it, so the contents left by the previous call are never used.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvarn.h"
#include "kvarn_launch.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device. The first call on a
// device looks it up (cudaGetSymbolAddress, with that device current) and keeps
// it; later calls reuse it.
kvarn_status static_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvarn::set_error(KVARN_ECUDA, "kvarn_decode_attention_static: no current device");
  if (dev < 0 || dev >= kMaxDevices)
    return kvarn::set_error(KVARN_EUNSUPPORTED, "kvarn_decode_attention_static: device ordinal >= 64");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr)
      return kvarn::set_error(KVARN_ECUDA, "kvarn_decode_attention_static: cudaGetSymbolAddress failed");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVARN_OK;
}

}  // namespace

extern "C" {

KVARN_API kvarn_status kvarn_decode_attention_static(const uint16_t* q, const uint8_t* cache,
                                                     const uint16_t* workspace, const int32_t* block_tables,
                                                     const int32_t* seq_lens, int32_t n_seqs, uint16_t* out,
                                                     const kvarn_meta* meta, void* stream) {
  kvarn::clear_error();
  // the same checks as kvarn_decode_attention: every preset of kvarn.h is served
  kvarn_status st = kvarn::check_meta_status(meta);
  if (st != KVARN_OK) return st;
  if (n_seqs < 0 || n_seqs > 65535) return kvarn::set_error(KVARN_EINVAL, "n_seqs must be in 0..65535");
  if (n_seqs == 0) return KVARN_OK;
  const struct {
    const void* p;
    const char* name;
  } need_aligned[] = {{q, "q"}, {seq_lens, "seq_lens"}, {out, "out"}};
  for (const auto& a : need_aligned)
    if ((st = kvarn::check_device_ptr(a.p, a.name)) != KVARN_OK) return st;
  if (meta->max_blocks_per_seq > 0) {
    if ((st = kvarn::check_device_ptr(cache, "cache")) != KVARN_OK) return st;
    if ((st = kvarn::check_device_ptr(block_tables, "block_tables")) != KVARN_OK) return st;
  }
  if (workspace != nullptr && (st = kvarn::check_device_ptr(workspace, "workspace")) != KVARN_OK) return st;

  const size_t need = kvarn::decode_scratch_bytes_for_ctas(n_seqs, meta->num_kv_heads, kvarn::decode_num_ctas());
  if (need > kStaticScratchBytes)
    return kvarn::set_error(KVARN_ESCRATCH,
                            "kvarn_decode_attention_static: n_seqs * num_kv_heads exceeds the 16 MiB built-in "
                            "scratch; use kvarn_decode_attention with a caller buffer");
  void* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != KVARN_OK) return st;
  unsigned* flags = nullptr;
  if (kvarn::flags_device_ptr(&flags) != cudaSuccess)
    return kvarn::set_error(KVARN_ECUDA, "kvarn_decode_attention_static: device flag word unavailable");
  const cudaError_t e = kvarn::launch_decode(q, cache, workspace, block_tables, seq_lens, n_seqs, meta->num_kv_heads,
                                             meta->num_q_heads / meta->num_kv_heads, meta->max_blocks_per_seq,
                                             meta->num_blocks, meta->k_bits, meta->v_bits,
                                             meta->layout == KVARN_LAYOUT_LEAN, out, scratch, flags,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return kvarn::set_error(KVARN_ECUDA, cudaGetErrorString(e));
  return KVARN_OK;
}

}  // extern "C"
