// KVarN paged decode attention over the packed cache (KVarN README, "How KVarN
// works": the scales are re-applied on read; the orthonormal rotation keeps
// attention scores, so q is rotated by the same H and the output un-rotated).
//
// Three launches:
//   decode_scan_kernel  - exclusive prefix of full tiles per sequence (scratch),
//     and every unit's first / last split-warp marks reset to -1;
//   decode_split_kernel - persistent, one CTA per SM. The flattened tile space
//     (sequence, kv-head, tile) is cut into one contiguous range per warp
//     (stream-K), so ragged batches balance to a tile. Each warp streams its range
//     through private record-sized (14336 bytes for k4v2) bulk-copy stages: one
//     stage in 12 warps (10 for k4v4) with the tile after next prefetched into L2,
//     for many (sequence, kv-head) units; two stages in 8 warps (6 for k4v4) for at
//     most as many units as SMs. It runs its GQA group (up to 8 q-heads) on
//     m16n8k16 tensor-core MMAs, with an online softmax in the log2 domain:
//       QK^T: A = q' = q_r r^K s^K per channel, fp16 hi part in rows 0-7 and fp16
//             lo part in rows 8-15 (q' carried to ~22 bits), B = 4-bit key codes
//             turned into fp16 in registers; score_j = c^K_j (D_hi + D_lo + beta),
//             beta = sum_i q_r,i r^K_i z^K_i;
//       PV:   A = p' = p_j c^V_j s^V_j (hi/lo rows), B = 2-bit value codes;
//             acc_i += r^V_i (D_hi + D_lo + gamma), gamma = sum_j p_j c^V_j z^V_j.
//     Four independent accumulator chains keep the MMA pipe busy. When a warp's
//     range crosses into a new (sequence, kv-head) it writes a partial record
//     (acc, running max, running sum) for the one it leaves; the warp that takes a
//     unit's first tile and the one that takes its last mark themselves;
//   decode_merge_kernel - per (sequence, kv-head): attends the fp16 workspace
//     tokens of the partial last tile (m16n8k16 MMAs over all q-heads of the
//     group), merges them online with the partial records of the warps between
//     those marks, un-rotates the records' part by H^T and normalises.
// decode_tc_split_kernel (decode_tc.cuh) is the split phase on tcgen05 for k4v2,
// chosen with KVARN_DECODE_SPLIT=tc; it writes the same partial records. The split
// and merge kernels are launched as programmatic dependents of the kernel before
// them, so their launch overlaps its tail.
#include <cstdlib>
#include <cstring>

#include "decode_tc.cuh"
#include "decode_tile.cuh"
#include "kvarn_common.cuh"
#include "kvarn_launch.h"

namespace kvarn {
namespace {

// Programmatic dependent launch: a kernel launched with the attribute may start
// while its predecessor in the stream runs; it waits for the predecessor's
// completion (and memory) before touching its outputs. Without the attribute both
// instructions do nothing.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ scan
// Exclusive prefix of full tiles per sequence: each thread a contiguous chunk of
// sequences, then a warp-shuffle scan and a scan of the 32 warp totals.
__global__ void __launch_bounds__(1024) decode_scan_kernel(DecodeArgs a) {
  griddep_launch_dependents();          // the split kernel waits for this grid itself
  __shared__ int64_t warp_sums[32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int per = (a.n_seqs + 1023) / 1024;
  const int s0 = min(t * per, a.n_seqs), s1 = min(s0 + per, a.n_seqs);
  int64_t sum = 0;
  bool clipped = false;
  for (int s = s0; s < s1; ++s) {
    sum += full_tiles(a, s);
    clipped |= max(a.seq_lens[s], 0) / kB > a.max_blocks;
  }
  if (clipped) raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
  int64_t incl = sum;                   // inclusive scan inside the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {                         // inclusive scan of the warp totals
    int64_t v = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    warp_sums[lane] = v;
  }
  __syncthreads();
  int64_t run = incl - sum + (w > 0 ? warp_sums[w - 1] : 0);
  for (int s = s0; s < s1; ++s) {
    a.prefix[s] = run;
    run += full_tiles(a, s);
  }
  if (t == 1023) a.prefix[a.n_seqs] = warp_sums[31];
  // no unit has a first or last split warp yet (the split kernel marks them)
  const int64_t n_cover = 2 * static_cast<int64_t>(a.n_seqs) * a.hkv;
  for (int64_t i = t; i < n_cover; i += 1024) a.cover[i] = -1;
}

template <int KB, int VB, bool kLean, class Cfg>
__global__ void __launch_bounds__(Cfg::kWarps * 32, 1) decode_split_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_launch_dependents();          // the merge kernel waits for this grid itself
  griddep_wait();                       // the scan's prefix
  split_body<KB, VB, kLean, Cfg>(a, smem, blockIdx.x);
}

template <bool kLean>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_split_kernel(DecodeArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  decode_tc_body<kLean>(a);
}

// The merge kernel's wait for the split kernel (its ranges, marks and records).
struct SplitWait {
  static constexpr bool kReady = false;
  __device__ void operator()() const { griddep_wait(); }
};

// One CTA of 8 kParts warps per (kv-head, sequence). For batches of many short units
// (a few partial records each): kParts 1 and kMinBlocks 4, so that 4 CTAs (at 64
// registers) share an SM. For a few long units (tens of records each): kParts 4, the
// records of a q-head split between 4 warps.

template <int kMinBlocks, int kParts>
__global__ void __launch_bounds__(256 * kParts, kMinBlocks) decode_merge_kernel(DecodeArgs a,
                                                                               const uint16_t* __restrict__ ws,
                                                                               uint16_t* __restrict__ out) {
  __shared__ WsPart sm;
  __shared__ RecShares<kParts> rs;
  // the workspace tokens first (inputs only), then wait for the split kernel's
  // ranges and partial records
  merge_body<8, kParts, SplitWait>(a, ws, out, blockIdx.x, blockIdx.y, sm, &rs, a.ranges);
}

// Launch with programmatic stream serialization (see griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                         Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

size_t decode_part_bytes(int n_seqs, int hkv, int max_blocks) {
  (void)max_blocks;
  const size_t records = static_cast<size_t>(kMaxCtas) * kMaxWarps + static_cast<size_t>(n_seqs) * hkv;
  return prefix_bytes(n_seqs) + kRangeBytes + records * kRecFloats * sizeof(float) + cover_bytes(n_seqs, hkv) +
         kServeBarrierBytes;
}

size_t decode_scratch_bytes_for_ctas(int n_seqs, int hkv, int n_ctas) {
  const size_t records = static_cast<size_t>(n_ctas) * kMaxWarps + static_cast<size_t>(n_seqs) * hkv;
  return prefix_bytes(n_seqs) + kRangeBytes + records * kRecFloats * sizeof(float) + cover_bytes(n_seqs, hkv);
}

int decode_num_ctas() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? (sms < kMaxCtas ? sms : kMaxCtas) : 1;
}

template <int KB, int VB, bool kLean, class C>
cudaError_t launch_split_cfg(const DecodeArgs& a, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(decode_split_kernel<KB, VB, kLean, C>, C::kSmem, smem_set);
  if (err != cudaSuccess) return err;
  return launch_after(decode_split_kernel<KB, VB, kLean, C>, dim3(a.n_ctas), dim3(C::kWarps * 32), C::kSmem, stream,
                      a);
}

// The split kernel in the shape a.warps was set for (SplitCfg, or SplitCfg2 for few units).
template <int KB, int VB, bool kLean>
cudaError_t launch_split(const DecodeArgs& a, bool few_units, cudaStream_t stream) {
  return few_units ? launch_split_cfg<KB, VB, kLean, SplitCfg2<KB, VB, kLean>>(a, stream)
                   : launch_split_cfg<KB, VB, kLean, SplitCfg<KB, VB, kLean>>(a, stream);
}

template <int KB, int VB, bool kLean>
int split_warps(bool few_units) {
  return few_units ? SplitCfg2<KB, VB, kLean>::kWarps : SplitCfg<KB, VB, kLean>::kWarps;
}

template <bool kLean>
cudaError_t launch_split_tc(const DecodeArgs& a, cudaStream_t stream) {
  using C = TcCfg<kLean>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(decode_tc_split_kernel<kLean>, C::kSmem, smem_set);
  if (err != cudaSuccess) return err;
  return launch_after(decode_tc_split_kernel<kLean>, dim3(a.n_ctas), dim3(kTcThreads), C::kSmem, stream, a);
}

// The warp-level split kernel serves every preset; KVARN_DECODE_SPLIT=tc selects the
// tcgen05 one for k4v2 (measured slower: 0.51 against 0.25 ms on 64 x 16384
// tokens). Read on every call, so one process can run both.
bool use_tc_split() {
  const char* e = std::getenv("KVARN_DECODE_SPLIT");
  return e != nullptr && std::strcmp(e, "tc") == 0;
}

cudaError_t launch_decode(const uint16_t* q, const uint8_t* cache, const uint16_t* ws, const int32_t* block_tables,
                          const int32_t* seq_lens, int n_seqs, int hkv, int group, int max_blocks, int64_t num_blocks,
                          int k_bits, int v_bits, bool lean, uint16_t* out, void* scratch, unsigned* flags,
                          cudaStream_t stream) {
  if (n_seqs <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  DecodeArgs a;
  a.q = q;
  a.cache = cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.prefix = static_cast<int64_t*>(scratch);
  a.ranges = reinterpret_cast<int64_t*>(static_cast<uint8_t*>(scratch) + prefix_bytes(n_seqs));
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + prefix_bytes(n_seqs) + kRangeBytes);
  a.flags = flags;
  a.num_blocks = num_blocks;
  a.n_seqs = n_seqs;
  a.hkv = hkv;
  a.group = group;
  a.max_blocks = max_blocks;
  a.n_ctas = sms > 0 ? (sms < kMaxCtas ? sms : kMaxCtas) : 1;
  a.cover = cover_ptr(a.part, n_seqs, hkv, a.n_ctas);
  const bool k4v2 = k_bits == 4 && v_bits == 2, k4v4 = k_bits == 4 && v_bits == 4, k2v2 = k_bits == 2 && v_bits == 2;
  if (!(k4v2 || ((k4v4 || k2v2) && !lean))) return cudaErrorInvalidValue;
  const bool tc = k4v2 && use_tc_split();
  // at most as many (sequence, kv-head) units as CTAs: 8 or more partial records per
  // unit with 8 split warps per CTA
  const int64_t units = static_cast<int64_t>(n_seqs) * hkv;
  const bool few_units = units <= a.n_ctas;
  a.warps = tc ? kTcTeams
            : k4v4 ? split_warps<4, 4, false>(few_units) : k2v2 ? split_warps<2, 2, false>(few_units)
            : lean ? split_warps<4, 2, true>(few_units) : split_warps<4, 2, false>(few_units);
  decode_scan_kernel<<<1, 1024, 0, stream>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (max_blocks > 0) {
    err = tc ? (lean ? launch_split_tc<true>(a, stream) : launch_split_tc<false>(a, stream))
          : k2v2 ? launch_split<2, 2, false>(a, few_units, stream)
          : k4v4 ? launch_split<4, 4, false>(a, few_units, stream)
          : lean ? launch_split<4, 2, true>(a, few_units, stream) : launch_split<4, 2, false>(a, few_units, stream);
    if (err != cudaSuccess) return err;
  }
  // units with 8 or more partial records on average: the records of a q-head split 4 ways
  // (a unit has no more records than tiles, so short block tables never qualify)
  const bool long_units = static_cast<int64_t>(a.n_ctas) * a.warps >= 8 * units && max_blocks >= 8;
  return long_units ? launch_after(decode_merge_kernel<1, 4>, dim3(hkv, n_seqs), dim3(1024), 0, stream, a, ws, out)
                    : launch_after(decode_merge_kernel<4, 1>, dim3(hkv, n_seqs), dim3(256), 0, stream, a, ws, out);
}

}  // namespace kvarn
