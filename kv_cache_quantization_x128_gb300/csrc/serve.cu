// One serving step of KVarN in a single launch: append one token per sequence to
// the fp16 decode workspace, quantize every tile the append completes into its
// paged block (KVarN README, "How KVarN works", stages 2-4, and the capacity tip's
// small fixed decode workspace), then paged GQA decode attention over the packed
// tiles plus the workspace tokens.
//
// A cooperative launch of one 256-thread CTA per SM runs three phases separated by
// grid-wide barriers (all CTAs are co-resident, so the barriers cannot wait on a
// CTA that never starts; each wait is bounded and reports KVARN_FLAG_WAIT_TIMEOUT):
//   A. CTA c takes items (sequence, kv-head) c, c + grid, ...: its threads copy the
//      new K and V rows into the workspace; an item whose tile the token completes
//      loads the workspace tile into shared memory (128-byte swizzled, K-major),
//      forms D1 = H X^T and D2 = X H on the tensor core into TMEM and quantizes it
//      with the same per-group code as the tile quantization kernel (one group of
//      8 warps, keys then values), storing the record parts with bulk copies.
//      CTA 0 also writes the per-sequence prefix of full tiles after the append.
//   B. the split phase of the decode (stream-K ranges of tiles per warp);
//   C. the merge of partial records with the workspace tokens, each warp taking
//      (sequence, kv-head, q-head) items on its own.
// Results are the same as kvarn_append_decode followed by kvarn_decode_attention.
#include <cuda.h>

#include <atomic>

#include "decode_tile.cuh"
#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_tc.cuh"
#include "quantize_group.cuh"

namespace kvarn {
namespace {

constexpr int kServeThreads = 256;
constexpr int kListCap = 16384;           // items whose tile completes, per CTA (at most)
constexpr int kOpBytes = kB * kD * 2;   // one fp16 128 x 128 operand (32 KB)

struct ServeArgs {
  DecodeArgs a;                // decode view; a.seq_lens = the lengths after the append
  unsigned* barrier;           // grid barrier words [arrivals, generation] in the caller's
                               // scratch, zeroed on the stream before every launch
  const uint16_t* k_new;       // [n_seqs][hkv][128] fp16
  const uint16_t* v_new;
  const int32_t* seq_lens_in;  // lengths before the append
  int32_t* seq_lens_out;
  uint16_t* ws;                // [n_seqs][hkv][2][128][128] fp16
  uint8_t* cache;              // the cache the append writes (a.cache reads it)
  uint16_t* out;               // [n_seqs][hq][128] fp16
  int n_iters;
  float eps;
};

// Shared memory: phase A (operands, stages, vectors, barrier, TMEM slot, scan
// scratch), then reused by the split stages and the merge scores.
template <int KB, int VB, bool kLean>
struct ServeSmem {
  static constexpr int kOffH = 0;
  static constexpr int kOffX = kOpBytes;
  static constexpr int kStageBytes = kD * kB * (KB > VB ? KB : VB) / 8 + 1024;
  static constexpr int kOffStage = 2 * kOpBytes;                    // [K, V]
  static constexpr int kOffVec = kOffStage + 2 * kStageBytes;
  static constexpr int kOffBar = kOffVec + kNumVec * kVec * 4;
  static constexpr int kOffTmem = kOffBar + 8;
  static constexpr int kOffScan = kOffTmem + 8;                     // int64 [256]
  static constexpr int kOffListN = kOffScan + kServeThreads * 8;    // int32: completed tiles listed
  static constexpr int kOffList = kOffListN + 16;                   // int32 [kListCap] item indices
  static constexpr int kAppendBytes = kOffList + kListCap * 4;
  static constexpr int kSplitBytes = SplitCfg2<KB, VB, kLean>::kSmem;
  static constexpr int kMergeBytes = static_cast<int>(sizeof(WsPart)) + kMaxCtas * kMaxWarps * 2 * 8;   // workspace part, range copy
  static constexpr int kBytes = kAppendBytes > kSplitBytes ? (kAppendBytes > kMergeBytes ? kAppendBytes : kMergeBytes)
                                                           : (kSplitBytes > kMergeBytes ? kSplitBytes : kMergeBytes);
  static_assert(kBytes <= 232448, "serving-step shared memory");
  static_assert(kOffStage % 1024 == 0 && kOffVec % 16 == 0 && kOffBar % 8 == 0 && kOffScan % 8 == 0, "align");
};

// All CTAs of the grid meet here. `barrier` = [arrivals, generation], zero before the
// launch's first barrier; the last CTA to arrive resets the arrivals and advances the
// generation. A CTA that waits longer than `limit_ns` raises KVARN_FLAG_WAIT_TIMEOUT
// and gets false: it must not start the next phase (its inputs may not be ready), so
// the caller returns. The words live in the call's own scratch, so a timeout in one
// call cannot disturb the barriers of another.
__device__ bool grid_sync(unsigned* barrier, unsigned n_ctas, unsigned* flags,
                          unsigned long long limit_ns = kWaitNs) {
  bool ok = true;
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* gen = &barrier[1];
    const unsigned g0 = *gen;   // read before arriving: it cannot advance without this CTA
    __threadfence();
    if (atomicAdd(&barrier[0], 1u) + 1u == n_ctas) {
      atomicExch(&barrier[0], 0u);
      __threadfence();
      atomicAdd(&barrier[1], 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (*gen == g0) {
        if (global_ns() - t0 > limit_ns) {
          raise_flag(flags, KVARN_FLAG_WAIT_TIMEOUT);
          ok = false;
          break;
        }
        __nanosleep(100);
      }
    }
    __threadfence();
  }
  return __syncthreads_and(ok) != 0;   // thread 0's result, for the whole CTA
}

// Length of sequence s after the append (a negative length is left as it is).
__device__ __forceinline__ int len_after(const ServeArgs& sa, int s) {
  const int L = sa.seq_lens_in[s];
  return L >= 0 ? L + 1 : L;
}

// CTA 0: exclusive prefix of full tiles per sequence after the append (the decode
// scan, from the lengths the append writes).
__device__ void serve_scan(const ServeArgs& sa, int64_t* part_sums) {
  const DecodeArgs& a = sa.a;
  const int t = threadIdx.x;
  const int per = (a.n_seqs + kServeThreads - 1) / kServeThreads;
  const int s0 = min(t * per, a.n_seqs), s1 = min(s0 + per, a.n_seqs);
  int64_t sum = 0;
  bool clipped = false;
  for (int s = s0; s < s1; ++s) {
    const int L = max(len_after(sa, s), 0);
    sum += min(L / kB, a.max_blocks);
    clipped |= L / kB > a.max_blocks;
  }
  if (clipped) raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
  part_sums[t] = sum;
  __syncthreads();
  for (int off = 1; off < kServeThreads; off <<= 1) {   // inclusive scan of the chunk sums
    const int64_t v = t >= off ? part_sums[t - off] : 0;
    __syncthreads();
    part_sums[t] += v;
    __syncthreads();
  }
  int64_t run = t > 0 ? part_sums[t - 1] : 0;
  for (int s = s0; s < s1; ++s) {
    a.prefix[s] = run;
    run += min(max(len_after(sa, s), 0) / kB, a.max_blocks);
  }
  if (t == kServeThreads - 1) a.prefix[a.n_seqs] = part_sums[kServeThreads - 1];
  // no unit has a first or last split warp yet (the split phase marks them)
  const int64_t n_cover = 2 * static_cast<int64_t>(a.n_seqs) * a.hkv;
  for (int64_t i = t; i < n_cover; i += kServeThreads) a.cover[i] = -1;
}

// Phase A for the items of this CTA.
template <int KB, int VB, bool kLean>
__device__ void serve_append(const ServeArgs& sa, uint8_t* smem) {
  using S = ServeSmem<KB, VB, kLean>;
  using L = RecordLayout<KB, VB, kLean>;
  const DecodeArgs& a = sa.a;
  const int tid = threadIdx.x;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffTmem);
  float* vec = reinterpret_cast<float*>(smem + S::kOffVec);
  uint8_t* xt = smem + S::kOffX;

  fill_hadamard_sw128(smem + S::kOffH, tid, kServeThreads);   // the +-1 Hadamard operand
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 256);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (blockIdx.x == 0) serve_scan(sa, reinterpret_cast<int64_t*>(smem + S::kOffScan));

  // this thread's half line in TMEM (as in the tile quantization kernel, group 0)
  const int gw = tid >> 5, t = tid & 31;
  const uint32_t lane0 = 32 * (gw & 3) + 16 * (gw >> 2);
  const int line = static_cast<int>(lane0) + (t >> 2) + 8 * (t & 1);
  const int p = (t >> 1) & 1;
  const uint32_t d1 = tmem_addr(tmem, 0, 0), d2 = d1 + 128;
  const uint32_t ta1 = tmem_addr(tmem, lane0, 0), ta2 = ta1 + 128;
  const uint32_t sh = smem_u32(smem + S::kOffH), sx = smem_u32(xt);
  constexpr uint32_t kIdesc = idesc_f16_f32(128, 128);

  uint32_t parity = 0;
  bool alive = true;          // no wait of this CTA has timed out
  bool mma_pending = false;   // thread 0: products whose completion was not seen
  uint32_t pending_parity = 0;
  const int64_t n_items = static_cast<int64_t>(a.n_seqs) * a.hkv;
  // The CTA's items w = c + grid * k: whole warps copy the new rows into the workspace
  // and list the items whose tile the token completes (with a valid block).
  int* list_n = reinterpret_cast<int*>(smem + S::kOffListN);
  int* list = reinterpret_cast<int*>(smem + S::kOffList);
  if (tid == 0) *list_n = 0;
  __syncthreads();
  {
    const int warp = tid >> 5, lane = tid & 31;
    for (int64_t w = blockIdx.x + static_cast<int64_t>(gridDim.x) * warp; w < n_items;
         w += static_cast<int64_t>(gridDim.x) * (kServeThreads / 32)) {
      const int s = static_cast<int>(w / a.hkv), h = static_cast<int>(w - static_cast<int64_t>(s) * a.hkv);
      const int Lin = sa.seq_lens_in[s];
      if (lane == 0 && h == 0) sa.seq_lens_out[s] = len_after(sa, s);
      if (Lin < 0) continue;
      {   // K (lanes 0-15) and V (16-31) rows of the new token, 16 bytes a lane
        const int g = lane >> 4, c = lane & 15;
        const uint16_t* src = (g ? sa.v_new : sa.k_new) + w * kD + c * 8;
        uint16_t* dst = sa.ws + ((w * 2 + g) * kB + Lin % kB) * kD + c * 8;
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      }
      if (lane != 0 || Lin % kB != kB - 1) continue;   // the tile is not complete yet
      const int bi = Lin / kB;
      if (bi >= a.max_blocks) {
        raise_flag(a.flags, KVARN_FLAG_BAD_LENGTH);
        continue;
      }
      const int64_t blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + bi];
      if (blk < 0 || blk >= a.num_blocks) {
        raise_flag(a.flags, KVARN_FLAG_BAD_BLOCK);
        continue;
      }
      const int k = atomicAdd(list_n, 1);
      if (k < kListCap) list[k] = static_cast<int>(w);   // the host keeps items per CTA within kListCap
    }
  }
  __syncthreads();   // the new rows are in the workspace, the list is complete
  const int n_list = min(*list_n, kListCap);
  for (int li = 0; li < n_list && alive; ++li) {
    const int64_t w = list[li];
    const int s = static_cast<int>(w / a.hkv), h = static_cast<int>(w - static_cast<int64_t>(s) * a.hkv);
    const int64_t blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + sa.seq_lens_in[s] / kB];
    uint8_t* rec = sa.cache + (blk * a.hkv + h) * static_cast<int64_t>(L::kBytes);
#pragma unroll 1
    for (int g = 0; g < 2; ++g) {
      // workspace tile (tokens x channels) into the swizzled operand: 16-byte chunk
      // c of row r goes where the TMA box of 64 channels would put it
      const uint16_t* tile = sa.ws + (w * 2 + g) * static_cast<int64_t>(kB * kD);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = tid + k * kServeThreads;   // chunk index, 16 per row
        const int r = e >> 4, c = e & 15;
        *reinterpret_cast<uint4*>(xt + sw_offset(r, 8 * c)) = *reinterpret_cast<const uint4*>(tile + r * kD + 8 * c);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t dh = smem_desc_sw128(sw_kstep(sh, k));
          const uint64_t dx = smem_desc_sw128(sw_kstep(sx, k));
          umma_f16(d1, dh, dx, kIdesc, k > 0);   // D1[i][j] = sum_k H[i][k] X[j][k]
          umma_f16(d2, dx, dh, kIdesc, k > 0);   // D2[j][i] = sum_k X[j][k] H[i][k]
        }
        umma_commit(bar);
      }
      bool ok = mbar_wait(bar, parity, a.flags);
      if (!ok && tid == 0) {
        mma_pending = true;
        pending_parity = parity;
      }
      parity ^= 1;
      tc_fence_after();
      uint8_t* stage = smem + S::kOffStage + g * S::kStageBytes;
      if (g == 0)
        ok = quantize_group<0, KB, kLean>(vec, stage, xt, ta1, ta2, line, p, sa.n_iters, sa.eps, 1, ok);
      else
        ok = quantize_group<1, VB, kLean>(vec, stage, xt, ta1, ta2, line, p, sa.n_iters, sa.eps, 1, ok);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (!ok) {   // a wait timed out (flag raised): the tensor core may still be busy
        alive = false;
        break;
      }
      if (tid == 0) {
        if (g == 0) {
          bulk_s2g(rec + L::kKCodeOff, stage, L::kKCodeBytes);
          bulk_s2g(rec + L::kKMetaOff, stage + L::kKCodeBytes, L::kMetaBytes);
        } else {
          bulk_s2g(rec + L::kVCodeOff, stage, L::kVCodeBytes);
          bulk_s2g(rec + L::kVMetaOff, stage + L::kVCodeBytes, L::kMetaBytes);
        }
        bulk_commit();
      }
    }
    if (tid == 0) bulk_wait_all();   // the stages are free and the records written
    __syncthreads();
  }
  if (tid == 0) {
    // after a timeout: let the products in flight finish (bounded) before the TMEM
    // and the shared memory are released
    if (mma_pending) mma_pending = !mbar_wait(bar, pending_parity, a.flags);
    bulk_wait_all();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    if (!mma_pending) mbar_inval(bar);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid < 32) tmem_dealloc(tmem, 256);
}

template <int KB, int VB, bool kLean>
__global__ void __launch_bounds__(kServeThreads, 1) serve_step_kernel(const ServeArgs sa) {
  extern __shared__ __align__(1024) uint8_t smem[];
  serve_append<KB, VB, kLean>(sa, smem);
  if (!grid_sync(sa.barrier, gridDim.x, sa.a.flags)) return;   // timed out (flag raised)
  // records written through the async proxy by other CTAs are read the same way
  asm volatile("fence.proxy.async.global;" ::: "memory");
  if (sa.a.max_blocks > 0) split_body<KB, VB, kLean, SplitCfg2<KB, VB, kLean>>(sa.a, smem, blockIdx.x);
  if (!grid_sync(sa.barrier, gridDim.x, sa.a.flags)) return;
  // merge: the block takes (sequence, kv-head) units in turn with its 8 warps; the
  // split warps' ranges are copied to shared memory for the record lookups
  WsPart& wsp = *reinterpret_cast<WsPart*>(smem);
  int64_t* rg = reinterpret_cast<int64_t*>(smem + sizeof(WsPart));
  const int n_range = 2 * sa.a.n_ctas * sa.a.warps;
  for (int i = threadIdx.x; i < n_range; i += kServeThreads) rg[i] = sa.a.ranges[i];
  __syncthreads();
  const int64_t n_units = static_cast<int64_t>(sa.a.n_seqs) * sa.a.hkv;
  for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int s = static_cast<int>(u / sa.a.hkv), h = static_cast<int>(u - static_cast<int64_t>(s) * sa.a.hkv);
    merge_body<8, 1>(sa.a, sa.ws, sa.out, h, s, wsp, nullptr, rg);
    __syncthreads();   // the next unit's workspace part reuses wsp
  }
}

template <int KB, int VB, bool kLean>
cudaError_t launch_serve_bits(const ServeArgs& sa, int grid, cudaStream_t stream) {
  using S = ServeSmem<KB, VB, kLean>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(serve_step_kernel<KB, VB, kLean>, S::kBytes, smem_set);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kServeThreads);
  cfg.dynamicSmemBytes = S::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, serve_step_kernel<KB, VB, kLean>, sa);
}

// Self-test of the bounded waits: waits that can never complete, each with a
// `limit_ns` limit. which = 0: every thread waits on an mbarrier whose phase expects
// 16 bytes that no copy delivers. which = 1: a cooperative grid whose barrier
// expects one CTA more than were launched. Either way each wait gives up, raises
// KVARN_FLAG_WAIT_TIMEOUT and the kernel returns; no copy or MMA is in flight.
__global__ void __launch_bounds__(32) wait_selftest_mbar_kernel(unsigned* flags, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar, 16);
  __syncwarp();
  mbar_wait(&bar, 0, flags, limit_ns);
}

__global__ void __launch_bounds__(32) wait_selftest_grid_kernel(unsigned* barrier, unsigned* flags,
                                                                unsigned long long limit_ns) {
  grid_sync(barrier, gridDim.x + 1, flags, limit_ns);
}

}  // namespace

size_t serve_barrier_offset(int n_seqs, int hkv, int max_blocks) {
  return decode_part_bytes(n_seqs, hkv, max_blocks) - kServeBarrierBytes;
}

unsigned* serve_barrier_words(void* scratch, int n_seqs, int hkv, int max_blocks) {
  return reinterpret_cast<unsigned*>(static_cast<uint8_t*>(scratch) + serve_barrier_offset(n_seqs, hkv, max_blocks));
}

cudaError_t launch_wait_selftest(int which, unsigned long long limit_ns, void* barrier_words, unsigned* flags,
                                 cudaStream_t stream) {
  if (which == 0) {
    wait_selftest_mbar_kernel<<<1, 32, 0, stream>>>(flags, limit_ns);
    return cudaGetLastError();
  }
  if (which != 1) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t err = cudaMemsetAsync(barrier_words, 0, 2 * sizeof(unsigned), stream);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms > 0 ? sms : 1));
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  unsigned* words = static_cast<unsigned*>(barrier_words);
  return cudaLaunchKernelEx(&cfg, wait_selftest_grid_kernel, words, flags, limit_ns);
}

cudaError_t launch_serve_step(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* seq_lens, int32_t* seq_lens_out, const int32_t* block_tables,
                              uint16_t* ws, uint8_t* cache, int n_seqs, int hkv, int group, int max_blocks,
                              int64_t num_blocks, int k_bits, int v_bits, bool lean, int n_iters, float eps,
                              uint16_t* out, void* scratch, unsigned* flags, cudaStream_t stream) {
  if (n_seqs <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms > 0 ? (sms < kMaxCtas ? sms : kMaxCtas) : 1;
  if ((static_cast<int64_t>(n_seqs) * hkv + grid - 1) / grid > kListCap) return cudaErrorInvalidValue;
  ServeArgs sa;
  DecodeArgs& a = sa.a;
  a.q = q;
  a.cache = cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens_out;
  a.prefix = static_cast<int64_t*>(scratch);
  a.ranges = reinterpret_cast<int64_t*>(static_cast<uint8_t*>(scratch) + prefix_bytes(n_seqs));
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + prefix_bytes(n_seqs) + kRangeBytes);
  a.flags = flags;
  a.num_blocks = num_blocks;
  a.n_seqs = n_seqs;
  a.hkv = hkv;
  a.group = group;
  a.max_blocks = max_blocks;
  a.n_ctas = grid;
  a.cover = cover_ptr(a.part, n_seqs, hkv, grid);
  sa.k_new = k_new;
  sa.v_new = v_new;
  sa.seq_lens_in = seq_lens;
  sa.seq_lens_out = seq_lens_out;
  sa.ws = ws;
  sa.cache = cache;
  sa.out = out;
  sa.n_iters = n_iters;
  sa.eps = eps;
  sa.barrier = serve_barrier_words(scratch, n_seqs, hkv, max_blocks);
  const cudaError_t zero = cudaMemsetAsync(sa.barrier, 0, 2 * sizeof(unsigned), stream);
  if (zero != cudaSuccess) return zero;
  if (k_bits == 4 && v_bits == 2 && !lean) {
    a.warps = SplitCfg2<4, 2>::kWarps;
    return launch_serve_bits<4, 2, false>(sa, grid, stream);
  }
  if (k_bits == 4 && v_bits == 2 && lean) {
    a.warps = SplitCfg2<4, 2, true>::kWarps;
    return launch_serve_bits<4, 2, true>(sa, grid, stream);
  }
  if (k_bits == 4 && v_bits == 4 && !lean) {
    a.warps = SplitCfg2<4, 4>::kWarps;
    return launch_serve_bits<4, 4, false>(sa, grid, stream);
  }
  if (k_bits == 2 && v_bits == 2 && !lean) {
    a.warps = SplitCfg2<2, 2>::kWarps;
    return launch_serve_bits<2, 2, false>(sa, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvarn
