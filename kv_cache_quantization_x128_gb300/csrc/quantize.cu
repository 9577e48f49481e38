// KVarN tile quantization (KVarN README, "How KVarN works", stages 2-4):
// Hadamard rotation along channels, log-space column/row variance normalisation,
// asymmetric round-to-nearest (4-bit keys per channel, 2-bit values per token) and
// packing into the 14336-byte record documented in kvarn.h.
//
// One persistent CTA per SM, 512 threads in two independent 8-warp groups: group 0
// quantizes the K tile and group 1 the V tile of each (block, kv-head) work item.
// Per item and group:
//   1. one thread starts two 2-D TMA copies (64 channels x 128 tokens each) of the
//      next item's tile into the group's spare buffer, in the 128-byte swizzled
//      K-major layout, completing on an mbarrier;
//   2. the same thread issues tcgen05.mma twice over K = 128: D1 = H X^T (TMEM
//      lanes = channels, columns = tokens) and D2 = X H (lanes = tokens, columns =
//      channels), with H the +-1 Sylvester matrix (exact in fp16) and fp32
//      accumulation; the 1/sqrt(128) factor is folded into the statistics;
//   3. each column pass reads D2 and each row pass reads D1 straight from TMEM
//      (tcgen05.ld 16x64b: two threads per line, 64 values each), so both passes
//      are thread-local loops plus one shuffle with the partner thread; every
//      sweep (the thread's 64 values) is loaded at the end of the sweep before it,
//      so its latency overlaps the reduction, the scale update and the barrier;
//   4. fp16 scales, group extremes (keys: a sweep of D1, whose lines are the key
//      groups, needing no barrier after the last row pass; values: a sweep of D2),
//      RTN, packing into a shared-memory stage, and two bulk stores of the group's
//      part of the record.
// The groups share only the Hadamard operand and the TMEM allocation (256 columns
// each), so one group's MMA latency and barriers overlap the other's arithmetic.
// The slot check of an item is agreed on at the barrier that ends the previous one.
// The decode append runs the same kernel over (sequence, kv-head) items: the block
// first writes the new tokens of its items into the workspace, then quantizes only
// the items whose sequence completes a tile (for batches of up to kRankItems items,
// those handed to it by rank, so that blocks get equal shares of them).
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_tc.cuh"
#include "quantize_group.cuh"

namespace kvarn {
namespace {

constexpr int kThreads = 2 * kGroupThreads;
constexpr int kTileOp = kB * kD * 2;              // 32768 B: one fp16 128x128 operand
constexpr int kOffH = 0;
constexpr int kOffIn = kOffH + kTileOp;                        // [group][buf] operands
static_assert(kOffIn % 1024 == 0, "align");

// Shared-memory layout after the operands, per preset: a stage (codes + metadata)
// of each tensor sized to its bit width, double buffered. Sizing the stages to the
// preset, not to the widest one, was measured 1.5 % faster for k4v2.
// The append hands the items that complete a tile out by rank (the k-th such item to
// block k mod grid) when the batch has at most kRankItems items and no block gets more
// than kRankList of them; each block keeps its list and the per-32-item counts here.
constexpr int kRankItems = 32768;
constexpr int kRankList = 216;
constexpr int kRankBytes = kRankList * 4 + (kRankItems / 32 + 1) * 4;

template <int KB, int VB, bool kRanked = false>
struct QSmem {
  static constexpr int kStageK = kD * kB * KB / 8 + 1024;
  static constexpr int kStageV = kD * kB * VB / 8 + 1024;
  static constexpr int kOffStageK = kOffIn + 4 * kTileOp;              // [buf]
  static constexpr int kOffStageV = kOffStageK + 2 * kStageK;           // [buf]
  static constexpr int kOffVec = kOffStageV + 2 * kStageV;              // [group][vector][kVec] fp32
  static constexpr int kOffBar = kOffVec + 2 * kNumVec * kVec * 4;      // mma [group], load [group][buf]
  static constexpr int kOffTmem = kOffBar + 48;
  static constexpr int kOffRank = kOffTmem + 16;                        // append: item list, chunk prefix
  static constexpr int kBytes = kOffRank + (kRanked ? kRankBytes : 0);
  static_assert(kBytes <= 232448, "quantize shared memory");
  static_assert(kOffStageV % 16 == 0 && kOffVec % 16 == 0, "align");
};

// ------------------------------------------------------------------ work sources
// A work item w is a (tile, kv-head) pair; both sources keep w below 2^31.
// w / d for 0 <= w < 2^31 by a multiply-high (the round-up method of Granlund and
// Montgomery, "Division by invariant integers using multiplication"):
// q = (umulhi(m, w) + w) >> l, l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
// Item indices split into (chunk or sequence, kv-head) without a division routine on
// the path to the next item's products.
struct ItemDiv {
  uint32_t d, m, l;
  __device__ __forceinline__ uint32_t div(int64_t w) const {
    const uint32_t x = static_cast<uint32_t>(w);
    return (__umulhi(m, x) + x) >> l;
  }
};
inline ItemDiv make_item_div(uint32_t d) {
  uint32_t l = 0;
  while ((1u << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
  return ItemDiv{d, static_cast<uint32_t>(m), l};
}

struct PrefillSource {
  CUtensorMap map[2];   // K, V as [n_tokens rows][hkv * 128 channels] fp16
  const int64_t* slot;
  int64_t n_items;      // (n_tokens / 128) * hkv
  int hkv;
  ItemDiv hd;           // division by hkv
  int64_t num_blocks;

  static constexpr bool kSparse = false;   // every item has a tile
  __device__ int scatter_all(int, uint8_t*) const { return 0; }
  // every item has a tile: the block's next one
  __device__ int64_t next_item(int64_t w, int) const { return w + gridDim.x; }
  __device__ int64_t next_of(int64_t w, int, int lane, const uint8_t*, int) const { return next_item(w, lane); }
  // TMA coordinates (channel, token) of the item's 128 x 128 tile of tensor g
  __device__ void coords(int64_t w, int, int& x, int& y) const {
    const uint32_t chunk = hd.div(w);
    x = static_cast<int>(static_cast<uint32_t>(w) - chunk * hkv) * kD;
    y = static_cast<int>(chunk) * kB;
  }
  struct Check {
    int64_t base = -1, mine = -1;
  };
  // Slot entries this thread checks for item w, loaded one item ahead of use.
  __device__ Check prepare(int64_t w, int gt) const {
    const int64_t t0 = static_cast<int64_t>(hd.div(w)) * kB;
    Check c;
    c.base = slot[t0];
    c.mine = slot[t0 + (gt & (kB - 1))];
    return c;
  }
  __device__ bool check_ok(const Check& c, int gt) const {
    return c.base >= 0 && (c.base % kB) == 0 && c.base / kB < num_blocks && c.mine == c.base + (gt & (kB - 1));
  }
  // Record index of item w once the group agreed its slots are valid.
  __device__ int64_t target(int64_t w, const Check& c, int, unsigned*) const {
    const uint32_t chunk = hd.div(w);
    return (c.base / kB) * hkv + (static_cast<uint32_t>(w) - chunk * hkv);
  }
};

struct AppendSource {
  CUtensorMap map;              // workspace as [n_seqs * hkv * 2 * 128 rows][128 channels] fp16
  const uint16_t* k_new;        // [n_seqs][hkv][128] fp16: the token appended to each sequence
  const uint16_t* v_new;
  uint16_t* ws;                 // the workspace the map describes
  int32_t* seq_lens_out;        // lengths after the append (may be NULL)
  const int32_t* seq_lens;      // lengths before the append
  const int32_t* block_tables;  // [n_seqs][max_blocks]
  int64_t n_items;              // n_seqs * hkv
  int hkv;
  ItemDiv hd;                   // division by hkv
  int max_blocks;
  int64_t num_blocks;
  int ranked;                   // the completing items are handed out by rank (see kRankItems)

  static constexpr bool kSparse = true;    // only items whose sequence completes a tile
  __device__ bool needs_load(int64_t w) const {
    const int L = seq_lens[hd.div(w)];
    return L >= 0 && (L % kB) == kB - 1;
  }
  __device__ void coords(int64_t w, int g, int& x, int& y) const {
    x = 0;
    y = (static_cast<int>(w) * 2 + g) * kB;
  }
  // Thread t < 16 copies 16 bytes of item w's new token (tensor g) into its
  // workspace row L % 128; thread 0 of tensor 0 also writes the new length of the
  // item's sequence (kv-head 0). The writers fence the global writes against the
  // async proxy.
  __device__ void scatter(int64_t w, int g, int t) const {
    const uint32_t s = hd.div(w);
    const uint32_t h = static_cast<uint32_t>(w) - s * hkv;
    const int L = seq_lens[s];
    if (L < 0) return;
    const uint16_t* src = (g ? v_new : k_new) + static_cast<int64_t>(w) * kD + t * 8;
    uint16_t* dst = ws + ((static_cast<int64_t>(w) * 2 + g) * kB + L % kB) * kD + t * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    if (g == 0 && h == 0 && t == 0 && seq_lens_out != nullptr) seq_lens_out[s] = L + 1;
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  // The block's items, 32 threads an item (both tensors), before the block barrier
  // that precedes its first tile copy. Without ranking these are w = blockIdx.x +
  // j gridDim.x. With ranking, the completing items of ranks blockIdx.x + k gridDim.x
  // (listed at `rank` in shared memory; their rows are the ones this block's tile
  // copies read) and the block's w that complete nothing. Returns the list's length.
  // Every thread of the block calls it.
  __device__ int scatter_all(int tid, uint8_t* rank) const {
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int kWarps = kThreads / 32;
    int n_mine = 0;
    if (ranked) {
      int32_t* list = reinterpret_cast<int32_t*>(rank);
      uint32_t* pref = reinterpret_cast<uint32_t*>(rank + kRankList * 4);   // [chunk]: completing items before it
      const int n_chunks = static_cast<int>((n_items + 31) / 32);
      for (int c = warp; c < n_chunks; c += kWarps) {
        const int64_t w = 32 * static_cast<int64_t>(c) + lane;
        const unsigned m = __ballot_sync(0xffffffffu, w < n_items && needs_load(w));
        if (lane == 0) pref[c] = __popc(m);
      }
      __syncthreads();
      if (warp == 0) {   // exclusive prefix over the chunks, lane l taking a contiguous run
        const int per = (n_chunks + 31) / 32, c0 = min(lane * per, n_chunks), c1 = min(c0 + per, n_chunks);
        uint32_t sum = 0;
        for (int c = c0; c < c1; ++c) sum += pref[c];
        uint32_t incl = sum;
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        uint32_t run = incl - sum;
        for (int c = c0; c < c1; ++c) {
          const uint32_t n = pref[c];
          pref[c] = run;
          run += n;
        }
        if (lane == 31) pref[n_chunks] = incl;
      }
      __syncthreads();
      const uint32_t total = pref[n_chunks];
      if (total > blockIdx.x) n_mine = static_cast<int>((total - blockIdx.x + gridDim.x - 1) / gridDim.x);
      for (int k = warp; k < n_mine; k += kWarps) {
        const uint32_t r = blockIdx.x + static_cast<uint32_t>(k) * gridDim.x;
        int lo = 0, hi = n_chunks - 1;   // the last chunk whose prefix is <= r holds rank r
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (pref[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int64_t w = 32 * static_cast<int64_t>(lo) + lane;
        unsigned m = __ballot_sync(0xffffffffu, w < n_items && needs_load(w));
        for (uint32_t i = pref[lo]; i < r; ++i) m &= m - 1;   // drop the lower-ranked items of the chunk
        if (lane == 0) list[k] = 32 * lo + __ffs(m) - 1;
      }
      __syncthreads();
      for (int k = warp; k < n_mine; k += kWarps) scatter(list[k], (tid >> 4) & 1, tid & 15);
    }
    for (int64_t j0 = 0; static_cast<int64_t>(blockIdx.x) + j0 * gridDim.x < n_items; j0 += kWarps) {
      const int64_t w = static_cast<int64_t>(blockIdx.x) + (j0 + warp) * gridDim.x;
      if (w < n_items && !(ranked && needs_load(w))) scatter(w, (tid >> 4) & 1, tid & 15);
    }
    return n_mine;
  }
  // The block's first item with a tile (n_items if none).
  __device__ int64_t first_item(int lane, const uint8_t* rank, int n_mine) const {
    if (ranked) return n_mine > 0 ? reinterpret_cast<const int32_t*>(rank)[0] : n_items;
    const int64_t w = blockIdx.x;
    return needs_load(w) ? w : next_item(w, lane);
  }
  // The item after the block's k-th (w).
  __device__ int64_t next_of(int64_t w, int k, int lane, const uint8_t* rank, int n_mine) const {
    if (ranked) return k + 1 < n_mine ? reinterpret_cast<const int32_t*>(rank)[k + 1] : n_items;
    return next_item(w, lane);
  }
  // The block's next item after w whose tile completes (n_items if none): 32 of the
  // block's items per round, one per lane, agreed by ballot (all 32 lanes call it).
  __device__ int64_t next_item(int64_t w, int lane) const {
    for (int64_t base = w + gridDim.x; base < n_items; base += 32 * static_cast<int64_t>(gridDim.x)) {
      const int64_t c = base + static_cast<int64_t>(lane) * gridDim.x;
      const unsigned m = __ballot_sync(0xffffffffu, c < n_items && needs_load(c));
      if (m) return base + static_cast<int64_t>(__ffs(m) - 1) * gridDim.x;
    }
    return n_items;
  }
  struct Check {};
  __device__ Check prepare(int64_t, int) const { return Check{}; }
  __device__ bool check_ok(const Check&, int) const { return true; }
  __device__ int64_t target(int64_t w, const Check&, int gt, unsigned* flags) const {
    if (!needs_load(w)) return -1;
    const uint32_t s = hd.div(w);
    const uint32_t h = static_cast<uint32_t>(w) - s * hkv;
    const int bi = seq_lens[s] / kB;
    if (bi >= max_blocks) {
      if (gt == 0) raise_flag(flags, KVARN_FLAG_BAD_LENGTH);
      return -1;
    }
    const int64_t blk = block_tables[static_cast<int64_t>(s) * max_blocks + bi];
    if (blk < 0 || blk >= num_blocks) {
      if (gt == 0) raise_flag(flags, KVARN_FLAG_BAD_BLOCK);
      return -1;
    }
    return blk * hkv + h;
  }
};

__device__ __forceinline__ const CUtensorMap* tensor_map(const PrefillSource& s, int g) { return &s.map[g]; }
__device__ __forceinline__ const CUtensorMap* tensor_map(const AppendSource& s, int) { return &s.map; }

// Thread gt == 0 of group g starts the two TMA copies (64 channels each) of item
// w's tile into `dst`, completing on `bar`.
template <class Src>
__device__ __forceinline__ void issue_tile(const Src& src, int64_t w, int g, uint8_t* dst, uint64_t* bar) {
  int x, y;
  src.coords(w, g, x, y);
  const CUtensorMap* map = tensor_map(src, g);
  mbar_arrive_expect_tx(bar, kTileOp);
  tma_load_2d(dst, map, x, y, bar);
  tma_load_2d(dst + kTileOp / 2, map, x + 64, y, bar);
}

// Thread gt == 0 issues the next item's Hadamard products once the group's last TMEM
// data of the current item is in registers, so that they run under its codes pass.
struct NextProducts {
  static constexpr bool kActive = true;
  bool go;
  int gt;
  uint64_t* load_bar;   // the next tile's copy
  uint32_t parity;
  uint32_t sx, sh, d1, d2;
  uint64_t* mma_bar;
  unsigned* flags;
  bool* inflight;
  __device__ void operator()() const {
    if (!go || gt != 0) return;
    if (!mbar_wait(load_bar, parity, flags)) return;
    constexpr uint32_t kIdesc = idesc_f16_f32(128, 128);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint64_t dh = smem_desc_sw128(sw_kstep(sh, s));
      const uint64_t dx = smem_desc_sw128(sw_kstep(sx, s));
      umma_f16(d1, dh, dx, kIdesc, s > 0);   // D1[i][j] = sum_k H[i][k] X[j][k]
      umma_f16(d2, dx, dh, kIdesc, s > 0);   // D2[j][i] = sum_k X[j][k] H[i][k]
    }
    umma_commit(mma_bar);
    *inflight = true;
  }
};

// 128 registers a thread (all that 512 threads can hold): a whole sweep in flight
// needs 64 of them; 112 spilled and measured 5 % slower.
template <class Src, int KB, int VB, bool kLean, bool kEarly>
__global__ void __maxnreg__(128)
    quantize_kernel(const __grid_constant__ Src src, uint8_t* __restrict__ cache, int n_iters, float eps,
                    unsigned* flags) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int grp = tid / kGroupThreads;     // 0 = K, 1 = V
  const int gt = tid % kGroupThreads;
  const int bar_id = 1 + grp;
  using S = QSmem<KB, VB, Src::kSparse>;
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* load_bar = mma_bar + 2 + 2 * grp;   // this group's [buf]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffTmem);
  if (static_cast<int64_t>(blockIdx.x) >= src.n_items) return;
  // Async work is spread over three threads of the group so that it overlaps:
  // gt == 0 issues the Hadamard products, gt == kTmaThread the tile copies and
  // gt == kStoreThread the record stores (bulk groups belong to the thread that
  // commits them, so it also waits for them).
  constexpr int kTmaThread = 64, kStoreThread = 32;
  uint8_t* tiles = smem + kOffIn + grp * 2 * kTileOp;   // this group's [buf]

  fill_hadamard_sw128(smem + kOffH, tid, kThreads);   // the +-1 Hadamard operand
  // appended tokens into the workspace (the block's items), ordered before any tile
  // copy by the barrier below
  uint8_t* rank = smem + S::kOffRank;
  const int n_mine = src.scatter_all(tid, rank);
  if (tid == 0) {
    for (int b = 0; b < 6; ++b) mbar_init(&mma_bar[b], 1);
    fence_mbar_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // this thread's half line in TMEM
  const int gw = gt >> 5, t = gt & 31;
  const uint32_t lane0 = 32 * (gw & 3) + 16 * (gw >> 2);
  const int line = static_cast<int>(lane0) + (t >> 2) + 8 * (t & 1);
  const int p = (t >> 1) & 1;
  const uint32_t d1 = tmem_addr(tmem, 0, 256 * grp);
  const uint32_t d2 = d1 + 128;
  const uint32_t ta1 = tmem_addr(tmem, lane0, 256 * grp);
  const uint32_t ta2 = ta1 + 128;
  float* vec = reinterpret_cast<float*>(smem + S::kOffVec) + grp * kNumVec * kVec;
  const uint32_t sh = smem_u32(smem + kOffH);
  constexpr uint32_t kIdesc = idesc_f16_f32(128, 128);

  // The block takes the items blockIdx.x + j gridDim.x that have a tile (all of them
  // for the prefill; for the append, those whose sequence completes one). The copy of
  // an item's tile is started one item ahead; the slot check of the next item is
  // agreed on at the barrier that ends the current one.
  int64_t item = blockIdx.x;
  if constexpr (Src::kSparse) item = src.first_item(t, rank, n_mine);
  uint32_t pend = 0;               // bit b: a copy into buffer b has not been waited for
  uint32_t load_parity = 0;        // bit b: phase parity of buffer b's barrier
  const bool has_first = !Src::kSparse || item < src.n_items;
  typename Src::Check check = has_first ? src.prepare(item, gt) : typename Src::Check{};
  int64_t dst = -1;
  if (named_bar_and(bar_id, kGroupThreads, !has_first || src.check_ok(check, gt))) {
    if (has_first) dst = src.target(item, check, gt, flags);
  } else if (gt == 0) {
    raise_flag(flags, KVARN_FLAG_BAD_SLOTS);
  }
  if (has_first) {
    if (gt == kTmaThread) issue_tile(src, item, grp, tiles, &load_bar[0]);
    pend = 1;
  }
  uint32_t mma_parity = 0;
  bool mma_inflight = false;       // thread gt == 0: an issued MMA not yet seen complete
  bool early = false;              // this item's products went out under the previous item's codes
  for (int k = 0; item < src.n_items; ++k) {
    const int buf = k & 1;
    const int64_t next = src.next_of(item, k, t, rank, n_mine);
    const bool has_next = next < src.n_items;
    bool ok = true;
    if ((pend >> buf) & 1u) {
      ok = mbar_wait(&load_bar[buf], (load_parity >> buf) & 1u, flags);
      if (ok) {
        load_parity ^= 1u << buf;
        pend &= ~(1u << buf);
      }
    }
    // the item's Hadamard products first, so the next item's bookkeeping below
    // (slot loads, the next tile copy) runs under them
    if (dst >= 0 && gt == 0 && ok && !early) {
      const uint32_t sx = smem_u32(tiles + buf * kTileOp);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t dh = smem_desc_sw128(sw_kstep(sh, s));
        const uint64_t dx = smem_desc_sw128(sw_kstep(sx, s));
        umma_f16(d1, dh, dx, kIdesc, s > 0);   // D1[i][j] = sum_k H[i][k] X[j][k]
        umma_f16(d2, dx, dh, kIdesc, s > 0);   // D2[j][i] = sum_k X[j][k] H[i][k]
      }
      umma_commit(&mma_bar[grp]);
      mma_inflight = true;
    }
    typename Src::Check check_next{};
    if (has_next) {
      // buffer buf ^ 1 was last read by the previous item
      if (gt == kTmaThread) issue_tile(src, next, grp, tiles + (buf ^ 1) * kTileOp, &load_bar[buf ^ 1]);
      pend |= 2u >> buf;
      check_next = src.prepare(next, gt);
    }
    // kEarly: the next item's products go out under this item's codes pass
    const bool go_next = kEarly && has_next && ((pend >> (buf ^ 1)) & 1u) != 0;
    if (dst < 0 && early && ok) {       // products of an item whose slots failed the check: consume them
      ok = mbar_wait(&mma_bar[grp], mma_parity, flags);
      if (ok) {
        mma_parity ^= 1;
        mma_inflight = false;
      }
    }
    bool early_next = false;
    if (dst >= 0) {
      uint8_t* stage = smem + (grp == 0 ? S::kOffStageK + buf * S::kStageK : S::kOffStageV + buf * S::kStageV);
      if (gt == kStoreThread) bulk_wait_read<1>();   // the stage written two items ago has been stored
      if (ok) {
        ok = mbar_wait(&mma_bar[grp], mma_parity, flags);
        if (ok) {
          mma_parity ^= 1;
          mma_inflight = false;
        }
      }
      tc_fence_after();
      const uint8_t* tile = tiles + buf * kTileOp;
      early_next = go_next && ok;
      if (!kEarly) {
        if (grp == 0)
          ok = quantize_group<0, KB, kLean>(vec, stage, tile, ta1, ta2, line, p, n_iters, eps, bar_id, ok);
        else
          ok = quantize_group<1, VB, kLean>(vec, stage, tile, ta1, ta2, line, p, n_iters, eps, bar_id, ok);
      } else {
        const NextProducts hook{early_next, gt, &load_bar[buf ^ 1], (load_parity >> (buf ^ 1)) & 1u,
                                smem_u32(tiles + (buf ^ 1) * kTileOp), sh, d1, d2, &mma_bar[grp], flags,
                                &mma_inflight};
        if (grp == 0)
          ok = quantize_group<0, KB, kLean>(vec, stage, tile, ta1, ta2, line, p, n_iters, eps, bar_id, ok, hook);
        else
          ok = quantize_group<1, VB, kLean>(vec, stage, tile, ta1, ta2, line, p, n_iters, eps, bar_id, ok, hook);
      }
      if (!ok) break;                     // a copy or the tensor core never signalled (flag raised)
      fence_proxy_async_smem();
      tc_fence_before();
    }
    // end of the item: its stage is complete, and the group agrees on the next item's slots
    const bool next_ok = named_bar_and(bar_id, kGroupThreads, !has_next || src.check_ok(check_next, gt));
    tc_fence_after();
    if (dst >= 0 && gt == kStoreThread) {
      using L = RecordLayout<KB, VB, kLean>;
      uint8_t* stage = smem + (grp == 0 ? S::kOffStageK + buf * S::kStageK : S::kOffStageV + buf * S::kStageV);
      uint8_t* rec = cache + dst * static_cast<int64_t>(L::kBytes);
      if (grp == 0) {
        bulk_s2g(rec + L::kKCodeOff, stage, L::kKCodeBytes);
        bulk_s2g(rec + L::kKMetaOff, stage + L::kKCodeBytes, L::kMetaBytes);
      } else {
        bulk_s2g(rec + L::kVCodeOff, stage, L::kVCodeBytes);
        bulk_s2g(rec + L::kVMetaOff, stage + L::kVCodeBytes, L::kMetaBytes);
      }
      bulk_commit();
    }
    if (has_next) {
      dst = -1;
      if (next_ok)
        dst = src.target(next, check_next, gt, flags);
      else if (gt == 0)
        raise_flag(flags, KVARN_FLAG_BAD_SLOTS);
    }
    item = next;
    early = early_next;
  }
  // after a timeout: let copies and MMAs still in flight finish (bounded) before the
  // shared memory and TMEM are released
  if (gt == kTmaThread)
    for (int b = 0; b < 2; ++b)
      if ((pend >> b) & 1u) mbar_wait(&load_bar[b], (load_parity >> b) & 1u, flags);
  if (gt == 0 && mma_inflight) mbar_wait(&mma_bar[grp], mma_parity, flags);
  if (gt == kStoreThread) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid < 32) tmem_dealloc(tmem, 512);
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <class Src, int KB, int VB, bool kLean>
cudaError_t launch_quantize_bits(const Src& src, uint8_t* cache, int n_iters, float eps, unsigned* flags,
                            cudaStream_t stream, int max_ctas) {
  if (src.n_items <= 0) return cudaSuccess;
  if (src.n_items > INT32_MAX) return cudaErrorInvalidValue;
  int64_t grid = sm_count();
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > src.n_items) grid = src.n_items;
  constexpr int kSmem = QSmem<KB, VB, Src::kSparse>::kBytes;
  // The prefill with 4-bit keys and more than one iteration issues each item's
  // products under the previous item's codes pass (measured slower for k2v2, for one
  // iteration and for the append, whose blocks get one or two items).
  if constexpr (!Src::kSparse && KB == 4) {
    if (n_iters > 1) {
      static std::atomic<unsigned long long> smem_set{0};
      cudaError_t err = set_smem_once(quantize_kernel<Src, KB, VB, kLean, true>, kSmem, smem_set);
      if (err != cudaSuccess) return err;
      quantize_kernel<Src, KB, VB, kLean, true><<<static_cast<unsigned>(grid), kThreads, kSmem, stream>>>(
          src, cache, n_iters, eps, flags);
      return cudaGetLastError();
    }
  }
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t err = set_smem_once(quantize_kernel<Src, KB, VB, kLean, false>, kSmem, smem_set);
  if (err != cudaSuccess) return err;
  quantize_kernel<Src, KB, VB, kLean, false><<<static_cast<unsigned>(grid), kThreads, kSmem, stream>>>(
      src, cache, n_iters, eps, flags);
  return cudaGetLastError();
}

// The kernel instance of a preset (k4v2, k4v4, k2v2; k4v2 with lean metadata).
template <class Src>
cudaError_t launch_quantize(const Src& src, uint8_t* cache, int k_bits, int v_bits, bool lean, int n_iters, float eps,
                            unsigned* flags, cudaStream_t stream, int max_ctas) {
  if (k_bits == 4 && v_bits == 2 && !lean)
    return launch_quantize_bits<Src, 4, 2, false>(src, cache, n_iters, eps, flags, stream, max_ctas);
  if (k_bits == 4 && v_bits == 2 && lean)
    return launch_quantize_bits<Src, 4, 2, true>(src, cache, n_iters, eps, flags, stream, max_ctas);
  if (k_bits == 4 && v_bits == 4 && !lean)
    return launch_quantize_bits<Src, 4, 4, false>(src, cache, n_iters, eps, flags, stream, max_ctas);
  if (k_bits == 2 && v_bits == 2 && !lean)
    return launch_quantize_bits<Src, 2, 2, false>(src, cache, n_iters, eps, flags, stream, max_ctas);
  return cudaErrorInvalidValue;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// TMA map of an fp16 matrix [rows][row_elems] read in boxes of 64 channels x 128
// rows with the 128-byte swizzle (row_elems a multiple of 64, base 16-byte aligned).
cudaError_t tile_map(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  if (rows > (1ull << 32) || row_elems > (1ull << 32)) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {row_elems * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                        elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quantize_prefill(const uint16_t* k, const uint16_t* v, const int64_t* slot, int64_t n_tokens,
                                    int hkv, int64_t num_blocks, uint8_t* cache, int k_bits, int v_bits, bool lean,
                                    int n_iters, float eps, unsigned* flags, cudaStream_t stream, int max_ctas) {
  PrefillSource src{};
  cudaError_t err = tile_map(&src.map[0], k, static_cast<uint64_t>(hkv) * kD, static_cast<uint64_t>(n_tokens));
  if (err == cudaSuccess)
    err = tile_map(&src.map[1], v, static_cast<uint64_t>(hkv) * kD, static_cast<uint64_t>(n_tokens));
  if (err != cudaSuccess) return err;
  src.slot = slot;
  src.n_items = (n_tokens / kB) * hkv;
  src.hkv = hkv;
  src.hd = make_item_div(static_cast<uint32_t>(hkv));
  src.num_blocks = num_blocks;
  return launch_quantize(src, cache, k_bits, v_bits, lean, n_iters, eps, flags, stream, max_ctas);
}

cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, const int32_t* seq_lens,
                          int32_t* seq_lens_out, const int32_t* block_tables, int n_seqs, int hkv, int max_blocks,
                          int64_t num_blocks, uint16_t* ws, uint8_t* cache, int k_bits, int v_bits, bool lean,
                          int n_iters, float eps, unsigned* flags, cudaStream_t stream) {
  if (n_seqs <= 0) return cudaSuccess;
  if (static_cast<int64_t>(n_seqs) * hkv * 2 * kB > INT32_MAX) return cudaErrorInvalidValue;
  AppendSource src{};
  const cudaError_t err = tile_map(&src.map, ws, kD, static_cast<uint64_t>(n_seqs) * hkv * 2 * kB);
  if (err != cudaSuccess) return err;
  src.k_new = k_new;
  src.v_new = v_new;
  src.ws = ws;
  src.seq_lens_out = seq_lens_out;
  src.seq_lens = seq_lens;
  src.block_tables = block_tables;
  src.n_items = static_cast<int64_t>(n_seqs) * hkv;
  src.hkv = hkv;
  src.hd = make_item_div(static_cast<uint32_t>(hkv));
  src.max_blocks = max_blocks;
  src.num_blocks = num_blocks;
  const int64_t grid = std::min<int64_t>(sm_count(), src.n_items);
  src.ranked = src.n_items <= kRankItems && (src.n_items + grid - 1) / grid <= kRankList;
  return launch_quantize(src, cache, k_bits, v_bits, lean, n_iters, eps, flags, stream, 0);
}

}  // namespace kvarn
