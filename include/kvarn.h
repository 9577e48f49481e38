/*
 * kvarn.h - C ABI of libkvarn: KVarN per-tile KV-cache quantization and paged
 * decode attention over the quantized cache, for NVIDIA GB300 (sm_103a).
 *
 * Method (KVarN README, huawei-csl/KVarN, "How KVarN works", stages 1-4): the KV
 * cache is quantized in tiles of 128 tokens per kv-head. Each fp16 tile
 * X [128 channels x 128 tokens] is (2) rotated along channels by an orthonormal
 * Hadamard matrix H, (3) variance-normalised by alternating column-wise and
 * row-wise std normalisation in log space (Sinkhorn style), keeping the row scale
 * vector r and column scale vector c, and (4) quantized by asymmetric
 * round-to-nearest: keys at 4 bits with (scale, zero) per channel, values at 2
 * bits with (scale, zero) per token. The default preset is kvarn_k4v2_g128 with block
 * size fixed at 128 (one paged block = one tile) and float16 compute (README,
 * quick start and note). Decode attention reads the packed blocks through the
 * block table, re-applies the scales on read (stage 4), rotates q by the same H
 * (scores are unchanged by an orthonormal rotation, stage 2) and un-rotates the
 * output by H^T. A partial last tile stays in a small fp16 decode workspace until
 * it holds 128 tokens (README, capacity tip: a small fixed decode workspace).
 *
 * Readings fixed by this library where the pages are silent:
 *   H = Sylvester Hadamard of order 128 / sqrt(128) (natural order, H = H^T).
 *   Normalisation: n_iters iterations (preset 4), each a column pass then a row
 *   pass; variance is the population variance about the mean; eps is added to
 *   the variance; data are divided, not centred.
 *   r, c, s clamped to [2^-14, 65504] and z to [-65504, 65504], then rounded to
 *   fp16 (nearest even). z = fp16(group min), s = fp16((group max - z)/(2^b-1)),
 *   code = clamp(floor((y - z)/s + 1/2), 0, 2^b - 1), y = X_r / (r_i c_j).
 *   Decode: softmax scale 1/sqrt(128); q-head h uses kv-head h / (Hq/Hkv); no
 *   mask (all seq_len tokens are attended).
 *
 * ---------------------------------------------------------------------------
 * Presets. kvarn_meta's (k_bits, v_bits) picks one of: k4v2 (the README's
 * kvarn_k4v2_g128, the default), k4v4 and k2v2 (the README reports 2-bit
 * results too). A record holds the key codes, then the value codes, then the key
 * and the value metadata (1024 bytes each); the layouts below are k4v2's, and
 * the two others use:
 *   2-bit K codes, token-major: token t owns bytes [32t, 32t+32) = four 8-byte
 *     groups g = (i>>1)&3, each two words u = i>>6; channel i sits in crumb
 *     p = 4((i>>4)&3) + 2(i&1) + ((i>>3)&1) (bits 2p..2p+1) of word u.
 *   4-bit V codes, channel-major: the 4-bit K layout with channel and token
 *     exchanged (channel i owns bytes [64i, 64i+64), groups g = (t>>1)&3, words
 *     w = t>>5, nibble p = 4((t>>3)&1) + 2(t&1) + ((t>>4)&1)).
 *   k4v4: K codes [0, 8192), V codes [8192, 16384), K meta [16384, 17408), V meta
 *     [17408, 18432). k2v2: K codes [0, 4096), V codes [4096, 8192), K meta
 *     [8192, 9216), V meta [9216, 10240).
 *   k4v2l (k4v2 with layout = KVARN_LAYOUT_LEAN): lean metadata. A key group is
 *     one channel, so the channel's r is constant inside it and is folded into
 *     its s and z (keys are quantized from X_r / c); a value group is one token,
 *     so c is folded likewise (values from X_r / r). K meta [12288, 13056) is fp16
 *     c, s, z x 128; V meta [13056, 13824) is r, s, z; 13824 bytes in all.
 * The decode kernel runs 8 warps with two record stages each for k4v2, k4v2l and
 * k2v2, and 6 warps for k4v4 (two of its 18432-byte records per warp fit only 6).
 *
 * Packed record (k4v2): 14336 bytes per (physical block, kv-head). The cache is
 * uint8 [num_blocks][num_kv_heads][record bytes], device memory owned by the
 * caller.
 *   [    0,  8192)  K codes, 4 bits, token-major: token t owns bytes
 *                   [64t, 64t+64) = four 16-byte groups g = (i>>1)&3, each four
 *                   little-endian 32-bit words w = i>>5; channel i sits in nibble
 *                   p = 4((i>>3)&1) + 2(i&1) + ((i>>4)&1) (bits 4p..4p+3) of word w.
 *   [ 8192, 12288)  V codes, 2 bits, channel-major: channel i lives in 512-byte
 *                   panel i>>4; 16-byte cell (i&7)*4 + ((t>>1)&3) of the panel
 *                   holds 8 bytes for the channel with bit 3 clear followed by 8
 *                   bytes for its partner i|8; each 8 bytes are two words
 *                   u = t>>6; token t sits in crumb
 *                   p = 4((t>>4)&3) + 2(t&1) + ((t>>3)&1) (bits 2p..2p+1).
 *   [12288, 13312)  K metadata, fp16 [4][128]: r (per channel), c (per token),
 *                   s (per channel), z (per channel).
 *   [13312, 14336)  V metadata, fp16 [4][128]: r (per channel), c (per token),
 *                   s (per token), z (per token).
 * Dequantised rotated tile: X_r[i][j] = r_i c_j (code_ij * s + z), (s, z) taken
 * per channel i for K and per token j for V; the tile is H * X_r.
 * The code orders follow the register fragments of the decode kernel's
 * m16n8k16 tensor-core operands, so a thread's operands are contiguous bytes.
 * Inside a word, the two codes of one operand register sit in the low nibbles of
 * the two bytes of a 16-bit half (4-bit) or at bits 0-1 and 4-5 of one byte
 * (2-bit), so one fp6 (e2m3: value code/8) or fp4 (e2m1: value code/2) conversion
 * instruction turns them into an fp16 pair.
 *
 * Decode workspace: fp16 [max_seqs][num_kv_heads][2 (K,V)][128 tokens][128 ch],
 * raw (unrotated, unquantised) tokens of each sequence's partial last tile;
 * token L of a sequence is at slot L % 128.
 * ---------------------------------------------------------------------------
 * Conventions for every call:
 *   - fp16 buffers are IEEE binary16 bit patterns (uint16_t), device memory.
 *   - All pointers are device pointers unless stated; all must be 16-byte
 *     aligned (KVARN_EALIGN otherwise). The library allocates nothing: every
 *     buffer is allocated and owned by the caller.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is queued
 *     asynchronously; a KVARN_OK return means the launches were queued.
 *   - Argument errors are detected on the host before anything is launched and
 *     leave device memory untouched. Data errors that only the device can see
 *     (a block index outside [0, num_blocks), a slot mapping that does not fill
 *     whole blocks, a sequence longer than its block table) make the kernels
 *     skip the affected tile and set a bit in a device flag word, read and
 *     cleared by kvarn_device_flags().
 *   - The calls keep no host state besides the per-thread error message, the
 *     device flag word's address and which kernels had their shared-memory
 *     limit raised (both looked up once per device); the flag word is shared by
 *     every call on a device.
 *   - kvarn_quantize_tiles, kvarn_append_decode and kvarn_decode_attention only
 *     queue kernels on `stream` (no allocation, no host synchronisation), so once
 *     each has been called on a device, a serving step made of them can be
 *     captured into a CUDA graph and replayed.
 */
#ifndef KVARN_H
#define KVARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVARN_API __attribute__((visibility("default")))
#else
#define KVARN_API
#endif

#define KVARN_HEAD_DIM 128
#define KVARN_BLOCK_SIZE 128
#define KVARN_RECORD_BYTES 14336
#define KVARN_MAX_GQA_GROUP 8
#define KVARN_LAYOUT_LEAN 1  /* kvarn_meta.layout: lean metadata (see presets)    */

typedef enum {
  KVARN_OK = 0,
  KVARN_EINVAL = 1,        /* null pointer, negative size, inconsistent sizes   */
  KVARN_EUNSUPPORTED = 2,  /* head_dim/block_size/bits/group outside the preset */
  KVARN_EALIGN = 3,        /* a pointer is not 16-byte aligned                   */
  KVARN_ESCRATCH = 4,      /* decode scratch smaller than the size query         */
  KVARN_ECUDA = 5          /* a CUDA call or launch failed (see kvarn_last_error) */
} kvarn_status;

/* Device flag bits reported by kvarn_device_flags(). */
#define KVARN_FLAG_BAD_SLOTS 0x1u      /* prefill chunk not one whole block: skipped  */
#define KVARN_FLAG_BAD_BLOCK 0x2u      /* block index outside [0, num_blocks): skipped */
#define KVARN_FLAG_BAD_LENGTH 0x4u     /* seq_len > max_blocks_per_seq*128: clipped   */
#define KVARN_FLAG_WAIT_TIMEOUT 0x8u   /* a bounded wait on a copy gave up            */

typedef struct {
  int32_t num_kv_heads;       /* Hkv >= 1                                         */
  int32_t num_q_heads;        /* Hq, a multiple of Hkv with Hq/Hkv <= 8           */
  int32_t head_dim;           /* must be 128                                      */
  int32_t block_size;         /* must be 128                                      */
  int32_t k_bits;             /* preset: 4 (k4v2, k4v4) or 2 (k2v2)               */
  int32_t v_bits;             /* preset: 2 (k4v2, k2v2) or 4 (k4v4)               */
  int32_t n_iters;            /* normalisation iterations, 1..16 (preset 4)       */
  float eps;                  /* added to each variance, > 0 (preset 1e-6)        */
  int64_t num_blocks;         /* physical blocks in the cache                     */
  int32_t max_blocks_per_seq; /* row length of block_tables                       */
  int32_t layout;             /* 0, or KVARN_LAYOUT_LEAN with k4v2 (preset k4v2l) */
} kvarn_meta;

/* Bytes of one (block, kv-head) record of the default preset k4v2: 14336. */
KVARN_API size_t kvarn_record_bytes(void);

/* Bytes of one (block, kv-head) record of the meta's preset:
 * 128 * 128 * (k_bits + v_bits) / 8 + 2048 (k4v2 14336, k4v4 18432, k2v2
 * 10240); 0 if meta is invalid. */
KVARN_API size_t kvarn_meta_record_bytes(const kvarn_meta* meta);

/* Bytes of the whole paged cache: num_blocks * num_kv_heads *
 * kvarn_meta_record_bytes(meta); 0 if meta is invalid. */
KVARN_API size_t kvarn_cache_bytes(const kvarn_meta* meta);

/* Bytes of a decode workspace for `max_seqs` sequences:
 * max_seqs * num_kv_heads * 2 * 128 * 128 * 2; 0 if meta is invalid. */
KVARN_API size_t kvarn_workspace_bytes(const kvarn_meta* meta, int32_t max_seqs);

/* Bytes of device scratch kvarn_decode_attention needs for `n_seqs` sequences
 * (partial softmax states of the context splits); depends on max_blocks_per_seq.
 * 0 if meta is invalid. */
KVARN_API size_t kvarn_decode_scratch_bytes(const kvarn_meta* meta, int32_t n_seqs);

/*
 * Prefill write. Quantizes whole tiles of fresh K/V into the paged cache
 * (stages 2-4 of "How KVarN works").
 *   k, v          fp16 [n_tokens][num_kv_heads][128], token-major (vLLM layout).
 *   slot_mapping  int64 [n_tokens]; every run of 128 tokens [t0, t0+128) must map
 *                 to one block at consecutive offsets: slot[t0+k] = 128*b + k.
 *                 A run that does not, or whose block b is outside
 *                 [0, num_blocks), is skipped and flagged.
 *   n_tokens      >= 0 and a multiple of 128 (partial tiles belong in the decode
 *                 workspace, see kvarn_append_decode), below 2^31, with
 *                 (n_tokens / 128) * num_kv_heads below 2^31 (KVARN_EINVAL otherwise).
 *                 Byte offsets into k, v and cache are 64-bit: inputs and caches
 *                 beyond 4 GiB are supported.
 *   cache         uint8 [num_blocks][num_kv_heads][14336]; written records only.
 */
KVARN_API kvarn_status kvarn_quantize_tiles(const uint16_t* k, const uint16_t* v,
                                  const int64_t* slot_mapping, int64_t n_tokens,
                                  uint8_t* cache, const kvarn_meta* meta, void* stream);

/*
 * Decode-step write. For each sequence s with L = seq_lens[s] stored tokens,
 * writes the new token into workspace[s][h][*][L % 128][*]; when that completes
 * the partial tile (L % 128 == 127) the tile is quantized into block
 * block_tables[s][L / 128] for every kv-head. One kernel launch: the
 * quantize kernel writes each (sequence, kv-head)'s token before it copies
 * that item's tile.
 *   k_new, v_new  fp16 [n_seqs][num_kv_heads][128].
 *   seq_lens      int32 [n_seqs], lengths before the append, >= 0.
 *   seq_lens_out  int32 [n_seqs] or NULL: receives seq_lens[s] + 1. Must not
 *                 alias seq_lens.
 *   block_tables  int32 [n_seqs][max_blocks_per_seq].
 *   workspace     fp16, see the workspace layout above; sequence s uses row s.
 */
KVARN_API kvarn_status kvarn_append_decode(const uint16_t* k_new, const uint16_t* v_new,
                                 const int32_t* seq_lens, int32_t* seq_lens_out,
                                 const int32_t* block_tables, int32_t n_seqs,
                                 uint16_t* workspace, uint8_t* cache,
                                 const kvarn_meta* meta, void* stream);

/*
 * Decode attention for one new query per sequence over its L = seq_lens[s]
 * tokens: floor(L/128) packed tiles read through block_tables, plus L % 128
 * workspace tokens. GQA: q-head h reads kv-head h / (Hq/Hkv).
 *   q             fp16 [n_seqs][num_q_heads][128].
 *   n_seqs        0..65535.
 *   workspace     fp16 workspace (may be NULL only if every L % 128 == 0; tail
 *                 tokens of a sequence without a workspace are not attended and
 *                 KVARN_FLAG_BAD_LENGTH is set).
 *   out           fp16 [n_seqs][num_q_heads][128]; a sequence with L == 0 gets 0.
 *   scratch       device buffer of >= kvarn_decode_scratch_bytes(meta, n_seqs).
 * Three kernels on the stream (a scan, the split phase, the merge); the last two
 * are programmatic dependent launches of the kernel before them. With the
 * environment variable KVARN_DECODE_SPLIT=tc (read on every call) the k4v2
 * presets run their split phase on the tcgen05 kernel instead of the warp-level
 * one (same results within the decode tolerance; measured slower).
 */
KVARN_API kvarn_status kvarn_decode_attention(const uint16_t* q, const uint8_t* cache,
                                    const uint16_t* workspace, const int32_t* block_tables,
                                    const int32_t* seq_lens, int32_t n_seqs, uint16_t* out,
                                    void* scratch, size_t scratch_bytes,
                                    const kvarn_meta* meta, void* stream);

/*
 * One serving step in one launch: kvarn_append_decode (the new token of every
 * sequence into the workspace; tiles it completes quantized into their blocks),
 * then kvarn_decode_attention over the lengths after the append, with the same
 * results as those two calls in order. A cooperative launch of one CTA per SM
 * whose phases (append and tile quantization; attention over the tiles; merge
 * with the workspace tokens) meet at grid-wide barriers; every wait is bounded
 * and reports KVARN_FLAG_WAIT_TIMEOUT instead of hanging (a CTA whose barrier wait
 * runs out stops there, so the outputs of such a call are not valid). The barrier
 * words are the last 256 bytes of `scratch`, zeroed on `stream` before each launch:
 * calls that overlap on the GPU must not share a scratch buffer (nor, as for the
 * two calls it fuses, a workspace or cache region). Capturable in a CUDA graph.
 * Measured on GB300 this one launch is slower than kvarn_append_decode followed by
 * kvarn_decode_attention (the grid-wide barriers between its phases, and its merge
 * phase at the split phase's one CTA per SM), so those two calls, captured in a CUDA
 * graph, are the recommended serving step; this entry point is kept for callers that
 * want a single launch.
 *   q             fp16 [n_seqs][num_q_heads][128], the new query of each sequence.
 *   k_new, v_new  fp16 [n_seqs][num_kv_heads][128].
 *   seq_lens      int32 [n_seqs], lengths before the append, >= 0.
 *   seq_lens_out  int32 [n_seqs] (required): receives seq_lens[s] + 1, the lengths
 *                 the attention uses. Must not alias seq_lens.
 *   block_tables  int32 [n_seqs][max_blocks_per_seq].
 *   workspace     fp16 workspace (required).
 *   n_seqs        0..65535.
 *   out           fp16 [n_seqs][num_q_heads][128].
 *   scratch       device buffer of >= kvarn_decode_scratch_bytes(meta, n_seqs).
 * Returns KVARN_ECUDA if the device cannot hold the grid co-resident.
 */
KVARN_API kvarn_status kvarn_serve_step(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                        const int32_t* seq_lens, int32_t* seq_lens_out,
                                        const int32_t* block_tables, int32_t n_seqs, uint16_t* workspace,
                                        uint8_t* cache, uint16_t* out, void* scratch, size_t scratch_bytes,
                                        const kvarn_meta* meta, void* stream);

/*
 * Decode attention that allocates nothing and needs no scratch from the caller.
 * This entry point has no counterpart in the KVarN paper or README; it exists for
 * callers that cannot allocate device memory: e.g. a serving engine whose free
 * device memory is all pre-reserved for its KV-cache pool and handed out only by
 * its own allocator, or a plain-C host with no device allocator for temporaries.
 * Same arguments, argument checks (every preset, KVARN_EALIGN for a misaligned
 * pointer) and results as kvarn_decode_attention minus scratch: the scratch
 * is a fixed 16 MiB array of device memory inside the library (held by every GPU
 * that loads the library until the process exits), shared by all calls on a device.
 *   - Sizes: returns KVARN_ESCRATCH, without launching, when the scratch needed for
 *     n_seqs * num_kv_heads (sequence, kv-head) pairs exceeds 16 MiB (about 2100
 *     pairs on a 152-SM GB300).
 *   - The first call on a device (with that device current) looks up the array's
 *     device address; make that first call before any stream capture.
 *   - Calls whose work overlaps on the GPU (different streams, not ordered) race on
 *     the shared array; order them. Nothing in the array needs to start at zero.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
KVARN_API kvarn_status kvarn_decode_attention_static(const uint16_t* q, const uint8_t* cache,
                                                     const uint16_t* workspace, const int32_t* block_tables,
                                                     const int32_t* seq_lens, int32_t n_seqs, uint16_t* out,
                                                     const kvarn_meta* meta, void* stream);

/*
 * Chunked-prefill attention, a reading of this library (the pages are silent on
 * prefill over a quantized cache): each sequence s has L0 = seq_lens[s] tokens
 * in the cache (floor(L0/128) packed tiles through block_tables, then L0 % 128
 * workspace tokens) and a chunk of fresh tokens cu_tokens[s] .. cu_tokens[s+1]-1
 * of k_new / v_new. Chunk token p attends the L0 cached tokens and chunk tokens
 * 0..p (causal), with the decode's softmax scale and GQA mapping; packed tiles
 * are read with their scales re-applied and q rotated by H (stage 2), fresh and
 * workspace tokens exactly. The chunk is not written to the cache (quantize it
 * with kvarn_quantize_tiles / kvarn_append_decode as it fills tiles).
 *   q, out        fp16 [n_tokens][num_q_heads][128], n_tokens = cu_tokens[n_seqs].
 *   k_new, v_new  fp16 [n_tokens][num_kv_heads][128].
 *   cu_tokens     int32 [n_seqs + 1], non-decreasing, cu_tokens[0] = 0.
 *   seq_lens      int32 [n_seqs], cached tokens before each chunk.
 *   n_seqs        0..65535. max_chunk: an upper bound of every chunk length
 *                 (sets the grid; the tokens of a longer chunk beyond max_chunk
 *                 rounded up to 16 are not computed, their out rows are left as
 *                 they were, and KVARN_FLAG_BAD_LENGTH is raised).
 *   workspace     fp16 workspace or NULL (then L0 % 128 tokens are not attended
 *                 and KVARN_FLAG_BAD_LENGTH is raised).
 * One launch; no scratch. Every preset of kvarn_meta is supported.
 */
KVARN_API kvarn_status kvarn_prefill_attention(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                     const int32_t* cu_tokens, const int32_t* seq_lens, int32_t n_seqs,
                                     int32_t max_chunk, const int32_t* block_tables, const uint8_t* cache,
                                     const uint16_t* workspace, uint16_t* out, const kvarn_meta* meta,
                                     void* stream);

/*
 * Self-test of the give-up path of the library's bounded waits (failure
 * detection): every wait of the kernels on a copy, a tensor-core commit or a grid
 * barrier gives up after a time limit (2 s in the kernels), raises
 * KVARN_FLAG_WAIT_TIMEOUT in the device flag word and returns instead of hanging.
 * This call runs the same device wait code against conditions that never complete,
 * with a limit of `limit_us` microseconds (1..1000000), so a caller can check on its
 * own device that a wait that runs out is reported and leaves the device usable:
 *   which = KVARN_WAIT_MBARRIER: one warp waits on an mbarrier phase that expects
 *           16 bytes no copy delivers;
 *   which = KVARN_WAIT_GRID: a cooperative grid of one CTA per SM waits at a grid
 *           barrier that expects one CTA more than were launched; its barrier
 *           words are the first 8 bytes of `scratch` (device memory, 16-byte
 *           aligned, scratch_bytes >= 8; ignored for KVARN_WAIT_MBARRIER).
 * Nothing is copied or multiplied while the waits run. Asynchronous on `stream`;
 * read the flag with kvarn_device_flags. The serving step keeps its own barrier
 * words in its scratch and zeroes them on the stream before each launch, so a
 * timed-out barrier of one call never affects another.
 */
#define KVARN_WAIT_MBARRIER 0
#define KVARN_WAIT_GRID 1
KVARN_API kvarn_status kvarn_check_bounded_waits(int32_t which, uint32_t limit_us, void* scratch,
                                                 size_t scratch_bytes, void* stream);

/* Copies the device flag word of the current device to *flags (host pointer)
 * after synchronising `stream`, then clears it. */
KVARN_API kvarn_status kvarn_device_flags(uint32_t* flags, void* stream);

/* Message of the last error returned on the calling host thread ("" if none). */
KVARN_API const char* kvarn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H */
