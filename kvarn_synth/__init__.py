"""Seeded synthetic inputs for the KVarN tile-quantization and paged-decode workloads.

This module only draws random numbers and lays out index arrays. It holds none of
the method's arithmetic (no rotation, normalisation, rounding to codes or
attention), so both the CPU oracle and the CUDA library can take their inputs
from here without sharing any code with each other.

Distributions (the pages name Qwen3-32B at 16K-context bursts as their workload,
KVarN README, introduction; no dataset or weights are available, these draws
stand in for them):

* K: per (kv-head, channel) a standard deviation sigma ~ LogNormal(0, 0.5),
  fixed over tokens, and a handful of outlier channels per head multiplied by a
  large factor; x = N(0, 1) * sigma.
* V: per (token, kv-head) sigma ~ LogNormal(0, 0.5); x = N(0, 1) * sigma.
* q: N(0, 1).
* Paged layout: physical blocks are a random permutation of [0, num_blocks).

All generators use numpy PCG64 with the given seed, draw in float32 and round to
fp16 (round-to-nearest-even, numpy's conversion).
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128
BLOCK = 128


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ----------------------------------------------------------------------------------
# Single tile (one kv-head, 128 channels x 128 tokens)
# ----------------------------------------------------------------------------------
def single_tile(seed: int = 0, n_outliers: int = 4, outlier_factor: float = 20.0):
    """One tile of K and V as fp16 arrays laid out [token, channel] (128 x 128),
    plus one fp16 query [1, 128].

    K: per-channel std LogNormal(0, 0.5), `n_outliers` random channels x factor.
    V: per-token std LogNormal(0, 0.5).
    """
    g = _rng(seed)
    sig_k = g.lognormal(0.0, 0.5, size=HEAD_DIM)
    out_ch = g.choice(HEAD_DIM, size=n_outliers, replace=False)
    sig_k[out_ch] *= outlier_factor
    k = (g.standard_normal((BLOCK, HEAD_DIM)) * sig_k[None, :]).astype(np.float16)
    sig_v = g.lognormal(0.0, 0.5, size=BLOCK)
    v = (g.standard_normal((BLOCK, HEAD_DIM)) * sig_v[:, None]).astype(np.float16)
    q = g.standard_normal((1, HEAD_DIM)).astype(np.float16)
    return k, v, q


# ----------------------------------------------------------------------------------
# Prefill batches [n_tokens, Hkv, 128]
# ----------------------------------------------------------------------------------
def head_channel_sigmas(seed: int, n_kv_heads: int, outliers=(1, 6), factor=(10.0, 50.0)):
    """Per (kv-head, channel) K standard deviations with outlier channels."""
    g = _rng(seed ^ 0x5EED)
    sig = g.lognormal(0.0, 0.5, size=(n_kv_heads, HEAD_DIM))
    for h in range(n_kv_heads):
        n_out = int(g.integers(outliers[0], outliers[1] + 1))
        ch = g.choice(HEAD_DIM, size=n_out, replace=False)
        sig[h, ch] *= g.uniform(factor[0], factor[1], size=n_out)
    return sig.astype(np.float32)


def prefill_kv(n_tokens: int, n_kv_heads: int, seed: int, chunk: int = 1 << 16,
               outliers=(1, 6), factor=(10.0, 50.0)):
    """fp16 K and V, each [n_tokens, n_kv_heads, 128] (vLLM's key/value layout).

    Drawn in chunks of `chunk` tokens so memory stays bounded; the result only
    depends on (n_tokens, n_kv_heads, seed, chunk)."""
    sig_k = head_channel_sigmas(seed, n_kv_heads, outliers, factor)
    k = np.empty((n_tokens, n_kv_heads, HEAD_DIM), np.float16)
    v = np.empty((n_tokens, n_kv_heads, HEAD_DIM), np.float16)
    for c0 in range(0, n_tokens, chunk):
        n = min(chunk, n_tokens - c0)
        g = _rng(seed * 1_000_003 + c0 // chunk)
        xk = g.standard_normal((n, n_kv_heads, HEAD_DIM), dtype=np.float32)
        xk *= sig_k[None]
        k[c0:c0 + n] = xk.astype(np.float16)
        xv = g.standard_normal((n, n_kv_heads, HEAD_DIM), dtype=np.float32)
        sv = g.lognormal(0.0, 0.5, size=(n, n_kv_heads, 1)).astype(np.float32)
        xv *= sv
        v[c0:c0 + n] = xv.astype(np.float16)
    return k, v


def block_permutation(num_blocks: int, seed: int) -> np.ndarray:
    return _rng(seed ^ 0xB10C).permutation(num_blocks).astype(np.int64)


def prefill_slot_mapping(n_tokens: int, num_blocks: int, seed: int) -> np.ndarray:
    """slot[t] = perm[t // 128] * 128 + t % 128: each run of 128 tokens fills one
    randomly chosen physical block, in order."""
    assert n_tokens % BLOCK == 0 and n_tokens // BLOCK <= num_blocks
    perm = block_permutation(num_blocks, seed)[: n_tokens // BLOCK]
    t = np.arange(n_tokens, dtype=np.int64)
    return perm[t // BLOCK] * BLOCK + t % BLOCK


def queries(n_seqs: int, n_q_heads: int, seed: int) -> np.ndarray:
    return _rng(seed ^ 0x0A11).standard_normal((n_seqs, n_q_heads, HEAD_DIM),
                                               dtype=np.float32).astype(np.float16)


# ----------------------------------------------------------------------------------
# Decode layouts
# ----------------------------------------------------------------------------------
def block_tables(n_seqs: int, max_blocks: int, num_blocks: int, seed: int) -> np.ndarray:
    """int32 [n_seqs, max_blocks]: distinct physical blocks, randomly permuted."""
    assert n_seqs * max_blocks <= num_blocks
    perm = block_permutation(num_blocks, seed)[: n_seqs * max_blocks]
    return perm.reshape(n_seqs, max_blocks).astype(np.int32)


def ragged_lengths(n_seqs: int, lo: int, hi: int, seed: int, avoid_multiple: int = BLOCK):
    """Lengths log-uniform in [lo, hi], redrawn while L % avoid_multiple == 0 so that
    every sequence has a partial last tile."""
    g = _rng(seed ^ 0x1E9)
    out = np.empty(n_seqs, np.int32)
    for i in range(n_seqs):
        while True:
            L = int(round(float(np.exp(g.uniform(np.log(lo), np.log(hi))))))
            if avoid_multiple == 0 or L % avoid_multiple != 0:
                break
        out[i] = L
    return out


def random_records(n: int, seed: int, record_bytes: int, code_bytes: int) -> np.ndarray:
    """`n` packed cache records of `record_bytes` each: uniformly random code bytes
    followed by fp16 metadata drawn in plausible ranges (positive scales near 1,
    zeros near -2 in normalised units). Used where a decode workload needs a valid
    packed cache but not one made by a quantizer."""
    g = _rng(seed ^ 0xCAC4E)
    rec = np.empty((n, record_bytes), np.uint8)
    rec[:, :code_bytes] = g.integers(0, 256, size=(n, code_bytes), dtype=np.uint8)
    n_meta = (record_bytes - code_bytes) // 2
    meta = np.empty((n, n_meta), np.float16)
    # the metadata area holds 8 vectors of 128 halves: (r, c, s, z) for K then V
    q = n_meta // 8
    for blk in range(8):
        kind = blk % 4
        if kind in (0, 1):          # row / column scales
            vals = g.lognormal(0.0, 0.4, size=(n, q))
        elif kind == 2:             # step sizes
            vals = g.uniform(0.2, 1.6, size=(n, q))
        else:                       # zeros (group minima)
            vals = g.normal(-2.0, 0.3, size=(n, q))
        meta[:, blk * q:(blk + 1) * q] = vals.astype(np.float16)
    rec[:, code_bytes:] = meta.view(np.uint8).reshape(n, -1)
    return rec


def workspace_tokens(n_seqs: int, n_kv_heads: int, seed: int):
    """fp16 [n_seqs, n_kv_heads, 2, 128, 128] (K/V x token x channel) drawn with the
    prefill distributions, for sequences whose last tile is still partial."""
    k, v = prefill_kv(n_seqs * BLOCK, n_kv_heads, seed)
    k = k.reshape(n_seqs, BLOCK, n_kv_heads, HEAD_DIM).transpose(0, 2, 1, 3)
    v = v.reshape(n_seqs, BLOCK, n_kv_heads, HEAD_DIM).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(np.stack([k, v], axis=2))


# ----------------------------------------------------------------------------------
# The five named workloads (sizes only; seeds fixed)
# ----------------------------------------------------------------------------------
WORKLOADS = {
    "single_tile": dict(n_kv_heads=1, n_q_heads=1, seed=0),
    "prefill_16x16k": dict(n_seqs=16, seq_len=16384, n_kv_heads=8, seed=1),
    "decode_64x16k": dict(n_seqs=64, seq_len=16384, n_kv_heads=8, n_q_heads=64, seed=2),
    "decode_4x128k": dict(n_seqs=4, seq_len=131072, n_kv_heads=8, n_q_heads=64, seed=3),
    "serve_256_ragged": dict(n_seqs=256, lo=1024, hi=32768, n_kv_heads=8, n_q_heads=64, seed=7),
}
