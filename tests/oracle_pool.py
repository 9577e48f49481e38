"""Oracle work spread over the host's cores for the full-size parity tests.

The oracle stays what it is (plain float64 NumPy, one tile at a time); this module
only runs independent pieces of it in a process pool started with `spawn` (safe
after CUDA is initialised in the test process). Each piece draws its own inputs
from kvarn_synth, quantizes them with the oracle and, where asked, computes the
oracle's decode attention over exactly those records, so nothing in it comes from
the CUDA path."""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def pair_draws(seed: int, n_tokens: int):
    """K and V of one (sequence, kv-head) pair: [n_tokens, 128] fp16 each, drawn like
    the prefill batch (per-channel key sigmas with 1-6 outlier channels x10-x50,
    per-token value sigmas)."""
    import kvarn_synth as synth
    k, v = synth.prefill_kv(n_tokens, 1, seed=seed)
    return k[:, 0], v[:, 0]


def pair_records_and_decode(seed: int, n_tokens: int, q_heads, preset: str = "k4v2"):
    """Oracle records of the pair's floor(n_tokens / 128) full tiles [n_full, bytes],
    its workspace tail [2, 128, 128] fp16 (the last n_tokens % 128 tokens, zero
    padded) and, if q_heads [G, 128] is given, the oracle's decode attention of those
    heads over the n_tokens tokens (records then tail)."""
    from oracle import kvarn_oracle as o
    k, v = pair_draws(seed, max(n_tokens, 1))
    n_full = n_tokens // 128
    recs = []
    for b0 in range(0, n_full, 32):
        b1 = min(n_full, b0 + 32)
        kt = k[b0 * 128:b1 * 128].reshape(-1, 128, 128)
        vt = v[b0 * 128:b1 * 128].reshape(-1, 128, 128)
        r, _, _ = o.quantize_tiles(kt, vt, preset=preset)
        recs.append(r)
    lay = o.LAYOUTS[preset]
    recs = np.concatenate(recs) if recs else np.zeros((0, lay.record_bytes), np.uint8)
    tail = np.zeros((2, 128, 128), np.float16)
    nw = n_tokens % 128
    tail[0, :nw] = k[n_full * 128:n_tokens]
    tail[1, :nw] = v[n_full * 128:n_tokens]
    out = None
    if q_heads is not None:
        out = o.decode_one(np.asarray(q_heads, np.float64), recs[:, None, :], tail if nw else None,
                           np.arange(n_full), n_tokens, 0)
    return recs, tail, out


def _call(args):
    return pair_records_and_decode(*args)


def run_pairs(jobs, workers: int | None = None):
    """jobs: list of (seed, n_tokens, q_heads or None, preset); returns the results in
    order. Uses up to os.cpu_count() (at most 32) spawned worker processes, each with
    single-threaded BLAS."""
    if not jobs:
        return []
    n = workers or min(32, os.cpu_count() or 1, len(jobs))
    if n <= 1:
        return [_call(j) for j in jobs]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
            return list(ex.map(_call, jobs, chunksize=1))
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
