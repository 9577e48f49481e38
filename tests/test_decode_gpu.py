"""Parity of kvarn_decode_attention (CUDA, through the C ABI) with the CPU oracle.
The packed caches are made by the oracle's quantizer (small cases, and every block
of the sampled pairs at full sizes; random valid records fill the rest of a
full-size cache), never by the CUDA quantizer."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import assert_decode_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()
    return kv, torch


def f16_to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()


def gpu_decode(env, q, cache, ws, bt, lens, hkv, num_blocks):
    kv, torch = env
    n_seqs, hq, _ = q.shape
    meta = kv.make_meta(hkv, hq, num_blocks, max_blocks_per_seq=bt.shape[1])
    out = torch.full((n_seqs, hq, 128), float("nan"), dtype=torch.float16, device="cuda")
    scratch = torch.empty(max(kv.decode_scratch_bytes(meta, n_seqs), 16), dtype=torch.uint8, device="cuda")
    cache_d = cache if hasattr(cache, "is_cuda") else torch.from_numpy(cache).cuda()
    kv.kvarn_decode_attention(f16_to_dev(torch, q), cache_d, None if ws is None else f16_to_dev(torch, ws),
                              torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(), out, scratch, meta)
    flags = kv.kvarn_device_flags()
    return out.float().cpu().numpy().astype(np.float64), flags


def oracle_cache(hkv, lens, seed, max_blocks):
    """Cache, block tables and workspace holding sequences of the given lengths,
    quantized by the oracle."""
    n_seqs = len(lens)
    num_blocks = n_seqs * max_blocks + 3
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    cache = np.zeros((num_blocks, hkv, o.RECORD_BYTES), np.uint8)
    ws = np.zeros((n_seqs, hkv, 2, 128, 128), np.float16)
    for s, L in enumerate(lens):
        nf = L // 128
        k, v = synth.prefill_kv(max(L, 1), hkv, seed=seed * 100 + s)
        if nf:
            slots = np.concatenate([bt[s, b] * 128 + np.arange(128) for b in range(nf)]).astype(np.int64)
            o.quantize_into_cache(k[:nf * 128], v[:nf * 128], slots, cache)
        nw = L % 128
        ws[s, :, 0, :nw] = k[nf * 128:L].transpose(1, 0, 2)
        ws[s, :, 1, :nw] = v[nf * 128:L].transpose(1, 0, 2)
    return cache, bt, ws, num_blocks


def test_single_tile_decode(env):
    k, v, q = synth.single_tile(0)
    rec, _, _ = o.quantize_tiles(k, v)
    cache = np.zeros((2, 1, o.RECORD_BYTES), np.uint8)
    cache[1, 0] = rec
    bt = np.array([[1]], np.int32)
    lens = np.array([128], np.int32)
    out, flags = gpu_decode(env, q[None], cache, None, bt, lens, 1, 2)
    assert flags == 0
    ref = o.decode(q[None].astype(np.float64), cache, None, bt, lens)
    assert_decode_close(out, ref, "single tile")


@pytest.mark.parametrize("group,hkv", [(1, 2), (2, 2), (4, 2), (8, 2), (8, 3), (3, 5)])
def test_ragged_lengths_and_groups(env, group, hkv):
    lens = np.array([1, 127, 128, 129, 300, 640, 1000, 2047, 2300, 0], np.int32)
    cache, bt, ws, nb = oracle_cache(hkv, lens, seed=30 + group, max_blocks=19)
    q = synth.queries(len(lens), hkv * group, seed=31)
    out, flags = gpu_decode(env, q, cache, ws, bt, lens, hkv, nb)
    assert flags == 0
    pairs = [(s, h) for s in range(len(lens)) if lens[s] > 0 for h in range(hkv)]
    ref = o.decode(q.astype(np.float64), cache, ws, bt, lens, pairs=pairs)
    ref[lens == 0] = 0.0                      # no tokens: the library writes zeros
    assert_decode_close(out, ref, f"group {group}")


def _config_case(env, n_seqs, seq_len, hkv, hq, seed, n_pairs):
    """A full-size decode workload whose sampled (sequence, kv-head) pairs hold K/V
    drawn like the prefill batch (outlier key channels x10-x50) and quantized by the
    oracle into every block of the pair; random valid records fill the rest of the
    cache. The oracle's decode of each sampled pair runs over exactly those records
    (in worker processes, tests/oracle_pool.py)."""
    from tests.oracle_pool import run_pairs
    kv, torch = env
    max_blocks = seq_len // 128
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    recs = synth.random_records(num_blocks * hkv, seed, o.RECORD_BYTES, 12288).reshape(num_blocks, hkv, -1)
    q = synth.queries(n_seqs, hq, seed)
    g = hq // hkv
    rng = np.random.default_rng(seed)
    all_pairs = [(s, h) for s in range(n_seqs) for h in range(hkv)]
    pick = rng.choice(len(all_pairs), size=min(n_pairs, len(all_pairs)), replace=False)
    pairs = sorted(all_pairs[int(i)] for i in pick)
    jobs = [(1_000_003 * seed + 64 * s + h, seq_len, q[s, h * g:(h + 1) * g], "k4v2") for s, h in pairs]
    res = run_pairs(jobs)
    for (s, h), (r, _, _) in zip(pairs, res):
        recs[bt[s], h] = r
    lens = np.full(n_seqs, seq_len, np.int32)
    out, flags = gpu_decode(env, q, torch.from_numpy(recs).cuda(), None, bt, lens, hkv, num_blocks)
    assert flags == 0
    worst = 0.0
    for (s, h), (_, _, ref) in zip(pairs, res):
        worst = max(worst, assert_decode_close(out[s, h * g:(h + 1) * g], ref, f"seq {s} head {h}"))
    assert np.isfinite(out).all()
    print(f"{len(pairs)} oracle-quantized pairs, max |err| {worst:.2e}")


def test_decode_64x16k_sampled(env):
    """Full decode workload: 64 sequences x 16384 tokens, 64 q-heads over 8 kv-heads;
    64 sampled (sequence, kv-head) pairs hold oracle-quantized K/V of the prefill
    distribution."""
    _config_case(env, 64, 16384, 8, 64, seed=2, n_pairs=64)


def test_decode_4x128k_sampled(env):
    """Long-context workload: 4 sequences x 131072 tokens, split-K; every one of the
    32 (sequence, kv-head) pairs holds oracle-quantized K/V of the prefill
    distribution."""
    _config_case(env, 4, 131072, 8, 64, seed=3, n_pairs=32)


@pytest.mark.parametrize("group", [1, 3, 8])
def test_ragged_lengths_many_units(env, group):
    """More (sequence, kv-head) units than SMs, so the split phase runs its 12-warp,
    one-stage shape with the L2 prefetch: 200 sequences cycling through empty, one-token,
    tile-edge and multi-tile lengths (with workspace tails), one kv-head with 1, 3 or 8
    q-heads; then the same batch with one block-table entry out of range."""
    kv, _ = env
    pattern = [0, 1, 127, 128, 129, 255, 256, 300, 383, 640]
    lens = np.array([pattern[i % len(pattern)] for i in range(200)], np.int32)
    cache, bt, ws, nb = oracle_cache(1, lens, seed=36, max_blocks=5)
    q = synth.queries(len(lens), group, seed=37)
    out, flags = gpu_decode(env, q, cache, ws, bt, lens, 1, nb)
    assert flags == 0
    pairs = [(s, 0) for s in range(len(lens)) if lens[s] > 0]
    ref = o.decode(q.astype(np.float64), cache, ws, bt, lens, pairs=pairs)
    ref[lens == 0] = 0.0
    assert_decode_close(out, ref, "many units")
    # one sequence's second block out of range: flagged, that tile skipped, the rest exact
    s_bad = int(np.nonzero(lens == 640)[0][0])
    bt_bad = bt.copy()
    bt_bad[s_bad, 1] = nb + 7
    out2, flags2 = gpu_decode(env, q, cache, ws, bt_bad, lens, 1, nb)
    assert flags2 & kv.FLAG_BAD_BLOCK
    assert np.isfinite(out2).all()
    keep = np.ones(len(lens), bool)
    keep[s_bad] = False
    assert_decode_close(out2[keep], ref[keep], "many units, other sequences")


def test_bad_block_is_skipped_and_flagged(env):
    kv, _ = env
    hkv = 1
    lens = np.array([384], np.int32)
    cache, bt, ws, nb = oracle_cache(hkv, lens, seed=33, max_blocks=3)
    bt_bad = bt.copy()
    bt_bad[0, 1] = nb + 5
    q = synth.queries(1, 8, seed=33)
    out, flags = gpu_decode(env, q, cache, ws, bt_bad, lens, hkv, nb)
    assert flags & kv.FLAG_BAD_BLOCK
    assert np.isfinite(out).all()
    # the output is attention over the two valid tiles
    kh, vh = o.dequant_record(cache[[bt[0, 0], bt[0, 2]], 0])
    kt = np.concatenate([kh[0].T, kh[1].T]); vt = np.concatenate([vh[0].T, vh[1].T])
    assert_decode_close(out[0], o.attend(q[0].astype(np.float64), kt, vt), "skipped block")


def test_length_beyond_block_table_is_clipped_and_flagged(env):
    kv, _ = env
    lens = np.array([256 + 5], np.int32)
    cache, bt, ws, nb = oracle_cache(1, lens, seed=34, max_blocks=2)
    q = synth.queries(1, 4, seed=34)
    lens_bad = np.array([3 * 128 + 5], np.int32)      # claims 3 full tiles, table holds 2
    out, flags = gpu_decode(env, q, cache, ws, bt, lens_bad, 1, nb)
    assert flags & kv.FLAG_BAD_LENGTH
    ref = o.decode(q.astype(np.float64), cache, ws, bt, lens)
    assert_decode_close(out, ref, "clipped")
