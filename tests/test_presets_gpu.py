"""Parity of the k4v4, k2v2 and k4v2l presets (quantize, decode, append; CUDA through the
C ABI) with the CPU oracle, under the same tolerances as the default preset."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import assert_decode_close, compare_records

pytestmark = pytest.mark.gpu

PRESETS = ["k4v4", "k2v2", "k4v2l"]


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()
    return kv, torch


def f16_to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()


def record_bytes(preset):
    return o.LAYOUTS[preset].record_bytes


@pytest.mark.parametrize("preset", PRESETS)
def test_quantize_single_and_multi_tile(env, preset):
    kv, torch = env
    # one tile with outlier channels
    k, v, _ = synth.single_tile(0)
    meta = kv.make_meta(1, 1, 2, preset=preset)
    cache = torch.zeros(2, 1, record_bytes(preset), dtype=torch.uint8, device="cuda")
    kv.kvarn_quantize_tiles(f16_to_dev(torch, k[:, None, :]), f16_to_dev(torch, v[:, None, :]),
                            torch.arange(128, 256, dtype=torch.int64, device="cuda"), cache, meta)
    assert kv.kvarn_device_flags() == 0
    _, kq, vq = o.quantize_tiles(k[None], v[None], preset=preset)
    got = cache.cpu().numpy()
    print(preset, "single", compare_records(got[1:2, 0], kq, vq))
    assert not got[0].any()
    # several tiles and heads, scattered blocks
    hkv, n_chunks, num_blocks = 4, 12, 16
    k, v = synth.prefill_kv(n_chunks * 128, hkv, seed=71)
    slots = synth.prefill_slot_mapping(n_chunks * 128, num_blocks, seed=71)
    meta = kv.make_meta(hkv, hkv, num_blocks, preset=preset)
    cache = torch.zeros(num_blocks, hkv, record_bytes(preset), dtype=torch.uint8, device="cuda")
    kv.kvarn_quantize_tiles(f16_to_dev(torch, k), f16_to_dev(torch, v), torch.from_numpy(slots).cuda(), cache, meta)
    assert kv.kvarn_device_flags() == 0
    pairs = [(c, h) for c in range(n_chunks) for h in range(hkv)]
    kt = np.stack([k[c * 128:(c + 1) * 128, h] for c, h in pairs])
    vt = np.stack([v[c * 128:(c + 1) * 128, h] for c, h in pairs])
    _, kq, vq = o.quantize_tiles(kt, vt, preset=preset)
    got = cache.cpu().numpy()
    blocks = np.array([slots[c * 128] // 128 for c, _ in pairs])
    heads = np.array([h for _, h in pairs])
    print(preset, "multi", compare_records(got[blocks, heads], kq, vq))


@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("n_iters", [1, 3])
def test_quantize_iteration_counts(env, preset, n_iters):
    """Other iteration counts per preset (with one iteration the keys' token scales
    are fixed straight after the first column pass)."""
    kv, torch = env
    hkv, n_chunks, num_blocks = 2, 6, 8
    k, v = synth.prefill_kv(n_chunks * 128, hkv, seed=77 + n_iters)
    slots = synth.prefill_slot_mapping(n_chunks * 128, num_blocks, seed=77)
    meta = kv.make_meta(hkv, hkv, num_blocks, n_iters=n_iters, preset=preset)
    cache = torch.zeros(num_blocks, hkv, record_bytes(preset), dtype=torch.uint8, device="cuda")
    kv.kvarn_quantize_tiles(f16_to_dev(torch, k), f16_to_dev(torch, v), torch.from_numpy(slots).cuda(), cache, meta)
    assert kv.kvarn_device_flags() == 0
    pairs = [(c, h) for c in range(n_chunks) for h in range(hkv)]
    kt = np.stack([k[c * 128:(c + 1) * 128, h] for c, h in pairs])
    vt = np.stack([v[c * 128:(c + 1) * 128, h] for c, h in pairs])
    _, kq, vq = o.quantize_tiles(kt, vt, n_iters, preset=preset)
    got = cache.cpu().numpy()
    blocks = np.array([slots[c * 128] // 128 for c, _ in pairs])
    heads = np.array([h for _, h in pairs])
    print(preset, n_iters, compare_records(got[blocks, heads], kq, vq))


def _gpu_decode(env, q, cache, ws, bt, lens, hkv, num_blocks, preset):
    kv, torch = env
    n_seqs, hq, _ = q.shape
    meta = kv.make_meta(hkv, hq, num_blocks, max_blocks_per_seq=bt.shape[1], preset=preset)
    out = torch.full((n_seqs, hq, 128), float("nan"), dtype=torch.float16, device="cuda")
    scratch = torch.empty(max(kv.decode_scratch_bytes(meta, n_seqs), 16), dtype=torch.uint8, device="cuda")
    cache_d = cache if hasattr(cache, "is_cuda") else torch.from_numpy(cache).cuda()
    kv.kvarn_decode_attention(f16_to_dev(torch, q), cache_d, None if ws is None else f16_to_dev(torch, ws),
                              torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(), out, scratch, meta)
    return out.float().cpu().numpy().astype(np.float64), kv.kvarn_device_flags()


@pytest.mark.parametrize("preset", PRESETS)
def test_decode_ragged_over_oracle_cache(env, preset):
    hkv, group, max_blocks = 2, 8, 12
    lens = np.array([1, 127, 128, 129, 300, 640, 1000, 1500, 0], np.int32)
    n_seqs = len(lens)
    num_blocks = n_seqs * max_blocks + 3
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, 72)
    cache = np.zeros((num_blocks, hkv, record_bytes(preset)), np.uint8)
    ws = np.zeros((n_seqs, hkv, 2, 128, 128), np.float16)
    for s, L in enumerate(lens):
        nf = L // 128
        k, v = synth.prefill_kv(max(L, 1), hkv, seed=7200 + s)
        if nf:
            slots = np.concatenate([bt[s, b] * 128 + np.arange(128) for b in range(nf)]).astype(np.int64)
            o.quantize_into_cache(k[:nf * 128], v[:nf * 128], slots, cache)
        nw = L % 128
        ws[s, :, 0, :nw] = k[nf * 128:L].transpose(1, 0, 2)
        ws[s, :, 1, :nw] = v[nf * 128:L].transpose(1, 0, 2)
    q = synth.queries(n_seqs, hkv * group, seed=73)
    out, flags = _gpu_decode(env, q, cache, ws, bt, lens, hkv, num_blocks, preset)
    assert flags == 0
    pairs = [(s, h) for s in range(n_seqs) if lens[s] > 0 for h in range(hkv)]
    ref = o.decode(q.astype(np.float64), cache, ws, bt, lens, pairs=pairs)
    ref[lens == 0] = 0.0
    print(preset, "decode max err", assert_decode_close(out, ref, preset))


@pytest.mark.parametrize("preset", PRESETS)
def test_decode_random_records_sampled(env, preset):
    """8 sequences x 4096 tokens, 64 q-heads over 8 kv-heads, random valid records;
    sampled (sequence, kv-head) pairs against the oracle."""
    kv, torch = env
    n_seqs, seq_len, hkv, hq, seed = 8, 4096, 8, 64, 74
    max_blocks = seq_len // 128
    num_blocks = n_seqs * max_blocks
    lay = o.LAYOUTS[preset]
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    recs = synth.random_records(num_blocks * hkv, seed, lay.record_bytes, lay.k_code_bytes + lay.v_code_bytes)
    recs = recs.reshape(num_blocks, hkv, -1)
    q = synth.queries(n_seqs, hq, seed)
    lens = np.full(n_seqs, seq_len, np.int32)
    out, flags = _gpu_decode(env, q, torch.from_numpy(recs).cuda(), None, bt, lens, hkv, num_blocks, preset)
    assert flags == 0 and np.isfinite(out).all()
    rng = np.random.default_rng(seed)
    pairs = sorted({(int(s), int(h)) for s, h in zip(rng.integers(0, n_seqs, 10), rng.integers(0, hkv, 10))})
    ref = o.decode(q.astype(np.float64), recs, None, bt, lens, pairs=pairs)
    g = hq // hkv
    for s, h in pairs:
        assert_decode_close(out[s, h * g:(h + 1) * g], ref[s, h * g:(h + 1) * g], f"{preset} seq {s} head {h}")


@pytest.mark.parametrize("preset", PRESETS)
def test_append_completes_tiles(env, preset):
    kv, torch = env
    hkv, n_seqs, max_blocks = 2, 6, 4
    lens = np.array([0, 5, 126, 127, 255, 383], np.int32)
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed=75)
    ws = synth.workspace_tokens(n_seqs, hkv, seed=75)
    cache = np.zeros((num_blocks, hkv, record_bytes(preset)), np.uint8)
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=76)
    meta = kv.make_meta(hkv, hkv, num_blocks, max_blocks_per_seq=max_blocks, preset=preset)
    ws_d = f16_to_dev(torch, ws)
    cache_d = torch.from_numpy(cache).cuda()
    lens_out = torch.full((n_seqs,), -7, dtype=torch.int32, device="cuda")
    kv.kvarn_append_decode(f16_to_dev(torch, k_new), f16_to_dev(torch, v_new), torch.from_numpy(lens).cuda(),
                           lens_out, torch.from_numpy(bt).cuda(), ws_d, cache_d, meta)
    assert kv.kvarn_device_flags() == 0
    assert (lens_out.cpu().numpy() == lens + 1).all()
    ws_ref, _, _ = o.append(k_new, v_new, lens, bt, ws, cache)
    assert np.array_equal(ws_d.cpu().view(torch.int16).numpy().view(np.float16), ws_ref)
    done = [s for s in range(n_seqs) if lens[s] % 128 == 127]
    kt = np.stack([ws_ref[s, :, 0] for s in done]).reshape(-1, 128, 128)
    vt = np.stack([ws_ref[s, :, 1] for s in done]).reshape(-1, 128, 128)
    _, kq, vq = o.quantize_tiles(kt, vt, preset=preset)
    got = cache_d.cpu().numpy()
    blocks = np.array([bt[s, lens[s] // 128] for s in done]).repeat(hkv)
    heads = np.tile(np.arange(hkv), len(done))
    print(preset, "append", compare_records(got[blocks, heads], kq, vq))


@pytest.mark.parametrize("preset", PRESETS)
def test_decode_64x16k_oracle_pairs(env, preset):
    """The full decode workload (64 sequences x 16384 tokens, 64 q-heads over 8
    kv-heads) in each preset's layout: 16 sampled (sequence, kv-head) pairs hold K/V
    drawn like the prefill batch (outlier key channels x10-x50), quantized by the
    oracle into every block of the pair; random valid records fill the rest. The
    oracle's decode of each sampled pair runs over exactly those records."""
    from tests.oracle_pool import run_pairs
    kv, torch = env
    n_seqs, seq_len, hkv, hq, seed = 64, 16384, 8, 64, 78
    max_blocks = seq_len // 128
    num_blocks = n_seqs * max_blocks
    lay = o.LAYOUTS[preset]
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    recs = synth.random_records(num_blocks * hkv, seed, lay.record_bytes, lay.k_code_bytes + lay.v_code_bytes)
    recs = recs.reshape(num_blocks, hkv, -1)
    q = synth.queries(n_seqs, hq, seed)
    g = hq // hkv
    rng = np.random.default_rng(seed)
    all_pairs = [(s, h) for s in range(n_seqs) for h in range(hkv)]
    pairs = sorted(all_pairs[int(i)] for i in rng.choice(len(all_pairs), size=16, replace=False))
    res = run_pairs([(1_000_003 * seed + 64 * s + h, seq_len, q[s, h * g:(h + 1) * g], preset) for s, h in pairs])
    for (s, h), (r, _, _) in zip(pairs, res):
        recs[bt[s], h] = r
    lens = np.full(n_seqs, seq_len, np.int32)
    out, flags = _gpu_decode(env, q, torch.from_numpy(recs).cuda(), None, bt, lens, hkv, num_blocks, preset)
    assert flags == 0 and np.isfinite(out).all()
    worst = 0.0
    for (s, h), (_, _, ref) in zip(pairs, res):
        worst = max(worst, assert_decode_close(out[s, h * g:(h + 1) * g], ref, f"{preset} seq {s} head {h}"))
    print(preset, f"{len(pairs)} oracle-quantized pairs at 64 x 16384, max |err| {worst:.2e}")


@pytest.mark.parametrize("preset", PRESETS)
def test_quantize_16x16k_sampled(env, preset):
    """The full prefill workload (16 sequences x 16384 tokens, 8 kv-heads) in each
    preset's layout, in the benchmark's launch configuration; 64 sampled tile-heads
    against the oracle."""
    kv, torch = env
    n_tokens, hkv = 16 * 16384, 8
    num_blocks = n_tokens // 128
    k, v = synth.prefill_kv(n_tokens, hkv, seed=1)
    slots = synth.prefill_slot_mapping(n_tokens, num_blocks, seed=1)
    meta = kv.make_meta(hkv, hkv, num_blocks, preset=preset)
    cache = torch.zeros(num_blocks, hkv, record_bytes(preset), dtype=torch.uint8, device="cuda")
    kv.kvarn_quantize_tiles(f16_to_dev(torch, k), f16_to_dev(torch, v), torch.from_numpy(slots).cuda(), cache, meta)
    assert kv.kvarn_device_flags() == 0
    rng = np.random.default_rng(79)
    pairs = [(int(c), int(h)) for c, h in zip(rng.integers(0, num_blocks, 64), rng.integers(0, hkv, 64))]
    kt = np.stack([k[c * 128:(c + 1) * 128, h] for c, h in pairs])
    vt = np.stack([v[c * 128:(c + 1) * 128, h] for c, h in pairs])
    _, kq, vq = o.quantize_tiles(kt, vt, preset=preset)
    got = cache.cpu().numpy()
    blocks = np.array([slots[c * 128] // 128 for c, _ in pairs])
    heads = np.array([h for _, h in pairs])
    print(preset, "16 x 16384", compare_records(got[blocks, heads], kq, vq))


@pytest.mark.parametrize("preset", PRESETS)
def test_decode_4x128k_oracle_pairs(env, preset):
    """The long-context decode (4 sequences x 131072 tokens, 64 q-heads over 8
    kv-heads: a few long units, the two-stage split shape and the merge that splits
    a unit's records four ways) in each preset's layout: 4 sampled (sequence, kv-head)
    pairs hold oracle-quantized K/V of the prefill distribution in every block, random
    valid records fill the rest."""
    from tests.oracle_pool import run_pairs
    kv, torch = env
    n_seqs, seq_len, hkv, hq, seed = 4, 131072, 8, 64, 81
    max_blocks = seq_len // 128
    num_blocks = n_seqs * max_blocks
    lay = o.LAYOUTS[preset]
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    recs = synth.random_records(num_blocks * hkv, seed, lay.record_bytes, lay.k_code_bytes + lay.v_code_bytes)
    recs = recs.reshape(num_blocks, hkv, -1)
    q = synth.queries(n_seqs, hq, seed)
    g = hq // hkv
    pairs = [(0, 3), (1, 0), (2, 7), (3, 5)]
    res = run_pairs([(1_000_003 * seed + 64 * s + h, seq_len, q[s, h * g:(h + 1) * g], preset) for s, h in pairs])
    for (s, h), (r, _, _) in zip(pairs, res):
        recs[bt[s], h] = r
    lens = np.full(n_seqs, seq_len, np.int32)
    out, flags = _gpu_decode(env, q, torch.from_numpy(recs).cuda(), None, bt, lens, hkv, num_blocks, preset)
    assert flags == 0 and np.isfinite(out).all()
    worst = 0.0
    for (s, h), (_, _, ref) in zip(pairs, res):
        worst = max(worst, assert_decode_close(out[s, h * g:(h + 1) * g], ref, f"{preset} seq {s} head {h}"))
    print(preset, f"{len(pairs)} oracle-quantized pairs at 4 x 131072, max |err| {worst:.2e}")
