"""Parity of kvarn_append_decode (CUDA, through the C ABI) with the CPU oracle, and
the mixed serving step (append one token per sequence, then decode)."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import assert_decode_close, compare_records

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


def dev_to_f16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.float16)


def gpu_append(env, k_new, v_new, lens, bt, ws, cache, num_blocks):
    kv, torch = env
    n_seqs, hkv, _ = k_new.shape
    meta = kv.make_meta(hkv, hkv, num_blocks, max_blocks_per_seq=bt.shape[1])
    ws_d = f16_to_dev(torch, ws)
    cache_d = cache if hasattr(cache, "is_cuda") else torch.from_numpy(cache).cuda()
    lens_out = torch.full((n_seqs,), -7, dtype=torch.int32, device="cuda")
    kv.kvarn_append_decode(f16_to_dev(torch, k_new), f16_to_dev(torch, v_new), torch.from_numpy(lens).cuda(),
                           lens_out, torch.from_numpy(bt).cuda(), ws_d, cache_d, meta)
    flags = kv.kvarn_device_flags()
    return ws_d, cache_d, lens_out.cpu().numpy(), flags


@pytest.mark.parametrize("hkv", [2, 3])
def test_append_small(env, hkv):
    n_seqs, max_blocks = 6, 4
    lens = np.array([0, 5, 126, 127, 255, 383], np.int32)
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed=40)
    ws = synth.workspace_tokens(n_seqs, hkv, seed=40)
    cache = np.zeros((num_blocks, hkv, o.RECORD_BYTES), np.uint8)
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=41)
    ws_d, cache_d, lens_out, flags = gpu_append(env, k_new, v_new, lens, bt, ws, cache, num_blocks)
    assert flags == 0
    assert (lens_out == lens + 1).all()
    ws_ref, cache_ref, _ = o.append(k_new, v_new, lens, bt, ws, cache)
    assert np.array_equal(dev_to_f16(ws_d), ws_ref)
    cache_g = cache_d.cpu().numpy()
    done = [s for s in range(n_seqs) if lens[s] % 128 == 127]
    assert len(done) == 3
    for s in done:
        blk = bt[s, lens[s] // 128]
        _, kq, vq = o.quantize_tiles(ws_ref[s, :, 0], ws_ref[s, :, 1])
        print("append tile", s, compare_records(cache_g[blk], kq, vq))
    untouched = np.ones(num_blocks, bool)
    untouched[[bt[s, lens[s] // 128] for s in done]] = False
    assert not cache_g[untouched].any()


def test_append_bad_block_flagged(env):
    kv, _ = env
    lens = np.array([127], np.int32)
    bt = np.array([[9]], np.int32)                        # outside num_blocks = 2
    ws = synth.workspace_tokens(1, 1, seed=42)
    k_new, v_new = synth.prefill_kv(1, 1, seed=42)
    _, cache_d, lens_out, flags = gpu_append(env, k_new, v_new, lens, bt, ws, np.zeros((2, 1, o.RECORD_BYTES), np.uint8), 2)
    assert flags & kv.FLAG_BAD_BLOCK
    assert not cache_d.cpu().numpy().any()
    assert lens_out[0] == 128


def test_serving_step_256_ragged(env):
    """Mixed serving step: 256 sequences, lengths log-uniform in [1024, 32768] with a
    partial last tile each (every 8th forced to L % 128 == 127 so the append
    completes a tile); append one token, then decode with 64 q-heads over 8
    kv-heads. Sampled sequences are checked against the oracle."""
    kv, torch = env
    cfg = synth.WORKLOADS["serve_256_ragged"]
    n_seqs, hkv, hq, seed = cfg["n_seqs"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["seed"]
    lens = synth.ragged_lengths(n_seqs, cfg["lo"], cfg["hi"], seed)
    lens[::8] = (lens[::8] // 128) * 128 + 127
    max_blocks = int(max((L + 1 + 127) // 128 for L in lens))
    n_full = lens // 128
    total_blocks = int(((lens + 1 + 127) // 128).sum())
    num_blocks = total_blocks + 16
    perm = synth.block_permutation(num_blocks, seed)
    bt = np.full((n_seqs, max_blocks), -1, np.int32)
    pos = 0
    for s in range(n_seqs):
        nb = (lens[s] + 1 + 127) // 128
        bt[s, :nb] = perm[pos:pos + nb]
        pos += nb
    recs = synth.random_records(num_blocks * hkv, seed, o.RECORD_BYTES, 12288).reshape(num_blocks, hkv, -1)
    ws = synth.workspace_tokens(n_seqs, hkv, seed)
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=seed + 1)
    ws_d, cache_d, lens_out, flags = gpu_append(env, k_new, v_new, lens, bt, ws, recs, num_blocks)
    assert flags == 0 and (lens_out == lens + 1).all()
    # completed tiles: GPU records vs oracle quantization of the completed workspace tile
    ws_g = dev_to_f16(ws_d)
    done = [s for s in range(n_seqs) if lens[s] % 128 == 127]
    kt = np.stack([ws_g[s, :, 0] for s in done]).reshape(-1, 128, 128)
    vt = np.stack([ws_g[s, :, 1] for s in done]).reshape(-1, 128, 128)
    for n, s in enumerate(done):                                   # workspace tile = old tokens + new one
        assert np.array_equal(ws_g[s, :, :, :127], ws[s, :, :, :127])
        assert np.array_equal(ws_g[s, :, 0, 127], k_new[s]) and np.array_equal(ws_g[s, :, 1, 127], v_new[s])
    recs_ref, kq, vq = o.quantize_tiles(kt, vt)
    cache_g = cache_d.cpu().numpy()
    blocks = np.array([bt[s, lens[s] // 128] for s in done]).repeat(hkv)
    heads = np.tile(np.arange(hkv), len(done))
    print("serving step", compare_records(cache_g[blocks, heads], kq, vq))
    # decode over the post-append state, with the oracle's records for the completed tiles
    cache_g[blocks, heads] = recs_ref
    lens_new = lens + 1
    meta = kv.make_meta(hkv, hq, num_blocks, max_blocks_per_seq=max_blocks)
    q = synth.queries(n_seqs, hq, seed)
    out = torch.empty((n_seqs, hq, 128), dtype=torch.float16, device="cuda")
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    kv.kvarn_decode_attention(f16_to_dev(torch, q), torch.from_numpy(cache_g).cuda(), ws_d,
                              torch.from_numpy(bt).cuda(), torch.from_numpy(lens_new).cuda(), out, scratch, meta)
    assert kv.kvarn_device_flags() == 0
    out = out.float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(seed)
    sample = sorted(set(rng.integers(0, n_seqs, 6).tolist()) | {done[0], int(np.argmin(lens)), int(np.argmax(lens))})
    pairs = [(s, h) for s in sample for h in (0, hkv - 1)]
    ref = o.decode(q.astype(np.float64), cache_g, ws_g, bt, lens_new, pairs=pairs)
    g = hq // hkv
    for s, h in pairs:
        assert_decode_close(out[s, h * g:(h + 1) * g], ref[s, h * g:(h + 1) * g], f"seq {s} head {h}")
    assert np.isfinite(out).all()


def test_append_many_items(env):
    """More (sequence, kv-head) items than 32 per block (1300 sequences x 4 kv-heads,
    ~34 items a block); every 7th sequence completes a tile, and the completing items
    are handed out to the blocks by rank (the batch is under 32768 items; the larger
    batches of tests/test_large_offsets_gpu.py take the ballot path). The new rows,
    the lengths, 64 sampled completed tiles against the oracle, and every other block
    untouched."""
    n_seqs, hkv, max_blocks = 1300, 4, 5
    rng = np.random.default_rng(43)
    lens = rng.integers(0, 600, n_seqs).astype(np.int32)
    lens[::7] = (lens[::7] // 128) * 128 + 127
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed=43)
    ws = synth.workspace_tokens(n_seqs, hkv, seed=43)
    cache = np.zeros((num_blocks, hkv, o.RECORD_BYTES), np.uint8)
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=44)
    ws_d, cache_d, lens_out, flags = gpu_append(env, k_new, v_new, lens, bt, ws, cache, num_blocks)
    assert flags == 0 and (lens_out == lens + 1).all()
    ws_g = dev_to_f16(ws_d)
    rows = lens % 128
    s_idx = np.arange(n_seqs)
    assert np.array_equal(ws_g[s_idx, :, 0, rows], k_new) and np.array_equal(ws_g[s_idx, :, 1, rows], v_new)
    keep = np.ones(ws.shape, bool)
    keep[s_idx, :, :, rows] = False
    assert np.array_equal(ws_g[keep].view(np.int16), ws[keep].view(np.int16))
    done = np.nonzero(lens % 128 == 127)[0]
    blocks = bt[done, lens[done] // 128]
    cache_g = cache_d.cpu().numpy()
    pick = rng.choice(len(done) * hkv, size=64, replace=False)
    ss, hh = done[pick // hkv], pick % hkv
    _, kq, vq = o.quantize_tiles(ws_g[ss, hh, 0], ws_g[ss, hh, 1])
    print("many items", compare_records(cache_g[blocks[pick // hkv], hh], kq, vq))
    untouched = np.ones(num_blocks, bool)
    untouched[blocks] = False
    assert not cache_g[untouched].any()
