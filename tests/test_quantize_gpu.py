"""Parity of kvarn_quantize_tiles (CUDA, through the C ABI) with the CPU oracle."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import compare_records

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()          # clear
    return kv, torch


def f16_to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()


def run_prefill(env, k, v, slots, num_blocks, n_iters=4, eps=1e-6):
    kv, torch = env
    n, hkv, _ = k.shape
    meta = kv.make_meta(hkv, hkv, num_blocks, n_iters=n_iters, eps=eps)
    cache = torch.zeros(num_blocks, hkv, o.RECORD_BYTES, dtype=torch.uint8, device="cuda")
    kv.kvarn_quantize_tiles(f16_to_dev(torch, k), f16_to_dev(torch, v),
                            torch.from_numpy(slots).cuda(), cache, meta)
    flags = kv.kvarn_device_flags()
    return cache.cpu().numpy(), flags


def oracle_tiles(k, v, pairs, n_iters=4, eps=1e-6):
    kt = np.stack([k[c * 128:(c + 1) * 128, h] for c, h in pairs])
    vt = np.stack([v[c * 128:(c + 1) * 128, h] for c, h in pairs])
    return o.quantize_tiles(kt, vt, n_iters, eps)


def test_single_tile(env):
    k, v, _ = synth.single_tile(0)
    cache, flags = run_prefill(env, k[:, None, :], v[:, None, :], np.arange(128, dtype=np.int64) + 128, 2)
    assert flags == 0
    _, kq, vq = o.quantize_tiles(k[None], v[None])
    compare_records(cache[1:2, 0], kq, vq)
    assert not cache[0].any()


@pytest.mark.parametrize("hkv", [8, 3, 5])
def test_multi_tile_random_slots(env, hkv):
    """40 chunks into 48 blocks in random order; 3 and 5 kv-heads split the item
    index by a divisor that is not a power of two."""
    n_chunks, num_blocks = 40, 48
    k, v = synth.prefill_kv(n_chunks * 128, hkv, seed=21)
    slots = synth.prefill_slot_mapping(n_chunks * 128, num_blocks, seed=21)
    cache, flags = run_prefill(env, k, v, slots, num_blocks)
    assert flags == 0
    pairs = [(c, h) for c in range(n_chunks) for h in range(hkv)]
    _, kq, vq = oracle_tiles(k, v, pairs)
    blocks = np.array([slots[c * 128] // 128 for c, _ in pairs])
    heads = np.array([h for _, h in pairs])
    stats = compare_records(cache[blocks, heads], kq, vq)
    used = set(blocks.tolist())
    for b in range(num_blocks):
        if b not in used:
            assert not cache[b].any()
    print(stats)


@pytest.mark.parametrize("n_iters,eps", [(1, 1e-6), (8, 1e-6), (16, 1e-6), (4, 1e-3)])
def test_iteration_count_and_eps(env, n_iters, eps):
    hkv, n_chunks = 2, 4
    k, v = synth.prefill_kv(n_chunks * 128, hkv, seed=22)
    slots = np.arange(n_chunks * 128, dtype=np.int64)
    cache, flags = run_prefill(env, k, v, slots, n_chunks, n_iters=n_iters, eps=eps)
    pairs = [(c, h) for c in range(n_chunks) for h in range(hkv)]
    _, kq, vq = oracle_tiles(k, v, pairs, n_iters=n_iters, eps=eps)
    compare_records(cache[[c for c, _ in pairs], [h for _, h in pairs]], kq, vq)


def test_degenerate_tiles(env):
    tiles_k, tiles_v = [], []
    rng = np.random.default_rng(23)
    zero = np.zeros((128, 128))
    const = np.full((128, 128), 3.0)
    spike = np.zeros((128, 128)); spike[5, 7] = 60000.0
    big = np.full((128, 128), 65504.0); big[::2] *= -1
    sub = rng.standard_normal((128, 128)) * 1e-6           # fp16 subnormals
    onecol = np.zeros((128, 128)); onecol[:, 3] = rng.standard_normal(128)
    for t in (zero, const, spike, big, sub, onecol):
        tiles_k.append(t.astype(np.float16))
        tiles_v.append(t.T.astype(np.float16))
    k = np.stack(tiles_k)[:, :, None, :].reshape(-1, 1, 128)
    v = np.stack(tiles_v)[:, :, None, :].reshape(-1, 1, 128)
    n = len(tiles_k)
    cache, flags = run_prefill(env, k, v, np.arange(n * 128, dtype=np.int64), n)
    assert flags == 0
    _, kq, vq = o.quantize_tiles(np.stack(tiles_k), np.stack(tiles_v))
    compare_records(cache[:, 0], kq, vq)


def test_bad_slot_mapping_is_skipped_and_flagged(env):
    kv, torch = env
    hkv, n_chunks, num_blocks = 2, 3, 4
    k, v = synth.prefill_kv(n_chunks * 128, hkv, seed=24)
    slots = np.arange(n_chunks * 128, dtype=np.int64)
    slots[128 + 5], slots[128 + 6] = slots[128 + 6], slots[128 + 5]   # chunk 1 not in order
    slots[256:384] += 10 * 128                                        # chunk 2 beyond num_blocks
    cache, flags = run_prefill(env, k, v, slots, num_blocks)
    assert flags & kv.FLAG_BAD_SLOTS
    assert not cache[1].any() and not cache[2].any() and not cache[3].any()
    _, kq, vq = oracle_tiles(k, v, [(0, 0), (0, 1)])
    compare_records(cache[0, [0, 1]], kq, vq)
    assert kv.kvarn_device_flags() == 0          # read clears


def test_prefill_16x16k_sampled(env):
    """Full prefill workload (16 sequences x 16384 tokens, 8 kv-heads) in the
    launch configuration the benchmark times; 192 sampled tile-heads vs oracle."""
    kv, torch = env
    n_tokens, hkv = 16 * 16384, 8
    num_blocks = n_tokens // 128
    k, v = synth.prefill_kv(n_tokens, hkv, seed=1)
    slots = synth.prefill_slot_mapping(n_tokens, num_blocks, seed=1)
    cache, flags = run_prefill(env, k, v, slots, num_blocks)
    assert flags == 0
    rng = np.random.default_rng(25)
    pairs = [(int(c), int(h)) for c, h in zip(rng.integers(0, num_blocks, 192), rng.integers(0, hkv, 192))]
    _, kq, vq = oracle_tiles(k, v, pairs)
    blocks = np.array([slots[c * 128] // 128 for c, _ in pairs])
    stats = compare_records(cache[blocks, [h for _, h in pairs]], kq, vq)
    # every record was written (metadata scales are positive fp16 values)
    kr = cache[:, :, o.K_META_OFF:o.K_META_OFF + 256].view(np.float16)
    assert (kr > 0).all()
    print(stats)
