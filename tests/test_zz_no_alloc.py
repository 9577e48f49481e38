"""kvarn_decode_attention_static: the decode entry point for callers that cannot
allocate device memory (for example a serving engine whose free device memory is
all pre-reserved for its KV-cache pool, or a plain-C host without a device
allocator for temporaries). It uses a built-in 16 MiB device array instead of a
caller scratch buffer. Checked through the C ABI against kvarn_decode_attention on
two calls in a row, with the decode tolerance of the other parity tests.

This file is collected last on purpose, so a stopping run has already run every
other test when it reaches these."""
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


def _case(torch, n_seqs, hkv, group, seed, preset="k4v2"):
    """Ragged lengths with partial tiles, random valid records, fp16 workspace."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 40 * 128, n_seqs).astype(np.int32)
    lens[0] = 128 * 7                      # whole tiles only
    max_blocks = int(lens.max()) // 128 + 1
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    lay = o.LAYOUTS[preset]
    recs = synth.random_records(num_blocks * hkv, seed, lay.record_bytes, lay.k_code_bytes + lay.v_code_bytes)
    recs = recs.reshape(num_blocks, hkv, -1)
    ws = synth.workspace_tokens(n_seqs, hkv, seed)
    q = synth.queries(n_seqs, hkv * group, seed)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    return dict(q=f16(q), cache=torch.from_numpy(recs).cuda(), ws=f16(ws), bt=torch.from_numpy(bt).cuda(),
                lens=torch.from_numpy(lens).cuda(), num_blocks=num_blocks, max_blocks=max_blocks, preset=preset)


def _both(env, c, hkv, group):
    kv, torch = env
    n_seqs = c["q"].shape[0]
    meta = kv.make_meta(hkv, hkv * group, c["num_blocks"], max_blocks_per_seq=c["max_blocks"], preset=c["preset"])
    out_ref = torch.empty_like(c["q"])
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    kv.kvarn_decode_attention(c["q"], c["cache"], c["ws"], c["bt"], c["lens"], out_ref, scratch, meta)
    out = torch.full_like(c["q"], float("nan"))
    kv.kvarn_decode_attention_static(c["q"], c["cache"], c["ws"], c["bt"], c["lens"], out, meta)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    return out.float().cpu().numpy().astype(np.float64), out_ref.float().cpu().numpy().astype(np.float64)


def test_static_scratch_matches_caller_scratch_twice(env):
    kv, torch = env
    # first call: 24 sequences, 4 kv-heads, groups of 8
    c1 = _case(torch, 24, 4, 8, seed=51)
    got, want = _both(env, c1, 4, 8)
    assert np.isfinite(got).all()
    assert_decode_close(got, want, "first call")
    # second call in a row, different shape and data: nothing from the first leaks
    c2 = _case(torch, 9, 2, 4, seed=52)
    got, want = _both(env, c2, 2, 4)
    assert np.isfinite(got).all()
    assert_decode_close(got, want, "second call")


@pytest.mark.parametrize("preset", ["k4v4", "k2v2", "k4v2l"])
def test_static_scratch_serves_every_preset(env, preset):
    """The other presets go through the same kernels as with a caller buffer: two
    calls in a row match kvarn_decode_attention."""
    kv, torch = env
    for seed, (n_seqs, hkv, group) in ((61, (10, 2, 8)), (62, (5, 4, 2))):
        c = _case(torch, n_seqs, hkv, group, seed=seed, preset=preset)
        got, want = _both(env, c, hkv, group)
        assert np.isfinite(got).all()
        assert_decode_close(got, want, f"{preset} seed {seed}")


def test_static_scratch_rejects_sizes_beyond_its_limit(env):
    kv, torch = env
    n_seqs, hkv, group = 4096, 8, 8          # 32768 (sequence, kv-head) pairs: far beyond 16 MiB
    meta = kv.make_meta(hkv, hkv * group, 16, max_blocks_per_seq=1)
    q = torch.zeros(n_seqs, hkv * group, 128, dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    lens = torch.full((n_seqs,), 128, dtype=torch.int32, device="cuda")
    bt = torch.zeros(n_seqs, 1, dtype=torch.int32, device="cuda")
    cache = torch.zeros(16, hkv, o.RECORD_BYTES, dtype=torch.uint8, device="cuda")
    with pytest.raises(kv.KvarnError) as e:
        kv.kvarn_decode_attention_static(q, cache, None, bt, lens, out, meta)
    assert e.value.status == kv.KVARN_ESCRATCH
    assert "16 MiB" in str(e.value)
    torch.cuda.synchronize()
    assert not out.any()                      # nothing was launched
