"""Parity of kvarn_prefill_attention (CUDA, through the C ABI) with the CPU oracle:
chunks of fresh tokens attending the packed cache, the fp16 workspace tail and the
chunk itself (causal), under the decode tolerance."""
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


def _case(lens, chunks, hkv, group, seed, preset="k4v2", random_cache=False):
    """Cached sequences of the given lengths (oracle-quantized, or random records),
    their workspace tails, and fresh chunks."""
    lay = o.LAYOUTS[preset]
    n_seqs = len(lens)
    max_blocks = max(1, max(L // 128 for L in lens))
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    ws = np.zeros((n_seqs, hkv, 2, 128, 128), np.float16)
    if random_cache:
        cache = synth.random_records(num_blocks * hkv, seed, lay.record_bytes,
                                     lay.k_code_bytes + lay.v_code_bytes).reshape(num_blocks, hkv, -1)
        for s, L in enumerate(lens):
            k, v = synth.prefill_kv(128, hkv, seed=seed * 10 + s)
            ws[s, :, 0, :L % 128] = k[:L % 128].transpose(1, 0, 2)
            ws[s, :, 1, :L % 128] = v[:L % 128].transpose(1, 0, 2)
    else:
        cache = np.zeros((num_blocks, hkv, lay.record_bytes), np.uint8)
        for s, L in enumerate(lens):
            k, v = synth.prefill_kv(max(L, 1), hkv, seed=seed * 10 + s)
            nf = L // 128
            if nf:
                slots = np.concatenate([bt[s, b] * 128 + np.arange(128) for b in range(nf)]).astype(np.int64)
                o.quantize_into_cache(k[:nf * 128], v[:nf * 128], slots, cache)
            ws[s, :, 0, :L % 128] = k[nf * 128:L].transpose(1, 0, 2)
            ws[s, :, 1, :L % 128] = v[nf * 128:L].transpose(1, 0, 2)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    kn, vn = synth.prefill_kv(max(int(cu[-1]), 1), hkv, seed=seed + 99)
    q = synth.queries(max(int(cu[-1]), 1), hkv * group, seed)
    return dict(q=q, kn=kn, vn=vn, cu=cu, lens=np.asarray(lens, np.int32), bt=bt, ws=ws, cache=cache,
                num_blocks=num_blocks, max_blocks=max_blocks, hkv=hkv, group=group, preset=preset)


def _gpu(env, c, use_ws=True, max_chunk=None):
    kv, torch = env
    meta = kv.make_meta(c["hkv"], c["hkv"] * c["group"], c["num_blocks"], max_blocks_per_seq=c["max_blocks"],
                        preset=c["preset"])
    q = f16_to_dev(torch, c["q"])
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    chunks = np.diff(c["cu"])
    kv.kvarn_prefill_attention(q, f16_to_dev(torch, c["kn"]), f16_to_dev(torch, c["vn"]),
                               torch.from_numpy(c["cu"]).cuda(), torch.from_numpy(c["lens"]).cuda(),
                               max_chunk if max_chunk is not None else int(chunks.max()) if len(chunks) else 0,
                               torch.from_numpy(c["bt"]).cuda(),
                               torch.from_numpy(c["cache"]).cuda(), f16_to_dev(torch, c["ws"]) if use_ws else None,
                               out, meta)
    flags = kv.kvarn_device_flags()
    return out.float().cpu().numpy().astype(np.float64), flags


@pytest.mark.parametrize("preset", ["k4v2", "k4v4", "k2v2", "k4v2l"])
def test_prefill_small_all_tokens(env, preset):
    c = _case([300, 0, 1000, 256], [37, 129, 8, 1], hkv=2, group=4, seed=81, preset=preset)
    out, flags = _gpu(env, c)
    assert flags == 0
    ref = o.prefill_attention(c["q"], c["kn"], c["vn"], c["cu"], c["lens"], c["bt"], c["ws"], c["cache"])
    n = int(c["cu"][-1])
    print(preset, "prefill max err", assert_decode_close(out[:n], ref[:n], preset))


@pytest.mark.parametrize("preset", ["k4v2", "k4v4", "k2v2", "k4v2l"])
def test_prefill_group_8_long_context_sampled(env, preset):
    """4 sequences with 4000-6000 cached tokens (random records of the preset) and
    chunks of 120-260 tokens, 64 q-heads over 8 kv-heads; sampled (token, kv-head)
    pairs."""
    lens, chunks = [4000, 6000, 4352, 5000], [260, 120, 256, 200]
    c = _case(lens, chunks, hkv=8, group=8, seed=82, preset=preset, random_cache=True)
    out, flags = _gpu(env, c)
    assert flags == 0 and np.isfinite(out).all()
    rng = np.random.default_rng(82)
    n = int(c["cu"][-1])
    toks = sorted({(int(t), int(h)) for t, h in zip(rng.integers(0, n, 24), rng.integers(0, 8, 24))})
    toks += [(0, 0), (n - 1, 7), (int(c["cu"][1]) - 1, 3)]          # first, last, end of a chunk
    ref = o.prefill_attention(c["q"], c["kn"], c["vn"], c["cu"], c["lens"], c["bt"], c["ws"], c["cache"],
                              tokens=toks)
    for t, h in toks:
        assert_decode_close(out[t, h * 8:(h + 1) * 8], ref[t, h * 8:(h + 1) * 8], f"token {t} head {h}")


def test_prefill_without_workspace_and_empty_chunk(env):
    """Cached lengths that are whole tiles need no workspace; an empty chunk is
    skipped; a missing workspace for a partial tile is flagged."""
    c = _case([256, 384, 0], [5, 0, 9], hkv=1, group=2, seed=83)
    out, flags = _gpu(env, c, use_ws=False)
    assert flags == 0
    ref = o.prefill_attention(c["q"], c["kn"], c["vn"], c["cu"], c["lens"], c["bt"], c["ws"], c["cache"])
    n = int(c["cu"][-1])
    assert_decode_close(out[:n], ref[:n], "no workspace")
    c = _case([200], [3], hkv=1, group=2, seed=84)
    _, flags = _gpu(env, c, use_ws=False)
    assert flags == 0x4                          # KVARN_FLAG_BAD_LENGTH


def test_prefill_chunk_longer_than_max_chunk_is_flagged(env):
    """A chunk longer than max_chunk (rounded up to 16 tokens) leaves its tail
    tokens uncomputed: the call raises KVARN_FLAG_BAD_LENGTH, the covered tokens
    still match the oracle and the rows past the grid stay untouched."""
    c = _case([300, 130], [40, 9], hkv=2, group=4, seed=85)
    out, flags = _gpu(env, c, max_chunk=20)          # grid: 2 CTAs x 16 tokens = 32 < 40
    assert flags == 0x4                              # KVARN_FLAG_BAD_LENGTH
    ref = o.prefill_attention(c["q"], c["kn"], c["vn"], c["cu"], c["lens"], c["bt"], c["ws"], c["cache"])
    assert_decode_close(out[:32], ref[:32], "covered tokens of the long chunk")
    assert np.isnan(out[32:40]).all()                # never written
    assert_decode_close(out[40:49], ref[40:49], "the short chunk")
    out, flags = _gpu(env, c, max_chunk=40)          # the bound is met: no flag
    assert flags == 0
