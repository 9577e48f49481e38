"""A serving step (append one token to every sequence, then decode) captured in a
CUDA graph and replayed: the replay must reproduce the eager step bit for bit,
and a second replay from the same state must do so again. The step runs the
library's launches on the capturing stream only (no allocation, no host
synchronisation, no runtime lookups after the first call on a device)."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()
    return kv, torch


def _serving_case(torch, n_seqs, hkv, group, seed):
    lens = synth.ragged_lengths(n_seqs, 1, 5000, seed)
    lens[::5] = (lens[::5] // 128) * 128 + 127          # these appends complete a tile
    max_blocks = int(max((L + 1 + 127) // 128 for L in lens))
    total_blocks = int(((lens + 1 + 127) // 128).sum())
    num_blocks = total_blocks + 8
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
    q = synth.queries(n_seqs, hkv * group, seed)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    return dict(lens=torch.from_numpy(lens).cuda(), bt=torch.from_numpy(bt).cuda(),
                cache=torch.from_numpy(recs).cuda(), ws=f16(ws), k_new=f16(k_new), v_new=f16(v_new), q=f16(q),
                num_blocks=num_blocks, max_blocks=max_blocks, n_done=int((lens % 128 == 127).sum()))


def test_serving_step_graph_replay_matches_eager(env):
    kv, torch = env
    n_seqs, hkv, group = 40, 4, 8
    c = _serving_case(torch, n_seqs, hkv, group, seed=61)
    assert c["n_done"] >= 8
    meta = kv.make_meta(hkv, hkv * group, c["num_blocks"], max_blocks_per_seq=c["max_blocks"])
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")

    # state the step mutates, and its initial copy
    init = {k: c[k].clone() for k in ("ws", "cache")}
    st = {k: c[k].clone() for k in ("ws", "cache")}
    lens_out = torch.empty_like(c["lens"])
    out = torch.empty_like(c["q"])

    def step():
        kv.kvarn_append_decode(c["k_new"], c["v_new"], c["lens"], lens_out, c["bt"], st["ws"], st["cache"], meta)
        kv.kvarn_decode_attention(c["q"], st["cache"], st["ws"], c["bt"], lens_out, out, scratch, meta)

    def reset():
        for k in st:
            st[k].copy_(init[k])
        lens_out.fill_(-1)
        out.fill_(float("nan"))

    # eager reference
    reset()
    step()
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    want = {k: v.clone() for k, v in st.items()}
    want_lens, want_out = lens_out.clone(), out.clone()
    assert (want_lens == c["lens"] + 1).all()
    assert torch.isfinite(want_out.float()).all()

    # warm-up on a side stream (first-call lookups happen here), then capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        reset()
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for replay in range(2):
        reset()
        graph.replay()
        torch.cuda.synchronize()
        assert kv.kvarn_device_flags() == 0
        for k in st:
            assert torch.equal(st[k], want[k]), (replay, k)
        assert torch.equal(lens_out, want_lens), replay
        assert torch.equal(out.view(torch.int16), want_out.view(torch.int16)), replay
