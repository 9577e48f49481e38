"""kvarn_serve_step (append + decode attention in one cooperative launch, CUDA
through the C ABI) against the two calls it fuses, kvarn_append_decode then
kvarn_decode_attention, on the same inputs: the workspace, the cache and the new
lengths must agree bit for bit. The attention outputs are compared within the decode
tolerance: the step's split phase runs 8 warps per SM with two record stages each,
the decode call's up to 12 with one (and its merge may split a unit's records between
warps), so the two sum the same terms in another order; each is checked against the
CPU oracle (the decode parity tests, and the oracle test of the step below). Also:
the step captured in a CUDA graph and replayed."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import assert_paths_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()
    return kv, torch


def _case(torch, n_seqs, hkv, group, seed, preset):
    lay = o.LAYOUTS[preset]
    lens = synth.ragged_lengths(n_seqs, 1, 5000, seed)
    lens[::5] = (lens[::5] // 128) * 128 + 127          # these appends complete a tile
    lens[1] = 0                                          # an empty sequence gets its first token
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
    recs = synth.random_records(num_blocks * hkv, seed, lay.record_bytes,
                                lay.k_code_bytes + lay.v_code_bytes).reshape(num_blocks, hkv, -1)
    ws = synth.workspace_tokens(n_seqs, hkv, seed)
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=seed + 1)
    q = synth.queries(n_seqs, hkv * group, seed)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    return dict(lens=torch.from_numpy(lens).cuda(), bt=torch.from_numpy(bt).cuda(),
                cache=torch.from_numpy(recs).cuda(), ws=f16(ws), k_new=f16(k_new), v_new=f16(v_new), q=f16(q),
                num_blocks=num_blocks, max_blocks=max_blocks, n_done=int((lens % 128 == 127).sum()))


def _meta(kv, c, hkv, group, preset):
    return kv.make_meta(hkv, hkv * group, c["num_blocks"], max_blocks_per_seq=c["max_blocks"], preset=preset)


def _serve(kv, torch, c, meta, scratch):
    ws, cache = c["ws"].clone(), c["cache"].clone()
    lens_out = torch.full_like(c["lens"], -7)
    out = torch.full_like(c["q"], float("nan"))
    kv.kvarn_serve_step(c["q"], c["k_new"], c["v_new"], c["lens"], lens_out, c["bt"], ws, cache, out, scratch, meta)
    torch.cuda.synchronize()
    return ws, cache, lens_out, out


def _two_calls(kv, torch, c, meta, scratch):
    ws, cache = c["ws"].clone(), c["cache"].clone()
    lens_out = torch.full_like(c["lens"], -7)
    out = torch.full_like(c["q"], float("nan"))
    kv.kvarn_append_decode(c["k_new"], c["v_new"], c["lens"], lens_out, c["bt"], ws, cache, meta)
    kv.kvarn_decode_attention(c["q"], cache, ws, c["bt"], lens_out, out, scratch, meta)
    torch.cuda.synchronize()
    return ws, cache, lens_out, out


@pytest.mark.parametrize("preset", ["k4v2", "k4v4", "k2v2", "k4v2l"])
def test_serve_step_matches_append_then_decode(env, preset):
    kv, torch = env
    n_seqs, hkv, group = 40, 4, 8
    c = _case(torch, n_seqs, hkv, group, seed=91, preset=preset)
    assert c["n_done"] >= 8
    meta = _meta(kv, c, hkv, group, preset)
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    want = _two_calls(kv, torch, c, meta, scratch)
    assert kv.kvarn_device_flags() == 0
    ws, cache = c["ws"].clone(), c["cache"].clone()
    lens_out = torch.full_like(c["lens"], -7)
    out = torch.full_like(c["q"], float("nan"))
    kv.kvarn_serve_step(c["q"], c["k_new"], c["v_new"], c["lens"], lens_out, c["bt"], ws, cache, out, scratch, meta)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    assert torch.equal(lens_out, c["lens"] + 1)
    assert torch.equal(lens_out, want[2])
    assert torch.equal(ws.view(torch.int16), want[0].view(torch.int16))
    assert torch.equal(cache, want[1])
    assert_paths_close(out.float().cpu().numpy(), want[3].float().cpu().numpy(), preset)
    assert torch.isfinite(out.float()).all()


def test_serve_step_graph_replay(env):
    """The fused step captured in a CUDA graph: two replays from the same state give
    the eager result bit for bit."""
    kv, torch = env
    n_seqs, hkv, group = 24, 2, 8
    c = _case(torch, n_seqs, hkv, group, seed=92, preset="k4v2")
    meta = _meta(kv, c, hkv, group, "k4v2")
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    init = {k: c[k].clone() for k in ("ws", "cache")}
    st = {k: c[k].clone() for k in ("ws", "cache")}
    lens_out = torch.empty_like(c["lens"])
    out = torch.empty_like(c["q"])

    def step():
        kv.kvarn_serve_step(c["q"], c["k_new"], c["v_new"], c["lens"], lens_out, c["bt"], st["ws"], st["cache"],
                            out, scratch, meta)

    def reset():
        for k in st:
            st[k].copy_(init[k])
        lens_out.fill_(-1)
        out.fill_(float("nan"))

    reset()
    step()
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    want = {k: v.clone() for k, v in st.items()}
    want_out = out.clone()
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
        assert torch.equal(lens_out, c["lens"] + 1)
        assert torch.equal(out.view(torch.int16), want_out.view(torch.int16)), replay


@pytest.mark.parametrize("preset", ["k4v2", "k4v4", "k2v2", "k4v2l"])
def test_serve_step_256_ragged_against_oracle(env, preset):
    """The mixed serving step at its full shape through the one-launch entry point,
    against the oracle: 256 sequences with lengths log-uniform in [1024, 32768] (every
    8th forced to L % 128 == 127, so the append completes its tile), 64 q-heads over
    8 kv-heads. 32 sampled (sequence, kv-head) pairs hold K/V drawn like the prefill
    batch and quantized by the oracle (all their full tiles, their workspace tail);
    random valid records and workspace tokens fill the rest. Checked against
    oracle.append + oracle.decode: the whole workspace and the new lengths bit for
    bit, every completed tile within the record tolerances, every other record
    untouched, and the attention of the sampled pairs within the decode tolerance.
    The other presets sample 8 sequences instead of 24."""
    from tests.oracle_pool import run_pairs
    from tests.parity import assert_decode_close, compare_records
    kv, torch = env
    cfg = synth.WORKLOADS["serve_256_ragged"]
    n_seqs, hkv, hq, seed = cfg["n_seqs"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["seed"]
    g = hq // hkv
    lens = synth.ragged_lengths(n_seqs, cfg["lo"], cfg["hi"], seed)
    lens[::8] = (lens[::8] // 128) * 128 + 127
    max_blocks = int(max((L + 1 + 127) // 128 for L in lens))
    num_blocks = int(((lens + 1 + 127) // 128).sum()) + 16
    perm = synth.block_permutation(num_blocks, seed)
    bt = np.full((n_seqs, max_blocks), -1, np.int32)
    pos = 0
    for s in range(n_seqs):
        nb = (lens[s] + 1 + 127) // 128
        bt[s, :nb] = perm[pos:pos + nb]
        pos += nb
    lay = o.LAYOUTS[preset]
    recs = synth.random_records(num_blocks * hkv, seed, lay.record_bytes, lay.k_code_bytes + lay.v_code_bytes)
    recs = recs.reshape(num_blocks, hkv, -1)
    ws = synth.workspace_tokens(n_seqs, hkv, seed)
    rng = np.random.default_rng(seed)
    done = [s for s in range(n_seqs) if lens[s] % 128 == 127]
    seqs = sorted(set(rng.choice(n_seqs, 24 if preset == "k4v2" else 8, replace=False).tolist()) | set(done[::4]))
    pairs = [(s, int(rng.integers(0, hkv))) for s in seqs]
    res = run_pairs([(7_000_001 + 64 * s + h, int(lens[s]), None, preset) for s, h in pairs])
    for (s, h), (r, tail, _) in zip(pairs, res):
        recs[bt[s, :lens[s] // 128], h] = r
        ws[s, h] = tail
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=seed + 1)
    q = synth.queries(n_seqs, hq, seed)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    meta = kv.make_meta(hkv, hq, num_blocks, max_blocks_per_seq=max_blocks, preset=preset)
    ws_d, cache_d = f16(ws), torch.from_numpy(recs).cuda()
    lens_out = torch.full((n_seqs,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((n_seqs, hq, 128), float("nan"), dtype=torch.float16, device="cuda")
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    kv.kvarn_serve_step(f16(q), f16(k_new), f16(v_new), torch.from_numpy(lens).cuda(), lens_out,
                        torch.from_numpy(bt).cuda(), ws_d, cache_d, out, scratch, meta)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    ws_ref, cache_ref, lens_ref = o.append(k_new, v_new, lens, bt, ws, recs)
    assert np.array_equal(lens_out.cpu().numpy(), lens_ref)
    ws_g = ws_d.view(torch.int16).cpu().numpy().view(np.float16)
    assert np.array_equal(ws_g.view(np.int16), ws_ref.view(np.int16))
    cache_g = cache_d.cpu().numpy()
    blocks = np.array([bt[s, lens[s] // 128] for s in done]).repeat(hkv)
    heads = np.tile(np.arange(hkv), len(done))
    _, kq, vq = o.quantize_tiles(np.stack([ws_ref[s, :, 0] for s in done]).reshape(-1, 128, 128),
                                 np.stack([ws_ref[s, :, 1] for s in done]).reshape(-1, 128, 128), preset=preset)
    print("completed tiles", compare_records(cache_g[blocks, heads], kq, vq))
    untouched = np.ones(cache_g.shape[:2], bool)
    untouched[blocks, heads] = False
    assert np.array_equal(cache_g[untouched], cache_ref[untouched])
    ref = o.decode(q.astype(np.float64), cache_ref, ws_ref, bt, lens_ref, pairs=pairs)
    out = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(out).all()
    worst = 0.0
    for s, h in pairs:
        worst = max(worst, assert_decode_close(out[s, h * g:(h + 1) * g], ref[s, h * g:(h + 1) * g],
                                               f"seq {s} head {h}"))
    print(f"{len(pairs)} sampled pairs ({sum(s in done for s, _ in pairs)} with a completed tile), "
          f"max |err| {worst:.2e}")
