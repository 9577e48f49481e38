"""Byte offsets past 2^31 and 2^32 (CUDA, through the C ABI, against the CPU
oracle). A 4.6 GB packed cache whose used blocks straddle the 2^31- and
2^32-byte marks and sit at its far end; a 4.3 GB decode workspace whose used
sequences lie past 2^32 bytes; a quantize input of 4.6 GB per tensor whose last
tiles start past 2^32 bytes. Every address the kernels form from a block,
sequence or token number has to be 64-bit for these to pass. The oracle sees
compact copies (the used blocks and sequences only); all inputs are seeded
synthetic data."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import assert_decode_close, assert_paths_close, compare_records

pytestmark = pytest.mark.gpu

HKV, GROUP = 8, 8
REC = o.RECORD_BYTES                          # 14336: k4v2
NUM_BLOCKS = 40000                            # 40000 x 8 x 14336 B = 4.59 GB
# (block 18724 holds the 2^31-byte mark, block 37449 the 2^32-byte mark)
MARK31, MARK32 = (1 << 31) // (HKV * REC), (1 << 32) // (HKV * REC)


def _f16(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()


def _np16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.float16)


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()
    return kv, torch


def test_block_marks():
    assert MARK31 * HKV * REC < (1 << 31) < (MARK31 + 1) * HKV * REC
    assert MARK32 * HKV * REC < (1 << 32) < (MARK32 + 1) * HKV * REC


def test_quantize_input_and_cache_past_4gb(env):
    kv, torch = env
    pool = 64 * 128
    n_tiles = 17408                                      # 2,228,224 tokens: 4.56 GB per tensor
    n_tokens = n_tiles * 128
    assert (n_tiles - 4) * 128 * HKV * 128 * 2 > (1 << 32)       # the last four tiles start past 2^32 bytes
    k = torch.empty(n_tokens, HKV, 128, dtype=torch.float16, device="cuda")
    v = torch.empty_like(k)
    pk, pv = synth.prefill_kv(pool, HKV, seed=61)
    reps = n_tokens // pool
    k.view(reps, pool, HKV, 128).copy_(_f16(torch, pk)[None].expand(reps, -1, -1, -1))
    v.view(reps, pool, HKV, 128).copy_(_f16(torch, pv)[None].expand(reps, -1, -1, -1))
    # tiles with data of their own, at both ends of the input, to blocks at the marks
    # and at both ends of the cache
    target = {0: NUM_BLOCKS - 1, 1: 0, n_tiles - 4: MARK31, n_tiles - 3: MARK32 - 1, n_tiles - 2: MARK32,
              n_tiles - 1: MARK32 + 1}
    special = sorted(target)
    sk, sv = synth.prefill_kv(len(special) * 128, HKV, seed=62)
    for i, c in enumerate(special):
        k[c * 128:(c + 1) * 128] = _f16(torch, sk[i * 128:(i + 1) * 128])
        v[c * 128:(c + 1) * 128] = _f16(torch, sv[i * 128:(i + 1) * 128])
    rng = np.random.default_rng(63)
    free = np.setdiff1d(np.arange(NUM_BLOCKS), list(target.values()))
    blocks = rng.permutation(free)[:n_tiles].astype(np.int64)
    for c, b in target.items():
        blocks[c] = b
    assert len(np.unique(blocks)) == n_tiles
    slots = (blocks[:, None] * 128 + np.arange(128)).reshape(-1)
    cache = torch.empty(NUM_BLOCKS, HKV, REC, dtype=torch.uint8, device="cuda")
    meta = kv.make_meta(HKV, HKV, NUM_BLOCKS)
    kv.kvarn_quantize_tiles(k, v, torch.from_numpy(slots).cuda(), cache, meta)
    assert kv.kvarn_device_flags() == 0
    # the special tiles (all heads) and one pool tile from the middle of the input
    mid = n_tiles // 2
    kt = [sk[i * 128:(i + 1) * 128, h] for i in range(len(special)) for h in range(HKV)]
    vt = [sv[i * 128:(i + 1) * 128, h] for i in range(len(special)) for h in range(HKV)]
    off = (mid * 128) % pool
    kt += [pk[off:off + 128, h] for h in range(HKV)]
    vt += [pv[off:off + 128, h] for h in range(HKV)]
    _, kq, vq = o.quantize_tiles(np.stack(kt), np.stack(vt))
    used = torch.from_numpy(np.array([target[c] for c in special] + [blocks[mid]], np.int64)).cuda()
    got = cache[used].cpu().numpy().reshape(-1, REC)
    print(compare_records(got, kq, vq))


def _serving_state(torch):
    """8200 sequences, three of them non-empty: 3 (before the 2^32-byte mark of the
    workspace) and 8195, 8199 (past it), with blocks at the cache's marks and ends.
    Returns the device state and the oracle's compact copy of the used part."""
    n_seqs, max_blocks = 8200, 5
    used = {3: (3 * 128 + 50, [0, MARK31, 5]),
            8195: (2 * 128 + 127, [NUM_BLOCKS - 1, MARK32 - 1, MARK32]),    # the append fills MARK32
            8199: (4 * 128 + 5, [MARK31 + 1, MARK32 + 1, NUM_BLOCKS - 2, NUM_BLOCKS - 3])}
    seqs = sorted(used)
    ws_row = HKV * 2 * 128 * 128 * 2
    assert seqs[0] * ws_row < (1 << 32) < seqs[1] * ws_row
    lens = np.zeros(n_seqs, np.int32)
    bt = np.full((n_seqs, max_blocks), -1, np.int32)
    # compact copy: used sequences 0..2, their blocks renumbered 0..n-1
    c_blocks = [b for s in seqs for b in used[s][1]]
    c_bt = np.full((len(seqs), max_blocks), -1, np.int32)
    c_lens = np.zeros(len(seqs), np.int32)
    c_cache = np.zeros((len(c_blocks), HKV, REC), np.uint8)
    c_ws = np.zeros((len(seqs), HKV, 2, 128, 128), np.float16)
    for i, s in enumerate(seqs):
        L, bl = used[s]
        lens[s] = c_lens[i] = L
        bt[s, :len(bl)] = bl
        c_bt[i, :len(bl)] = [c_blocks.index(b) for b in bl]
        k, v = synth.prefill_kv(L, HKV, seed=70 + i)
        nf = L // 128
        slots = np.concatenate([c_bt[i, b] * 128 + np.arange(128) for b in range(nf)]).astype(np.int64)
        o.quantize_into_cache(k[:nf * 128], v[:nf * 128], slots, c_cache)
        c_ws[i, :, 0, :L % 128] = k[nf * 128:].transpose(1, 0, 2)
        c_ws[i, :, 1, :L % 128] = v[nf * 128:].transpose(1, 0, 2)
    cache = torch.empty(NUM_BLOCKS, HKV, REC, dtype=torch.uint8, device="cuda")
    cache[torch.tensor(c_blocks, device="cuda")] = torch.from_numpy(c_cache).cuda()
    ws = torch.empty(n_seqs, HKV, 2, 128, 128, dtype=torch.float16, device="cuda")
    ws[torch.tensor(seqs, device="cuda")] = _f16(torch, c_ws)
    q = synth.queries(n_seqs, HKV * GROUP, seed=71)
    kn, vn = synth.prefill_kv(n_seqs, HKV, seed=72)
    return dict(n_seqs=n_seqs, max_blocks=max_blocks, seqs=seqs, lens=lens, bt=bt, cache=cache, ws=ws, q=q,
                kn=kn, vn=vn, c_bt=c_bt, c_lens=c_lens, c_cache=c_cache, c_ws=c_ws, c_blocks=c_blocks)


@pytest.fixture(scope="module")
def state(env):
    _, torch = env
    return _serving_state(torch)


def _meta(kv, st):
    return kv.make_meta(HKV, HKV * GROUP, NUM_BLOCKS, max_blocks_per_seq=st["max_blocks"])


def test_decode_past_4gb(env, state):
    kv, torch = env
    st = state
    meta = _meta(kv, st)
    out = torch.full((st["n_seqs"], HKV * GROUP, 128), float("nan"), dtype=torch.float16, device="cuda")
    scratch = torch.empty(kv.decode_scratch_bytes(meta, st["n_seqs"]), dtype=torch.uint8, device="cuda")
    kv.kvarn_decode_attention(_f16(torch, st["q"]), st["cache"], st["ws"], torch.from_numpy(st["bt"]).cuda(),
                              torch.from_numpy(st["lens"]).cuda(), out, scratch, meta)
    assert kv.kvarn_device_flags() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    ref = o.decode(st["q"][st["seqs"]].astype(np.float64), st["c_cache"], st["c_ws"], st["c_bt"], st["c_lens"])
    for i, s in enumerate(st["seqs"]):
        assert_decode_close(got[s], ref[i], f"sequence {s}")
    empty = np.ones(st["n_seqs"], bool)
    empty[st["seqs"]] = False
    assert not got[empty].any()                       # length 0: zero output


def test_append_and_serve_step_past_4gb(env, state):
    kv, torch = env
    st = state
    meta = _meta(kv, st)
    lens_d = torch.from_numpy(st["lens"]).cuda()
    bt_d = torch.from_numpy(st["bt"]).cuda()
    kn, vn = _f16(torch, st["kn"]), _f16(torch, st["vn"])
    q = _f16(torch, st["q"])
    scratch = torch.empty(kv.decode_scratch_bytes(meta, st["n_seqs"]), dtype=torch.uint8, device="cuda")
    # two calls
    ws2, cache2 = st["ws"].clone(), st["cache"].clone()
    lens2 = torch.full_like(lens_d, -7)
    out2 = torch.full_like(q, float("nan"))
    kv.kvarn_append_decode(kn, vn, lens_d, lens2, bt_d, ws2, cache2, meta)
    kv.kvarn_decode_attention(q, cache2, ws2, bt_d, lens2, out2, scratch, meta)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    assert torch.equal(lens2, lens_d + 1)
    # the used sequences against the oracle's append on the compact copy
    seqs = st["seqs"]
    c_ws, c_cache, c_lens = o.append(st["kn"][seqs], st["vn"][seqs], st["c_lens"], st["c_bt"], st["c_ws"],
                                     st["c_cache"])
    assert np.array_equal(_np16(ws2[torch.tensor(seqs, device="cuda")]), c_ws)
    s_done = seqs[1]                                  # 383 -> 384 tokens: its third tile is quantized
    blk = st["bt"][s_done, 2]
    assert blk == MARK32
    _, kq, vq = o.quantize_tiles(c_ws[1, :, 0], c_ws[1, :, 1])
    print(compare_records(cache2[blk].cpu().numpy(), kq, vq))
    # an empty sequence past the 2^32-byte mark got its first token in row 0
    row = _np16(ws2[8196, :, :, 0])
    assert np.array_equal(row[:, 0], st["kn"][8196]) and np.array_equal(row[:, 1], st["vn"][8196])
    got = out2.float().cpu().numpy().astype(np.float64)
    c_q = st["q"][seqs].astype(np.float64)
    ref = o.decode(c_q, c_cache, c_ws, st["c_bt"], c_lens)
    for i, s in enumerate(seqs):
        assert_decode_close(got[s], ref[i], f"sequence {s} after the append")
    # the same step in one launch: the two calls' workspace, cache and lengths bit for
    # bit; its output (the warp-level split kernel) within the decode tolerance of the
    # two calls' (the tensor-core one) and of the oracle
    ws1, cache1 = st["ws"].clone(), st["cache"].clone()
    lens1 = torch.full_like(lens_d, -7)
    out1 = torch.full_like(q, float("nan"))
    kv.kvarn_serve_step(q, kn, vn, lens_d, lens1, bt_d, ws1, cache1, out1, scratch, meta)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    assert torch.equal(lens1, lens2)
    assert torch.equal(ws1.view(torch.int16), ws2.view(torch.int16))
    assert torch.equal(cache1, cache2)
    got1 = out1.float().cpu().numpy().astype(np.float64)
    assert_paths_close(got1, got, "serve step vs two calls")
    for i, s in enumerate(seqs):
        assert_decode_close(got1[s], ref[i], f"sequence {s}, serve step")


def test_prefill_past_4gb(env, state):
    kv, torch = env
    st = state
    seqs = st["seqs"]
    chunks = np.zeros(st["n_seqs"], np.int64)
    chunks[seqs[0]], chunks[seqs[2]] = 20, 9
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    n_tok = int(cu[-1])
    kn, vn = synth.prefill_kv(n_tok, HKV, seed=73)
    q = synth.queries(n_tok, HKV * GROUP, seed=74)
    meta = _meta(kv, st)
    out = torch.full((n_tok, HKV * GROUP, 128), float("nan"), dtype=torch.float16, device="cuda")
    kv.kvarn_prefill_attention(_f16(torch, q), _f16(torch, kn), _f16(torch, vn), torch.from_numpy(cu).cuda(),
                               torch.from_numpy(st["lens"]).cuda(), int(chunks.max()),
                               torch.from_numpy(st["bt"]).cuda(), st["cache"], st["ws"], out, meta)
    assert kv.kvarn_device_flags() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    c_cu = np.array([0, 20, 20, 29], np.int32)         # the compact copy's three sequences
    ref = o.prefill_attention(q.astype(np.float64), kn, vn, c_cu, st["c_lens"], st["c_bt"], st["c_ws"],
                              st["c_cache"])
    for t in range(n_tok):
        assert_decode_close(got[t], ref[t], f"chunk token {t}")
