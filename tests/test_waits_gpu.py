"""Failure detection without a GPU fault: the library's bounded waits give up,
report KVARN_FLAG_WAIT_TIMEOUT and leave the device usable.

kvarn_check_bounded_waits runs the kernels' own wait code (the mbarrier wait of the
copy and tensor-core paths, the grid barrier of the serving step) against a wait
that never completes, with a limit of a few milliseconds. Each test checks the
flag, then that the next normal call on the same device is still exact: a quantize
call against the oracle, and a serving step whose scratch held the barrier words
the timed-out barrier left behind, against the two calls it fuses."""
import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o
from tests.parity import compare_records

pytestmark = pytest.mark.gpu

LIMIT_US = 3000


@pytest.fixture(scope="module")
def env():
    import torch
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    kv.kvarn_device_flags()
    return kv, torch


def _quantize_small(kv, torch):
    hkv, n_chunks, num_blocks = 2, 5, 8
    k, v = synth.prefill_kv(n_chunks * 128, hkv, seed=95)
    slots = synth.prefill_slot_mapping(n_chunks * 128, num_blocks, seed=95)
    meta = kv.make_meta(hkv, hkv, num_blocks)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    cache = torch.zeros(num_blocks, hkv, o.RECORD_BYTES, dtype=torch.uint8, device="cuda")
    kv.kvarn_quantize_tiles(f16(k), f16(v), torch.from_numpy(slots).cuda(), cache, meta)
    flags = kv.kvarn_device_flags()
    pairs = [(c, h) for c in range(n_chunks) for h in range(hkv)]
    kt = np.stack([k[c * 128:(c + 1) * 128, h] for c, h in pairs])
    vt = np.stack([v[c * 128:(c + 1) * 128, h] for c, h in pairs])
    _, kq, vq = o.quantize_tiles(kt, vt)
    got = cache.cpu().numpy()
    blocks = np.array([slots[c * 128] // 128 for c, _ in pairs])
    heads = np.array([h for _, h in pairs])
    return flags, got[blocks, heads], kq, vq


def test_mbarrier_wait_gives_up_and_reports(env):
    kv, torch = env
    kv.kvarn_check_bounded_waits(kv.KVARN_WAIT_MBARRIER, LIMIT_US)
    assert kv.kvarn_device_flags() == kv.FLAG_WAIT_TIMEOUT
    assert kv.kvarn_device_flags() == 0                     # reading clears it
    # the device is still usable: a quantize call right after is exact
    flags, rec, kq, vq = _quantize_small(kv, torch)
    assert flags == 0
    compare_records(rec, kq, vq)


def test_grid_barrier_gives_up_and_later_steps_are_exact(env):
    """A grid barrier that expects one CTA more than were launched runs out; its
    words are left in the last 256 bytes of a scratch buffer, exactly where a
    serving step keeps its own. A serving step on that same scratch right after
    still matches the same step run before the timeout bit for bit: the step zeroes
    its barrier words before it starts."""
    kv, torch = env
    from tests.test_serve_gpu import _case, _meta, _serve
    n_seqs, hkv, group = 24, 2, 8
    c = _case(torch, n_seqs, hkv, group, seed=96, preset="k4v2")
    meta = _meta(kv, c, hkv, group, "k4v2")
    need = kv.decode_scratch_bytes(meta, n_seqs)
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = _serve(kv, torch, c, meta, scratch)
    assert kv.kvarn_device_flags() == 0
    kv.kvarn_check_bounded_waits(kv.KVARN_WAIT_GRID, LIMIT_US, scratch[need - 256:])
    assert kv.kvarn_device_flags() == kv.FLAG_WAIT_TIMEOUT
    left = scratch[need - 256:need - 248].view(torch.int32).cpu().numpy()
    assert left[0] > 0                                       # arrivals the timed-out barrier left
    ws, cache = c["ws"].clone(), c["cache"].clone()
    lens_out = torch.full_like(c["lens"], -7)
    out = torch.full_like(c["q"], float("nan"))
    kv.kvarn_serve_step(c["q"], c["k_new"], c["v_new"], c["lens"], lens_out, c["bt"], ws, cache, out, scratch, meta)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    assert torch.equal(lens_out, want[2])
    assert torch.equal(ws.view(torch.int16), want[0].view(torch.int16))
    assert torch.equal(cache, want[1])
    assert torch.equal(out.view(torch.int16), want[3].view(torch.int16))
