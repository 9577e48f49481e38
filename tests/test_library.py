"""libkvarn loads, exports every entry point declared in include/kvarn.h, and rejects
bad arguments on the host before touching the GPU (these calls return before any
CUDA call, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def kv():
    import __graft_entry__
    if not os.path.exists(os.path.join(ROOT, "kv_cache_quantization_x128_gb300", "libkvarn.so")):
        __graft_entry__.build()
    import kv_cache_quantization_x128_gb300 as kv
    return kv


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            names += re.findall(r"KVARN_API\s+[\w\s\*]+?\b(kvarn_\w+)\s*\(", text)
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("kvarn_quantize_tiles", "kvarn_append_decode", "kvarn_decode_attention",
                 "kvarn_decode_scratch_bytes", "kvarn_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(kv):
    lib = ctypes.CDLL(kv.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) <= set(kv._SIGS)


def test_meta_struct_layout(kv):
    assert ctypes.sizeof(kv.KvarnMeta) == 48
    assert kv.KvarnMeta.num_blocks.offset == 32


def test_size_queries(kv):
    m = kv.make_meta(8, 64, num_blocks=2048, max_blocks_per_seq=128)
    assert kv.record_bytes() == 14336
    assert kv.cache_bytes(m) == 2048 * 8 * 14336
    assert kv.workspace_bytes(m, 4) == 4 * 8 * 2 * 128 * 128 * 2
    assert kv.decode_scratch_bytes(m, 64) > 0
    bad = kv.make_meta(8, 64, 16)
    bad.head_dim = 64
    assert kv.cache_bytes(bad) == 0


def _raw(kv, name):
    return getattr(kv._lib, name)


A = ctypes.c_void_p(0x10000)          # aligned fake device address (never dereferenced)
MIS = ctypes.c_void_p(0x10008)        # not 16-byte aligned
B = ctypes.c_void_p(0x20000)          # a second aligned fake address


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, 2), ("block_size", 16, 2), ("k_bits", 3, 2), ("v_bits", 3, 2), ("v_bits", 8, 2),
    ("num_q_heads", 12, 1), ("n_iters", 0, 1), ("n_iters", 17, 1), ("num_kv_heads", 0, 1),
    ("layout", 2, 1),
])
def test_quantize_rejects_bad_meta(kv, field, value, status):
    m = kv.make_meta(8, 64, 16)
    setattr(m, field, value)
    st = _raw(kv, "kvarn_quantize_tiles")(A, A, A, 128, A, ctypes.byref(m), None)
    assert st == status
    assert kv._lib.kvarn_last_error().decode()


def test_group_larger_than_eight_unsupported(kv):
    m = kv.make_meta(2, 32, 16)
    assert _raw(kv, "kvarn_decode_attention")(A, A, A, A, A, 1, A, A, 1 << 20, ctypes.byref(m), None) == 2


def test_quantize_rejects_partial_tiles_and_nulls(kv):
    m = kv.make_meta(8, 64, 16)
    q = _raw(kv, "kvarn_quantize_tiles")
    assert q(A, A, A, 100, A, ctypes.byref(m), None) == 1          # not a multiple of 128
    assert q(A, A, A, -128, A, ctypes.byref(m), None) == 1
    assert q(None, A, A, 128, A, ctypes.byref(m), None) == 1       # NULL k
    assert q(A, MIS, A, 128, A, ctypes.byref(m), None) == 3        # misaligned v
    assert q(A, A, A, 128, A, None, None) == 1                     # NULL meta
    assert q(A, A, A, 0, A, ctypes.byref(m), None) == 0            # nothing to do
    assert q(A, A, A, 1 << 31, A, ctypes.byref(m), None) == 1      # token index beyond 32 bits
    m1 = kv.make_meta(512, 512, 16)
    assert q(A, A, A, 1 << 30, A, ctypes.byref(m1), None) == 1     # 2^23 tiles x 512 kv-heads: items beyond 2^31


def test_append_rejects_aliasing_and_nulls(kv):
    m = kv.make_meta(8, 64, 16, max_blocks_per_seq=4)
    ap = _raw(kv, "kvarn_append_decode")
    assert ap(A, A, A, A, A, 4, A, A, ctypes.byref(m), None) == 1   # seq_lens_out aliases seq_lens
    assert ap(A, A, None, None, A, 4, A, A, ctypes.byref(m), None) == 1
    assert ap(A, A, A, None, A, -1, A, A, ctypes.byref(m), None) == 1
    m0 = kv.make_meta(8, 64, 16, max_blocks_per_seq=0)
    assert ap(A, A, A, None, A, 4, A, A, ctypes.byref(m0), None) == 1
    assert ap(A, A, A, B, A, 0, A, A, ctypes.byref(m), None) == 0      # no sequences: nothing to do


def test_decode_rejects_small_scratch(kv):
    m = kv.make_meta(8, 64, 1024, max_blocks_per_seq=128)
    need = kv.decode_scratch_bytes(m, 4)
    dec = _raw(kv, "kvarn_decode_attention")
    assert dec(A, A, A, A, A, 4, A, A, need - 16, ctypes.byref(m), None) == 4
    assert dec(A, A, A, A, A, 0, A, A, 0, ctypes.byref(m), None) == 0          # no sequences: nothing to do
    assert dec(A, A, A, A, A, 4, A, None, need, ctypes.byref(m), None) == 1     # NULL scratch
    assert dec(A, A, A, A, A, 4, None, A, need, ctypes.byref(m), None) == 1     # NULL out


def test_serve_step_rejects_bad_arguments(kv):
    """kvarn_serve_step: seq_lens_out is required and must not alias seq_lens, the
    workspace is required, and the scratch must hold the decode's partial records."""
    m = kv.make_meta(8, 64, 1024, max_blocks_per_seq=128)
    need = kv.decode_scratch_bytes(m, 4)
    sv = _raw(kv, "kvarn_serve_step")
    mm = ctypes.byref(m)
    #        q  kn vn lens out_lens bt  n  ws cache out scratch bytes meta stream
    assert sv(A, A, A, A, None, A, 4, A, A, A, A, need, mm, None) == 1       # NULL seq_lens_out
    assert sv(A, A, A, A, A, A, 4, A, A, A, A, need, mm, None) == 1          # seq_lens_out aliases seq_lens
    assert sv(A, A, A, A, B, A, 4, None, A, A, A, need, mm, None) == 1       # NULL workspace
    assert sv(A, A, A, A, B, A, 4, A, A, A, A, need - 16, mm, None) == 4     # scratch too small
    assert sv(A, A, A, A, B, A, 70000, A, A, A, A, need, mm, None) == 1      # n_seqs > 65535
    assert sv(A, A, A, A, B, A, 0, A, A, A, A, 0, mm, None) == 0             # nothing to do
    m0 = kv.make_meta(8, 64, 16, max_blocks_per_seq=0)
    assert sv(A, A, A, A, B, A, 4, A, A, A, A, need, ctypes.byref(m0), None) == 1


def test_prefill_rejects_bad_arguments(kv):
    """kvarn_prefill_attention: sequence count and chunk bound are checked, empty work
    returns before any pointer is looked at, pointers must be non-NULL and 16-byte
    aligned (cache and block tables only when the meta allows cached blocks, the
    workspace only when given)."""
    m = kv.make_meta(8, 64, 1024, max_blocks_per_seq=128)
    pf = _raw(kv, "kvarn_prefill_attention")
    mm = ctypes.byref(m)
    #        q  kn vn cu lens  n  max  bt cache ws  out meta stream
    assert pf(A, A, A, A, A, -1, 16, A, A, A, A, mm, None) == 1           # n_seqs < 0
    assert pf(A, A, A, A, A, 65536, 16, A, A, A, A, mm, None) == 1        # n_seqs > 65535
    assert pf(A, A, A, A, A, 4, -1, A, A, A, A, mm, None) == 1            # max_chunk < 0
    assert pf(None, None, None, None, None, 0, 16, None, None, None, None, mm, None) == 0   # no sequences
    assert pf(None, None, None, None, None, 4, 0, None, None, None, None, mm, None) == 0    # empty chunks
    assert pf(None, A, A, A, A, 4, 16, A, A, A, A, mm, None) == 1         # NULL q
    assert pf(A, MIS, A, A, A, 4, 16, A, A, A, A, mm, None) == 3          # misaligned k_new
    assert pf(A, A, A, A, A, 4, 16, A, None, A, A, mm, None) == 1         # NULL cache with cached blocks
    assert pf(A, A, A, A, A, 4, 16, A, A, MIS, A, mm, None) == 3          # misaligned workspace
    assert pf(A, A, A, A, A, 4, 16, A, A, A, None, mm, None) == 1         # NULL out
    assert pf(A, A, A, A, A, 4, 16, A, A, A, A, None, None) == 1          # NULL meta
    assert kv._lib.kvarn_last_error().decode()


def test_presets_are_accepted_and_sized(kv):
    for preset, (kb, vb), rec in (("k4v2", (4, 2), 14336), ("k4v4", (4, 4), 18432), ("k2v2", (2, 2), 10240),
                                  ("k4v2l", (4, 2), 13824)):
        meta = kv.make_meta(8, 64, 10, preset=preset)
        assert (meta.k_bits, meta.v_bits) == (kb, vb)
        assert kv.meta_record_bytes(meta) == rec
        assert kv.cache_bytes(meta) == 10 * 8 * rec
    meta = kv.make_meta(8, 64, 10)
    meta.k_bits, meta.v_bits = 2, 4            # not a preset
    assert kv.meta_record_bytes(meta) == 0 and kv.cache_bytes(meta) == 0


def test_lean_layout_only_with_k4v2(kv):
    meta = kv.make_meta(2, 2, 4, preset="k4v4")
    meta.layout = kv.KVARN_LAYOUT_LEAN
    assert kv.meta_record_bytes(meta) == 0
    st = _raw(kv, "kvarn_quantize_tiles")(None, None, None, 0, None, ctypes.byref(meta), None)
    assert st == 2                      # KVARN_EUNSUPPORTED


def test_static_decode_checks_like_the_scratch_decode(kv):
    """kvarn_decode_attention_static takes the same argument checks as
    kvarn_decode_attention: a misaligned pointer is KVARN_EALIGN, a NULL one
    KVARN_EINVAL, and every preset passes the meta check (these calls return
    before touching a device)."""
    st = _raw(kv, "kvarn_decode_attention_static")
    for preset in ("k4v2", "k4v4", "k2v2", "k4v2l"):
        m = kv.make_meta(8, 64, 1024, max_blocks_per_seq=128, preset=preset)
        mm = ctypes.byref(m)
        #          q    cache ws  bt  lens n  out  meta stream
        assert st(MIS, A, None, A, A, 4, A, mm, None) == 3, preset        # misaligned q
        assert st(A, A, None, A, MIS, 4, A, mm, None) == 3, preset        # misaligned seq_lens
        assert st(A, A, None, A, A, 4, MIS, mm, None) == 3, preset        # misaligned out
        assert st(A, MIS, None, A, A, 4, A, mm, None) == 3, preset        # misaligned cache
        assert st(A, A, MIS, A, A, 4, A, mm, None) == 3, preset           # misaligned workspace
        assert st(None, A, None, A, A, 4, A, mm, None) == 1, preset       # NULL q
        assert st(A, A, None, A, A, 0, A, mm, None) == 0, preset          # nothing to do
    bad = kv.make_meta(8, 64, 1024, max_blocks_per_seq=128)
    bad.k_bits = 3
    assert st(A, A, None, A, A, 4, A, ctypes.byref(bad), None) == 2     # not a preset


def test_bounded_wait_check_rejects_bad_arguments(kv):
    chk = _raw(kv, "kvarn_check_bounded_waits")
    assert chk(2, 1000, A, 256, None) == 1              # unknown wait kind
    assert chk(0, 0, None, 0, None) == 1                # limit below 1 us
    assert chk(0, 2000000, None, 0, None) == 1          # limit above 1 s
    assert chk(1, 1000, None, 0, None) == 1             # grid barrier needs scratch
    assert chk(1, 1000, MIS, 256, None) == 3            # misaligned scratch
    assert chk(1, 1000, A, 4, None) == 4                # scratch smaller than the barrier words
