"""Python binding of libkvarn (KVarN tile quantization + paged decode attention on
GB300). Argument marshalling only: every step runs in the CUDA library, whose C
ABI is declared in include/kvarn.h. Tensors are torch CUDA tensors; PyTorch only
provides device memory and streams.

Importing this module loads ``libkvarn.so`` built in-tree by ``build_lib.build()``;
if the library is missing the import fails (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvarn.so")

RECORD_BYTES = 14336
HEAD_DIM = 128
BLOCK_SIZE = 128

KVARN_OK, KVARN_EINVAL, KVARN_EUNSUPPORTED, KVARN_EALIGN, KVARN_ESCRATCH, KVARN_ECUDA = range(6)
FLAG_BAD_SLOTS, FLAG_BAD_BLOCK, FLAG_BAD_LENGTH, FLAG_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
KVARN_WAIT_MBARRIER, KVARN_WAIT_GRID = 0, 1

# exported entry points and their C signatures (include/kvarn.h)
_SIGS = {
    "kvarn_record_bytes": (ctypes.c_size_t, []),
    "kvarn_meta_record_bytes": (ctypes.c_size_t, [ctypes.c_void_p]),
    "kvarn_cache_bytes": (ctypes.c_size_t, [ctypes.c_void_p]),
    "kvarn_workspace_bytes": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32]),
    "kvarn_decode_scratch_bytes": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32]),
    "kvarn_quantize_tiles": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvarn_append_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p]),
    "kvarn_decode_attention": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "kvarn_decode_attention_static": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvarn_serve_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p, ctypes.c_void_p]),
    "kvarn_prefill_attention": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p]),
    "kvarn_check_bounded_waits": (ctypes.c_int, [ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t,
                                                 ctypes.c_void_p]),
    "kvarn_device_flags": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]),
    "kvarn_last_error": (ctypes.c_char_p, []),
}


class KvarnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libkvarn status {status}: {message}")
        self.status = status


class KvarnMeta(ctypes.Structure):
    """Mirror of ``kvarn_meta`` (include/kvarn.h)."""
    _fields_ = [
        ("num_kv_heads", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("k_bits", ctypes.c_int32),
        ("v_bits", ctypes.c_int32),
        ("n_iters", ctypes.c_int32),
        ("eps", ctypes.c_float),
        ("num_blocks", ctypes.c_int64),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("layout", ctypes.c_int32),
    ]


# bit widths (keys, values) and metadata layout of the presets; k4v2 is
# kvarn_k4v2_g128, k4v2l the same with lean metadata (KVARN_LAYOUT_LEAN)
PRESETS = {"k4v2": (4, 2, 0), "k4v4": (4, 4, 0), "k2v2": (2, 2, 0), "k4v2l": (4, 2, 1)}
KVARN_LAYOUT_LEAN = 1


def make_meta(num_kv_heads: int, num_q_heads: int, num_blocks: int, max_blocks_per_seq: int = 0,
              n_iters: int = 4, eps: float = 1e-6, preset: str = "k4v2") -> KvarnMeta:
    """Head_dim 128, block 128; preset k4v2 (4-bit K, 2-bit V: kvarn_k4v2_g128),
    k4v4, k2v2, or k4v2l (k4v2 with lean metadata)."""
    kb, vb, layout = PRESETS[preset]
    return KvarnMeta(num_kv_heads, num_q_heads, HEAD_DIM, BLOCK_SIZE, kb, vb, n_iters, eps,
                     num_blocks, max_blocks_per_seq, layout)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


def _check(status: int):
    if status != KVARN_OK:
        raise KvarnError(status, _lib.kvarn_last_error().decode())


def _ptr(t, name, dtype=None, numel=None):
    """Device address of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def record_bytes() -> int:
    return int(_lib.kvarn_record_bytes())


def meta_record_bytes(meta: KvarnMeta) -> int:
    """Bytes of one (block, kv-head) record for the meta's preset."""
    return int(_lib.kvarn_meta_record_bytes(ctypes.byref(meta)))


def cache_bytes(meta: KvarnMeta) -> int:
    return int(_lib.kvarn_cache_bytes(ctypes.byref(meta)))


def workspace_bytes(meta: KvarnMeta, max_seqs: int) -> int:
    return int(_lib.kvarn_workspace_bytes(ctypes.byref(meta), max_seqs))


def decode_scratch_bytes(meta: KvarnMeta, n_seqs: int) -> int:
    return int(_lib.kvarn_decode_scratch_bytes(ctypes.byref(meta), n_seqs))


def kvarn_quantize_tiles(k, v, slot_mapping, cache, meta: KvarnMeta, stream=None):
    """k, v: fp16 [n_tokens, Hkv, 128]; slot_mapping: int64 [n_tokens];
    cache: uint8 [num_blocks, Hkv, meta_record_bytes(meta)]."""
    import torch
    n = int(k.shape[0])
    _check(_lib.kvarn_quantize_tiles(_ptr(k, "k", torch.float16), _ptr(v, "v", torch.float16),
                                     _ptr(slot_mapping, "slot_mapping", torch.int64, n), n,
                                     _ptr(cache, "cache", torch.uint8), ctypes.byref(meta), _stream(stream)))


def kvarn_append_decode(k_new, v_new, seq_lens, seq_lens_out, block_tables, workspace, cache,
                        meta: KvarnMeta, stream=None):
    """k_new, v_new: fp16 [n_seqs, Hkv, 128]; seq_lens (before) / seq_lens_out
    (after, may be None): int32 [n_seqs]; block_tables: int32 [n_seqs,
    max_blocks]; workspace: fp16 [>= n_seqs, Hkv, 2, 128, 128]."""
    import torch
    n = int(k_new.shape[0])
    _check(_lib.kvarn_append_decode(_ptr(k_new, "k_new", torch.float16), _ptr(v_new, "v_new", torch.float16),
                                    _ptr(seq_lens, "seq_lens", torch.int32, n),
                                    _ptr(seq_lens_out, "seq_lens_out", torch.int32, n),
                                    _ptr(block_tables, "block_tables", torch.int32), n,
                                    _ptr(workspace, "workspace", torch.float16),
                                    _ptr(cache, "cache", torch.uint8), ctypes.byref(meta), _stream(stream)))


def kvarn_decode_attention(q, cache, workspace, block_tables, seq_lens, out, scratch, meta: KvarnMeta,
                           stream=None):
    """q, out: fp16 [n_seqs, Hq, 128]; scratch: any CUDA tensor of at least
    decode_scratch_bytes(meta, n_seqs) bytes."""
    import torch
    n = int(q.shape[0])
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(_lib.kvarn_decode_attention(_ptr(q, "q", torch.float16), _ptr(cache, "cache", torch.uint8),
                                       _ptr(workspace, "workspace", torch.float16),
                                       _ptr(block_tables, "block_tables", torch.int32),
                                       _ptr(seq_lens, "seq_lens", torch.int32, n), n,
                                       _ptr(out, "out", torch.float16), _ptr(scratch, "scratch"), nbytes,
                                       ctypes.byref(meta), _stream(stream)))


def kvarn_serve_step(q, k_new, v_new, seq_lens, seq_lens_out, block_tables, workspace, cache, out, scratch,
                     meta: KvarnMeta, stream=None):
    """One serving step in one launch: kvarn_append_decode then
    kvarn_decode_attention over seq_lens_out. q, out: fp16 [n_seqs, Hq, 128];
    k_new, v_new: fp16 [n_seqs, Hkv, 128]; seq_lens / seq_lens_out: int32 [n_seqs];
    scratch: at least decode_scratch_bytes(meta, n_seqs) bytes."""
    import torch
    n = int(q.shape[0])
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(_lib.kvarn_serve_step(_ptr(q, "q", torch.float16), _ptr(k_new, "k_new", torch.float16),
                                 _ptr(v_new, "v_new", torch.float16), _ptr(seq_lens, "seq_lens", torch.int32, n),
                                 _ptr(seq_lens_out, "seq_lens_out", torch.int32, n),
                                 _ptr(block_tables, "block_tables", torch.int32), n,
                                 _ptr(workspace, "workspace", torch.float16), _ptr(cache, "cache", torch.uint8),
                                 _ptr(out, "out", torch.float16), _ptr(scratch, "scratch"), nbytes,
                                 ctypes.byref(meta), _stream(stream)))


def kvarn_decode_attention_static(q, cache, workspace, block_tables, seq_lens, out, meta: KvarnMeta, stream=None):
    """kvarn_decode_attention without a scratch argument, for callers that cannot
    allocate device memory: the library's built-in 16 MiB device array is used
    instead (shared by all calls on a device; calls overlapping on the GPU race).
    The first call on a device looks up that array's address."""
    import torch
    n = int(q.shape[0])
    _check(_lib.kvarn_decode_attention_static(_ptr(q, "q", torch.float16), _ptr(cache, "cache", torch.uint8),
                                              _ptr(workspace, "workspace", torch.float16),
                                              _ptr(block_tables, "block_tables", torch.int32),
                                              _ptr(seq_lens, "seq_lens", torch.int32, n), n,
                                              _ptr(out, "out", torch.float16), ctypes.byref(meta), _stream(stream)))


def kvarn_prefill_attention(q, k_new, v_new, cu_tokens, seq_lens, max_chunk: int, block_tables, cache, workspace,
                            out, meta: KvarnMeta, stream=None):
    """Chunked prefill: q, out fp16 [n_tokens, Hq, 128]; k_new, v_new fp16
    [n_tokens, Hkv, 128]; cu_tokens int32 [n_seqs + 1]; seq_lens int32 [n_seqs]
    (cached tokens before each chunk); max_chunk >= every chunk length."""
    import torch
    n = int(seq_lens.shape[0])
    _check(_lib.kvarn_prefill_attention(_ptr(q, "q", torch.float16), _ptr(k_new, "k_new", torch.float16),
                                        _ptr(v_new, "v_new", torch.float16),
                                        _ptr(cu_tokens, "cu_tokens", torch.int32, n + 1),
                                        _ptr(seq_lens, "seq_lens", torch.int32, n), n, int(max_chunk),
                                        _ptr(block_tables, "block_tables", torch.int32),
                                        _ptr(cache, "cache", torch.uint8), _ptr(workspace, "workspace", torch.float16),
                                        _ptr(out, "out", torch.float16), ctypes.byref(meta), _stream(stream)))


def kvarn_check_bounded_waits(which: int, limit_us: int, scratch=None, stream=None):
    """Runs the library's bounded-wait code against a wait that never completes
    (KVARN_WAIT_MBARRIER or KVARN_WAIT_GRID), giving up after limit_us; the
    timeout shows as FLAG_WAIT_TIMEOUT in kvarn_device_flags(). scratch: a device
    buffer of at least 8 bytes for the grid barrier's words."""
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(_lib.kvarn_check_bounded_waits(int(which), int(limit_us), _ptr(scratch, "scratch"), nbytes,
                                          _stream(stream)))


def kvarn_device_flags(stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib.kvarn_device_flags(ctypes.byref(v), _stream(stream)))
    return int(v.value)
