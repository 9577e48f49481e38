"""KVarN CPU oracle: plain float64 NumPy restatement of the method.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The CUDA library never calls it and shares no code with it.

Sources (the method is only described in prose; every constant below that the
pages leave open is a stated reading, marked [R]):

* KVarN README (huawei-csl/KVarN), "How KVarN works", stages 1-4: tiles of fp16
  KV (channels x tokens) are (2) Hadamard-rotated along channels, (3) iteratively
  variance-normalised in log space, alternating column-wise and row-wise std
  normalisation, Sinkhorn style, and (4) quantised by asymmetric round-to-nearest
  at low bit width, with the scales re-applied on read: per channel for keys, per
  token for values.
* KVarN README, quick start and note: preset ``kvarn_k4v2_g128`` (4-bit keys,
  2-bit values, tile 128), block size fixed at 128 (one vLLM block = one tile),
  float16 compute, and a small fixed decode workspace.

Readings [R] fixed here (the pages are silent on them):

* H is the Sylvester Hadamard matrix of order 128 in natural order, scaled by
  1/sqrt(128) so that H = H^T = H^-1; the same H for K and V and for q.
* Tile matrix X is [128 channels (rows i) x 128 tokens (columns j)].
* "std" is the population standard deviation (ddof 0) about the mean; the data
  are divided, never centred (the offset is left to the asymmetric zero point).
* One iteration = a column pass (each token's std over channels) followed by a
  row pass (each channel's std over tokens); 4 iterations; eps = 1e-6 is added to
  the variance before the log; only the log scales are accumulated and
  exponentiated once at the end.
* Stored scales r, c, s, z are fp16 (round to nearest even); r, c and s are held
  inside the normal fp16 range [2^-14, 65504], z inside [-65504, 65504].
* RTN: z = fp16(group min), s = fp16((group max - z) / (2^b - 1)), code =
  clamp(floor((y - z) / s + 1/2), 0, 2^b - 1). Key groups are rows (one per
  channel, over tokens), value groups are columns (one per token, over channels).
* Decode attention: q is a [heads x 128] fp16 query, softmax scale 1/sqrt(128),
  q-head h reads kv-head h // (Hq / Hkv), every stored token is attended (no
  mask), and the tokens of a partial last tile are taken exactly from the fp16
  decode workspace (unrotated, unquantised).

The packed record layout (14336 bytes per (block, kv-head) for the default
preset) is documented in the C header of the CUDA library and restated by the
position functions below. Besides the README's preset k4v2, the library offers
k4v4 and k2v2 (the pages report 2-bit results as well); a record is the key codes,
then the value codes, then 1024 bytes of key metadata and 1024 of value metadata.
"""
from __future__ import annotations

import numpy as np

D = 128            # channels per head
B = 128            # tokens per tile (= block size)
K_BITS = 4
V_BITS = 2
N_ITERS = 4
EPS = 1e-6
FP16_MIN_NORMAL = 2.0 ** -14
FP16_MAX = 65504.0

K_CODE_OFF, K_CODE_BYTES = 0, 8192
V_CODE_OFF, V_CODE_BYTES = 8192, 4096
K_META_OFF = 12288
V_META_OFF = 13312
RECORD_BYTES = 14336

# bit widths (keys, values) of the presets; the default one is the README's
PRESETS = {"k4v2": (4, 2), "k4v4": (4, 4), "k2v2": (2, 2), "k4v2l": (4, 2)}
DEFAULT_PRESET = "k4v2"
# Presets with lean metadata [R]: a key group is one channel, so the channel's
# row scale r_i is one constant inside it and folds into the group's (s, z); a
# value group is one token, so c_j folds into the value (s, z). Such records store
# (c, s, z) for keys and (r, s, z) for values: 768 bytes each instead of 1024.
LEAN = {"k4v2l"}


# ----------------------------------------------------------------------------------
# Stage 2: Hadamard rotation along channels
# ----------------------------------------------------------------------------------
def sylvester_hadamard(n: int = D) -> np.ndarray:
    """Orthonormal Sylvester Hadamard matrix H_n / sqrt(n) (KVarN README, "How KVarN
    works", stage 2: an orthonormal Hadamard rotation along channels, which keeps
    attention scores unchanged). Built by the doubling H_2m = [[H, H], [H, -H]]."""
    assert n >= 1 and n & (n - 1) == 0
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)


_H = sylvester_hadamard(D)


def rotate(x: np.ndarray) -> np.ndarray:
    """X_r = H @ X for tiles X [..., 128 channels, 128 tokens]."""
    return _H @ x


def fp16_rne(x) -> np.ndarray:
    """Round float64 values to IEEE binary16, nearest even; returned as float64."""
    return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)


# ----------------------------------------------------------------------------------
# Stage 3: iterative log-space variance normalisation
# ----------------------------------------------------------------------------------
def normalise(xr: np.ndarray, n_iters: int = N_ITERS, eps: float = EPS, trace: list | None = None):
    """Log row / column scales (lr [..., 128 channels], lc [..., 128 tokens]) of the
    Sinkhorn-style normalisation (KVarN README, "How KVarN works", stage 3:
    alternate column-wise and row-wise std normalisation in log space).

    Z = X_r / (exp(lr)_i * exp(lc)_j). Each iteration first adds half the log of
    every column's variance (over channels) plus eps to lc, then, with the new lc,
    half the log of every row's variance (over tokens) plus eps to lr.
    If `trace` is a list, the per-iteration column log-stds of Z measured at the
    start of each column pass are appended to it."""
    lr = np.zeros(xr.shape[:-1])
    lc = np.zeros(xr.shape[:-2] + xr.shape[-1:])
    for _ in range(n_iters):
        z = xr * np.exp(-lr)[..., :, None] * np.exp(-lc)[..., None, :]
        col_var = z.var(axis=-2)
        if trace is not None:
            trace.append(0.5 * np.log(col_var + eps))
        lc = lc + 0.5 * np.log(col_var + eps)
        z = xr * np.exp(-lr)[..., :, None] * np.exp(-lc)[..., None, :]
        lr = lr + 0.5 * np.log(z.var(axis=-1) + eps)
    return lr, lc


# ----------------------------------------------------------------------------------
# Stage 4: asymmetric round-to-nearest
# ----------------------------------------------------------------------------------
def rtn(y: np.ndarray, bits: int, axis: int):
    """Asymmetric RTN of y in groups along `axis` (KVarN README, "How KVarN works",
    stage 4). Returns (codes uint8, s, z, pre) where s, z are fp16 values and
    pre = (y - z) / s is the value before rounding to a code."""
    levels = (1 << bits) - 1
    ymin = y.min(axis=axis)
    ymax = y.max(axis=axis)
    z = fp16_rne(np.clip(ymin, -FP16_MAX, FP16_MAX))
    s_pre = np.maximum(ymax - z, 0.0) / levels
    s = fp16_rne(np.clip(s_pre, FP16_MIN_NORMAL, FP16_MAX))
    pre = (y - np.expand_dims(z, axis)) / np.expand_dims(s, axis)
    codes = np.clip(np.floor(pre + 0.5), 0, levels).astype(np.uint8)
    return codes, s, z, dict(zmin=ymin, zmax=ymax, s_pre=s_pre, pre=pre)


def quantize_tensor(x: np.ndarray, kind: str, n_iters: int = N_ITERS, eps: float = EPS, bits: int | None = None,
                    lean: bool = False):
    """Stages 2-4 for tiles x [..., 128 channels, 128 tokens] (float64 holding fp16
    values). kind 'K': s and z per channel (row); kind 'V': s and z per token
    (column); `bits` codes (default: 4 for K, 2 for V, the README's preset).

    With `lean`, the scale that is constant inside a group is folded into the
    group's (s, z): keys are quantized from X_r / c_j (groups are channels) and
    values from X_r / r_i (groups are tokens); the result's `stored` names the
    scale vectors a lean record keeps.

    Returns a dict with fp16-valued r [.., 128], c [.., 128], s, z, the codes
    [.., 128 ch, 128 tok] and the pre-rounding values needed to decide ties."""
    assert kind in ("K", "V")
    if bits is None:
        bits = K_BITS if kind == "K" else V_BITS
    xr = rotate(np.asarray(x, np.float64))
    lr, lc = normalise(xr, n_iters, eps)
    r_pre, c_pre = np.exp(lr), np.exp(lc)
    r = fp16_rne(np.clip(r_pre, FP16_MIN_NORMAL, FP16_MAX))
    c = fp16_rne(np.clip(c_pre, FP16_MIN_NORMAL, FP16_MAX))
    if not lean:
        y = xr / (r[..., :, None] * c[..., None, :])
        stored = ("r", "c", "s", "z")
    elif kind == "K":
        y = xr / c[..., None, :]
        stored = ("c", "s", "z")
    else:
        y = xr / r[..., :, None]
        stored = ("r", "s", "z")
    codes, s, z, info = rtn(y, bits, axis=-1 if kind == "K" else -2)
    return dict(kind=kind, bits=bits, codes=codes, r=r, c=c, s=s, z=z, r_pre=r_pre, c_pre=c_pre,
                z_pre=info["zmin"], s_pre=info["s_pre"], code_pre=info["pre"], xr=xr, y=y, stored=stored)


def dequant_tensor(codes, r, c, s, z, kind: str, rotated: bool = False):
    """Inverse of stage 4 (scales re-applied on read) and of stage 2:
    X_r_hat[i, j] = r_i c_j (code_ij s + z) with (s, z) per row for K and per
    column for V; returns H @ X_r_hat unless `rotated`."""
    codes = np.asarray(codes, np.float64)
    if kind == "K":
        inner = codes * s[..., :, None] + z[..., :, None]
    else:
        inner = codes * s[..., None, :] + z[..., None, :]
    xr_hat = r[..., :, None] * c[..., None, :] * inner
    return xr_hat if rotated else _H @ xr_hat


# ----------------------------------------------------------------------------------
# Packed record layout (one (block, kv-head))
# ----------------------------------------------------------------------------------
def k4_position(i: int, t: int):
    """(byte, bit shift) of the 4-bit key code of channel i, token t, counted from
    the start of the key codes.

    Token t owns bytes [64 t, 64 t + 64): four 16-byte groups g4 = (i >> 1) & 3,
    each four little-endian 32-bit words w = i >> 5. Within a word, nibble
    p = 4 ((i >> 3) & 1) + 2 (i & 1) + ((i >> 4) & 1), nibble p at bits 4p..4p+3:
    the low nibbles of bytes (0, 1) and (2, 3) hold channels 2c + {0, 1} and
    2c + {8, 9} of the word's first 16 channels, the high nibbles those of its last 16
    (c = g4), so one 16-bit half of the word masked to low nibbles is a pair of
    fp6 (e2m3) values code / 8."""
    g4 = (i >> 1) & 3
    w = i >> 5
    p = 4 * ((i >> 3) & 1) + 2 * (i & 1) + ((i >> 4) & 1)
    return t * 64 + g4 * 16 + w * 4 + p // 2, 4 * (p % 2)


def k2_position(i: int, t: int):
    """(byte, bit shift) of the 2-bit key code of channel i, token t, counted from
    the start of the key codes.

    Token t owns bytes [32 t, 32 t + 32): four 8-byte groups g4 = (i >> 1) & 3,
    each two little-endian words u = i >> 6. Within a word, crumb
    p = 4 ((i >> 4) & 3) + 2 (i & 1) + ((i >> 3) & 1), crumb p at bits 2p..2p+1:
    byte k of the word holds the 16-channel step k, channels 2c + {0, 1} at bits
    {0, 4} and 2c + {8, 9} at bits {2, 6} of the byte (c = g4), so a byte masked to
    bits {0, 1, 4, 5} is a pair of fp4 (e2m1) values code / 2."""
    g4 = (i >> 1) & 3
    u = i >> 6
    p = 4 * ((i >> 4) & 3) + 2 * (i & 1) + ((i >> 3) & 1)
    return t * 32 + g4 * 8 + u * 4 + p // 4, 2 * (p % 4)


def v2_position(i: int, t: int):
    """(byte, bit shift) of the 2-bit value code of channel i, token t, counted from
    the start of the value codes.

    Channel i lives in 512-byte panel m = i >> 4 (16 channels). Inside a panel,
    16-byte cell (i & 7) * 4 + g4 with g4 = (t >> 1) & 3 holds 8 bytes for channel
    i with (i >> 3) & 1 == 0 followed by 8 bytes for its partner i + 8; each 8
    bytes are two little-endian words u = t >> 6. Within a word, crumb
    p = 4 ((t >> 4) & 3) + 2 (t & 1) + ((t >> 3) & 1), crumb p at bits 2p..2p+1
    (the 2-bit key order with the token in the channel's place)."""
    m = i >> 4
    cell = (i & 7) * 4 + ((t >> 1) & 3)
    which = (i >> 3) & 1
    u = t >> 6
    p = 4 * ((t >> 4) & 3) + 2 * (t & 1) + ((t >> 3) & 1)
    return m * 512 + cell * 16 + which * 8 + u * 4 + p // 4, 2 * (p % 4)


def v4_position(i: int, t: int):
    """(byte, bit shift) of the 4-bit value code of channel i, token t, counted from
    the start of the value codes: the 4-bit key layout with the roles of channel
    and token exchanged. Channel i owns bytes [64 i, 64 i + 64): four 16-byte
    groups g4 = (t >> 1) & 3, each four words w = t >> 5; nibble
    p = 4 ((t >> 3) & 1) + 2 (t & 1) + ((t >> 4) & 1) at bits 4p..4p+3."""
    g4 = (t >> 1) & 3
    w = t >> 5
    p = 4 * ((t >> 3) & 1) + 2 * (t & 1) + ((t >> 4) & 1)
    return i * 64 + g4 * 16 + w * 4 + p // 2, 4 * (p % 2)


def k_code_position(i: int, t: int):
    """(byte, bit shift) of the key code of channel i, token t in a k4v2 record."""
    b, sh = k4_position(i, t)
    return K_CODE_OFF + b, sh


def v_code_position(i: int, t: int):
    """(byte, bit shift) of the value code of channel i, token t in a k4v2 record."""
    b, sh = v2_position(i, t)
    return V_CODE_OFF + b, sh


def _source_table(position, bits: int) -> np.ndarray:
    """For each byte of a code area, the flat (i * 128 + t) index of the code in
    each of its 8 / bits slots (slot n at bits n*bits..)."""
    per = 8 // bits
    nbytes = D * B * bits // 8
    src = np.full((nbytes, per), -1, np.int64)
    for i in range(D):
        for t in range(B):
            b, sh = position(i, t)
            assert src[b, sh // bits] == -1
            src[b, sh // bits] = i * B + t
    assert (src >= 0).all()
    return src


class Layout:
    """Byte layout of the records of one preset."""

    def __init__(self, name: str):
        self.name = name
        self.k_bits, self.v_bits = PRESETS[name]
        self.lean = name in LEAN
        # scale vectors kept per tensor, in record order (fp16 x 128 each)
        self.k_meta = ("c", "s", "z") if self.lean else ("r", "c", "s", "z")
        self.v_meta = ("r", "s", "z") if self.lean else ("r", "c", "s", "z")
        self.k_code_off, self.k_code_bytes = 0, D * B * self.k_bits // 8
        self.v_code_off, self.v_code_bytes = self.k_code_bytes, D * B * self.v_bits // 8
        self.k_meta_off = self.v_code_off + self.v_code_bytes
        self.v_meta_off = self.k_meta_off + 256 * len(self.k_meta)
        self.record_bytes = self.v_meta_off + 256 * len(self.v_meta)
        self.k_src = _source_table(k4_position if self.k_bits == 4 else k2_position, self.k_bits)
        self.v_src = _source_table(v4_position if self.v_bits == 4 else v2_position, self.v_bits)


LAYOUTS = {name: Layout(name) for name in PRESETS}
K_SRC, V_SRC = LAYOUTS[DEFAULT_PRESET].k_src, LAYOUTS[DEFAULT_PRESET].v_src


def layout_of(record_bytes: int) -> Layout:
    """The preset layout whose records have `record_bytes` bytes."""
    for lay in LAYOUTS.values():
        if lay.record_bytes == record_bytes:
            return lay
    raise ValueError(f"no preset has {record_bytes}-byte records")


def _f16_bytes(vals) -> np.ndarray:
    a = np.asarray(vals, np.float64).astype("<f2")
    return a.view(np.uint8).reshape(a.shape[:-1] + (a.shape[-1] * 2,))


def _pack_codes(codes: np.ndarray, src: np.ndarray, bits: int) -> np.ndarray:
    out = np.zeros(codes.shape[:-1] + (src.shape[0],), np.uint8)
    for n in range(src.shape[1]):
        out |= (codes[..., src[:, n]] << (bits * n)).astype(np.uint8)
    return out


def _unpack_codes(area: np.ndarray, src: np.ndarray, bits: int) -> np.ndarray:
    codes = np.zeros(area.shape[:-1] + (D * B,), np.uint8)
    for n in range(src.shape[1]):
        codes[..., src[:, n]] = (area >> (bits * n)) & ((1 << bits) - 1)
    return codes


def pack_record(kq: dict, vq: dict, preset: str = DEFAULT_PRESET) -> np.ndarray:
    """Records [..., record bytes] uint8 from quantize_tensor results for K and V."""
    lay = LAYOUTS[preset]
    assert kq.get("bits", lay.k_bits) == lay.k_bits and vq.get("bits", lay.v_bits) == lay.v_bits
    assert kq.get("stored", lay.k_meta) == lay.k_meta and vq.get("stored", lay.v_meta) == lay.v_meta
    kc = kq["codes"].reshape(kq["codes"].shape[:-2] + (D * B,)).astype(np.uint8)
    vc = vq["codes"].reshape(vq["codes"].shape[:-2] + (D * B,)).astype(np.uint8)
    rec = np.zeros(kc.shape[:-1] + (lay.record_bytes,), np.uint8)
    rec[..., lay.k_code_off:lay.k_code_off + lay.k_code_bytes] = _pack_codes(kc, lay.k_src, lay.k_bits)
    rec[..., lay.v_code_off:lay.v_code_off + lay.v_code_bytes] = _pack_codes(vc, lay.v_src, lay.v_bits)
    for off, q, names in ((lay.k_meta_off, kq, lay.k_meta), (lay.v_meta_off, vq, lay.v_meta)):
        for n, name in enumerate(names):
            rec[..., off + 256 * n: off + 256 * (n + 1)] = _f16_bytes(q[name])
    return rec


def unpack_record(rec: np.ndarray):
    """Inverse of pack_record (the preset follows from the record size): dicts for
    K and V with codes [.., 128 ch, 128 tok], bits and r, c, s, z (float64
    holding fp16); a scale a lean record does not keep is returned as ones, which
    is what it was folded against, and `stored` names the kept ones."""
    rec = np.asarray(rec, np.uint8)
    lay = layout_of(rec.shape[-1])
    lead = rec.shape[:-1]
    kc = _unpack_codes(rec[..., lay.k_code_off:lay.k_code_off + lay.k_code_bytes], lay.k_src, lay.k_bits)
    vc = _unpack_codes(rec[..., lay.v_code_off:lay.v_code_off + lay.v_code_bytes], lay.v_src, lay.v_bits)
    out = []
    for off, codes, kind, bits, names in ((lay.k_meta_off, kc, "K", lay.k_bits, lay.k_meta),
                                          (lay.v_meta_off, vc, "V", lay.v_bits, lay.v_meta)):
        meta = np.ascontiguousarray(rec[..., off:off + 256 * len(names)]).view("<f2").astype(np.float64)
        d = dict(kind=kind, bits=bits, codes=codes.reshape(lead + (D, B)), stored=names)
        for name in ("r", "c"):
            d[name] = np.ones(lead + (D,))
        for n, name in enumerate(names):
            d[name] = meta[..., 128 * n:128 * (n + 1)]
        out.append(d)
    return out[0], out[1]


def dequant_record(rec: np.ndarray, rotated: bool = False):
    """(K_hat, V_hat) tiles [.., 128 ch, 128 tok] of packed records."""
    k, v = unpack_record(rec)
    return (dequant_tensor(k["codes"], k["r"], k["c"], k["s"], k["z"], "K", rotated),
            dequant_tensor(v["codes"], v["r"], v["c"], v["s"], v["z"], "V", rotated))


# ----------------------------------------------------------------------------------
# Whole-tile and paged-cache operations
# ----------------------------------------------------------------------------------
def quantize_tiles(k_tok: np.ndarray, v_tok: np.ndarray, n_iters: int = N_ITERS, eps: float = EPS,
                   preset: str = DEFAULT_PRESET):
    """k_tok, v_tok: fp16 tiles [..., 128 tokens, 128 channels] (vLLM row layout).
    Returns (records [..., record bytes], K result, V result)."""
    kb, vb = PRESETS[preset]
    lean = preset in LEAN
    kx = np.swapaxes(np.asarray(k_tok, np.float64), -1, -2)
    vx = np.swapaxes(np.asarray(v_tok, np.float64), -1, -2)
    kq = quantize_tensor(kx, "K", n_iters, eps, bits=kb, lean=lean)
    vq = quantize_tensor(vx, "V", n_iters, eps, bits=vb, lean=lean)
    return pack_record(kq, vq, preset), kq, vq


def quantize_into_cache(k, v, slot_mapping, cache, tiles=None, batch: int = 32):
    """Prefill write (kvarn_quantize_tiles): every run of 128 tokens [t0, t0+128)
    goes to block slot_mapping[t0] // 128, token t0 + k at offset k. k, v: fp16
    [n_tokens, Hkv, 128]; cache: uint8 [num_blocks, Hkv, record bytes] (the preset
    follows from the record size), updated in place. `tiles`, if given, restricts
    the work to a list of (chunk, head) pairs."""
    preset = layout_of(cache.shape[-1]).name
    n_tokens, hkv, _ = k.shape
    assert n_tokens % B == 0
    work = tiles if tiles is not None else [(ch, h) for ch in range(n_tokens // B) for h in range(hkv)]
    for b0 in range(0, len(work), batch):
        part = work[b0:b0 + batch]
        kt = np.stack([k[ch * B:(ch + 1) * B, h, :] for ch, h in part])
        vt = np.stack([v[ch * B:(ch + 1) * B, h, :] for ch, h in part])
        recs, _, _ = quantize_tiles(kt, vt, preset=preset)
        for (ch, h), rec in zip(part, recs):
            blk = int(slot_mapping[ch * B]) // B
            cache[blk, h] = rec
    return cache


def attend(q: np.ndarray, k_tok: np.ndarray, v_tok: np.ndarray) -> np.ndarray:
    """Softmax attention of queries q [G, 128] over tokens k_tok, v_tok [L, 128]
    with scale 1/sqrt(128), in float64."""
    s = (q @ k_tok.T) / np.sqrt(D)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ v_tok


def decode_one(q_heads, cache, workspace_sh, block_table, seq_len: int, kv_head: int):
    """Decode attention for the q-heads of one GQA group over one sequence.

    q_heads: [G, 128]; cache: [num_blocks, Hkv, record bytes]; workspace_sh: fp16
    [2, 128 tok, 128 ch] for this (sequence, kv-head) or None; block_table:
    [max_blocks]. Full tiles come from the packed cache (dequantised, un-rotated),
    the last seq_len % 128 tokens from the workspace."""
    n_full, n_ws = seq_len // B, seq_len % B
    ks, vs = [], []
    if n_full:
        recs = cache[np.asarray(block_table[:n_full], np.int64), kv_head]
        kh, vh = dequant_record(recs)                     # [n_full, ch, tok]
        ks.append(np.swapaxes(kh, -1, -2).reshape(-1, D))
        vs.append(np.swapaxes(vh, -1, -2).reshape(-1, D))
    if n_ws:
        ks.append(np.asarray(workspace_sh[0, :n_ws], np.float64))
        vs.append(np.asarray(workspace_sh[1, :n_ws], np.float64))
    return attend(np.asarray(q_heads, np.float64), np.concatenate(ks), np.concatenate(vs))


def decode(q, cache, workspace, block_tables, seq_lens, pairs=None):
    """Decode attention (kvarn_decode_attention) for q [n_seqs, Hq, 128]; returns
    float64 [n_seqs, Hq, 128]. `pairs`, if given, restricts the work to a list of
    (sequence, kv-head) pairs (other outputs are NaN)."""
    n_seqs, hq, _ = q.shape
    hkv = cache.shape[1]
    g = hq // hkv
    out = np.full(q.shape, np.nan)
    work = pairs if pairs is not None else [(s, h) for s in range(n_seqs) for h in range(hkv)]
    for s, h in work:
        ws = None if workspace is None else workspace[s, h]
        out[s, h * g:(h + 1) * g] = decode_one(q[s, h * g:(h + 1) * g], cache, ws,
                                               block_tables[s], int(seq_lens[s]), h)
    return out


def prefill_attention(q, k_new, v_new, cu_tokens, seq_lens, block_tables, workspace, cache, tokens=None):
    """Chunked-prefill attention (kvarn_prefill_attention) [R]: sequence s has
    L0 = seq_lens[s] tokens in the cache (floor(L0/128) packed tiles read through
    its block table, then L0 % 128 tokens in its fp16 workspace) and appends the
    chunk of fresh fp16 tokens cu_tokens[s] .. cu_tokens[s+1] - 1 of k_new, v_new
    [n_tokens, Hkv, 128]. Chunk token p (0-based) attends the L0 cached tokens and
    chunk tokens 0..p (causal), with the decode's softmax scale and GQA mapping.

    q: [n_tokens, Hq, 128]; returns float64 [n_tokens, Hq, 128]. `tokens`, if given,
    restricts the work to a list of (token, kv-head) pairs (other rows are NaN)."""
    n_tokens, hq, _ = q.shape
    hkv = k_new.shape[1]
    g = hq // hkv
    out = np.full(q.shape, np.nan)
    seq_of = np.searchsorted(np.asarray(cu_tokens), np.arange(n_tokens), side="right") - 1
    work = tokens if tokens is not None else [(t, h) for t in range(n_tokens) for h in range(hkv)]
    ctx = {}
    for t, h in work:
        s = int(seq_of[t])
        if (s, h) not in ctx:                    # cached tokens of (s, h), un-rotated
            L0 = int(seq_lens[s])
            n_full, n_ws = L0 // B, L0 % B
            ks, vs = [np.zeros((0, D))], [np.zeros((0, D))]
            if n_full:
                kh, vh = dequant_record(cache[np.asarray(block_tables[s, :n_full], np.int64), h])
                ks.append(np.swapaxes(kh, -1, -2).reshape(-1, D))
                vs.append(np.swapaxes(vh, -1, -2).reshape(-1, D))
            if n_ws:
                ks.append(np.asarray(workspace[s, h, 0, :n_ws], np.float64))
                vs.append(np.asarray(workspace[s, h, 1, :n_ws], np.float64))
            ctx[(s, h)] = (np.concatenate(ks), np.concatenate(vs))
        kc, vc = ctx[(s, h)]
        t0 = int(cu_tokens[s])
        kf = np.asarray(k_new[t0:t + 1, h], np.float64)
        vf = np.asarray(v_new[t0:t + 1, h], np.float64)
        out[t, h * g:(h + 1) * g] = attend(np.asarray(q[t, h * g:(h + 1) * g], np.float64),
                                           np.concatenate([kc, kf]), np.concatenate([vc, vf]))
    return out


def append(k_new, v_new, seq_lens, block_tables, workspace, cache):
    """Decode-step write (kvarn_append_decode): for each sequence s with L =
    seq_lens[s] tokens, store the new token in workspace[s, :, :, L % 128]; when
    that fills the partial tile (L % 128 == 127), quantize the workspace tile into
    block block_tables[s, L // 128]. Returns (workspace, cache, new lengths); the
    inputs are not modified."""
    ws = np.array(workspace, copy=True)
    cache = np.array(cache, copy=True)
    preset = layout_of(cache.shape[-1]).name
    n_seqs = k_new.shape[0]
    for s in range(n_seqs):
        L = int(seq_lens[s])
        pos = L % B
        ws[s, :, 0, pos] = k_new[s]
        ws[s, :, 1, pos] = v_new[s]
        if pos == B - 1:
            blk = int(block_tables[s, L // B])
            recs, _, _ = quantize_tiles(ws[s, :, 0], ws[s, :, 1], preset=preset)
            cache[blk] = recs
    return ws, cache, np.asarray(seq_lens) + 1


def compression_ratio(preset: str = DEFAULT_PRESET) -> float:
    """fp16 bytes of one (K, V) tile-head over its packed record."""
    return (2 * D * B * 2) / LAYOUTS[preset].record_bytes
