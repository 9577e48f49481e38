"""Pins for the CPU oracle: each check ties the oracle to something other than
itself (a hand-written table, a closed form, an invariant the pages state, a brute
force search, or an independent restatement in plain Python loops)."""
import math
import os

import numpy as np
import pytest

import kvarn_synth as synth
from oracle import kvarn_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def _tile(seed=0):
    k, v, q = synth.single_tile(seed)
    return k.T.astype(np.float64), v.T.astype(np.float64), q.astype(np.float64)


# ------------------------------------------------------------------ Hadamard (stage 2)
def test_hadamard_matches_hand_written_order_8():
    want = np.array([[float(x) for x in r] for r in _golden_rows("hadamard_8.txt")])
    assert np.array_equal(o.sylvester_hadamard(8) * np.sqrt(8), want)


def test_hadamard_orthonormal_symmetric():
    h = o.sylvester_hadamard(128)
    assert np.abs(h @ h.T - np.eye(128)).max() < 1e-14
    assert np.array_equal(h, h.T)
    assert np.all(np.abs(np.abs(h) * np.sqrt(128) - 1) < 1e-14)


def test_hadamard_is_kron_power_of_h2():
    h2 = np.array([[1.0, 1.0], [1.0, -1.0]])
    h = np.ones((1, 1))
    for _ in range(7):
        h = np.kron(h2, h)
    assert np.array_equal(o.sylvester_hadamard(128) * np.sqrt(128), h)


def test_rotation_preserves_norms_and_scores():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((128, 40))
    q = rng.standard_normal((5, 128))
    xr = o.rotate(x)
    assert np.allclose(np.linalg.norm(xr, axis=0), np.linalg.norm(x, axis=0), rtol=1e-13)
    qr = o.rotate(q.T).T
    assert np.allclose(qr @ xr, q @ x, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ fp16 rounding
def _all_finite_halves():
    bits = np.arange(0, 0x7C00, dtype=np.uint16)          # +0 .. largest finite
    pos = bits.view(np.float16).astype(np.float64)
    return pos, bits


def _brute_rne(x):
    """Nearest binary16 by search over every finite positive half; ties -> even bits."""
    vals, bits = _all_finite_halves()
    out = np.empty_like(x)
    for n, xv in enumerate(x):
        a = abs(xv)
        j = np.searchsorted(vals, a)
        if j == 0:
            r = vals[0]
        elif j >= len(vals):
            r = vals[-1] if a <= 65520.0 else np.inf
        else:
            lo, hi = vals[j - 1], vals[j]
            if a - lo < hi - a:
                r = lo
            elif a - lo > hi - a:
                r = hi
            else:
                r = lo if bits[j - 1] % 2 == 0 else hi
        out[n] = math.copysign(r, xv)
    return out


def test_fp16_golden_encodings():
    for val, bits in _golden_rows("fp16_bits.txt"):
        got = np.array([o.fp16_rne(float(val))]).astype(np.float16).view(np.uint16)[0]
        assert got == int(bits, 16), (val, hex(got), bits)


def test_fp16_rne_matches_brute_force():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.uniform(-7, 4.5, 3000),
        # exact midpoints between neighbouring halves, both parities
        (np.arange(1000, 1100, dtype=np.uint16).view(np.float16).astype(np.float64)
         + np.arange(1001, 1101, dtype=np.uint16).view(np.float16).astype(np.float64)) / 2,
    ])
    assert np.array_equal(o.fp16_rne(x), _brute_rne(x))


# ------------------------------------------------------------------ normalisation (stage 3)
def test_first_column_pass_closed_form():
    """With no row scale yet, a rotated column's mean is x_0 / sqrt(n) and its mean
    square is |x|^2 / n (H orthonormal, first Sylvester row all ones), so its
    variance is sum_{k >= 1} x_k^2 / n, computed here from the unrotated tile."""
    kx, vx, _ = _tile(0)
    for x in (kx, vx):
        lr, lc = o.normalise(o.rotate(x), n_iters=1)
        var = (x[1:] ** 2).sum(axis=0) / 128.0
        assert np.allclose(lc, 0.5 * np.log(var + o.EPS), rtol=0, atol=1e-12)


def test_final_pass_is_a_row_pass_to_unit_variance():
    kx, vx, _ = _tile(3)
    for x in (kx, vx):
        xr = o.rotate(x)
        lr, lc = o.normalise(xr)
        z = xr * np.exp(-lr)[:, None] * np.exp(-lc)[None, :]
        assert np.abs(z.var(axis=1) - 1.0).max() < 1e-4       # rows: exactly v / (v + eps)


def test_column_scaling_equivariance_fixes_order_and_sign():
    """With eps = 0, scaling token j by beta_j shifts lc_j by log beta_j and changes
    nothing else, because the first pass is a column pass."""
    kx, _, _ = _tile(4)
    xr = o.rotate(kx)
    beta = np.exp(np.random.default_rng(5).uniform(-2, 2, 128))
    lr0, lc0 = o.normalise(xr, eps=0.0)
    lr1, lc1 = o.normalise(xr * beta[None, :], eps=0.0)
    assert np.allclose(lr1, lr0, atol=1e-10)
    assert np.allclose(lc1 - lc0, np.log(beta), atol=1e-10)


def test_normalisation_equalises_column_spread():
    """Stage 3 equalises the variance inside the tile: the spread of the column
    log-stds, measured before each column pass, never grows."""
    k, v = synth.prefill_kv(128, 8, seed=11)
    for h in range(8):
        for x in (k[:, h, :].T, v[:, h, :].T):
            trace = []
            o.normalise(o.rotate(x.astype(np.float64)), trace=trace)
            spread = [t.std() for t in trace]
            assert all(b <= a * (1 + 1e-9) for a, b in zip(spread, spread[1:])), spread


def test_many_iterations_reach_doubly_normalised_tile():
    kx, _, _ = _tile(6)
    xr = o.rotate(kx)
    lr, lc = o.normalise(xr, n_iters=60, eps=0.0)
    z = xr * np.exp(-lr)[:, None] * np.exp(-lc)[None, :]
    assert np.abs(z.var(axis=1) - 1).max() < 1e-9
    assert np.abs(z.var(axis=0) - 1).max() < 1e-3


# ------------------------------------------------------------------ RTN (stage 4)
def _brute_codes(y, s, z, bits, axis):
    levels = np.arange(2 ** bits, dtype=np.float64)
    zz, ss = np.expand_dims(z, axis), np.expand_dims(s, axis)
    grid = zz[..., None] + ss[..., None] * levels            # [..., levels]
    err = np.abs(y[..., None] - grid)
    # nearest grid point; on an exact tie floor(x + 1/2) takes the upper level
    best = err.shape[-1] - 1 - np.argmin(err[..., ::-1], axis=-1)
    return best


@pytest.mark.parametrize("kbits,vbits", sorted(set(o.PRESETS.values())))
def test_rtn_is_nearest_grid_point_and_bounded(kbits, vbits):
    kx, vx, _ = _tile(7)
    for x, kind, bits, axis in ((kx, "K", kbits, -1), (vx, "V", vbits, -2)):
        qd = o.quantize_tensor(x, kind, bits=bits)
        codes, s, z, y = qd["codes"], qd["s"], qd["z"], qd["y"]
        assert codes.max() <= 2 ** bits - 1
        assert np.array_equal(codes, _brute_codes(y, s, z, bits, axis))
        assert np.array_equal(o.fp16_rne(s), s) and np.array_equal(o.fp16_rne(z), z)
        deq = np.expand_dims(z, axis) + codes * np.expand_dims(s, axis)
        ulp = lambda a: np.spacing(np.abs(a).astype(np.float16)).astype(np.float64)
        bound = (np.expand_dims(s / 2 + ulp(z) / 2 + (2 ** bits - 1) * ulp(s) / 2, axis))
        assert (np.abs(y - deq) <= bound * (1 + 1e-12)).all()
        # the group extremes land on the end codes
        assert (np.take_along_axis(codes, np.expand_dims(y.argmin(axis), axis), axis) == 0).all()
        assert (np.take_along_axis(codes, np.expand_dims(y.argmax(axis), axis), axis) == 2 ** bits - 1).all()


def test_key_groups_are_channels_and_value_groups_are_tokens():
    """Stage 4: key scales per channel, value scales per token. Scaling one token's
    values or one channel's keys only moves that group's (s, z)."""
    kx, vx, _ = _tile(8)
    kq = o.quantize_tensor(kx, "K")
    vq = o.quantize_tensor(vx, "V")
    assert kq["s"].shape == (128,) and vq["s"].shape == (128,)
    y = kq["y"]
    assert np.allclose(kq["z"], o.fp16_rne(y.min(axis=1)))
    y = vq["y"]
    assert np.allclose(vq["z"], o.fp16_rne(y.min(axis=0)))


def test_method_beats_plain_rtn_on_outlier_keys():
    """The rotation and normalisation exist to cut quantisation error on keys with
    outlier channels (KVarN README, stages 2 and 3)."""
    k, v = synth.prefill_kv(128, 8, seed=12)
    worse = 0
    for h in range(8):
        x = k[:, h, :].T.astype(np.float64)
        qd = o.quantize_tensor(x, "K")
        xhat = o.dequant_tensor(qd["codes"], qd["r"], qd["c"], qd["s"], qd["z"], "K")
        e_kvarn = np.linalg.norm(xhat - x)
        # plain asymmetric 4-bit RTN per channel, no rotation or normalisation
        codes, s, z, _ = o.rtn(x, 4, axis=-1)
        e_plain = np.linalg.norm(z[:, None] + codes * s[:, None] - x)
        worse += e_kvarn >= e_plain
    assert worse == 0


def test_dequant_error_bounded_by_half_step():
    kx, vx, _ = _tile(9)
    for x, kind in ((kx, "K"), (vx, "V")):
        qd = o.quantize_tensor(x, kind)
        xr_hat = o.dequant_tensor(qd["codes"], qd["r"], qd["c"], qd["s"], qd["z"], kind, rotated=True)
        s = qd["s"][:, None] if kind == "K" else qd["s"][None, :]
        scale = qd["r"][:, None] * qd["c"][None, :]
        assert (np.abs(qd["xr"] - xr_hat) <= scale * s * 0.5 * (1 + 2e-3) + 1e-9).all()


def test_degenerate_tiles_stay_finite():
    zero = np.zeros((128, 128))
    const = np.full((128, 128), 3.0)
    spike = np.zeros((128, 128)); spike[5, 7] = 60000.0
    big = np.full((128, 128), 65504.0); big[::2] *= -1
    for x in (zero, const, spike, big):
        for kind in ("K", "V"):
            qd = o.quantize_tensor(x, kind)
            for name in ("r", "c", "s", "z"):
                assert np.all(np.isfinite(qd[name])), (kind, name)
            xhat = o.dequant_tensor(qd["codes"], qd["r"], qd["c"], qd["s"], qd["z"], kind)
            assert np.all(np.isfinite(xhat))
    qd = o.quantize_tensor(zero, "K")
    assert (qd["codes"] == 0).all() and (qd["z"] == 0).all()


# ------------------------------------------------------------------ packed layout
def test_layout_spots_match_hand_computed_table():
    for tensor, ch, tok, byte, shift in _golden_rows("record_layout_spots.txt"):
        f = o.k_code_position if tensor == "K" else o.v_code_position
        assert f(int(ch), int(tok)) == (int(byte), int(shift)), (tensor, ch, tok)


def test_k2_and_v4_layout_spots_match_hand_computed_table():
    """The 2-bit key layout (k2v2) and the 4-bit value layout (k4v4) at hand-computed
    spots: the position function and the packer (a single code written alone lands
    at exactly those bits of a whole record) both agree with the table."""
    zero = {n: np.zeros(128) for n in ("r", "c", "s", "z")}
    for preset, tensor, ch, tok, byte, shift in _golden_rows("record_layout_spots_k2_v4.txt"):
        ch, tok, byte, shift = int(ch), int(tok), int(byte), int(shift)
        lay = o.LAYOUTS[preset]
        if tensor == "K":
            b, sh = o.k2_position(ch, tok)
            b += lay.k_code_off
        else:
            b, sh = o.v4_position(ch, tok)
            b += lay.v_code_off
        assert (b, sh) == (byte, shift), (preset, tensor, ch, tok)
        bits = lay.k_bits if tensor == "K" else lay.v_bits
        val = (1 << bits) - 1
        kc = np.zeros((128, 128), np.uint8)
        vc = np.zeros((128, 128), np.uint8)
        (kc if tensor == "K" else vc)[ch, tok] = val
        rec = o.pack_record(dict(codes=kc, bits=lay.k_bits, **zero), dict(codes=vc, bits=lay.v_bits, **zero), preset)
        codes = rec[:lay.k_meta_off]
        assert codes[byte] == val << shift and np.count_nonzero(codes) == 1, (preset, tensor, ch, tok)


def test_pack_roundtrip_and_single_code_positions():
    rng = np.random.default_rng(13)
    kq = dict(codes=rng.integers(0, 16, (3, 128, 128)).astype(np.uint8))
    vq = dict(codes=rng.integers(0, 4, (3, 128, 128)).astype(np.uint8))
    for d in (kq, vq):
        for n in ("r", "c", "s", "z"):
            d[n] = o.fp16_rne(rng.standard_normal((3, 128)))
    rec = o.pack_record(kq, vq)
    k2, v2 = o.unpack_record(rec)
    assert np.array_equal(k2["codes"], kq["codes"]) and np.array_equal(v2["codes"], vq["codes"])
    for n in ("r", "c", "s", "z"):
        assert np.array_equal(k2[n], kq[n]) and np.array_equal(v2[n], vq[n])
    # every code value at a sample of positions lands alone at its documented bits
    for (i, t) in [(0, 0), (9, 100), (127, 1), (64, 64), (33, 17)]:
        for val in range(16):
            kc = np.zeros((128, 128), np.uint8); kc[i, t] = val
            vc = np.zeros((128, 128), np.uint8); vc[i, t] = val & 3
            zero = {n: np.zeros(128) for n in ("r", "c", "s", "z")}
            r = o.pack_record(dict(codes=kc, **zero), dict(codes=vc, **zero))
            b, sh = o.k_code_position(i, t)
            assert r[b] == val << sh and np.count_nonzero(r[:8192]) == (val != 0)
            b, sh = o.v_code_position(i, t)
            assert r[b] == (val & 3) << sh and np.count_nonzero(r[8192:12288]) == ((val & 3) != 0)


def test_compression_ratio_within_pages_claim():
    """14336 bytes per (K, V) tile-head vs 65536 fp16 bytes: 4.571x, inside the
    3-5x KV-capacity claim (KVarN README, introduction)."""
    assert o.RECORD_BYTES == 14336
    assert abs(o.compression_ratio() - 65536 / 14336) < 1e-12
    assert 3.0 <= o.compression_ratio() <= 5.0


# ------------------------------------------------------------------ attention
def _loop_attention(q, k, v):
    out = []
    for qh in q:
        scores = [sum(qh[c] * kt[c] for c in range(len(qh))) / math.sqrt(len(qh)) for kt in k]
        mx = max(scores)
        w = [math.exp(s - mx) for s in scores]
        tot = sum(w)
        out.append([sum(w[t] * v[t][c] for t in range(len(k))) / tot for c in range(len(qh))])
    return np.array(out)


def test_attend_matches_plain_loops():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((2, 128)); k = rng.standard_normal((5, 128)) * 3; v = rng.standard_normal((5, 128))
    assert np.allclose(o.attend(q, k, v), _loop_attention(q.tolist(), k.tolist(), v.tolist()), atol=1e-12)


def test_rotated_domain_attention_equals_plain():
    """q rotated by H against rotated dequantised tiles, then output un-rotated by
    H^T, equals attention over the un-rotated tiles (the rotation is orthonormal)."""
    kx, vx, q = _tile(15)
    rec, _, _ = o.quantize_tiles(kx.T, vx.T)
    kr, vr = o.dequant_record(rec, rotated=True)
    k, v = o.dequant_record(rec)
    plain = o.attend(q, k.T, v.T)
    h = o.sylvester_hadamard(128)
    rot = o.attend(q @ h.T, kr.T, vr.T) @ h
    assert np.allclose(plain, rot, atol=1e-12)


def test_split_merge_identity():
    """Attention over two token sets merged by log-sum-exp equals the whole."""
    rng = np.random.default_rng(16)
    q = rng.standard_normal((8, 128)); k = rng.standard_normal((300, 128)); v = rng.standard_normal((300, 128))
    parts = []
    for sl in (slice(0, 128), slice(128, 300)):
        s = q @ k[sl].T / np.sqrt(128)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        parts.append((m, p.sum(axis=1, keepdims=True), p @ v[sl]))
    M = np.maximum(parts[0][0], parts[1][0])
    L = sum(l * np.exp(m - M) for m, l, _ in parts)
    A = sum(a * np.exp(m - M) for m, _, a in parts)
    assert np.allclose(A / L, o.attend(q, k, v), atol=1e-12)


def test_decode_reads_cache_and_workspace():
    k, v = synth.prefill_kv(300, 2, seed=17)
    q = synth.queries(1, 4, seed=17).astype(np.float64)
    cache = np.zeros((4, 2, o.RECORD_BYTES), np.uint8)
    slots = np.concatenate([np.arange(128) + 3 * 128, np.arange(128) + 1 * 128])
    o.quantize_into_cache(k[:256], v[:256], slots, cache)
    ws = np.zeros((1, 2, 2, 128, 128), np.float16)
    ws[0, :, 0, :44] = k[256:].transpose(1, 0, 2)
    ws[0, :, 1, :44] = v[256:].transpose(1, 0, 2)
    out = o.decode(q, cache, ws, np.array([[3, 1, 0, 0]]), np.array([300]))
    for h in range(2):
        kh, vh = o.dequant_record(cache[[3, 1], h])
        kt = np.concatenate([kh[0].T, kh[1].T, k[256:, h].astype(np.float64)])
        vt = np.concatenate([vh[0].T, vh[1].T, v[256:, h].astype(np.float64)])
        assert np.allclose(out[0, 2 * h:2 * h + 2], o.attend(q[0, 2 * h:2 * h + 2], kt, vt), atol=1e-13)


def test_append_builds_same_cache_as_prefill():
    hkv = 2
    k, v = synth.prefill_kv(300, hkv, seed=18)
    bt = np.array([[2, 0, 3]], np.int32)
    ws = np.zeros((1, hkv, 2, 128, 128), np.float16)
    cache = np.zeros((4, hkv, o.RECORD_BYTES), np.uint8)
    L = np.array([0])
    for t in range(300):
        ws, cache, L = o.append(k[t:t + 1], v[t:t + 1], L, bt, ws, cache)
    assert L[0] == 300
    ref = np.zeros_like(cache)
    slots = np.concatenate([np.arange(128) + 2 * 128, np.arange(128) + 0 * 128])
    o.quantize_into_cache(k[:256], v[:256], slots, ref)
    assert np.array_equal(cache, ref)
    assert np.array_equal(ws[0, :, 0, :44], k[256:].transpose(1, 0, 2))
    assert np.array_equal(ws[0, :, 1, :44], v[256:].transpose(1, 0, 2))


# ----------------------------------------------------------------------------------
# Other bit presets (k4v4, k2v2): layouts, sizes, and what the bit width leaves alone
# ----------------------------------------------------------------------------------
def _random_quantized(rng, n, kbits, vbits):
    kq = dict(bits=kbits, codes=rng.integers(0, 2 ** kbits, (n, 128, 128)).astype(np.uint8))
    vq = dict(bits=vbits, codes=rng.integers(0, 2 ** vbits, (n, 128, 128)).astype(np.uint8))
    for d in (kq, vq):
        for name in ("r", "c", "s", "z"):
            d[name] = o.fp16_rne(rng.standard_normal((n, 128)))
    return kq, vq


@pytest.mark.parametrize("preset", sorted(o.PRESETS))
def test_preset_record_sizes_and_roundtrip(preset):
    kbits, vbits = o.PRESETS[preset]
    lay = o.LAYOUTS[preset]
    # code areas hold 128 x 128 codes at their width, then 4 (lean: 3) vectors of 128
    # fp16 scales per tensor
    n_vec = 3 if preset in o.LEAN else 4
    assert lay.record_bytes == 128 * 128 * (kbits + vbits) // 8 + 2 * n_vec * 128 * 2
    assert abs(o.compression_ratio(preset) - 65536 / lay.record_bytes) < 1e-12
    assert o.layout_of(lay.record_bytes) is lay
    kq, vq = _random_quantized(np.random.default_rng(17), 2, kbits, vbits)
    if preset in o.LEAN:                      # the folded scales are ones after unpacking
        kq["r"] = np.ones_like(kq["r"])
        vq["c"] = np.ones_like(vq["c"])
    rec = o.pack_record(kq, vq, preset)
    assert rec.shape == (2, lay.record_bytes)
    k2, v2 = o.unpack_record(rec)
    assert k2["bits"] == kbits and v2["bits"] == vbits
    assert np.array_equal(k2["codes"], kq["codes"]) and np.array_equal(v2["codes"], vq["codes"])
    for name in ("r", "c", "s", "z"):
        assert np.array_equal(k2[name], kq[name]) and np.array_equal(v2[name], vq[name])


def test_preset_compression_ratios():
    """fp16 K and V of a tile (65536 bytes) over the record: 4-bit + 2-bit codes
    (12 KiB) + 2 KiB of scales; 4 + 4 bits (16 KiB + 2 KiB); 2 + 2 bits (8 + 2 KiB)."""
    assert o.compression_ratio("k4v2") == 65536 / 14336
    assert o.compression_ratio("k4v4") == 65536 / 18432
    assert o.compression_ratio("k2v2") == 65536 / 10240 == 6.4


def _word(area, off):
    return int.from_bytes(bytes(area[off:off + 4]), "little")


def _fragment_codes_4bit(word, c, m):
    """The eight 4-bit codes a decode thread with column c of an m16n8k16 operand
    takes from word m of its 16-byte group (k-steps 2m and 2m + 1): the word shifted
    by 4h and masked to the low nibble of each byte gives k-step 2m + h, byte b
    holding row 2c + (b & 1) + 8 (b >> 1); returns {16 ks + row: code}."""
    out = {}
    for h in (0, 1):
        masked = (word >> (4 * h)) & 0x0F0F0F0F
        for b in range(4):
            out[16 * (2 * m + h) + 2 * c + (b & 1) + 8 * (b >> 1)] = (masked >> (8 * b)) & 15
    return out


def _fragment_codes_2bit(word, c, u):
    """The sixteen 2-bit codes a decode thread with column c takes from word u of
    its 8-byte group (k-steps 4u..4u + 3): the word shifted by 2r and masked to bits
    {0, 1, 4, 5} of each byte gives, in byte k, rows 2c + 8r (low nibble) and
    2c + 8r + 1 (high nibble) of k-step 4u + k; returns {16 ks + row: code}."""
    out = {}
    for r in (0, 1):
        masked = (word >> (2 * r)) & 0x33333333
        for k in range(4):
            byte = (masked >> (8 * k)) & 0xFF
            out[16 * (4 * u + k) + 2 * c + 8 * r] = byte & 3
            out[16 * (4 * u + k) + 2 * c + 8 * r + 1] = byte >> 4
    return out


def _check_fragment_reads(area, codes, offsets, bits):
    """Every (line, element) code comes back exactly once through the fragment reads
    listed in `offsets`: (line, c, word index, byte offset of the word)."""
    seen = np.zeros((128, 128), int)
    for line, c, wi, off in offsets:
        read = _fragment_codes_4bit if bits == 4 else _fragment_codes_2bit
        for e, val in read(_word(area, off), c, wi).items():
            assert val == codes[line, e], (line, e)
            seen[line, e] += 1
    assert (seen == 1).all()


def test_code_layouts_serve_the_mma_fragments():
    """Every code layout is read by tensor-core fragments: a thread with column c of
    an m16n8k16 operand needs rows 2c, 2c+1, 2c+8, 2c+9 of each 16-row k-step, and
    converts each register's pair of codes with one fp6 (4-bit) or fp4 (2-bit)
    conversion. Read that way, every (channel, token) code of a packed record comes
    back exactly once: keys by token line (elements = channels), values by channel
    line (elements = tokens)."""
    rng = np.random.default_rng(23)
    k4q, v4q = _random_quantized(rng, 1, 4, 4)
    k2q, v2q = dict(k4q, bits=2, codes=k4q["codes"] & 3), dict(v4q, bits=2, codes=v4q["codes"] & 3)
    for preset, kk, vv in (("k4v2", k4q, v2q), ("k2v2", k2q, v2q), ("k4v4", k4q, v4q)):
        lay = o.LAYOUTS[preset]
        rec = o.pack_record(kk, vv, preset)[0]
        karea = rec[lay.k_code_off:lay.k_code_off + lay.k_code_bytes]
        varea = rec[lay.v_code_off:lay.v_code_off + lay.v_code_bytes]
        if lay.k_bits == 4:   # token row of 64 bytes: group c, words m
            offs = [(t, c, m, t * 64 + c * 16 + m * 4) for t in range(128) for c in range(4) for m in range(4)]
        else:                 # token row of 32 bytes: group c, words u
            offs = [(t, c, u, t * 32 + c * 8 + u * 4) for t in range(128) for c in range(4) for u in range(2)]
        _check_fragment_reads(karea, kk["codes"][0].T, offs, lay.k_bits)
        if lay.v_bits == 4:   # channel row of 64 bytes
            offs = [(i, c, m, i * 64 + c * 16 + m * 4) for i in range(128) for c in range(4) for m in range(4)]
        else:                 # 512-byte panel of 16 channels, 16-byte cell (i & 7, c), partner half, words u
            offs = [(i, c, u, (i >> 4) * 512 + ((i & 7) * 4 + c) * 16 + ((i >> 3) & 1) * 8 + u * 4)
                    for i in range(128) for c in range(4) for u in range(2)]
        _check_fragment_reads(varea, vv["codes"][0], offs, lay.v_bits)


def test_bit_width_changes_only_the_step_and_zero():
    """Stages 2-3 do not depend on the bit width: the same tile gives the same r and
    c in every preset; only s, z and the codes change (s shrinks with more levels)."""
    k, v, _ = synth.single_tile(5)
    _, k42, v42 = o.quantize_tiles(k, v, preset="k4v2")
    _, k44, v44 = o.quantize_tiles(k, v, preset="k4v4")
    _, k22, v22 = o.quantize_tiles(k, v, preset="k2v2")
    for a, b in ((k42, k44), (k42, k22), (v42, v44), (v42, v22)):
        assert np.array_equal(a["r"], b["r"]) and np.array_equal(a["c"], b["c"])
        assert np.array_equal(a["z"], b["z"])           # z is the group minimum in every preset
    assert (v44["s"] < v42["s"]).all() and (k22["s"] > k42["s"]).all()
    assert v44["codes"].max() == 15 and k22["codes"].max() == 3


def test_lean_preset_folds_the_in_group_scale():
    """Lean metadata: keys are quantized from X_r / c (the channel's r is constant in
    a key group), values from X_r / r (the token's c is constant in a value group).
    Recomputed from the full-format quantization's y = X_r / (r c): multiplying a
    key row by r_i (a value column by c_j) and rounding gives the lean result."""
    k, v, _ = synth.single_tile(9)
    rec, kq, vq = o.quantize_tiles(k, v, preset="k4v2l")
    _, kf, vf = o.quantize_tiles(k, v, preset="k4v2")
    assert rec.shape[-1] == 13824 and abs(o.compression_ratio("k4v2l") - 65536 / 13824) < 1e-12
    assert abs(o.compression_ratio("k4v2l") - 4.74) < 0.005            # 2048 -> 1536 bytes of scales
    assert np.array_equal(kq["c"], kf["c"]) and np.array_equal(vq["r"], vf["r"])
    for lq, f, kind, axis, bits in ((kq, kf, "K", -1, 4), (vq, vf, "V", -2, 2)):
        y = f["y"] * (f["r"][:, None] if kind == "K" else f["c"][None, :])
        assert np.allclose(y, lq["y"], rtol=1e-14, atol=0)
        assert np.array_equal(lq["codes"], _brute_codes(lq["y"], lq["s"], lq["z"], bits, axis))
        assert np.array_equal(lq["z"], o.fp16_rne(np.clip(y.min(axis=axis), -o.FP16_MAX, o.FP16_MAX)))
    k2, v2 = o.unpack_record(rec)
    assert k2["stored"] == ("c", "s", "z") and v2["stored"] == ("r", "s", "z")
    assert (k2["r"] == 1).all() and (v2["c"] == 1).all()
    # both formats dequantize to nearly the same tile (each within its own step)
    kl, vl = o.dequant_record(rec)
    kfull, vfull = o.dequant_record(o.pack_record(kf, vf))
    for a, b in ((kl, kfull), (vl, vfull)):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert rel < 0.05, rel


def _fwht_rows(x):
    """Orthonormal Walsh-Hadamard transform along axis 0 by the butterfly recursion
    (independent of the oracle's dense H)."""
    x = np.array(x, np.float64)
    h = 1
    while h < x.shape[0]:
        for i in range(0, x.shape[0], 2 * h):
            a, b = x[i:i + h].copy(), x[i + h:i + 2 * h].copy()
            x[i:i + h], x[i + h:i + 2 * h] = a + b, a - b
        h *= 2
    return x / np.sqrt(x.shape[0])


def test_lean_groups_quantize_the_rotated_tile_over_the_other_scale():
    """Lean metadata against the tile itself: with X_r from an independent butterfly
    transform, a lean key group (channel i) holds X_r[i, :] / c within half a step of
    its (s_i, z_i) grid, and a lean value group (token j) holds X_r[:, j] / r likewise;
    the group extremes land on the end codes. Dropping the division, dividing by the
    wrong scale or grouping along the wrong axis breaks the bound."""
    k, v, _ = synth.single_tile(10)
    rec, kq, vq = o.quantize_tiles(k, v, preset="k4v2l")
    k2, v2 = o.unpack_record(rec)
    ulp = lambda a: np.spacing(np.abs(a).astype(np.float16)).astype(np.float64)
    for x, g, kind, bits in ((k, k2, "K", 4), (v, v2, "V", 2)):
        xr = _fwht_rows(np.asarray(x, np.float64).T)             # [channel, token]
        if kind == "K":
            y = xr / g["c"][None, :]
            axis = 1
        else:
            y = xr / g["r"][:, None]
            axis = 0
        s, z, codes = g["s"], g["z"], g["codes"]
        deq = np.expand_dims(z, axis) + codes * np.expand_dims(s, axis)
        bound = np.expand_dims(s / 2 + ulp(z) / 2 + (2 ** bits - 1) * ulp(s) / 2, axis)
        assert (np.abs(y - deq) <= bound * (1 + 1e-9) + 1e-12).all(), kind
        assert (np.take_along_axis(codes, np.expand_dims(y.argmin(axis), axis), axis) == 0).all(), kind
        assert (np.take_along_axis(codes, np.expand_dims(y.argmax(axis), axis), axis) == 2 ** bits - 1).all(), kind
        # z is the fp16 group minimum of exactly this y
        assert np.array_equal(z, o.fp16_rne(y.min(axis=axis))), kind


# ----------------------------------------------------------------------------------
# Chunked-prefill attention over the packed cache plus the fresh chunk
# ----------------------------------------------------------------------------------
def _prefill_case(seed, lens, chunks, hkv=2, g=2, preset="k4v2"):
    rng = np.random.default_rng(seed)
    n_seqs = len(lens)
    max_blocks = max(1, max(L // 128 for L in lens))
    num_blocks = n_seqs * max_blocks
    bt = synth.block_tables(n_seqs, max_blocks, num_blocks, seed)
    cache = np.zeros((num_blocks, hkv, o.LAYOUTS[preset].record_bytes), np.uint8)
    ws = np.zeros((n_seqs, hkv, 2, 128, 128), np.float16)
    for s, L in enumerate(lens):
        k, v = synth.prefill_kv(max(L, 1), hkv, seed=seed * 10 + s)
        nf = L // 128
        if nf:
            slots = np.concatenate([bt[s, b] * 128 + np.arange(128) for b in range(nf)]).astype(np.int64)
            o.quantize_into_cache(k[:nf * 128], v[:nf * 128], slots, cache)
        ws[s, :, 0, :L % 128] = k[nf * 128:L].transpose(1, 0, 2)
        ws[s, :, 1, :L % 128] = v[nf * 128:L].transpose(1, 0, 2)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    kn, vn = synth.prefill_kv(int(cu[-1]), hkv, seed=seed + 99)
    q = rng.standard_normal((int(cu[-1]), hkv * g, 128)).astype(np.float16)
    return q, kn, vn, cu, np.asarray(lens, np.int32), bt, ws, cache


def test_prefill_one_token_chunk_equals_append_then_decode():
    """A chunk of one token is a decode step: append the token, then decode over
    L0 + 1 tokens (when L0 % 128 < 127 the token stays in the workspace)."""
    q, kn, vn, cu, lens, bt, ws, cache = _prefill_case(3, [300, 0, 17], [1, 1, 1])
    got = o.prefill_attention(q, kn, vn, cu, lens, bt, ws, cache)
    ws2, cache2, lens2 = o.append(kn, vn, lens, bt, ws, cache)
    want = o.decode(q.astype(np.float64), cache2, ws2, bt, lens2)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_prefill_on_empty_cache_is_causal_attention():
    """With nothing cached the chunk attends itself with a causal mask: compare with
    softmax(Q K^T / sqrt(128) + mask) V written out on the fp16 inputs."""
    q, kn, vn, cu, lens, bt, ws, cache = _prefill_case(4, [0], [37], hkv=1, g=3)
    got = o.prefill_attention(q, kn, vn, cu, lens, bt, ws, cache)
    k = kn[:, 0].astype(np.float64)
    v = vn[:, 0].astype(np.float64)
    for h in range(3):
        qq = q[:, h].astype(np.float64)
        sc = qq @ k.T / math.sqrt(128) + np.triu(np.full((37, 37), -np.inf), 1)
        p = np.exp(sc - sc.max(axis=1, keepdims=True))
        want = (p / p.sum(axis=1, keepdims=True)) @ v
        assert np.allclose(got[:, h], want, rtol=1e-12, atol=1e-12)


def test_prefill_is_causal_and_reads_the_cache():
    """Changing chunk token p's key and value moves outputs p.. only; a chunk token
    sees every cached token (changing one cached tile moves the first output)."""
    q, kn, vn, cu, lens, bt, ws, cache = _prefill_case(5, [256 + 40], [9])
    base = o.prefill_attention(q, kn, vn, cu, lens, bt, ws, cache)
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[4] *= -1
    vn2[4] += np.float16(1)
    moved = o.prefill_attention(q, kn2, vn2, cu, lens, bt, ws, cache)
    assert np.array_equal(moved[:4], base[:4]) and not np.allclose(moved[4:], base[4:])
    cache2 = cache.copy()
    cache2[bt[0, 1]] = cache[bt[0, 0]]            # tile 1 := tile 0
    assert not np.allclose(o.prefill_attention(q, kn, vn, cu, lens, bt, ws, cache2)[0], base[0])
