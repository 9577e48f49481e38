"""Comparison rules between the CUDA library's outputs and the CPU oracle.

Tolerances (stated once, used by every parity test):
* fp16 metadata (r, c, s, z): bit-exact, except a +-1 ulp flip where the oracle's
  float64 value before rounding lies within 1e-3 ulp of the rounding midpoint.
* codes: bit-exact, except a +-1 flip where the oracle's value before rounding,
  (y - z) / s + 1/2, lies within 1e-3 of an integer; at most 1e-4 of all codes may
  flip. In a group whose metadata flipped (allowed above), codes are instead
  checked for validity against the oracle's rotated tile: each GPU code must be the
  nearest grid point of the GPU's own (s, z) within 1e-3 of a step.
* dequantised tiles: relative Frobenius error <= 1e-3 against the oracle's, over
  the elements whose codes agree (a permitted flip of one 2-bit code alone moves a
  128 x 128 tile by ~1e-2 relative; flips are bounded by the code budget instead).
* decode outputs (fp16): |gpu - oracle| <= 2e-3 + half an fp16 ulp of the oracle
  value (the output's own rounding). Two GPU paths that each hold that bound are
  compared with each other at twice the absolute part plus one ulp.
"""
from __future__ import annotations

import numpy as np

from oracle import kvarn_oracle as o

META_WINDOW_ULP = 1e-3
CODE_WINDOW = 1e-3
MAX_CODE_FLIP_FRACTION = 1e-4
DEQUANT_REL = 1e-3
DECODE_ATOL = 2e-3


def to_np_f16(t):
    return t.detach().cpu().contiguous().view(dtype=__import__("torch").int16).numpy().view(np.float16)


def _meta_ok(gpu, ref, pre):
    """Boolean mask of acceptable fp16 values (exact, or a window flip)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    pre = np.asarray(pre, np.float64)
    exact = gpu == ref
    g16 = gpu.astype(np.float16)
    r16 = ref.astype(np.float16)
    adjacent = np.nextafter(r16, g16).astype(np.float64) == gpu
    mid = (gpu + ref) / 2
    near = np.abs(pre - mid) <= META_WINDOW_ULP * np.abs(gpu - ref)
    return exact | (adjacent & near)


def compare_records(gpu_rec: np.ndarray, kq: dict, vq: dict) -> dict:
    """Check GPU records [N, record bytes] against oracle results for the same N tiles.
    Raises AssertionError with a description on the first violation; returns
    counts of the flips it accepted."""
    gk, gv = o.unpack_record(gpu_rec)
    stats = dict(meta_flips=0, code_flips=0, codes=0, groups_by_property=0)
    for g, r, kind in ((gk, kq, "K"), (gv, vq, "V")):
        n = g["codes"].shape[0]
        bits = g["bits"]
        assert r["bits"] == bits
        gaxis = -1 if kind == "K" else -2      # axis inside a group
        # r, c
        stored = g["stored"]                   # a lean record keeps one of r, c
        assert tuple(r.get("stored", stored)) == tuple(stored)
        tile_rc_flip = np.zeros(g["codes"].shape[0], bool)
        for name, pre in (("r", np.clip(r["r_pre"], o.FP16_MIN_NORMAL, o.FP16_MAX)),
                          ("c", np.clip(r["c_pre"], o.FP16_MIN_NORMAL, o.FP16_MAX))):
            if name not in stored:
                continue
            ok = _meta_ok(g[name], r[name], pre)
            assert ok.all(), f"{kind}.{name}: {np.count_nonzero(~ok)} values outside tolerance"
            stats["meta_flips"] += int(np.count_nonzero(g[name] != r[name]))
            tile_rc_flip |= (g[name] != r[name]).any(axis=-1)                 # [N]
        # s, z (only meaningful where r, c agree)
        z_pre = np.clip(r["z_pre"], -o.FP16_MAX, o.FP16_MAX)
        s_pre = np.clip(r["s_pre"], o.FP16_MIN_NORMAL, o.FP16_MAX)
        same = ~tile_rc_flip
        okz = _meta_ok(g["z"], r["z"], z_pre)
        assert okz[same].all(), f"{kind}.z outside tolerance"
        z_eq = g["z"] == r["z"]
        oks = _meta_ok(g["s"], r["s"], s_pre)      # s_pre used the oracle's rounded z
        assert oks[same[:, None] & z_eq].all(), f"{kind}.s outside tolerance"
        stats["meta_flips"] += int(np.count_nonzero((g["z"] != r["z"]) & same[:, None]))
        stats["meta_flips"] += int(np.count_nonzero((g["s"] != r["s"]) & same[:, None]))
        group_exact = same[:, None] & (g["s"] == r["s"]) & (g["z"] == r["z"])    # [N, 128]
        # codes in groups with identical metadata: exact or window flips
        gc = g["codes"].astype(np.int64)
        rc = r["codes"].astype(np.int64)
        mask = np.expand_dims(group_exact, gaxis)
        mask = np.broadcast_to(mask, gc.shape)
        diff = (gc != rc) & mask
        if diff.any():
            pre = r["code_pre"][diff] + 0.5
            lo = np.minimum(gc[diff], rc[diff]) + 1.0
            okc = (np.abs(gc[diff] - rc[diff]) == 1) & (np.abs(pre - lo) <= CODE_WINDOW)
            assert okc.all(), f"{kind} codes: {np.count_nonzero(~okc)} flips outside the window"
        stats["code_flips"] += int(np.count_nonzero(diff))
        stats["codes"] += int(gc.size)
        # groups whose metadata differs: validity of the GPU's own quantisation
        prop = ~group_exact
        if prop.any():
            stats["groups_by_property"] += int(np.count_nonzero(prop))
            y = r["xr"] / (g["r"][..., :, None] * g["c"][..., None, :])     # oracle x_r, GPU scales
            s = np.expand_dims(g["s"], gaxis)
            z = np.expand_dims(g["z"], gaxis)
            v = (y - z) / s
            best = np.clip(np.floor(v + 0.5), 0, 2 ** bits - 1)
            frac_ok = np.abs(v - (np.minimum(best, gc) + 0.5)) <= CODE_WINDOW
            okp = (gc == best) | ((np.abs(gc - best) == 1) & frac_ok)
            pm = np.broadcast_to(np.expand_dims(prop, gaxis), gc.shape)
            assert okp[pm].all(), f"{kind}: {np.count_nonzero(~okp[pm])} invalid codes in flipped groups"
    assert stats["code_flips"] <= MAX_CODE_FLIP_FRACTION * stats["codes"] + 1, stats
    # dequantised tiles (rotated domain; elements whose codes flipped are covered by
    # the code-flip budget above, a single 2-bit flip alone moves a tile by ~1e-2)
    for g, r, kind in ((gk, kq, "K"), (gv, vq, "V")):
        # the scales a record does not keep are ones on both sides (they were folded)
        rr = {n: (r[n] if n in g["stored"] else np.ones_like(r[n])) for n in ("r", "c")}
        a = o.dequant_tensor(g["codes"], g["r"], g["c"], g["s"], g["z"], kind, rotated=True)
        b = o.dequant_tensor(r["codes"], rr["r"], rr["c"], r["s"], r["z"], kind, rotated=True)
        keep = g["codes"] == r["codes"]
        num = np.sqrt(((a - b) ** 2 * keep).reshape(a.shape[0], -1).sum(axis=1))
        den = np.maximum(np.sqrt((b ** 2 * keep).reshape(b.shape[0], -1).sum(axis=1)), 1e-30)
        rel = num / den
        assert (rel <= DEQUANT_REL).all(), f"{kind} dequant rel err {rel.max():.2e}"
        stats[f"{kind}_dequant_rel_max"] = float(rel.max())
    return stats


def assert_decode_close(gpu_out: np.ndarray, ref: np.ndarray, what: str = ""):
    gpu_out = np.asarray(gpu_out, np.float64)
    ulp_half = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64) / 2
    err = np.abs(gpu_out - ref)
    tol = DECODE_ATOL + ulp_half
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {np.count_nonzero(bad)} outputs off, max err {err.max():.3e}"
    return float(err.max())


def assert_paths_close(a, b, what: str = ""):
    """Two GPU decode outputs of the same inputs computed by different kernels (the
    tensor-core split phase of kvarn_decode_attention and the warp-level one of the
    fused serving step): each is within DECODE_ATOL + half an ulp of the oracle, so
    they differ by at most 2 * DECODE_ATOL + one fp16 ulp."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert np.isfinite(a).all() and np.isfinite(b).all(), f"{what}: non-finite outputs"
    ulp = np.spacing(np.abs(b).astype(np.float16)).astype(np.float64)
    err = np.abs(a - b)
    bad = ~(err <= 2 * DECODE_ATOL + ulp)
    assert not bad.any(), f"{what}: {np.count_nonzero(bad)} outputs apart, max {err.max():.3e}"
    return float(err.max())
