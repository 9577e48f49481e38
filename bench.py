"""Benchmark of the KVarN hot path on GB300.

One step = one pass of the whole path over one batch:
  1. kvarn_quantize_tiles: prefill quantize of 16 sequences x 16384 tokens, 8
     kv-heads, head_dim 128 (1.074 GB of fp16 K+V in, 235 MB of records out);
  2. kvarn_decode_attention: GQA decode (64 q-heads over 8 kv-heads) for 64
     sequences x 16384 tokens over the packed cache (939.5 MB of records read).
The cache holds K/V drawn and quantized like the prefill batch. Metric:
(fp16 K+V bytes consumed + packed bytes read) / step time, in GB/s; per-kernel
GB/s, decode tokens/s and fractions of the measured HBM peak are reported beside
it. Every input is larger than L2 (129 MB), so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) each rank runs the same per-GPU workload on its own GPU
(weak scaling, no data-path collective); timing is the max over ranks.
--impl reference times the CPU oracle (float64 NumPy restatement of the method)
in a process pool over all of this host's cores; each of its steps is a bounded,
scaled-down copy of the GPU step with the same quantize/decode mix.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = dict(n_seqs=16, seq_len=16384, n_kv_heads=8, seed=1)
DECODE = dict(n_seqs=64, seq_len=16384, n_kv_heads=8, n_q_heads=64, seed=2)
RECORD = 14336
PRESET = "k4v2"             # `--preset`: k4v2 (the headline), k4v4, k2v2 or k4v2l
PRESET_RECORD = {"k4v2": 14336, "k4v4": 18432, "k2v2": 10240, "k4v2l": 13824}
WORKLOAD = "prefill_quantize_16x16k + decode_attn_64x16k_gqa64/8"
E2E_CHUNKS = 8             # slices of the prefill batch in the end-to-end leg
E2E_WINDOWS = 5            # end-to-end windows of K steps each; the median is reported
# Reduced shapes for profiler captures (`--case small`): still larger than L2, a
# few hundred MB on the device, and more (sequence, kv-head) units than SMs so that
# the decode runs the split kernel in the full bench's shape. Not a bench line.
SMALL = dict(prefill=dict(n_seqs=4, seq_len=16384, n_kv_heads=8, seed=1),
             decode=dict(n_seqs=20, seq_len=16384, n_kv_heads=8, n_q_heads=64, seed=2),
             workload="profiling case: prefill_quantize_4x16k + decode_attn_20x16k_gqa64/8")


def reduce_max(values, world: int):
    """Max over ranks of per-rank timings (gloo all-reduce on CPU tensors)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


# The quantize kernel's work counted as fp32 operations per fp16 element by this
# implementation's scheme (a secondary view of the roofline, derived, not measured):
# 4 iterations x 2 passes x (deviation FMA 2 + running sum 1 + square FMA 2) = 40,
# plus y, group extremes and the code (10). The Hadamard runs on tensor cores.
Q_FLOP_PER_ELEMENT = 50
# Algorithmic HBM bytes of the quantize kernel per token per kv-head: K and V fp16
# read (2 x 128 x 2) and the packed record written (14336 / 128 = 112 for k4v2).
Q_BYTES_READ_PER_TOKEN_HEAD = 512


def fp32_peak_tflops():
    # 152 SMs x 128 fp32 lanes x 2 flop per FMA x 2.07 GHz maximum SM clock
    return round(152 * 128 * 2 * 2.07e9 / 1e12, 2)


def step_config(world: int):
    """The `config` object of both arms' JSON lines (the same workload)."""
    return {"workload": WORKLOAD, "quantize": PREFILL, "decode": DECODE, "preset": f"kvarn_{PRESET}_g128",
            "n_iters": 4, "l2": "every input > L2 (129 MB); no flush", "parallelism": f"replicas x{world}"}


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- traffic from profiles
# sources a kernel's profile summary was captured from (hashed together, in order)
PROFILE_SOURCES = {
    "quantize": ["quantize.cu", "quantize_group.cuh", "kvarn_tc.cuh", "kvarn_common.cuh"],
    "decode": ["decode.cu", "decode_tile.cuh", "kvarn_common.cuh", "kvarn_frag.cuh"],
}


def source_sha16(kernel: str) -> str:
    """First 16 hex digits of the sha256 of the kernel's sources, concatenated."""
    h = hashlib.sha256()
    for name in PROFILE_SOURCES["quantize" if kernel.startswith("quantize") else "decode"]:
        with open(os.path.join(ROOT, "kv_cache_quantization_x128_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch recorded in profiles/<kernel>.md for the current source
    (null when the kernel source changed since the capture)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}.md")
    try:
        text = open(path).read()
        sha = source_sha16(kernel)
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != sha:
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------- GPU arm
def setup_gpu(torch, kv, synth, dev):
    import numpy as np
    p, d = PREFILL, DECODE
    n_tok = p["n_seqs"] * p["seq_len"]
    hkv = p["n_kv_heads"]
    k, v = synth.prefill_kv(n_tok, hkv, seed=p["seed"])
    kh = torch.from_numpy(k.view(np.int16)).view(torch.float16).pin_memory()
    vh = torch.from_numpy(v.view(np.int16)).view(torch.float16).pin_memory()
    kd, vd = kh.to(dev), vh.to(dev)
    n_blocks = d["n_seqs"] * d["seq_len"] // 128
    max_blocks = d["seq_len"] // 128
    perm = synth.block_permutation(n_blocks, d["seed"])
    cache = torch.zeros(n_blocks, hkv, RECORD, dtype=torch.uint8, device=dev)
    meta = kv.make_meta(hkv, d["n_q_heads"], n_blocks, max_blocks_per_seq=max_blocks, preset=PRESET)
    # fill the whole cache by quantizing the prefill batch into 4 disjoint block sets
    per = n_tok // 128
    slot_sets = []
    for r in range(n_blocks // per):
        blocks = perm[r * per:(r + 1) * per]
        t = np.arange(n_tok, dtype=np.int64)
        slot_sets.append(torch.from_numpy(blocks[t // 128] * 128 + t % 128).to(dev))
        kv.kvarn_quantize_tiles(kd, vd, slot_sets[-1], cache, meta)
    bt = torch.from_numpy(perm.reshape(d["n_seqs"], max_blocks).astype(np.int32)).to(dev)
    lens = torch.full((d["n_seqs"],), d["seq_len"], dtype=torch.int32, device=dev)
    q = torch.from_numpy(synth.queries(d["n_seqs"], d["n_q_heads"], d["seed"]).view(np.int16)).view(torch.float16)
    qh = q.pin_memory()
    qd = qh.to(dev)
    out = torch.empty_like(qd)
    scratch = torch.empty(kv.decode_scratch_bytes(meta, d["n_seqs"]), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert kv.kvarn_device_flags() == 0
    return dict(kd=kd, vd=vd, kh=kh, vh=vh, slots=slot_sets[0], cache=cache, meta=meta, bt=bt, lens=lens,
                qd=qd, qh=qh, out=out, out_h=torch.empty(out.shape, dtype=torch.float16).pin_memory(),
                scratch=scratch, slots_h=slot_sets[0].cpu().pin_memory(), bt_h=bt.cpu().pin_memory(),
                lens_h=lens.cpu().pin_memory())


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import kv_cache_quantization_x128_gb300 as kv
    import kvarn_synth as synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    S = setup_gpu(torch, kv, synth, dev)
    stream = torch.cuda.current_stream()

    def step(events=None):
        if events:
            events[0].record(stream)
        kv.kvarn_quantize_tiles(S["kd"], S["vd"], S["slots"], S["cache"], S["meta"])
        if events:
            events[1].record(stream)
        kv.kvarn_decode_attention(S["qd"], S["cache"], None, S["bt"], S["lens"], S["out"], S["scratch"], S["meta"])
        if events:
            events[2].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    total_ms = t0.elapsed_time(t1)
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    d_ms = [e[1].elapsed_time(e[2]) for e in evs]
    assert kv.kvarn_device_flags() == 0

    # the host link on this machine: the prefill batch's K (pinned) copied to the device alone
    h2d_ms = []
    for _ in range(4):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        S["kd"].copy_(S["kh"], non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        h2d_ms.append(c0.elapsed_time(c1))
    h2d_gbs = S["kh"].numel() * 2 / (min(h2d_ms[1:]) * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: inputs H2D, result D2H inside the
    # region. The prefill batch moves in E2E_CHUNKS slices on two copy streams; each
    # slice is quantized (one kvarn_quantize_tiles call) as soon as it is resident, so
    # copies overlap the kernels; decode follows, then its output goes back to the host.
    # A slice's copy for the next step waits only for this step's quantization of that
    # slice, and the small inputs wait for this step's decode, so the next step's
    # copies run under this step's decode.
    copy_streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    n_tok = S["kd"].shape[0]
    piece = n_tok // E2E_CHUNKS
    prev = {"quant": [None] * E2E_CHUNKS, "decode": None}

    def e2e_step():
        with torch.cuda.stream(copy_streams[0]):
            if prev["decode"] is not None:
                copy_streams[0].wait_event(prev["decode"])   # the last decode read these
            for name in ("qd", "bt", "lens"):
                S[name].copy_(S[{"qd": "qh", "bt": "bt_h", "lens": "lens_h"}[name]], non_blocking=True)
        small = torch.cuda.Event()
        small.record(copy_streams[0])
        ready = []
        for i in range(E2E_CHUNKS):
            cs = copy_streams[i % 2]
            sl = slice(i * piece, (i + 1) * piece)
            with torch.cuda.stream(cs):
                if prev["quant"][i] is not None:
                    cs.wait_event(prev["quant"][i])         # the last quantization of this slice
                S["kd"][sl].copy_(S["kh"][sl], non_blocking=True)
                S["vd"][sl].copy_(S["vh"][sl], non_blocking=True)
                S["slots"][sl].copy_(S["slots_h"][sl], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            ready.append(ev)
        for i in range(E2E_CHUNKS):
            sl = slice(i * piece, (i + 1) * piece)
            stream.wait_event(ready[i])
            kv.kvarn_quantize_tiles(S["kd"][sl], S["vd"][sl], S["slots"][sl], S["cache"], S["meta"])
            done = torch.cuda.Event()
            done.record(stream)
            prev["quant"][i] = done
        stream.wait_event(small)
        kv.kvarn_decode_attention(S["qd"], S["cache"], None, S["bt"], S["lens"], S["out"], S["scratch"], S["meta"])
        dec = torch.cuda.Event()
        dec.record(stream)
        prev["decode"] = dec
        S["out_h"].copy_(S["out"], non_blocking=True)
    for _ in range(max(1, args.warmup)):
        e2e_step()
    # A window of K steps moves ~K GB over the host link in tens of milliseconds, so
    # it is timed E2E_WINDOWS times (each bracketed like the device-timed steps) and
    # the median window is reported, every window listed beside it.
    e2e_windows = []
    for _ in range(E2E_WINDOWS):
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_windows.append(e0.elapsed_time(e1))
    h2d = sum(S[n].numel() * S[n].element_size() for n in ("kh", "vh", "slots_h", "qh", "bt_h", "lens_h"))
    d2h = S["out_h"].numel() * 2

    # the decode with its tcgen05 split kernel (KVARN_DECODE_SPLIT=tc) on the same batch,
    # outside the timed step, beside the default warp-level split kernel
    tc_ms = None
    if PRESET == "k4v2":
        saved = os.environ.get("KVARN_DECODE_SPLIT")
        os.environ["KVARN_DECODE_SPLIT"] = "tc"
        try:
            call = lambda: kv.kvarn_decode_attention(S["qd"], S["cache"], None, S["bt"], S["lens"], S["out"],
                                                     S["scratch"], S["meta"])
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            ts = []
            for _ in range(10):
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                call()
                a1.record(stream)
                torch.cuda.synchronize()
                ts.append(a0.elapsed_time(a1))
            tc_ms = float(np.median(ts))
        finally:
            if saved is None:
                del os.environ["KVARN_DECODE_SPLIT"]
            else:
                os.environ["KVARN_DECODE_SPLIT"] = saved
        assert kv.kvarn_device_flags() == 0

    # max over ranks
    total_ms, *e2e_windows = reduce_max([total_ms, *e2e_windows], world)
    e2e_ms = float(np.median(e2e_windows))

    p, d = PREFILL, DECODE
    q_bytes = p["n_seqs"] * p["seq_len"] * p["n_kv_heads"] * 128 * 2 * 2
    q_out_bytes = p["n_seqs"] * p["seq_len"] // 128 * p["n_kv_heads"] * RECORD
    d_bytes = d["n_seqs"] * (d["seq_len"] // 128) * d["n_kv_heads"] * RECORD
    step_bytes = q_bytes + d_bytes
    ms = total_ms / args.steps
    peak, peak_kind = hbm_peak()
    qm, dm = float(np.median(q_ms)), float(np.median(d_ms))
    q_avg, d_avg = float(np.mean(q_ms)), float(np.mean(d_ms))
    q_gbs, d_gbs = q_bytes / (qm * 1e-3) / 1e9, d_bytes / (dm * 1e-3) / 1e9
    # Roofline of each kernel on HBM bandwidth: algorithmic bytes per launch (quantize:
    # fp16 K+V read + records written; decode: records read) over the kernel's average
    # launch time in the timed region, against the measured copy bandwidth. The
    # quantize kernel's fp32-ALU view is reported beside it (derived peak).
    q_alg = q_bytes + q_out_bytes
    q_tflops = Q_FLOP_PER_ELEMENT * (q_bytes // 2) / (q_avg * 1e-3) / 1e12
    fp32_peak = fp32_peak_tflops()
    q_hbm = q_alg / (q_avg * 1e-3) / 1e9
    kq = dict(bound="hbm", achieved=round(q_hbm, 1), peak=peak, unit="GB/s", frac=round(q_hbm / peak, 4),
              traffic=profiled_traffic("quantize_kernel") if PRESET == "k4v2" else None,
              kernel="quantize_kernel", algorithmic_bytes_per_launch=q_alg,
              algorithmic_bytes_per_unit="512 B read + 112 B written per token per kv-head",
              launch_ms=round(q_avg, 4), peak_kind=peak_kind,
              alu_view=dict(achieved=round(q_tflops, 2), peak=fp32_peak, unit="TFLOP/s",
                            frac=round(q_tflops / fp32_peak, 4),
                            flops_per_launch=Q_FLOP_PER_ELEMENT * (q_bytes // 2),
                            peak_kind="derived: 152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz; flops counted "
                                      "by this implementation's scheme (50 per fp16 element)"))
    d_hbm = d_bytes / (d_avg * 1e-3) / 1e9
    kd = dict(bound="hbm", achieved=round(d_hbm, 1), peak=peak, unit="GB/s", frac=round(d_hbm / peak, 4),
              traffic=profiled_traffic("decode_split_kernel") if PRESET == "k4v2" else None,
              kernel="decode_split_kernel+decode_merge_kernel",
              algorithmic_bytes_per_launch=d_bytes, algorithmic_bytes_per_unit="112 B per cached token per kv-head",
              launch_ms=round(d_avg, 4), peak_kind=peak_kind)
    dominant = kq if qm >= dm else kd
    res = {
        "metric": "quantize GB/s (fp16 KV in) + paged decode-attn GB/s, % of GB300 HBM peak",
        "value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": step_config(world),
        "quantize_gbs": round(q_gbs, 1),
        "quantize_frac_hbm": round(q_gbs / peak, 4),
        "decode_gbs": round(d_gbs, 1),
        "decode_frac_hbm": round(d_gbs / peak, 4),
        "decode_tokens_per_s": round(d["n_seqs"] / (dm * 1e-3), 1),
        "quantize_ms": round(qm, 4),
        "decode_ms": round(dm, 4),
        "compression_ratio": round(2 * 128 * 128 * 2 / RECORD, 4),
        "roofline": dominant,
        "roofline_kernels": [kq, kd],
        "e2e": {"value": round(world * step_bytes / (e2e_ms / args.steps * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "windows": E2E_WINDOWS,
                "windows_gbs": [round(world * step_bytes / (w / args.steps * 1e-3) / 1e9, 2) for w in e2e_windows],
                "h2d_gbs": round(h2d_gbs, 1),
                "h2d_bound": round(world * step_bytes / (h2d / (h2d_gbs * 1e9)) / 1e9, 1),
                "h2d_note": "h2d_gbs: a pinned-host to device copy of the prefill batch's K (512 MiB) timed "
                            "alone on this box; h2d_bound: the metric if the step took only its "
                            "host-to-device copies at that rate"},
        "decode_variants": None if tc_ms is None else {
            "tcgen05_split_ms": round(tc_ms, 4),
            "tcgen05_split_gbs": round(d_bytes / (tc_ms * 1e-3) / 1e9, 1),
            "note": "the same decode with KVARN_DECODE_SPLIT=tc (tcgen05 split kernel, then the same merge), "
                    "timed after the step (median of 10, inputs > L2); decode_ms is the default "
                    "warp-level split kernel"},
        "gpu_launches": args.steps * 4,
        "e2e_pipeline": f"{E2E_CHUNKS} slices on 2 copy streams, quantize per slice; the next step's copies "
                        "overlap this step's decode",
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle arms
# The oracle (float64 NumPy, one tile at a time, as it stands) on this host's cores.
# A step of the oracle arm is a scaled-down copy of the GPU step with the same mix:
# every worker process quantizes ORACLE_TILES_PER_UNIT tile-heads of the prefill
# batch and decodes one (sequence, kv-head) pair over 16384 tokens, per unit, and
# the workload has PREFILL tile-heads / DECODE pairs = 16384 / 512 = 32 tile-heads
# per decode pair, so a unit is 1/512 of the full step's bytes.
ORACLE_TILES_PER_UNIT = 32
_ORACLE_STATE = {}


def _oracle_worker(job):
    """One worker's share of an oracle step: `units` units (see above). Runs in a
    spawned process with single-threaded BLAS; returns (seconds, tile-heads, pairs)."""
    wid, units = job
    import numpy as np
    if not _ORACLE_STATE:
        import kvarn_synth as synth
        from oracle import kvarn_oracle as o
        p, d = PREFILL, DECODE
        heads = p["n_kv_heads"]
        chunks = ORACLE_TILES_PER_UNIT // heads
        k, v = synth.prefill_kv((wid + 1) * chunks * 128, heads, seed=p["seed"])
        k, v = k[wid * chunks * 128:], v[wid * chunks * 128:]
        kt = np.stack([k[c * 128:(c + 1) * 128, h] for c in range(chunks) for h in range(heads)])
        vt = np.stack([v[c * 128:(c + 1) * 128, h] for c in range(chunks) for h in range(heads)])
        max_blocks = d["seq_len"] // 128
        recs = synth.random_records(max_blocks, d["seed"] + wid, 14336, 12288).reshape(max_blocks, 1, -1)
        g = d["n_q_heads"] // d["n_kv_heads"]
        q = synth.queries(1, d["n_q_heads"], d["seed"]).astype(np.float64)[0, :g]
        _ORACLE_STATE.update(o=o, kt=kt, vt=vt, recs=recs, q=q, max_blocks=max_blocks)
    st = _ORACLE_STATE
    t0 = time.perf_counter()
    for _ in range(units):
        st["o"].quantize_tiles(st["kt"], st["vt"])
        st["o"].decode_one(st["q"], st["recs"], None, np.arange(st["max_blocks"]), DECODE["seq_len"], 0)
    return time.perf_counter() - t0, units * ORACLE_TILES_PER_UNIT, units


class OraclePool:
    """Persistent spawned worker processes (one per host core unless told otherwise),
    BLAS limited to one thread each."""

    def __init__(self, workers: int):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        self.workers = workers
        self.ex = ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))

    def step(self, units_per_worker: int):
        """Wall seconds of one step (every worker runs its units) and the units done."""
        t0 = time.perf_counter()
        res = list(self.ex.map(_oracle_worker, [(w, units_per_worker) for w in range(self.workers)]))
        wall = time.perf_counter() - t0
        return wall, sum(r[1] for r in res), sum(r[2] for r in res)

    def close(self):
        self.ex.shutdown()


def _unit_bytes():
    """Bytes of the metric one unit stands for: its tile-heads' fp16 K+V and its
    decode pair's packed records."""
    return ORACLE_TILES_PER_UNIT * 2 * 128 * 128 * 2 + (DECODE["seq_len"] // 128) * RECORD


def _full_step_units():
    n_pairs = DECODE["n_seqs"] * DECODE["n_kv_heads"]
    n_tiles = PREFILL["n_seqs"] * PREFILL["seq_len"] // 128 * PREFILL["n_kv_heads"]
    assert n_tiles == ORACLE_TILES_PER_UNIT * n_pairs
    return n_pairs


def oracle_rate(workers: int, units_per_worker: int, steps: int, warmup: int = 1):
    """Oracle GB/s of the metric on `workers` host cores: median over `steps` timed
    steps after `warmup` untimed ones (which also start the workers and draw their
    inputs). Returns (GB/s, per-step walls, units per step)."""
    pool = OraclePool(workers)
    try:
        for _ in range(warmup):
            pool.step(1)
        walls, units = [], 0
        for _ in range(steps):
            w, _, u = pool.step(units_per_worker)
            walls.append(w)
            units = u
    finally:
        pool.close()
    walls.sort()
    med = walls[len(walls) // 2]
    return units * _unit_bytes() / med / 1e9, walls, units


def cpu_baseline(seconds: float):
    """The oracle on all host cores (process pool) and on one core, each on a bounded
    sample of the step's workload with the step's mix."""
    cores = os.cpu_count() or 1
    per = max(1, int(seconds / 2 / 0.1 / 3))       # a unit is ~0.1 s of one core; 3 timed steps
    gbs_all, walls_all, units_all = oracle_rate(cores, max(1, per // 4), steps=3)
    gbs_one, walls_one, units_one = oracle_rate(1, per, steps=3)
    full = _full_step_units()
    return {"value": round(gbs_all, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": (f"float64 NumPy oracle in a process pool of {cores} workers (one per host core, "
                       f"single-threaded BLAS); each timed step {units_all} units of {ORACLE_TILES_PER_UNIT} "
                       f"tile-heads quantized plus one (sequence, kv-head) decode over 16384 tokens, i.e. "
                       f"{units_all}/{full} of the full step with its mix; median of 3 steps"),
            "step_s": round(walls_all[len(walls_all) // 2], 3),
            "single_core": {"value": round(gbs_one, 6), "unit": "GB/s", "cores": 1,
                            "sample": f"the same oracle in one worker, {units_one} units per timed step, median of 3",
                            "step_s": round(walls_one[len(walls_one) // 2], 3)}}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    units_per_worker = 4
    pool = OraclePool(cores)
    try:
        for _ in range(args.warmup):
            pool.step(1)
        t0 = time.perf_counter()
        walls, units = [], 0
        for _ in range(args.steps):
            w, _, units = pool.step(units_per_worker)
            walls.append(w)
        wall = time.perf_counter() - t0
    finally:
        pool.close()
    step_bytes = units * _unit_bytes()
    ms = 1e3 * sum(walls) / len(walls)
    value = step_bytes / (ms * 1e-3) / 1e9
    full = _full_step_units()
    sample = (f"float64 NumPy oracle in a process pool of {cores} workers (one per host core, single-threaded "
              f"BLAS); a step is {units} units of {ORACLE_TILES_PER_UNIT} tile-heads quantized plus one "
              f"(sequence, kv-head) decode over 16384 tokens: {units}/{full} of the GPU step, same mix")
    res = {
        "impl": "reference",
        "metric": "quantize GB/s (fp16 KV in) + paged decode-attn GB/s, % of GB300 HBM peak",
        "value": round(value, 6), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(world),
        "step_fraction_of_gpu_step": f"{units}/{full}",
        "extrapolated_full_step_ms": round(ms * full / units, 1),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 1),
    }
    print(json.dumps(res), flush=True)


# `--case prefill_attn`: the chunked-prefill attention kernel alone (not the headline
# line): 16 sequences x (4096 cached tokens in 32 packed k4v2 tiles + a 512-token
# chunk), 64 q-heads over 8 kv-heads, random valid records; flops 4 x 128 per (q-head,
# attended token). L2 is flushed before every timed call.
PREFILL_ATTN = dict(n_seqs=16, cached=4096, chunk=512, n_kv_heads=8, group=8, seed=5)


def run_prefill_attn(args):
    import numpy as np
    import torch
    import kvarn_synth as synth
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    c = PREFILL_ATTN
    n_seqs, hkv, group = c["n_seqs"], c["n_kv_heads"], c["group"]
    mb = c["cached"] // 128
    nb = n_seqs * mb
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    rec = torch.from_numpy(synth.random_records(nb * hkv, c["seed"], 14336, 12288)).cuda().reshape(nb, hkv, 14336)
    bt = torch.from_numpy(synth.block_tables(n_seqs, mb, nb, c["seed"])).cuda()
    lens = torch.full((n_seqs,), c["cached"], dtype=torch.int32, device="cuda")
    cu = torch.arange(0, (n_seqs + 1) * c["chunk"], c["chunk"], dtype=torch.int32, device="cuda")
    n = n_seqs * c["chunk"]
    k, v = synth.prefill_kv(n, hkv, seed=c["seed"] + 1)
    q = f16(synth.queries(n, hkv * group, c["seed"]))
    kd, vd = f16(k), f16(v)
    out = torch.empty_like(q)
    meta = kv.make_meta(hkv, hkv * group, nb, max_blocks_per_seq=mb)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    call = lambda: kv.kvarn_prefill_attention(q, kd, vd, cu, lens, c["chunk"], bt, rec, None, out, meta)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if kv.kvarn_device_flags() != 0:
        raise SystemExit("prefill attention raised a device flag")
    ms = float(np.median(times))
    pairs = n_seqs * sum(c["cached"] + p + 1 for p in range(c["chunk"]))    # (query, key) pairs per q-head
    flops = 4.0 * 128 * hkv * group * pairs
    print(json.dumps({"metric": "chunked_prefill_attention_tflops", "value": round(flops / (ms * 1e-3) / 1e12, 1),
                      "unit": "TFLOP/s", "ms_per_call": round(ms, 4), "steps": args.steps, "warmup": args.warmup,
                      "higher_is_better": True, "dtype": "f16 operands (hi + lo pairs), f32 accumulate",
                      "data": "synthetic", "config": {"workload": "prefill_attn_16x(4096+512)_gqa64/8", "l2": "flushed"},
                      "prefill_tokens_per_s": round(n / (ms * 1e-3))}), flush=True)


# `--case serve`: the mixed serving step (not the headline line): 256 sequences with
# lengths log-uniform in [1024, 32768] and a partial last tile each (every 8th at
# L % 128 == 127, so that the append completes 33 tiles), 64 q-heads over 8 kv-heads,
# k4v2, random valid records in the cache and fp16 tokens in the workspace. One step
# appends a token to every sequence and decodes over the result; the append is
# idempotent on the same inputs, so steps repeat without a reset. L2 is flushed
# before every timed call.
SERVE = "serve_256_ragged"


def run_serve(args):
    import numpy as np
    import torch
    import kvarn_synth as synth
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    cfg = synth.WORKLOADS[SERVE]
    n_seqs, hkv, hq, seed = cfg["n_seqs"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["seed"]
    lens = synth.ragged_lengths(n_seqs, cfg["lo"], cfg["hi"], seed)
    lens[::8] = (lens[::8] // 128) * 128 + 127
    max_blocks = int(max((L + 1 + 127) // 128 for L in lens))
    num_blocks = int(((lens + 1 + 127) // 128).sum()) + 16
    perm = synth.block_permutation(num_blocks, seed)
    bt = np.full((n_seqs, max_blocks), -1, np.int32)
    pos = 0
    for i in range(n_seqs):
        nb = (lens[i] + 1 + 127) // 128
        bt[i, :nb] = perm[pos:pos + nb]
        pos += nb
    recs = synth.random_records(num_blocks * hkv, seed, RECORD, 12288).reshape(num_blocks, hkv, -1)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    k_new, v_new = synth.prefill_kv(n_seqs, hkv, seed=seed + 1)
    ws, cache = f16(synth.workspace_tokens(n_seqs, hkv, seed)), torch.from_numpy(recs).cuda()
    lens_d, bt_d = torch.from_numpy(lens).cuda(), torch.from_numpy(bt).cuda()
    q, kn, vn = f16(synth.queries(n_seqs, hq, seed)), f16(k_new), f16(v_new)
    lens_out = torch.empty((n_seqs,), dtype=torch.int32, device="cuda")
    out = torch.empty((n_seqs, hq, 128), dtype=torch.float16, device="cuda")
    meta = kv.make_meta(hkv, hq, num_blocks, max_blocks_per_seq=max_blocks)
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def append():
        kv.kvarn_append_decode(kn, vn, lens_d, lens_out, bt_d, ws, cache, meta)

    def decode():
        kv.kvarn_decode_attention(q, cache, ws, bt_d, lens_out, out, scratch, meta)

    def two():
        append()
        decode()

    def fused():
        kv.kvarn_serve_step(q, kn, vn, lens_d, lens_out, bt_d, ws, cache, out, scratch, meta)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    two()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        two()
    res = {"graph": timed(graph.replay), "two_calls": timed(two), "append": timed(append),
           "decode": timed(decode), "fused": timed(fused)}
    if kv.kvarn_device_flags() != 0:
        raise SystemExit("the serving step raised a device flag")
    peak, peak_kind = hbm_peak()
    tiles = int(sum((L + 1) // 128 for L in lens)) * hkv          # full tiles the decode reads
    decode_gbs = tiles * RECORD / (res["decode"] * 1e-3) / 1e9
    ms = res["graph"]
    print(json.dumps({"metric": "serving_step_sequences_per_s", "value": round(n_seqs / (ms * 1e-3)),
                      "unit": "sequences/s", "ms_per_step": round(ms, 4), "steps": args.steps,
                      "warmup": args.warmup, "higher_is_better": True,
                      "dtype": "f32 statistics and accumulation on fp16 inputs", "data": "synthetic",
                      "config": {"workload": f"{SERVE}: 256 sequences, lengths log-uniform 1024-32768, "
                                             "gqa64/8, one token appended and decoded",
                                 "preset": "kvarn_k4v2_g128", "l2": "flushed", "step": "append + decode "
                                 "captured in one CUDA graph"},
                      "append_us": round(res["append"] * 1e3, 1), "decode_us": round(res["decode"] * 1e3, 1),
                      "two_calls_eager_us": round(res["two_calls"] * 1e3, 1),
                      "graph_us": round(res["graph"] * 1e3, 1), "serve_step_one_launch_us": round(res["fused"] * 1e3, 1),
                      "decode_gbs": round(decode_gbs, 1), "decode_frac_hbm": round(decode_gbs / peak, 4),
                      "peak_kind": peak_kind, "decode_bytes": tiles * RECORD}), flush=True)


# `--case decode_long`: long-context decode alone (not the headline line): 4 sequences
# x 131072 tokens, 64 q-heads over 8 kv-heads, k4v2, random valid records (decode time
# does not depend on the code values), stream-K over 32 (sequence, kv-head) units.
# L2 is flushed before every timed call.
DECODE_LONG = "decode_4x128k"


def run_decode_long(args):
    import numpy as np
    import torch
    import kvarn_synth as synth
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    cfg = synth.WORKLOADS[DECODE_LONG]
    n_seqs, L, hkv, hq, seed = cfg["n_seqs"], cfg["seq_len"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["seed"]
    mb = L // 128
    nb = n_seqs * mb
    recs = torch.from_numpy(synth.random_records(nb * hkv, seed, RECORD, 12288)).cuda().reshape(nb, hkv, RECORD)
    bt = torch.from_numpy(synth.block_tables(n_seqs, mb, nb, seed)).cuda()
    lens = torch.full((n_seqs,), L, dtype=torch.int32, device="cuda")
    q = torch.from_numpy(synth.queries(n_seqs, hq, seed).view(np.int16)).view(torch.float16).cuda()
    out = torch.empty_like(q)
    meta = kv.make_meta(hkv, hq, nb, max_blocks_per_seq=mb)
    scratch = torch.empty(kv.decode_scratch_bytes(meta, n_seqs), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    call = lambda: kv.kvarn_decode_attention(q, recs, None, bt, lens, out, scratch, meta)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if kv.kvarn_device_flags() != 0:
        raise SystemExit("the decode raised a device flag")
    ms = float(np.median(times))
    peak, peak_kind = hbm_peak()
    nbytes = nb * hkv * RECORD
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"metric": "decode_attention_gbs", "value": round(gbs, 1), "unit": "GB/s",
                      "ms_per_call": round(ms, 4), "steps": args.steps, "warmup": args.warmup,
                      "higher_is_better": True, "dtype": "f32 accumulation on fp16 operands (hi + lo q', p')",
                      "data": "synthetic (random valid records)",
                      "config": {"workload": f"{DECODE_LONG}: 4 sequences x 131072 tokens, gqa64/8",
                                 "preset": "kvarn_k4v2_g128", "l2": "flushed"},
                      "frac_hbm": round(gbs / peak, 4), "peak_kind": peak_kind, "bytes": nbytes,
                      "tokens_per_s": round(n_seqs / (ms * 1e-3), 1)}), flush=True)


# `--case tile`: one tile-head, the latency case (not the headline line): quantize
# one 128 x 128 fp16 K and V tile (4 outlier key channels x20) into its record, and
# decode one query over it; each call timed alone (median), L2 flushed before it.
def run_tile(args):
    import numpy as np
    import torch
    import kvarn_synth as synth
    import kv_cache_quantization_x128_gb300 as kv
    torch.cuda.set_device(0)
    k, v, q = synth.single_tile(0)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    kd, vd, qd = f16(k[:, None, :]), f16(v[:, None, :]), f16(q[None])
    cache = torch.zeros((1, 1, RECORD), dtype=torch.uint8, device="cuda")
    slots = torch.arange(128, dtype=torch.int64, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.full((1,), 128, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)
    meta = kv.make_meta(1, 1, 1, max_blocks_per_seq=1)
    scratch = torch.empty(kv.decode_scratch_bytes(meta, 1), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    tq = timed(lambda: kv.kvarn_quantize_tiles(kd, vd, slots, cache, meta))
    td = timed(lambda: kv.kvarn_decode_attention(qd, cache, None, bt, lens, out, scratch, meta))
    if kv.kvarn_device_flags() != 0:
        raise SystemExit("the tile case raised a device flag")
    print(json.dumps({"metric": "single_tile_latency_us", "value": round((tq + td) * 1e3, 1), "unit": "us",
                      "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
                      "dtype": "f32 statistics and accumulation on fp16 inputs", "data": "synthetic",
                      "config": {"workload": "single_tile: one 128 x 128 tile-head quantized, one query decoded over it",
                                 "preset": "kvarn_k4v2_g128", "l2": "flushed"},
                      "quantize_us": round(tq * 1e3, 1), "decode_us": round(td * 1e3, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default="full", choices=["full", "small", "prefill_attn", "serve", "decode_long", "tile"],
                    help="small: reduced shapes for profiler captures (not a bench line); "
                         "prefill_attn: the chunked-prefill attention kernel alone; "
                         "serve: the 256-sequence serving step (append + decode); "
                         "decode_long: the 4 x 131072-token decode alone; "
                         "tile: one tile-head quantized and decoded (latency)")
    ap.add_argument("--preset", default="k4v2", choices=sorted(PRESET_RECORD),
                    help="bit preset of the gb300 arm; the default k4v2 is the headline workload")
    args = ap.parse_args()
    global PRESET, RECORD, PREFILL, DECODE, WORKLOAD
    PRESET, RECORD = args.preset, PRESET_RECORD[args.preset]
    if args.case == "small":
        PREFILL, DECODE, WORKLOAD = SMALL["prefill"], SMALL["decode"], SMALL["workload"]
        args.no_cpu_baseline = True
    if PRESET != "k4v2":
        WORKLOAD = f"{WORKLOAD} (preset {PRESET})"
        args.no_cpu_baseline = True
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case == "prefill_attn":
        run_prefill_attn(args)
    elif args.case == "serve":
        run_serve(args)
    elif args.case == "decode_long":
        run_decode_long(args)
    elif args.case == "tile":
        run_tile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
