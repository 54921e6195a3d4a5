"""Benchmark of the W4A16 INT4 MoE layer (align + gate/up + SiLU + down + combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T]
                    [--impl ours|reference] [--flags F] [--weights plain|packed]

Prints ONE JSON line.  A step is one pass of the whole hot path (moe_align +
the indexed layer) over one batch of synthetic inputs already resident in HBM,
replayed from a CUDA graph; the weights (1.19 GB for the EP8 workloads) are
far larger than L2, so every step streams them from HBM.  By default they are
packed once with chord_w4a16_prepack before anything is timed, as a server
does when it loads them (--weights plain keeps the [E, N, K/8] layout).  `value` is
microseconds per layer call (lower is better).

--impl reference times the CPU oracle (test infrastructure, plain C) on the
host cores on the same workload: the reference arm of this benchmark.
Under torchrun each rank runs an independent replica (the layer has no
cross-GPU step); rank 0 prints the max over ranks.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from w4a16_int4_mixture_gb300 import synth  # noqa: E402

METRIC = "MoE layer us/call; decode HBM TB/s and prefill BF16 TFLOPS as % of roofline"
UNIT = "us/call"
KERNEL_SOURCES = ["gemm_kernel.cuh", "gemm_instances.cuh", "device.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", choices=synth.WORKLOADS, default="ep8-decode")
    ap.add_argument("--weights", choices=("plain", "packed"), default="packed",
                    help="plain [E,N,K/8] codes + scales, or chord_w4a16_prepack packs "
                         "(packed once before timing, like loading the weights)")
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the headline configuration, and its align only as part of "
                         "the step (default: also every other configuration, under the "
                         "`configs` key, and each indexed configuration's align alone)")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def workload_bytes_flops(inp):
    """Algorithmic work of one layer call: each touched expert's codes + scales
    once, each distinct routed token read once, each token output written once;
    FLOPs 2 * pairs * (2I*H + H*I)."""
    from w4a16_int4_mixture_gb300 import synth
    s = inp.shape
    lid = synth.local_ids(inp)
    touched = np.unique(lid[lid >= 0])
    pairs = int(np.count_nonzero(lid >= 0))
    tokens = int(np.count_nonzero((lid >= 0).any(axis=1)))
    # scale bytes per group of 32: bf16 (INT4) or one E8M0 byte (MXFP4; its pack
    # holds them widened to bf16, but the format's own traffic is counted)
    sb = 1 if getattr(inp.w13_s, "dtype", None) == np.uint8 else 2
    w13 = 2 * s.I * s.H // 2 + 2 * s.I * (s.H // 32) * sb
    w2 = s.H * s.I // 2 + s.H * (s.I // 32) * sb
    n = len(touched)
    gate_up = {"weights": n * w13, "x": tokens * s.H * 2, "h": pairs * s.I * 2,
               "flops": 2 * pairs * 2 * s.I * s.H}
    down = {"weights": n * w2, "h": pairs * s.I * 2, "flops": 2 * pairs * s.H * s.I}
    layer = {"bytes": n * (w13 + w2) + tokens * s.H * 2 + s.T * s.H * 2,
             "flops": gate_up["flops"] + down["flops"]}
    return {"touched": n, "pairs": pairs, "tokens": tokens, "gate_up": gate_up, "down": down,
            "layer": layer}


def kernel_source_hash():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "w4a16_int4_mixture_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, when it was taken on
    the current kernel source (its hash) and this workload; else None."""
    pat = re.compile(r"traffic_per_launch\s+kernel=(\S+)\s+workload=(\S+)\s+source=(\S+)\s+"
                     r"bytes=(\d+)")
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        with open(path) as f:
            for m in pat.finditer(f.read()):
                if m.group(1) == kernel and m.group(2) == workload and m.group(3) == src_hash:
                    return int(m.group(4))
    return None


class Clocks:
    """SM clock, power and clock-event reasons sampled every millisecond during
    the timed region, read through NVML (libnvidia-ml via ctypes); nvidia-smi
    at its fastest period when NVML cannot be loaded."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, uuid: str | None = None):
        self.index = index
        self.uuid = uuid
        self.samples = []  # (sm_mhz, reasons_mask, power_w)
        self.max_mhz = None
        self.source = None
        self._stop = None
        self._thread = None
        self._smi = None

    def _nvml_handle(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            for u in (self.uuid, "GPU-" + self.uuid):
                if lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                    ok = True
                    break
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return lib, h

    def __enter__(self):
        import ctypes
        import threading
        try:
            lib, h = self._nvml_handle()
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self._stop = threading.Event()
            started = threading.Event()

            def run():
                mhz, rs, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
                while True:
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                        r = rs.value if reasons_fn(h, ctypes.byref(rs)) == 0 else 0
                        p = mw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else None
                        self.samples.append((float(mhz.value), r, p))
                    started.set()
                    if self._stop.wait(0.001):
                        break

            self._thread = threading.Thread(target=run, daemon=True)
            self._thread.start()
            started.wait(2.0)
            self.source = "nvml, 1 ms"
        except Exception:
            self._thread = None
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.SMI_Q}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi, 20 ms"
            except Exception:
                self._smi = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(5.0)
        if self._smi is not None:
            self._smi.terminate()
            try:
                out, _ = self._smi.communicate(timeout=5)
            except Exception:
                self._smi.kill()
                out = ""
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
                    "sw_power_cap": 0x4}
            for ln in out.splitlines():
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 9:
                    continue
                try:
                    mhz = float(f[1])
                    self.max_mhz = float(f[2])
                    pw = float(f[3])
                except ValueError:
                    continue
                mask = 0
                for nm, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        mask |= bits[nm]
                self.samples.append((mhz, mask, pw))
        return False

    def summary(self):
        sm = [m for m, _, _ in self.samples]
        reasons = set()
        for _, r, _ in self.samples:
            for bit, nm in self.REASONS.items():
                if r & bit:
                    reasons.add(nm)
        pw = [p for _, _, p in self.samples if p is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None, "sampler": self.source}


def device_inputs(inp, torch, dev, weights=True):
    def t(a, bf16=False):
        a = np.ascontiguousarray(a)
        x = torch.from_numpy(a.view(np.int16) if bf16 else a)
        return (x.view(torch.bfloat16) if bf16 else x).to(dev)
    d = {"x": t(inp.x, True), "ids": t(inp.topk_ids), "tw": t(inp.topk_weights)}
    if weights:
        d.update({"w13_q": t(inp.w13_q), "w13_s": t(inp.w13_s, True), "w2_q": t(inp.w2_q),
                  "w2_s": t(inp.w2_s, True)})
    d["emap"] = None if inp.expert_map is None else t(inp.expert_map)
    return d


L2_BYTES = 129 * 10**6          # GB300 L2
L2_FLUSH_BYTES = 256 * 2**20    # written between replays when a step could stay in L2
SPREAD_REPLAYS = 50             # single replays behind each median / p10 / p90 (after the timed region)


def needs_l2_flush(step_bytes: int) -> bool:
    """A step that moves less than twice the L2 could be served from it on
    the next replay."""
    return step_bytes < 2 * L2_BYTES


def replay_spread_us(ms_list):
    """Median, 10th and 90th percentile of single-replay times (ms in, us out)."""
    v = sorted(float(x) * 1e3 for x in ms_list)
    if not v:
        return None

    def pct(q):
        i = min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))
        return round(v[i], 2)
    return {"median": round(statistics.median(v), 2), "p10": pct(0.1), "p90": pct(0.9),
            "replays": len(v)}


def kernels_per_call(pairs: int, e_local: int) -> int:
    """Kernels of one align + indexed layer call: the align runs as one CTA up to
    4096 pairs and 512 local experts (aux_kernels.cu), else as three kernels;
    the layer is prep, gate_up, down and the combine / finalize."""
    align = 1 if (pairs <= 4096 and e_local <= 512) else 3
    return align + 4


def max_over_ranks(local_ms: float, world: int, device) -> float:
    """The slowest rank's time (every rank gets it); the plain value for one rank."""
    if world <= 1:
        return local_ms
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_call(max_ms: float, world: int) -> float:
    """Whole-job µs per layer call: N replicas each complete one call per step,
    so the job completes N calls in the slowest rank's step time."""
    return round(max_ms * 1e3 / max(world, 1), 2)


def layer_weights(chord, d, packed: bool):
    """The four weight arguments of the layer calls: plain device tensors, or
    packed once with chord_w4a16_prepack (before anything is timed, like
    loading the weights)."""
    import torch
    w = (d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"])
    if packed:
        w = (chord.prepack_weights(*w), None, None, None)
        torch.cuda.synchronize()
    return w


def capture(step, stream):
    """Three eager calls, then one CUDA graph of `step` on `stream`."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    return graph


def time_graph(graph, stream, steps, warmup, flush, barrier=None):
    """Mean ms of one replay over `steps` timed replays after `warmup` untimed
    ones: CUDA events around the whole run, or (flush given: a step that could
    stay in L2) around each replay with the flush buffer written in between,
    outside the events."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        if flush is None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
        else:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(steps)]
            for a, b in pairs:
                flush.zero_()
                a.record(stream)
                graph.replay()
                b.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    if flush is None:
        return e0.elapsed_time(e1) / steps
    return sum(a.elapsed_time(b) for a, b in pairs) / steps


def replay_spread(graph, stream, steps, flush):
    """Single-replay times (after the timed region; not part of `value`)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            if flush is not None:
                flush.zero_()
            ev[2 * i].record(stream)
            graph.replay()
            ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    return replay_spread_us([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)])


def stage_times(chord, step, stream, calls):
    """Per-stage ms (prepare, gate_up, down, combine) of eager calls, from the
    library's stage events on the same stream."""
    import torch
    chord.stage_timing_enable(True)
    with torch.cuda.stream(stream):
        for _ in range(calls):
            step()
    stage_ms, n = chord.stage_timing_read()
    chord.stage_timing_enable(False)
    return [v / max(n, 1) for v in stage_ms]


ALIGN_REPS = 20


def align_time_ms(align_call, stream, steps=20):
    """Per-call ms of the align alone: a CUDA graph of ALIGN_REPS back-to-back
    calls (after three eager ones), replayed `steps` times; the median replay
    over ALIGN_REPS.  (The layer's own stages come from the library's stage
    events; the align is a separate call, so it is timed this way.)"""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            align_call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(ALIGN_REPS):
                align_call()
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            ev[2 * i].record(stream)
            g.replay()
            ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    return float(np.median([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)])) / ALIGN_REPS


STAGES_HOW = ("align: a CUDA graph of 20 back-to-back align calls, replayed, per call; prepare, "
              "gate_up, down, combine: the library's per-stage CUDA events over eager layer calls")


def stages_record(stage, align_ms=None):
    rec = {} if align_ms is None else {"align": round(align_ms, 5)}
    rec.update({"prepare": round(stage[0], 5), "gate_up": round(stage[1], 5),
                "down": round(stage[2], 5), "combine": round(stage[3], 5)})
    return rec


def roofline(work, stage, layer_ms, decode, label):
    """The dominant kernel's roofline (the gate/up GEMM: HBM-bound for decode
    shapes, tensor-bound for prefill) and the layer's achieved fractions."""
    hbm, tfl, tfl_sus, src = peaks()
    gu = work["gate_up"]
    gu_bytes = gu["weights"] + gu["x"] + gu["h"]
    gu_s = stage[1] / 1e3
    if decode:
        ach = gu_bytes / gu_s / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4)}
    else:
        ach = gu["flops"] / gu_s / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": tfl, "unit": "TFLOP/s",
                "frac": round(ach / tfl, 4)}
    roof["kernel"] = f"w4a16_gemm_kernel (gate_up, fused SiLU*up; {label})"
    roof["peak_source"] = (f"{src} (MEASURED_PEAKS.json burst; 'of measured')" if src == "measured"
                           else "fallback (6.8 TB/s, 1.9 PFLOP/s)")
    roof["algorithmic_bytes_per_launch"] = int(gu_bytes)
    roof["algorithmic_flops_per_launch"] = int(gu["flops"])
    roof["launch_ms"] = round(stage[1], 5)
    layer_s = layer_ms / 1e3
    layer_tbs = work["layer"]["bytes"] / layer_s / 1e12
    layer_tflops = work["layer"]["flops"] / layer_s / 1e12
    layer = {"hbm_tbs": round(layer_tbs, 3), "hbm_frac": round(layer_tbs * 1e3 / hbm, 4),
             "tflops": round(layer_tflops, 2), "tensor_frac": round(layer_tflops / tfl, 4),
             "tensor_frac_sustained": round(layer_tflops / tfl_sus, 4),
             "algorithmic_bytes": int(work["layer"]["bytes"]),
             "algorithmic_flops": int(work["layer"]["flops"])}
    return roof, layer


def is_decode(work):
    """HBM-bound (weight streaming) below 80 routed rows per touched expert."""
    return work["pairs"] / max(work["touched"], 1) < 80


class IndexedCase:
    """Device state of one align + indexed-layer step: routing buffers and
    workspaces sized for `cap_T` tokens (over-allocated, like a server that
    serves every batch size from one set), reused for any T <= cap_T."""

    def __init__(self, chord, torch, dev, s, cap_T, flags):
        self.chord, self.s, self.flags = chord, s, flags
        self.bm = chord.select_block_m(cap_T, s.k, s.E_global, s.E_local, s.H, s.I)
        self.cap = chord.moe_align_capacity(cap_T, s.k, s.E_local, self.bm)
        self.si = torch.empty(self.cap, dtype=torch.int32, device=dev)
        self.ei = torch.empty(self.cap // self.bm, dtype=torch.int32, device=dev)
        self.ntp = torch.empty(1, dtype=torch.int32, device=dev)
        self.out = torch.empty((cap_T, s.H), dtype=torch.bfloat16, device=dev)
        self.ws_a = torch.empty(chord.ops.align_workspace_size(cap_T, s.k, s.E_local),
                                dtype=torch.uint8, device=dev)
        self.ws_l = torch.empty(chord.moe_workspace_size(cap_T, s.k, s.E_global, s.E_local, s.H,
                                                         s.I, self.bm, self.cap, flags),
                                dtype=torch.uint8, device=dev)

    def align_fn(self, d, T):
        chord, s = self.chord, self.s
        ids = d["ids"][:T]

        def call():
            chord.moe_align(ids, s.E_global, s.E_local, self.bm, expert_map=d["emap"],
                            capacity=self.cap, workspace=self.ws_a, out=(self.si, self.ei, self.ntp))
        return call

    def step_fn(self, d, w, T):
        chord, s = self.chord, self.s
        x, ids, tw, out = d["x"][:T], d["ids"][:T], d["tw"][:T], self.out[:T]

        def step():
            chord.moe_align(ids, s.E_global, s.E_local, self.bm, expert_map=d["emap"],
                            capacity=self.cap, workspace=self.ws_a, out=(self.si, self.ei, self.ntp))
            chord.w4a16_moe_indexed(x, *w, tw, self.si, self.ei, self.ntp, self.bm, s.E_global,
                                    out=out, workspace=self.ws_l, flags=self.flags)
        return step


def config_record(chord, torch, dev, stream, step, graph, work, steps, warmup, label, extra,
                  dev_index, uuid, align_call=None):
    """Timing record of one extra configuration (same rules as the headline)."""
    flush = None
    if needs_l2_flush(work["layer"]["bytes"]):
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    with Clocks(dev_index, uuid) as clk:
        ms = time_graph(graph, stream, steps, warmup, flush)
    replay_us = replay_spread(graph, stream, max(steps, SPREAD_REPLAYS), flush)
    stage = stage_times(chord, step, stream, max(3, min(steps, 10)))
    align_ms = align_time_ms(align_call, stream) if align_call is not None else None
    roof, layer = roofline(work, stage, ms, is_decode(work), label)
    rec = {"value": round(ms * 1e3, 2), "unit": UNIT, "ms_per_step": round(ms, 5),
           "steps": steps, "warmup": warmup,
           "timing": ("CUDA events over K CUDA-graph replays" if flush is None else
                      "CUDA events around each of K CUDA-graph replays, L2 flushed between them "
                      "outside the events"),
           "replay_us": replay_us,
           "routed_pairs": work["pairs"], "touched_experts": work["touched"],
           "roofline": roof, "layer": layer,
           "stages_ms": stages_record(stage, align_ms), "stages_how": STAGES_HOW,
           "clocks": clk.summary()}
    rec.update(extra)
    return rec


def run_configs(args, chord, torch, dev, stream, ep8_inp, ep8_dev, dev_index, uuid):
    """Every other configuration of the benchmark, each timed like the headline
    one: the tiny case, EP8 decode with MXFP4 weights, EP8 prefill (the EP8
    weights), TP8 at T = 1, 16, 128 and 2048 from one weight set and one set of
    routing buffers and workspaces sized for 2048 tokens, and the skewed
    decode on the indexed and the masked layouts (the EP8 weights)."""
    from w4a16_int4_mixture_gb300 import synth
    steps = max(5, min(args.steps, 50))
    warmup = max(3, args.warmup)
    packed = args.weights == "packed"
    recs = {}

    def indexed(s, inp, d, w, label, cap_T=None, T=None):
        case = IndexedCase(chord, torch, dev, s, cap_T or s.T, args.flags)
        T = s.T if T is None else T
        step = case.step_fn(d, w, T)
        graph = capture(step, stream)
        work = workload_bytes_flops(inp)
        extra = {"T": T, "k": s.k, "E_global": s.E_global, "E_local": s.E_local, "H": s.H,
                 "I": s.I, "weights": label,
                 "schedule": chord.describe_schedule(T, s.k, s.E_global, s.E_local, s.H, s.I,
                                                     args.flags),
                 "gpu_launches_per_step": kernels_per_call(T * s.k, s.E_local)}
        if cap_T:
            extra["buffers"] = f"routing buffers and workspaces sized for {cap_T} tokens"
        return config_record(chord, torch, dev, stream, step, graph, work, steps, warmup, label,
                             extra, dev_index, uuid, align_call=case.align_fn(d, T))

    # tiny: K = 128 of its down GEMM is below the prepack's 256-deep blocks
    s = synth.workload("tiny")
    inp = synth.make_inputs(s)
    d = device_inputs(inp, torch, dev)
    recs[s.name] = indexed(s, inp, d, layer_weights(chord, d, False),
                           "plain weights (the prepack needs K % 256 == 0)")

    # EP8 decode with MXFP4 weights: the EP8 codes read as E2M1 numbers, one
    # E8M0 scale byte per 32 inputs (synth.mx_scales), packed once
    s = synth.workload("ep8-decode")
    rng = np.random.default_rng(101)
    mx13 = synth.mx_scales(rng, s.E_local, 2 * s.I, s.H)
    mx2 = synth.mx_scales(rng, s.E_local, s.H, s.I)
    w_mx = (chord.prepack_weights(ep8_dev["w13_q"], torch.from_numpy(mx13).to(dev),
                                  ep8_dev["w2_q"], torch.from_numpy(mx2).to(dev)),
            None, None, None)
    torch.cuda.synchronize()
    inp = synth.MoEInputs(s, ep8_inp.x, ep8_inp.w13_q, mx13, ep8_inp.w2_q, mx2,
                          ep8_inp.topk_ids, ep8_inp.topk_weights, ep8_inp.expert_map)
    recs[s.name + "-mxfp4"] = indexed(s, inp, ep8_dev, w_mx, "MXFP4 packs (chord_mxfp4_prepack)")
    del w_mx

    # EP8 prefill and skewed decode on the EP8 weights
    w_ep8 = layer_weights(chord, ep8_dev, packed)
    label = f"{args.weights} weights"
    for wl in ("ep8-prefill", "skewed"):
        s = synth.workload(wl)
        inp = synth.make_inputs(s, weights=False)
        inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s = (ep8_inp.w13_q, ep8_inp.w13_s, ep8_inp.w2_q,
                                                    ep8_inp.w2_s)
        d = device_inputs(inp, torch, dev, weights=False)
        recs[s.name + ("-indexed" if wl == "skewed" else "")] = indexed(s, inp, d, w_ep8, label)
        if wl == "skewed":
            recs[s.name + "-masked"] = masked(args, chord, torch, dev, stream, s, inp, w_ep8,
                                              label, steps, warmup, dev_index, uuid)
    del w_ep8

    # TP8: one weight set, buffers for 2048 tokens, T = 1, 16, 128, 2048
    s = synth.workload("tp8", T=2048)
    inp = synth.make_inputs(s)
    d = device_inputs(inp, torch, dev)
    w = layer_weights(chord, d, packed)
    for k in ("w13_q", "w13_s", "w2_q", "w2_s"):
        d[k] = None
    for T in (1, 16, 128, 2048):
        sT = synth.workload("tp8", T=T)
        sub = synth.MoEInputs(sT, inp.x[:T], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                              inp.topk_ids[:T], inp.topk_weights[:T], inp.expert_map)
        recs[sT.name] = indexed(sT, sub, d, w, label, cap_T=2048, T=T)
    return recs


def masked(args, chord, torch, dev, stream, s, inp, w, label, steps, warmup, dev_index, uuid):
    """The grouped masked layout of a draw ([E, max_m, H], max_m = T): the
    layer with the token combine, timed like the indexed step."""
    from w4a16_int4_mixture_gb300 import synth
    a3, mm, r2p = synth.grouped_masked_layout(inp)

    def t(a, bf16=False):
        a = np.ascontiguousarray(a)
        x = torch.from_numpy(a.view(np.int16) if bf16 else a)
        return (x.view(torch.bfloat16) if bf16 else x).to(dev)
    da3, dmm, dr2p, dtw = t(a3, True), t(mm), t(r2p), t(inp.topk_weights)
    exp_m = int(np.ceil(mm.sum() / s.E_local))
    M = a3.shape[0] * a3.shape[1]
    out_rows = torch.empty((M, s.H), dtype=torch.bfloat16, device=dev)
    out_tok = torch.empty((s.T, s.H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(chord.ops.grouped_workspace_size(1, M, s.H, s.I, s.E_local, s.T, s.k, True,
                                                      exp_m), dtype=torch.uint8, device=dev)

    def step():
        chord.w4a16_moe_grouped("masked", da3, *w, masked_m=dmm, expected_m=exp_m,
                                row_to_pair=dr2p, topk_weights=dtw, out_rows=out_rows,
                                out_tokens=out_tok, workspace=ws, flags=args.flags)
    graph = capture(step, stream)
    work = workload_bytes_flops(inp)
    rows = int(mm.sum())
    # the masked call reads each valid row of a3 and writes its bf16 row output
    # as well as the token rows
    work["layer"]["bytes"] += rows * s.H * 2 * 2 - work["tokens"] * s.H * 2
    work["gate_up"]["x"] = rows * s.H * 2
    extra = {"T": s.T, "k": s.k, "E_local": s.E_local, "H": s.H, "I": s.I, "weights": label,
             "layout": f"grouped masked [{s.E_local}, {a3.shape[1]}, {s.H}], expected_m={exp_m}",
             "algorithmic_bytes_note": "valid rows of a3 read once, their bf16 row outputs and "
                                       "the token outputs written once, plus the touched "
                                       "experts' weights",
             "gpu_launches_per_step": 4}
    return config_record(chord, torch, dev, stream, step, graph, work, steps, warmup, label,
                         extra, dev_index, uuid)


def e2e_pipelined(chord, torch, dev, inp, d, w, s, bm, args, graphed=True):
    """ms per step of the end-to-end loop (host inputs -> chord.w4a16_moe ->
    host output), and the bytes copied in and out per step.  graphed: the
    layer call is replayed from a CUDA graph captured once per input buffer,
    as a serving engine replays its decode step; else it is called eagerly."""
    hx = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    hids = torch.from_numpy(inp.topk_ids).pin_memory()
    htw = torch.from_numpy(inp.topk_weights).pin_memory()
    hout = [torch.empty((s.T, s.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx = [torch.empty_like(d["x"]) for _ in range(2)]
    dids = [torch.empty_like(d["ids"]) for _ in range(2)]
    dtw = [torch.empty_like(d["tw"]) for _ in range(2)]
    dout = [torch.empty((s.T, s.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_in, s_comp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def layer(b):
        return lambda: chord.w4a16_moe(dx[b], dids[b], dtw[b], *w, s.E_global, expert_map=d["emap"],
                                       block_m=bm, flags=args.flags, out=dout[b])
    graphs = None
    if graphed:
        for b in range(2):  # (captured on the real inputs)
            dx[b].copy_(hx)
            dids[b].copy_(hids)
            dtw[b].copy_(htw)
        graphs = [capture(layer(b), s_comp) for b in range(2)]
    torch.cuda.synchronize()
    n = args.warmup + args.steps
    for i in range(n):
        b = i % 2
        if i == args.warmup:
            # exactly K steps in the timed region: the warm-up steps have ended
            torch.cuda.synchronize()
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[b])  # the layer of step i-2 has read buffer b
            if i == args.warmup:
                e0.record(s_in)
            dx[b].copy_(hx, non_blocking=True)
            dids[b].copy_(hids, non_blocking=True)
            dtw[b].copy_(htw, non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            if i >= 2:
                s_comp.wait_event(out_done[b])  # step i-2's output has been copied out
            if graphs is not None:
                graphs[b].replay()
            else:
                layer(b)()
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            hout[b].copy_(dout[b], non_blocking=True)
            out_done[b].record(s_out)
            if i == n - 1:
                e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    h2d = hx.numel() * 2 + hids.numel() * 4 + htw.numel() * 4
    d2h = hout[0].numel() * 2
    return e2e_ms, h2d, d2h


def run_ours(args, rank, world, dev_index):
    import torch
    import w4a16_int4_mixture_gb300 as chord
    from w4a16_int4_mixture_gb300 import synth

    chord.build()
    torch.cuda.set_device(dev_index)
    dev = torch.device("cuda", dev_index)
    s = synth.workload(args.workload, T=args.T)
    inp = synth.make_inputs(s)
    work = workload_bytes_flops(inp)
    d = device_inputs(inp, torch, dev)
    packed = args.weights == "packed"
    w = layer_weights(chord, d, packed)
    case = IndexedCase(chord, torch, dev, s, s.T, args.flags)
    bm, cap = case.bm, case.cap
    step = case.step_fn(d, w, s.T)
    stream = torch.cuda.Stream(device=dev)
    graph = capture(step, stream)
    launches_per_step = kernels_per_call(s.T * s.k, s.E_local)
    if s.T * s.k == 0:
        launches_per_step = 1

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    try:
        uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
    except Exception:
        uuid = None
    # A step whose bytes could stay in L2 between replays is timed replay by
    # replay, with a write of twice the L2 between them (outside the events).
    flush = None
    if needs_l2_flush(work["layer"]["bytes"]):
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    with Clocks(dev_index, uuid) as clk:
        local_ms = time_graph(graph, stream, args.steps, args.warmup, flush, barrier)
    ms = max_over_ranks(local_ms, world, dev)
    replay_us = replay_spread(graph, stream, max(args.steps, SPREAD_REPLAYS), flush)
    stage = stage_times(chord, step, stream, args.steps)
    # (the align-only graph adds ~460 align launches: left out of the short
    # single-configuration runs that the ncu launch lists capture)
    align_ms = None if args.no_configs else align_time_ms(case.align_fn(d, s.T), stream)

    # end to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory and its output back; the copies
    # run on their own streams, double-buffered, so step i's output copy and
    # step i+1's input copies overlap the layer of the step between them (as
    # a server pipelines them).  The events bracket the first timed input copy
    # and the last output copy.
    e2e_ms, h2d, d2h = e2e_pipelined(chord, torch, dev, inp, d, w, s, bm, args)
    e2e_eager_ms, _, _ = e2e_pipelined(chord, torch, dev, inp, d, w, s, bm, args, graphed=False)
    src_hash = kernel_source_hash()
    roof, layer = roofline(work, stage, ms, is_decode(work), f"{args.weights} weights")
    roof["traffic"] = ncu_traffic("gate_up" + (".packed" if packed else ""), s.name, src_hash)
    res = {
        "metric": METRIC, "value": whole_job_us_per_call(ms, world), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random INT4 codes / bf16 scales / bf16 activations; "
                "routing per workload recipe)",
        "config": {"workload": s.name, "T": s.T, "k": s.k, "E_global": s.E_global,
                   "E_local": s.E_local, "H": s.H, "I": s.I, "block_m": bm,
                   "routed_pairs": work["pairs"], "touched_experts": work["touched"],
                   "schedule": chord.describe_schedule(s.T, s.k, s.E_global, s.E_local, s.H, s.I,
                                                       args.flags),
                   "l2": ("inputs larger than L2 (weights of the touched experts "
                          f"{work['layer']['bytes'] / 1e9:.2f} GB per step)") if flush is None else
                         (f"L2 flushed between replays ({L2_FLUSH_BYTES >> 20} MB written, outside "
                          f"the timed events; the step touches {work['layer']['bytes'] / 1e6:.0f} MB)"),
                   "weights": args.weights,
                   "timing": ("CUDA events over K CUDA-graph replays on the launching stream"
                              if flush is None else
                              "CUDA events around each of K CUDA-graph replays on the launching "
                              "stream, summed"),
                   "parallelism": f"replicas x{world}",
                   "value": "whole job: the slowest rank's step time / the N layer calls the "
                            "N replicas complete per step"},
        "layer": layer,
        "replay_us": replay_us,
        "stages_ms": stages_record(stage, align_ms), "stages_how": STAGES_HOW,
        "roofline": roof,
        "e2e": {"value": round(e2e_ms * 1e3, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "how": "chord.w4a16_moe on inputs copied in from pinned host memory each step, "
                       "output copied back each step; copies on their own streams, double-buffered "
                       "(step i's output copy and step i+1's input copies overlap the layer); the "
                       "layer call replayed from a CUDA graph captured once per input buffer, as a "
                       "serving engine replays its decode step",
                "eager_value": round(e2e_eager_ms * 1e3, 2),
                "eager_how": "the same loop with chord.w4a16_moe called eagerly every step"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "kernel_source": src_hash,
    }
    if rank == 0 and not args.no_configs and args.workload == "ep8-decode" and args.T is None:
        del graph, case
        res["configs"] = run_configs(args, chord, torch, dev, stream, inp, d, dev_index, uuid)
        res["configs_note"] = ("the other configurations, timed in the same process after the "
                               "headline one, each with its own roofline and clock record; "
                               "`value` is the headline configuration's")
    return res, inp


REF_BUDGET_S = 150.0


def cpu_oracle_time(inp, max_tokens=None):
    """Wall time of the CPU oracle on (a sample of) the workload: align + layer."""
    import oracle
    from w4a16_int4_mixture_gb300 import synth
    s = inp.shape
    T = s.T if max_tokens is None else min(s.T, max_tokens)
    sub = inp
    if T < s.T:
        shp = synth.MoEShape(s.name, T=T, k=s.k, E_global=s.E_global, E_local=s.E_local,
                             H=s.H, I=s.I, block_m=s.block_m)
        sub = synth.MoEInputs(shp, inp.x[:T], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                              inp.topk_ids[:T], inp.topk_weights[:T], inp.expert_map)
    t0 = time.perf_counter()
    oracle.run_workload(sub)
    dt = time.perf_counter() - t0
    return dt, T, oracle.num_threads()


def cpu_baseline(inp, single_thread_tokens=16):
    """The oracle on the host cores, on the whole workload when it has at most
    1024 tokens, else on its first 512 tokens scaled by tokens (a bounded sample
    of about 10-30 s); and on one thread over the first few tokens."""
    import oracle
    s = inp.shape
    max_tok = s.T if s.T <= 1024 else 512
    dt, T, cores = cpu_oracle_time(inp, max_tok)
    per_call_us = dt * 1e6 * (s.T / T)
    sample = (f"CPU oracle (plain C, fp32) on {T} of {s.T} tokens of {s.name}: align + "
              f"gate/up + SiLU + down + combine, {dt:.2f} s wall; scaled by tokens to one call")
    res = {"value": round(per_call_us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": sample}
    oracle.set_threads(1)
    try:
        dt1, T1, _ = cpu_oracle_time(inp, single_thread_tokens)
    finally:
        oracle.set_threads(0)
    res["single_thread"] = {
        "value": round(dt1 * 1e6 * (s.T / T1), 1), "unit": UNIT, "cores": 1,
        "sample": f"the first {T1} tokens on one thread, {dt1:.2f} s wall; scaled by tokens "
                  f"(each touched expert is dequantised once per call, so a short sample "
                  f"overstates the per-token cost)"}
    return res


def run_reference(args):
    """The oracle timed on the host cores.  Each step is a bounded sample: the
    first T' tokens of the workload, T' sized from one untimed calibration run
    so that all warm-up and timed steps take about REF_BUDGET_S together; its
    time is scaled by tokens to one call."""
    from w4a16_int4_mixture_gb300 import synth
    import oracle
    oracle.build()
    s = synth.workload(args.workload, T=args.T)
    inp = synth.make_inputs(s)
    cap = s.T if s.T <= 1024 else 256
    t_cal, T_cal, _ = cpu_oracle_time(inp, cap)
    per_step = REF_BUDGET_S / max(1, args.warmup + args.steps)
    T_step = max(1, min(T_cal, int(T_cal * per_step / max(t_cal, 1e-9))))
    times = []
    for i in range(args.warmup + args.steps):
        dt, T, cores = cpu_oracle_time(inp, T_step)
        if i >= args.warmup:
            times.append(dt * (s.T / T))
    per_call_us = statistics.median(times) * 1e6
    sample = (f"CPU oracle (plain C, fp32) on the first {T} of {s.T} tokens of {s.name} per step "
              f"(sized for a {REF_BUDGET_S:.0f} s run; calibration {T_cal} tokens in "
              f"{t_cal:.2f} s), scaled by tokens to one call")
    return {
        "impl": "reference", "metric": METRIC, "value": round(per_call_us, 1), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_call_us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 (oracle)", "data": "synthetic",
        "config": {"workload": s.name, "T": s.T, "k": s.k, "E_global": s.E_global,
                   "E_local": s.E_local, "H": s.H, "I": s.I},
        "cpu_baseline": {"value": round(per_call_us, 1), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(per_call_us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    res, inp = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(inp)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
