"""Benchmark of the sparse MoE layer on one GB300 (or N replicas under torchrun).

Headline: Qwen-shaped decode layer (H=2048, E=256 routed experts, top-8,
SwiGLU intermediate 512, one shared expert, bf16 experts, fp32 router), T=1:
microseconds per layer call, over 64 different seeded tokens per step, with
the L2 cache flushed (a 256 MiB write) before every call, outside the timed
events. The same line also reports, as secondary workloads: the verify window (T=4),
a decode T-sweep 1..8, the MXFP4 Ling layer (T=1, T=4), int4 routed experts
(T=1), the online-FP8 LM head (T=1, 4) and the prefill chunks (T=4096: bf16,
int4 and MXFP4 routed experts).

  python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--quick]

Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

METRIC = "MoE layer µs at T=1/4 (HBM GB/s, % peak); prefill tokens/s at T=4096 (TC % peak)"
HEADLINE = "qwen_decode"
L2_FLUSH_BYTES = 256 << 20  # 2x the 129 MB L2


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every PERIOD_MS with their own timestamps. Sampling is
    running before the caller's region starts (__enter__ waits for the first
    sample), and summary() keeps the samples stamped inside the region marked by
    begin() / end(), widened by one period on each side."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, exe: str = "nvidia-smi", first_sample_timeout_s: float = 5.0):
        self.gpu = gpu_index
        self.exe = exe
        self.first_timeout = first_sample_timeout_s
        self.lines = []
        self.proc = None
        self.t_begin = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                [self.exe, f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            t0 = time.time()
            while not self.lines and self.proc.poll() is None and time.time() - t0 < self.first_timeout:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(self.PERIOD_MS / 1000.0)   # the sample that closes the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.th.join(timeout=5)

    @staticmethod
    def _stamp(text: str):
        from datetime import datetime
        try:
            return datetime.strptime(text, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        pad = self.PERIOD_MS / 1000.0
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((self._stamp(f[0]), float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        if self.t_begin is not None and self.t_end is not None:
            inside = [r for r in rows if r[0] is not None and self.t_begin - pad <= r[0] <= self.t_end + pad]
        else:
            inside = rows
        reasons = set()
        for r in inside:
            for n, v in zip(self.REASONS, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": inside[-1][2] if inside else (rows[-1][2] if rows else None),
                "reasons": sorted(reasons), "samples": len(inside), "samples_total": len(rows),
                "period_ms": self.PERIOD_MS}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Bench:
    def __init__(self, device):
        import torch
        self.torch = torch
        self.dev = device
        self.flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_sink = torch.empty(1, dtype=torch.float32, device=device)
        self.layers = {}

    def flush_l2(self):
        """Write a buffer twice the size of L2, then read another one: the write evicts the
        layer's lines, the read evicts the written (dirty) lines so that their write-back
        to HBM happens here, outside the timed region, and the timed call starts with a
        cold, clean L2."""
        self.flush_w.zero_()
        torch = self.torch
        torch.sum(self.flush_r, dim=0, keepdim=True, out=self.flush_sink)

    def layer(self, spec: mi.LayerSpec, max_tokens: int):
        from sparse_mixture_experts_gemv_gb300 import MoeLayer, weights_from_raw
        key = (spec, max_tokens)
        if key not in self.layers:
            for k in list(self.layers):
                if k[0] != spec:
                    self.layers.pop(k).close()
            S = mi.SynthLayer(spec)
            w = weights_from_raw(S.router(), S.router_bias(), S.stacked(), S.shared_raw())
            self.layers[key] = MoeLayer(spec.H, spec.E, spec.k, spec.I, spec.Is, w, fmt=spec.fmt,
                                        max_tokens=max_tokens, device=self.dev)
        return self.layers[key]

    def inputs(self, w: mi.Workload, calls: int):
        torch = self.torch
        xs = [torch.from_numpy(mi.workload_tokens(w, c).view(np.int16)).to(self.dev) for c in range(calls)]
        lbs = [None] * calls
        if w.logit_bias_sigma:
            lbs = [torch.from_numpy(mi.workload_logit_bias(w, c)).to(self.dev) for c in range(calls)]
        return xs, lbs

    def time_calls(self, L, xs, lbs, outs, flush=True, profile=False):
        """Per-call device time (ms) of each forward, L2 flushed before each call."""
        torch = self.torch
        from sparse_mixture_experts_gemv_gb300 import _native as N
        n = len(xs)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        stages = []
        if profile:
            N.moe_layer_profile_enable(L.handle, True)
        torch.cuda._sleep(20_000_000)  # let the host queue the whole loop ahead of the GPU
        for i in range(n):
            if flush:
                self.flush_l2()
            ev[i][0].record()
            L.forward(xs[i], outs[i], lbs[i])
            ev[i][1].record()
            if profile:
                stages.append(N.moe_layer_profile_read(L.handle))
        torch.cuda.synchronize()
        if profile:
            N.moe_layer_profile_enable(L.handle, False)
        return [a.elapsed_time(b) for a, b in ev], stages

    def launch_floor(self, n=64):
        """Event-to-event time (ms) of the same loop as time_calls (L2 flush, queued ahead behind a
        sleep, no host sync between calls) with nothing between the events, and with one one-thread
        kernel between them: the part of a single-launch call's time that is not the kernel's work."""
        torch = self.torch
        tiny = torch.zeros(1, device=self.dev)
        res = {}
        for name, body in (("events_only", None), ("one_tiny_kernel", lambda: tiny.add_(1.0))):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            if body is not None:   # the first launch loads the kernel's module: keep it out of the timing
                body()
                torch.cuda.synchronize()
            torch.cuda._sleep(20_000_000)
            for i in range(n):
                self.flush_l2()
                ev[i][0].record()
                if body is not None:
                    body()
                ev[i][1].record()
            torch.cuda.synchronize()
            res[name] = float(np.mean([a.elapsed_time(b) for a, b in ev]))
        return res

    def warm_back_to_back(self, L, xs, lbs, outs, reps=4):
        torch = self.torch
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(50_000_000)
        s.record()
        for _ in range(reps):
            for i in range(len(xs)):
                L.forward(xs[i], outs[i], lbs[i])
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / (reps * len(xs))

    def e2e(self, L, w: mi.Workload, calls: int):
        """Host-buffer calls through moe_layer_forward_host: H2D + layer + D2H + sync, wall clock."""
        torch = self.torch
        xh = [torch.from_numpy(mi.workload_tokens(w, c).view(np.int16)).pin_memory() for c in range(calls)]
        oh = [torch.empty_like(x).pin_memory() for x in xh]
        lb = [None] * calls
        if w.logit_bias_sigma:
            lb = [torch.from_numpy(mi.workload_logit_bias(w, c)).pin_memory() for c in range(calls)]
        for i in range(min(3, calls)):
            L.forward_host(xh[i], oh[i], lb[i])
        tot = 0.0
        for i in range(calls):
            self.flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            L.forward_host(xh[i], oh[i], lb[i])
            tot += time.perf_counter() - t0
        h2d = xh[0].numel() * 2 + (lb[0].numel() * 4 if lb[0] is not None else 0)
        d2h = oh[0].numel() * 2
        return tot / calls * 1e6, h2d, d2h


def decode_workload(B: Bench, wname: str, steps: int, warmup: int, peaks, profile=True):
    """Returns a result dict for one small-T workload (per-call us, GB/s, per-kernel roofline)."""
    torch = B.torch
    w = mi.WORKLOADS[wname]
    L = B.layer(w.layer, max_tokens=4096 if w.layer.fmt == "bf16" else 8)
    calls = w.calls
    xs, lbs = B.inputs(w, calls)
    outs = [torch.empty_like(x) for x in xs]
    # routed-expert bytes per call from the realised routing
    stats = []
    for i in range(calls):
        L.forward(xs[i], outs[i], lbs[i])
        stats.append(L.stats())
    for _ in range(warmup):
        B.time_calls(L, xs, lbs, outs)
    times = []
    for _ in range(steps):
        t, _ = B.time_calls(L, xs, lbs, outs)
        times += t
    us = float(np.mean(times) * 1e3)
    alg_bytes = float(np.mean([s.algorithmic_bytes for s in stats]))
    distinct = float(np.mean([s.distinct_experts for s in stats]))
    warm_us = B.warm_back_to_back(L, xs, lbs, outs) * 1e3
    res = {"workload": wname, "T": w.T, "us_per_call": us, "us_p50": float(np.median(times) * 1e3),
           "us_p90": float(np.percentile(times, 90) * 1e3), "warm_us_per_call": warm_us,
           "distinct_experts_mean": distinct, "algorithmic_bytes": alg_bytes,
           "layer_gbs": alg_bytes / (us * 1e-6) / 1e9,
           "layer_frac_of_hbm": alg_bytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
           "calls_timed": len(times), "launches_per_call": 1}
    if profile:
        st_all = []
        for _ in range(max(1, steps // 2)):
            _, st = B.time_calls(L, xs, lbs, outs, profile=True)
            st_all += st
        k_us = float(np.mean([x[0] for x in st_all]) * 1e3)
        res["kernel_us"] = k_us
        res["kernel_gbs"] = alg_bytes / (k_us * 1e-6) / 1e9
        res["kernel_frac_of_hbm"] = res["kernel_gbs"] / peaks["hbm_gbs"]
    return res


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over all ranks (the slowest replica
    sets the job's time); the identity when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def run_ours(args):
    import torch
    peaks = _peaks()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B = Bench(dev)

    # ---- headline: Qwen decode T=1, flushed L2, per-call CUDA events
    w = mi.WORKLOADS[HEADLINE]
    L = B.layer(w.layer, max_tokens=4096)
    xs, lbs = B.inputs(w, w.calls)
    outs = [torch.empty_like(x) for x in xs]
    stats = []
    for i in range(w.calls):
        L.forward(xs[i], outs[i], lbs[i])
        stats.append(L.stats())
    for _ in range(args.warmup):
        B.time_calls(L, xs, lbs, outs)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.begin()
        t0 = time.perf_counter()
        times = []
        for _ in range(args.steps):
            t, _ = B.time_calls(L, xs, lbs, outs)
            times += t
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        clk.end()
    if world > 1:
        torch.distributed.barrier()
    us = float(np.mean(times) * 1e3)
    step_ms = float(np.sum(times) / args.steps)
    us, step_ms = max_over_ranks([us, step_ms], dev)
    alg_bytes = float(np.mean([s.algorithmic_bytes for s in stats]))
    distinct = float(np.mean([s.distinct_experts for s in stats]))

    # the decode path is one kernel per call (moe_decode_stream_kernel): time that
    # launch with CUDA events recorded on the launching stream around it
    stage_all = []
    for _ in range(max(1, args.steps // 2)):
        _, st = B.time_calls(L, xs, lbs, outs, profile=True)
        stage_all += st
    k_us = float(np.mean([x[0] for x in stage_all]) * 1e3)
    achieved = alg_bytes / (k_us * 1e-6) / 1e9
    warm_us = B.warm_back_to_back(L, xs, lbs, outs) * 1e3
    e2e_us, h2d, d2h = B.e2e(L, w, min(w.calls, 32))
    floor = B.launch_floor()

    result = {
        "metric": METRIC, "value": round(us, 3), "unit": "us", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "qwen_decode: H=2048 E=256 top-8 I=512 + shared expert I=512, bf16 experts, "
                               "fp32 router, T=1, 64 seeded tokens per step",
                   "tokens_per_call": 1, "calls_per_step": w.calls, "l2": "flushed before every call (256 MiB write, then a 256 MiB read so dirty lines are written back outside the timed region)",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu"},
        "layer": {"algorithmic_bytes_per_call": alg_bytes, "gbs": alg_bytes / (us * 1e-6) / 1e9,
                  "frac_of_measured_hbm": alg_bytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
                  "warm_us_per_call": warm_us, "us_p50": float(np.median(times) * 1e3),
                  "us_p90": float(np.percentile(times, 90) * 1e3),
                  "distinct_experts_mean": distinct,
                  "launch_floor_us": {k: round(v * 1e3, 3) for k, v in floor.items()}},
        "roofline": {"kernel": "moe_decode_stream_kernel<1>", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": None, "peak_source": peaks["source"],
                     "bytes_per_launch": alg_bytes, "launch_us": round(k_us, 3)},
        "e2e": {"value": round(e2e_us, 3), "unit": "us", "h2d_bytes_per_step": h2d * w.calls,
                "d2h_bytes_per_step": d2h * w.calls},
        "gpu_launches": 1 * w.calls * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 3),
    }
    traffic = _profile_traffic("moe_decode_stream_kernel")
    if traffic is not None:
        result["roofline"]["traffic"] = traffic

    # ---- secondary workloads
    extra = {}
    if not args.quick:
        for wname in ("qwen_verify", "qwen_tsweep", "ling_mxfp4_t1", "ling_mxfp4_t4"):
            try:
                if wname == "qwen_tsweep":   # same layer as the headline: runs before the Ling layer replaces it
                    extra[wname] = tsweep_workload(B, max(2, args.steps // 4), peaks)
                else:
                    extra[wname] = decode_workload(B, wname, max(2, args.steps // 2), 2, peaks)
            except Exception as ex:  # report, never hide
                extra[wname] = {"error": repr(ex)}
        try:
            extra["lmhead_fp8"] = lmhead_workload(B, max(2, args.steps // 4), peaks)
        except Exception as ex:
            extra["lmhead_fp8"] = {"error": repr(ex)}
        for wname in ("qwen_int4_decode",):
            try:
                extra[wname] = decode_workload(B, wname, max(2, args.steps // 2), 2, peaks)
            except Exception as ex:
                extra[wname] = {"error": repr(ex)}
        for wname in ("qwen_prefill", "qwen_int4_prefill", "ling_mxfp4_prefill"):
            try:
                extra[wname] = prefill_workload(B, wname, max(2, args.steps // 2), 2, peaks)
            except Exception as ex:
                extra[wname] = {"error": repr(ex)}
    result["workloads"] = extra

    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def tsweep_workload(B: Bench, steps: int, peaks, tmax: int = 8, calls: int = 16):
    """Per-call time of the Qwen-shaped layer for windows of T = 1..tmax rows (verify
    windows of 2-5 rows, 2-token MTP batches), L2 flushed before every call; T > the
    weight-streaming limit would take the grouped path and is reported as such."""
    torch = B.torch
    spec = mi.QWEN_LAYER
    L = B.layer(spec, max_tokens=4096)
    rows = []
    for T in range(1, tmax + 1):
        xs = [torch.from_numpy(mi.tokens(spec, T, stream=900_000 + 100 * T + c).view(np.int16)).to(B.dev)
              for c in range(calls)]
        outs = [torch.empty_like(x) for x in xs]
        stats = []
        for i in range(calls):
            L.forward(xs[i], outs[i])
            stats.append(L.stats())
        B.time_calls(L, xs, [None] * calls, outs)
        times = []
        for _ in range(steps):
            times += B.time_calls(L, xs, [None] * calls, outs)[0]
        us = float(np.mean(times) * 1e3)
        alg = float(np.mean([s.algorithmic_bytes for s in stats]))
        rows.append({"T": T, "us_per_call": round(us, 3), "path": int(stats[0].path),
                     "distinct_experts_mean": float(np.mean([s.distinct_experts for s in stats])),
                     "algorithmic_bytes": alg, "frac_of_hbm": round(alg / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                     "us_per_token": round(us / T, 3)})
    return {"workload": "qwen_tsweep: Qwen-shaped layer, T = 1..8 seeded tokens per call (no logit bias)",
            "calls_per_T": calls, "rows": rows}


def lmhead_workload(B: Bench, steps: int, peaks, calls: int = 16):
    """Online-FP8 LM head, 157,184 x 2,560, T = 1 and 4: per-call time with the L2
    flushed before every call; algorithmic bytes = codes + scales + x + logits."""
    torch = B.torch
    from sparse_mixture_experts_gemv_gb300 import LmHead
    spec = mi.LMHEAD
    head = LmHead(mi.lmhead_weights(spec), device=B.dev)
    res = {"workload": f"lmhead_fp8: online-FP8 (E4M3, per-row fp32 scale) output projection "
                       f"{spec.V} x {spec.H}, bf16 activations", "rows": []}
    try:
        for T in (1, 4):
            xs = [torch.from_numpy(mi.lmhead_tokens(spec, T, stream=100 * T + c).view(np.int16)).to(B.dev)
                  for c in range(calls)]
            outs = [torch.empty((T, spec.V), dtype=torch.float32, device=B.dev) for _ in range(calls)]
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
            times = []
            for it in range(steps + 1):
                torch.cuda._sleep(20_000_000)
                for i in range(calls):
                    B.flush_l2()
                    ev[i][0].record()
                    head.forward(xs[i], outs[i])
                    ev[i][1].record()
                torch.cuda.synchronize()
                if it:  # the first pass warms up
                    times += [a.elapsed_time(b) for a, b in ev]
            us = float(np.mean(times) * 1e3)
            alg = spec.V * spec.H + 4 * spec.V + 2 * T * spec.H + 4 * T * spec.V
            gbs = alg / (us * 1e-6) / 1e9
            res["rows"].append({"T": T, "us_per_call": round(us, 3), "algorithmic_bytes": alg,
                                "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                                "launches_per_call": 1})
    finally:
        head.close()
    return res


def prefill_workload(B: Bench, wname: str, steps: int, warmup: int, peaks):
    torch = B.torch
    w = mi.WORKLOADS[wname]
    L = B.layer(w.layer, max_tokens=4096)
    x = torch.from_numpy(mi.workload_tokens(w, 0).view(np.int16)).to(B.dev)
    out = torch.empty_like(x)
    L.forward(x, out)
    st = L.stats()
    hist = L.dispatch(w.T)[0].cpu().numpy()          # rows routed to each expert by this chunk
    for _ in range(warmup):
        L.forward(x, out)
    times = []
    for _ in range(steps):
        t, _ = B.time_calls(L, [x], [None], [out])
        times += t
    ms = float(np.mean(times))
    tok_s = w.T / (ms * 1e-3)
    tflops = st.flops / (ms * 1e-3) / 1e12
    _, stages = B.time_calls(L, [x] * 3, [None] * 3, [out] * 3, profile=True)
    st_us = np.mean(np.array(stages), axis=0) * 1e3
    names = ["router", "dispatch", "grouped_gateup", "grouped_down", "combine"]
    return {"workload": wname, "T": w.T, "ms_per_call": ms, "tokens_per_s": tok_s,
            "useful_tflops": tflops, "frac_of_measured_bf16": tflops / peaks["bf16_tflops"],
            "mma": ("routed f16 x f16 (MXFP4 rows decoded in the GEMM), shared bf16 x bf16"
                    if w.layer.fmt == "mxfp4" else "bf16 x bf16"),
            "touched_experts": st.distinct_experts, "max_expert_rows": st.max_expert_rows,
            "expert_rows_summary": {"min": int(hist.min()), "median": float(np.median(hist)), "max": int(hist.max()),
                                    "mean": float(hist.mean()), "experts_over_128_rows": int((hist > 128).sum())},
            "expert_rows_histogram": [int(v) for v in hist],
            "algorithmic_bytes": st.algorithmic_bytes,
            "hbm_frac": st.algorithmic_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "stage_us": {n: round(float(v), 2) for n, v in zip(names, st_us)}}


def _profile_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary for `kernel`, if present and current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    v = d.get(kernel)
    return None if v is None or v.get("stale") else v.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
class StackedLayer:
    """Oracle accessor over pre-drawn stacked arrays (so timing excludes random draws)."""

    def __init__(self, S: mi.SynthLayer):
        self.spec = S.spec
        self._r = S.router()
        self._b = S.router_bias()
        self._st = S.stacked()
        self._sh = S.shared_raw()

    def router(self):
        return self._r

    def router_bias(self):
        return self._b

    def expert_raw(self, e):
        return {k: v[e] for k, v in self._st.items()}

    def shared_raw(self):
        return self._sh


class CachedLayer:
    """Oracle accessor that draws each expert once (lazily) and keeps it, so the
    timed calls exclude random draws; only the experts a sample touches are drawn."""

    def __init__(self, S: mi.SynthLayer):
        self.spec = S.spec
        self._S = S
        self._r = S.router()
        self._b = S.router_bias()
        self._sh = S.shared_raw()
        self._e = {}

    def router(self):
        return self._r

    def router_bias(self):
        return self._b

    def expert_raw(self, e):
        if e not in self._e:
            self._e[e] = self._S.expert_raw(e)
        return self._e[e]

    def shared_raw(self):
        return self._sh


# CPU-oracle legs: (name, workload, rows of one call or None for the workload's T, calls in the sample)
CPU_LEGS = [("t1", "qwen_decode", None, 8), ("t4", "qwen_verify", None, 4), ("t4096_256rows", "qwen_prefill", 256, 1)]


def _oracle_leg(wname: str, rows, ncalls: int, seconds: float) -> dict:
    """Per-call seconds of the oracle on a bounded sample of one workload."""
    from oracle import moe_oracle as o
    w = mi.WORKLOADS[wname]
    SL = CachedLayer(mi.SynthLayer(w.layer))
    calls = []
    for c in range(ncalls):
        x = mi.workload_tokens(w, c)
        lb = mi.workload_logit_bias(w, c) if w.logit_bias_sigma else None
        if rows is not None:   # a seeded subset of the chunk's rows (the layer is row-independent)
            sel = np.sort(np.random.default_rng(c).choice(x.shape[0], size=rows, replace=False))
            x = x[sel]
            lb = None if lb is None else lb[sel]
        calls.append((x, lb))
    for x, lb in calls:   # draws every touched expert once, outside the timing
        o.moe_forward(SL, x, logit_bias=lb)
    n, t0 = 0, time.perf_counter()
    while True:
        x, lb = calls[n % len(calls)]
        o.moe_forward(SL, x, logit_bias=lb)
        n += 1
        if time.perf_counter() - t0 >= seconds and n >= 2:
            break
    el = time.perf_counter() - t0
    return {"s_per_call": el / n, "calls": n, "rows_per_call": int(calls[0][0].shape[0]), "elapsed_s": el}


def _single_thread_legs(seconds: float) -> dict:
    """The same legs in a child process with one BLAS/OpenMP thread."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-legs-child", str(seconds)],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout)[-300:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_legs(seconds: float) -> list:
    """Oracle timings at T=1, T=4 and on a 256-row subset of the T=4096 prefill chunk,
    on all host cores (numpy/BLAS threads) and on one thread."""
    allc = {name: _oracle_leg(wn, rows, nc, seconds) for name, wn, rows, nc in CPU_LEGS}
    one = _single_thread_legs(seconds)
    out = []
    for name, wn, rows, nc in CPU_LEGS:
        for cores, r in ((os.cpu_count(), allc.get(name)), (1, one.get(name))):
            if not r or "s_per_call" not in r:
                out.append({"leg": name, "workload": wn, "cores": cores, "error": str(one.get("error", "missing"))})
                continue
            T_full = mi.WORKLOADS[wn].T
            leg = {"leg": name, "workload": wn, "cores": cores, "us_per_call": round(r["s_per_call"] * 1e6, 1),
                   "rows_per_call": r["rows_per_call"], "calls_timed": r["calls"]}
            if rows is not None:
                leg["sample"] = f"{rows} seeded rows of each T={T_full} chunk (the layer is row-independent)"
                leg["us_per_full_chunk_scaled"] = round(r["s_per_call"] * 1e6 * T_full / rows, 1)
                leg["tokens_per_s"] = round(rows / r["s_per_call"], 1)
            out.append(leg)
    return out


def cpu_baseline(seconds: float, wname: str = HEADLINE):
    from oracle import moe_oracle as o
    w = mi.WORKLOADS[wname]
    SL = StackedLayer(mi.SynthLayer(w.layer))
    xs = [mi.workload_tokens(w, c) for c in range(w.calls)]
    o.moe_forward(SL, xs[0])
    n, t0 = 0, time.perf_counter()
    while True:
        o.moe_forward(SL, xs[n % len(xs)])
        n += 1
        if time.perf_counter() - t0 >= seconds and n >= 2:
            break
    el = time.perf_counter() - t0
    res = {"value": round(el / n * 1e6, 1), "unit": "us", "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"{n} T=1 calls of the {wname} layer (fp64 numpy oracle, {el:.1f} s)"}
    try:
        res["legs"] = cpu_legs(max(2.0, seconds / 3))
    except Exception as ex:  # report, never hide
        res["legs"] = [{"error": repr(ex)}]
    return res


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import moe_oracle as o
    w = mi.WORKLOADS[HEADLINE]
    SL = StackedLayer(mi.SynthLayer(w.layer))
    xs = [mi.workload_tokens(w, c) for c in range(w.calls)]
    per_step = max(1, args.ref_calls_per_step)
    for i in range(args.warmup):
        o.moe_forward(SL, xs[i % len(xs)])
    t0 = time.perf_counter()
    n = 0
    for s in range(args.steps):
        for c in range(per_step):
            o.moe_forward(SL, xs[n % len(xs)])
            n += 1
    el = time.perf_counter() - t0
    us = el / n * 1e6
    cb = {"value": round(us, 1), "unit": "us", "cores": os.cpu_count(), "kind": "oracle",
          "sample": f"{per_step} T=1 calls per step of the {HEADLINE} layer, {args.steps} steps"}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": "qwen_decode: H=2048 E=256 top-8 I=512 + shared, T=1 "
                                                    "(fp64 CPU oracle, the layer's plain definition)"},
        "cpu_baseline": cb, "e2e": {"value": round(us, 1), "unit": "us", "h2d_bytes_per_step": 0,
                                    "d2h_bytes_per_step": 0}}), flush=True)


def run_profile_driver(args):
    """Untimed forward calls of one workload (for ncu captures): builds the layer,
    then runs --profile-calls calls with the L2 flushed before each."""
    import torch
    dev = torch.device("cuda", 0)
    B = Bench(dev)
    if args.profile == "lmhead_fp8":   # the online-FP8 LM head GEMV at T=1
        from sparse_mixture_experts_gemv_gb300 import LmHead
        head = LmHead(mi.lmhead_weights(mi.LMHEAD), device=dev)
        x = torch.from_numpy(mi.lmhead_tokens(mi.LMHEAD, 1, stream=3).view(np.int16)).to(dev)
        for c in range(args.profile_calls):
            B.flush_l2()
            head.forward(x)
        torch.cuda.synchronize()
        head.close()
        print(json.dumps({"profile_driver": args.profile, "calls": args.profile_calls, "status": 0}))
        return
    w = mi.WORKLOADS[args.profile]
    L = B.layer(w.layer, max_tokens=max(8, w.T) if w.layer.fmt != "bf16" else 4096)
    xs, lbs = B.inputs(w, min(w.calls, args.profile_calls))
    for c in range(args.profile_calls):
        B.flush_l2()
        L.forward(xs[c % len(xs)], logit_bias=lbs[c % len(lbs)])
    torch.cuda.synchronize()
    st = L.sync_status()
    print(json.dumps({"profile_driver": args.profile, "calls": args.profile_calls, "status": st}))
    if st != 0:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-calls-per-step", type=int, default=8)
    ap.add_argument("--profile", default=None, choices=sorted(mi.WORKLOADS) + ["lmhead_fp8"],
                    help="untimed calls of one workload, for ncu captures")
    ap.add_argument("--profile-calls", type=int, default=6)
    ap.add_argument("--cpu-legs-child", type=float, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_legs_child is not None:   # one-thread oracle legs (run by cpu_legs in a child process)
        print(json.dumps({name: _oracle_leg(wn, rows, nc, args.cpu_legs_child) for name, wn, rows, nc in CPU_LEGS}))
        return
    if args.profile:
        run_profile_driver(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
