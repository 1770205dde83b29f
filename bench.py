"""Benchmark of the single-GPU MoE layer forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload v3] [--extras LIST|none] [--no-cpu-baseline]

One step = one whole layer forward (router GEMM, scoring/Top-k, statistics, dispatch, grouped
SwiGLU expert GEMMs, shared experts, combine) over one batch of synthetic tokens already in HBM.
The headline workload is the largest single-GPU layer, the DeepSeek-V3-shaped prefill layer
(T=8192, d=7168, 256 routed experts + 1 shared, top-8 of 8 groups keep 4).  The timed step is
moe_forward_timed: moe_forward's kernels, with two CUDA events recorded around the routed expert
GEMM launches (the shared experts' two run on a side stream beside the router, outside them) so
that the grouped GEMM's share is measured live.
After the headline, the same JSON line carries the other prefill layers (`per_config`: the
Mixtral-8x7B-shaped layer balanced and collapsed, DeepSeekMoE-16B token choice and expert
choice) and the decode-batch sweep (`decode`: B = 1, 8, 64, 256 on the V3- and Mixtral-shaped
layers, HBM bandwidth on the expert bytes each step touched).
Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica on its own token
batch (the layer shards over tokens with no exchange), so the work scales weakly.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd tokens/s on 1 B300; % of tensor-peak (prefill) / HBM BW (decode)"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the expert GEMM launches that
# the roofline times (the routed gate/up and down launches of one step), keyed by (workload,
# T, E), from an ncu capture of the bench command on the current kernel build; a workload
# without a capture on the current build reports null.
GEMM_TRAFFIC_BYTES = {
    ("v3", 8192, 256): (16824082688 + 266261504) + (7862229760 + 929332992),
    ("mixtral", 4096, 8): (1948641024 + 226491136) + (1553855744 + 122539776),
    ("mixtral_collapsed", 4096, 8): (1963653888 + 229137664) + (1768455936 + 124471808),
    ("dsmoe16b", 8192, 64): (953357056 + 125698560) + (517015552 + 171648256),
    ("dsmoe16b_ec", 8192, 64): (939601152 + 123286272) + (507836160 + 171243520),
}


def workload_flops_bytes(wl):
    """Algorithmic FLOPs and bytes of one layer forward (per step).

    FLOPs = T * (2 d E  +  (k + shared) * 3 * 2 d F)  (router + SwiGLU experts)
    bytes = touched expert weights + router weights + x read + out write.
    """
    T, d, E, k, F, Fs = wl.T, wl.d, wl.E, wl.k, wl.F, wl.F_sh
    routed = T * k * 3 * 2 * d * F
    ffn = routed + T * 3 * 2 * d * Fs
    router = T * 2 * d * E
    weights = (E * 3 * d * F + 3 * d * Fs + E * d) * 2
    act = 2 * T * d * 2
    return {"flops": ffn + router, "ffn_flops": ffn, "routed_flops": routed,
            "bytes": weights + act}


def shared_on_side_stream(wl):
    """Mirrors the library's rule: a bf16 prefill layer's shared experts run on a side stream
    beside the router and the gather (outside the expert-stage events) unless
    MOE_B300_SHARED=serial runs them after the routed GEMMs (inside the events)."""
    if wl.F_sh <= 0 or wl.dtype != "bf16" or os.environ.get("MOE_B300_SHARED") == "serial":
        return False
    path = os.environ.get("MOE_B300_PATH")
    decode = (wl.routing != "expert_choice" and wl.d % 256 == 0
              and (path == "decode" or (path != "prefill" and wl.T * wl.k <= 64 * wl.E)))
    return not decode


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml.so.1 ships with the driver)."""
    CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")

    def handle(self, cuda_index):
        ct = self.ct
        h = ct.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ct.byref(h)) == 0:
                return h
        except Exception:
            pass
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(cuda_index), ct.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex failed")
        return h

    def clock(self, h, maximum=False):
        v = self.ct.c_uint()
        fn = self.lib.nvmlDeviceGetMaxClockInfo if maximum else self.lib.nvmlDeviceGetClockInfo
        if fn(h, self.ct.c_int(self.CLOCK_SM), self.ct.byref(v)) != 0:
            raise RuntimeError("nvml clock query failed")
        return v.value

    def reasons(self, h):
        v = self.ct.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if fn is None or fn(h, self.ct.byref(v)) != 0:
            if self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, self.ct.byref(v)) != 0:
                raise RuntimeError("nvml reasons query failed")
        return v.value

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of the benchmarked GPU
    through NVML (read-only) every few milliseconds while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, interval_s: float = 0.002):
        self.cuda_index = cuda_index
        self.interval = interval_s
        self.samples = []
        self.max_mhz = None
        self.error = None
        self.recording = False

    def start(self):
        """Begin recording (call right before the timed region)."""
        self.recording = True

    def _run(self):
        try:
            nv = _Nvml()
            h = nv.handle(self.cuda_index)
            self.max_mhz = nv.clock(h, maximum=True)
            while not self._stop.is_set():
                if self.recording:
                    self.samples.append((nv.clock(h), nv.reasons(h)))
                self._stop.wait(self.interval)
            nv.close()
        except Exception as e:          # sampling is best effort; reported as unsampled
            self.error = repr(e)

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        time.sleep(0.05)                 # first sample before the timed region starts
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0, "error": self.error}
        count = {}
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    count[name] = count.get(name, 0) + 1
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(count),
                "reason_share": {n: c / len(self.samples) for n, c in sorted(count.items())},
                "samples": len(self.samples)}


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (every rank processes its own token batch; the job is done when
    the last one is).  Single process: returns ms."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms_max / 1e3)


def runs_reference_arm(rank: int) -> bool:
    """Under torchrun only rank 0 times the oracle; the other ranks exit without work."""
    return rank == 0


def cpu_cores():
    """Host threads the oracle's loops use."""
    from oracle import moe_oracle as O
    return O.threads()


def oracle_sample(wl, inp_host, S):
    """The oracle (as it stands, the C++ library) on an independent batch of the first S tokens;
    returns the seconds it took.  inp_host: host tensors (bf16 passed as its 16 bits), the
    routed weights stacked or one tensor per expert."""
    from oracle import moe_oracle as O
    h = dict(inp_host)
    x = h["x"][:S]
    sub = wl.replace(T=S)
    t0 = time.perf_counter()
    if wl.routing == "expert_choice":
        O.moe_forward_expert_choice(sub, x, h["w_gate"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    else:
        O.moe_forward(sub, x, h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    return time.perf_counter() - t0


def host_inputs(inp):
    """Host copies of the device inputs (same dtype: bf16 stays 2 bytes per value)."""
    return {k: (None if v is None else v.detach().to("cpu")) for k, v in inp.items()}


def run_cpu_baseline(wl, inp, target_s=12.0, max_reps=8):
    """Sizes the oracle's sample so that it takes about target_s seconds (two probe sizes give
    the per-token cost) and times it; when even the whole batch is shorter, the batch is timed
    again until about target_s has passed (at most max_reps passes)."""
    hi = host_inputs(inp)
    lo = -(-wl.E // wl.k) if wl.routing == "expert_choice" else 1   # C = S k / E >= 1
    s1, s2 = min(max(8, lo), wl.T), min(max(64, 2 * lo), wl.T)
    t1 = oracle_sample(wl, hi, s1)
    t2 = oracle_sample(wl, hi, s2) if s2 > s1 else t1
    per_tok = max((t2 - t1) / max(s2 - s1, 1), 1e-6)
    S = int(min(wl.T, max(s2, s1 + (target_s - t1) / per_tok)))
    times = [oracle_sample(wl, hi, S)]
    while sum(times) < target_s * 0.8 and len(times) < max_reps:
        times.append(oracle_sample(wl, hi, S))
    return S, times


def reference_inputs(wl, S):
    """Host inputs of the reference arm's sample, drawn on the CPU: the router inputs of S
    tokens, the shared experts, and only the routed experts the oracle's routing of those S
    tokens selects (each drawn from its own generator), so that a layer with 22.6 GB of expert
    weights is not drawn in full.  Expert choice lets every expert choose: all are drawn."""
    import moe_inputs
    from oracle import moe_oracle as O
    sub = wl.replace(T=S)
    r = moe_inputs.make_router_inputs(sub)
    if wl.routing == "expert_choice":
        need = range(wl.E)
    else:
        need = sorted({int(e) for e in O.route(sub, r["x"], r["w_gate"], r["bias"])["idx"].ravel()})
    w13, w2 = [None] * wl.E, [None] * wl.E
    for e in need:
        w13[e], w2[e] = moe_inputs.expert_weights(wl, e)
    ws13, ws2 = moe_inputs.shared_weights(wl)
    return {**r, "w13": w13, "w2": w2, "ws13": ws13, "ws2": ws2}, len(need)


def reference_sample_tokens(wl):
    """Tokens per reference-arm step: about 1.6 G multiply-adds of oracle work (~1-3 s on the
    host cores), at least 16 (and enough for one expert-choice token per expert)."""
    macs = 3 * wl.d * wl.F * wl.k + 3 * wl.d * wl.F_sh + wl.d * wl.E
    S = max(16, int(1.6e9 / macs) // 8 * 8)
    if wl.routing == "expert_choice":
        S = max(S, -(-wl.E // wl.k))
    return min(wl.T, S)


def layer_config(m, wl, T=None):
    return m.make_config(wl.T if T is None else T, wl.d, wl.E, wl.k, wl.F, wl.F_sh, wl.score,
                         wl.routing, wl.n_groups, wl.topk_groups, wl.renormalize,
                         wl.route_scale, wl.capacity_factor, wl.dtype)


def decode_case(m, wl0, weights, B, steps, hbm, peak_kind, graphs=True, fp8=False, q=None):
    """One decode batch size: B tokens per step, `steps` seeded steps with fresh x and router
    weights (expert weights fixed), timed through moe_forward (one CUDA graph per step,
    captured outside the timed region).  Returns the result dict: tokens/s and the HBM
    bandwidth reached on the bytes a step must read -- the experts it actually touched (counted
    from its own selection), the shared experts, the router, x and the output -- plus the
    distinct experts touched per step against E(1-(1-k/E)^B), as configured (with the
    workload's selection bias, if any) and with a zero selection bias (exchangeable experts,
    where the formula holds in expectation)."""
    import math
    import torch
    import moe_inputs
    if fp8:
        per_expert = 3 * wl0.d * wl0.F + (2 * wl0.F + wl0.d) * 4
        shared_bytes = 3 * wl0.d * wl0.F_sh + ((2 * wl0.F_sh + wl0.d) * 4 if wl0.F_sh else 0)
    else:
        per_expert = 3 * wl0.d * wl0.F * 2
        shared_bytes = 3 * wl0.d * wl0.F_sh * 2
    wl = wl0.replace(T=B)
    cfg = layer_config(m, wl)
    routers = [moe_inputs.make_router_inputs(wl, seed=1000 + i, device="cuda")
               for i in range(steps)]
    ws = m.fp8_workspace(cfg) if fp8 else m.workspace(cfg)
    out = torch.empty((B, wl.d), dtype=torch.float32, device="cuda")
    idx_all = torch.empty((steps, B, wl.k), dtype=torch.int32, device="cuda")

    def fwd(i):
        r = routers[i]
        if fp8:
            m.moe_forward_fp8(cfg, r["x"], r["w_gate"], r["bias"], *q["w13"], *q["w2"],
                              *q["ws13"], *q["ws2"], out, topk_idx=idx_all[i], ws=ws)
        else:
            m.moe_forward(cfg, r["x"], r["w_gate"], r["bias"], weights["w13"], weights["w2"],
                          weights["ws13"], weights["ws2"], out, topk_idx=idx_all[i], ws=ws)
    for i in range(min(5, steps)):
        fwd(i)
    torch.cuda.synchronize()
    grs = []
    if graphs:
        for i in range(steps):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                fwd(i)
            grs.append(gr)
        torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.start()
        ev[0].record()
        for i in range(steps):
            if grs:
                grs[i].replay()
            else:
                fwd(i)
            ev[i + 1].record()
        torch.cuda.synchronize()
    st = m.sync_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st}: {m.status_string(st)}")
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    distinct = [int(torch.unique(idx_all[i]).numel()) for i in range(steps)]
    step_bytes = [dn * per_expert + shared_bytes + wl.E * wl.d * 2 + B * wl.d * 2 +
                  B * wl.d * 4 for dn in distinct]
    total_s = sum(ms) / 1e3
    gbs = sum(step_bytes) / total_s / 1e9
    # routing-only statistic with the selection bias at zero
    zero = wl.replace(bias_range=0.0)
    logits = torch.empty((B, wl.E), dtype=torch.float32, device="cuda")
    w0 = torch.empty((B, wl.k), dtype=torch.float32, device="cuda")
    dz = []
    for i in range(steps):
        r = moe_inputs.make_router_inputs(zero, seed=5000 + i, device="cuda")
        m.moe_router_topk(cfg, r["x"], r["w_gate"], None, logits, idx_all[i], w0, ws)
        dz.append(int(torch.unique(idx_all[i]).numel()))
    formula = wl.E * (1 - (1 - wl.k / wl.E) ** B)
    mean_z = sum(dz) / len(dz)
    se_z = (sum((v - mean_z) ** 2 for v in dz) / max(len(dz) - 1, 1)) ** 0.5 / math.sqrt(len(dz))
    res = {
        "workload": f"{wl0.name} B={B}", "B": B, "steps": steps,
        "value": B * steps / total_s, "unit": "tokens/s", "ms_per_step": sum(ms) / steps,
        "dtype": "e4m3 expert weights and activations, bf16 router" if fp8 else "bf16",
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_kind": f"{peak_kind} copy bandwidth",
                     "bytes": "touched expert weights (from each step's own selection) + "
                              "shared experts + router + x + out"},
        "bytes_per_step_mean": sum(step_bytes) / steps,
        "distinct_experts": {"as_configured_mean": sum(distinct) / steps,
                             "selection_bias": (f"U(-{wl0.bias_range}, {wl0.bias_range})"
                                                if wl0.bias_range > 0 else "none"),
                             "zero_bias_mean": mean_z, "zero_bias_se": se_z,
                             "formula": formula},
        "clocks": clk.summary(), "cuda_graphs": bool(grs),
        "l2": "each step reads >= 0.35 GB of expert weights (> 126 MB L2)"}
    del routers, ws, grs
    torch.cuda.empty_cache()
    return res


def decode_sweep(args):
    """Decode-sized batches, one JSON line per (workload, B); see decode_case."""
    import torch
    import moe_inputs
    import top_routing_expert_scoring_b300 as m
    torch.cuda.set_device(0)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    fp8 = args.fp8
    for name in args.decode_workloads.split(","):
        wl0 = moe_inputs.workload(name)
        weights = moe_inputs.make_expert_weights(wl0, device="cuda")
        q = None
        if fp8:
            # one-byte E4M3 codes plus one fp32 scale per weight row, quantised once up front
            q = {key: (m.quantize_fp8(weights[key]) if weights[key] is not None else (None, None))
                 for key in ("w13", "w2", "ws13", "ws2")}
            torch.cuda.synchronize()
            del weights
            weights = None
            torch.cuda.empty_cache()
        for B in [int(b) for b in args.decode_batches.split(",")]:
            res = decode_case(m, wl0, weights, B, args.decode_steps, hbm, peak_kind,
                              graphs=not args.no_graphs, fp8=fp8, q=q)
            print(json.dumps({
                "metric": "MoE layer fwd tokens/s, decode batch; % of HBM BW on touched expert "
                          "weights", "mode": "decode_fp8" if fp8 else "decode",
                "data": "synthetic", **res}))
        del weights, q
        torch.cuda.empty_cache()


def router_backward_bytes_flops(wl):
    """Algorithmic bytes and FLOPs of one router-side backward (moe_router_backward with every
    output): reads logits, selection, d_topk_w, f, x and W_gate; writes dL/dg, dW_gate and dx
    (float32).  FLOPs: the two gradient products, 2 T d E each."""
    T, d, E, k = wl.T, wl.d, wl.E, wl.k
    rd = T * E * 4 + T * k * 8 + E * 4 + T * d * 2 + E * d * 2
    wr = T * E * 4 + E * d * 4 + T * d * 4
    return {"bytes": rd + wr, "flops": 4 * T * d * E}


def router_backward_sweep(args):
    """Router-side backward (dL/dg, dW_gate, dx) per workload: CUDA events around each call
    (replayed from a CUDA graph), L2 flushed (256 MB write) between calls outside the events.
    The routing inputs come from the forward's own router call."""
    import torch
    import moe_inputs
    import top_routing_expert_scoring_b300 as m
    torch.cuda.set_device(0)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks["bf16_tflops"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for name in args.backward_workloads.split(","):
        wl = moe_inputs.workload(name)
        T, E, k, d = wl.T, wl.E, wl.k, wl.d
        cfg = m.make_config(T, d, E, k, wl.F, wl.F_sh, wl.score, wl.routing, wl.n_groups,
                            wl.topk_groups, wl.renormalize, wl.route_scale, wl.capacity_factor,
                            wl.dtype)
        inp = moe_inputs.make_router_inputs(wl, device="cuda")
        gi = moe_inputs.make_grad_inputs(wl, device="cuda")
        ws_f = m.workspace(cfg)
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        f = torch.empty(E, dtype=torch.float32, device="cuda")
        P = torch.empty(E, dtype=torch.float32, device="cuda")
        lb = torch.empty(1, dtype=torch.float32, device="cuda")
        z = torch.empty(1, dtype=torch.float32, device="cuda")
        m.moe_router_topk(cfg, inp["x"], inp["w_gate"], inp["bias"], logits, idx, w, ws_f)
        m.moe_aux_stats(cfg, logits, idx, f, P, lb, z, ws_f)
        del ws_f
        ws = m.router_backward_workspace(cfg)
        d_logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        dW = torch.empty((E, d), dtype=torch.float32, device="cuda")
        dx = torch.empty((T, d), dtype=torch.float32, device="cuda")

        def call():
            m.moe_router_backward(cfg, inp["x"], inp["w_gate"], logits, idx, gi["d_topk_w"], f,
                                  0.01, 0.001, d_logits, dW, dx, ws)
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        # one CUDA graph per call, so that the events time the kernels and not the host's
        # marshalling and launch of three short kernels
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        graph.replay()
        torch.cuda.synchronize()
        reps = args.backward_steps
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.start()
            for a, b in ev:
                flush.fill_(1)
                a.record()
                graph.replay()
                b.record()
            torch.cuda.synchronize()
        st = m.sync_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st}: {m.status_string(st)}")
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        bf = router_backward_bytes_flops(wl)
        gbs = bf["bytes"] / (ms / 1e3) / 1e9
        tfs = bf["flops"] / (ms / 1e3) / 1e12
        hbm_ms = bf["bytes"] / (hbm * 1e9) * 1e3
        tc_ms = 4 * T * d * ((E + 63) // 64 * 64) / (tflops * 1e12) * 1e3
        print(json.dumps({
            "metric": "router-side backward (dL/dg, dW_gate, dx) tokens/s; % of HBM roofline",
            "mode": "router_backward", "workload": name, "value": T / (ms / 1e3),
            "unit": "tokens/s", "ms_per_call_median": ms, "steps": reps, "dtype": wl.dtype,
            "data": "synthetic",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_kind": f"{peak_kind} copy bandwidth",
                         "algorithmic_bytes": bf["bytes"]},
            "floors_ms": {"hbm": hbm_ms, "tensor_padded_E64": tc_ms},
            "tflops_algorithmic": tfs,
            "clocks": clk.summary(), "l2": "256 MB buffer written between calls"}))
        del inp, gi, ws, logits, idx, w, d_logits, dW, dx
        torch.cuda.empty_cache()


def router_in_gemm(wl):
    """The library's rule for running scoring and Top-k in the router GEMM's epilogue: a bf16
    token-choice router with E a multiple of 32 up to 256, k <= 8, more than 512 tokens, and
    groups (if limited) of whole 32-expert chunks; by default only from 128 experts up.
    MOE_B300_ROUTER=fused takes it for every such router, =separate for none."""
    if wl.dtype != "bf16" or wl.routing != "token_choice":
        return False
    if wl.E < 32 or wl.E > 256 or wl.E % 32 or wl.k > 8 or wl.T <= 512:
        return False
    limit = wl.score == "sigmoid" and wl.n_groups > 1 and wl.topk_groups < wl.n_groups
    if limit and (wl.E // wl.n_groups) % 32:
        return False
    env = os.environ.get("MOE_B300_ROUTER")
    if env in ("fused", "separate"):
        return env == "fused"
    return wl.E >= 128


def launches_per_step(wl):
    """Our kernels per forward: router logits and Top-k (+statistics partials; one kernel when
    the router GEMM's epilogue does the Top-k), dispatch (1 kernel for T <= 256, else 4),
    2 expert GEMMs, 2 shared-expert GEMMs, combine, statistics final.  A k <= 2 bf16 layer
    without shared experts and with a float32 output has no combine kernel: the down GEMM adds
    the weighted rows into the output itself."""
    shared = wl.F_sh > 0
    if wl.routing == "expert_choice":
        return 1 + 5 + 2 + 2 + (2 if shared else 0) + 1 + 2
    combine_in_gemm = (wl.k <= 2 and not shared and wl.dtype == "bf16"
                       and os.environ.get("MOE_B300_COMBINE") != "separate")
    return ((1 if router_in_gemm(wl) else 2) + (1 if wl.T <= 256 else 4) + 2
            + (2 if shared else 0) + (0 if combine_in_gemm else 1) + 1)


class Prefill:
    """Device buffers of one prefill layer forward and its timed step (moe_forward_timed)."""

    def __init__(self, m, wl, inp, dev, stream):
        import torch
        self.m, self.wl, self.inp, self.stream = m, wl, inp, stream
        T, E, k, d = wl.T, wl.E, wl.k, wl.d
        self.cfg = layer_config(m, wl)
        self.ws = m.workspace(self.cfg, dev)
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.idx, self.w = torch.empty((T, k), **i32), torch.empty((T, k), **f32)
        self.f, self.P = torch.empty(E, **f32), torch.empty(E, **f32)
        self.lb, self.z = torch.empty(1, **f32), torch.empty(1, **f32)
        self.nd = torch.empty(1, **i32)
        self.out = torch.empty((T, d), **f32)      # fp32 layer output (out_dtype f32)

    def step(self, ev_pair):
        inp = self.inp
        self.m.moe_forward_timed(self.cfg, inp["x"], inp["w_gate"], inp["bias"], inp["w13"],
                                 inp["w2"], inp["ws13"], inp["ws2"], self.out, self.idx, self.w,
                                 self.f, self.P, self.lb, self.z, self.nd, self.ws, self.stream,
                                 ev_pair[0], ev_pair[1])

    def check(self):
        st = self.m.sync_status(self.ws)
        if st != 0:
            raise RuntimeError(f"device status {st}: {self.m.status_string(st)}")

    def timed(self, steps, warmup, barrier):
        """Returns (ms over the timed steps, per-step expert-stage ms, clock summary)."""
        import torch
        warm = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for ev_ in warm:
            ev_.record(self.stream)          # torch creates the event handle on first record
        for _ in range(max(warmup, 3)):
            self.step(warm)
        barrier()
        self.check()
        pairs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for pair in pairs:
            for ev_ in pair:
                ev_.record(self.stream)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            barrier()
            clk.start()
            t0.record(self.stream)
            for i in range(steps):
                self.step(pairs[i])
            t1.record(self.stream)
            barrier()
        self.check()
        return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in pairs], clk.summary()


def choose_peak(peaks, peak_kind, clocks):
    """Burst bf16 peak while the GPU held its clock; the sustained (power-capped) peak when the
    timed region ran under the power cap: its median SM clock sat materially below the maximum,
    or the power-cap reason was active in at least half of its clock samples while the median
    clock sat below the maximum (a cap flag at full clock does not count)."""
    mhz, top = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    low = bool(mhz and top and mhz < 0.95 * top)
    below = bool(mhz and top and mhz < 0.99 * top)
    cap_share = clocks.get("reason_share", {}).get("sw_power_cap", 0.0)
    if (low or (below and cap_share >= 0.5)) and "bf16_tflops_sustained" in peaks:
        why = ("timed region ran below 95% of the maximum SM clock" if low else
               f"power cap active in {cap_share:.0%} of the timed region's clock samples")
        return float(peaks["bf16_tflops_sustained"]), f"{peak_kind} bf16 sustained ({why})"
    return float(peaks["bf16_tflops"]), f"{peak_kind} bf16 burst"


def prefill_figures(wl, ms_step, gemm_ms, clocks, peaks, peak_kind):
    """Roofline of the expert GEMM stage (the SwiGLU FLOPs of the launches between the two
    CUDA events on the launching stream: the routed gate/up and down, plus the shared experts'
    two when they run on that stream after them) and of the whole layer."""
    fb = workload_flops_bytes(wl)
    side = shared_on_side_stream(wl)
    stage_flops = fb["routed_flops"] if side else fb["ffn_flops"]
    gemm_avg = sum(gemm_ms) / len(gemm_ms)
    tflops = stage_flops / (gemm_avg / 1e3) / 1e12
    peak, peak_name = choose_peak(peaks, peak_kind, clocks)
    layer_roof_ms = max(fb["flops"] / (peak * 1e12),
                        fb["bytes"] / (peaks["hbm_gbs"] * 1e9)) * 1e3
    kernel = ("grouped GEMM kernel: the routed gate/up + down launches of one step"
              + ("; the shared experts' two launches run on a side stream beside the router and "
                 "the gather, outside the timed pair" if side else
                 (", then the shared experts' gate/up + down launches" if wl.F_sh > 0 else "")))
    return {
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak,
                     "traffic": (GEMM_TRAFFIC_BYTES.get((wl.name, wl.T, wl.E))
                                 if side or wl.F_sh == 0 else None),
                     "traffic_unit": "bytes per step (the timed expert GEMM launches)",
                     "kernel": kernel, "peak_kind": peak_name,
                     "flops_per_step": stage_flops},
        "layer_roofline": {"roofline_ms": layer_roof_ms, "frac": layer_roof_ms / ms_step,
                           "flops_per_step": fb["flops"], "bytes_per_step": fb["bytes"]},
        "stage_ms": {"expert_ffn": gemm_avg, "rest": ms_step - gemm_avg},
    }


def workload_config(wl, world):
    return {"workload": f"{wl.name}-shaped MoE layer: T={wl.T} d={wl.d} E={wl.E} k={wl.k} "
                        f"F={wl.F} shared={wl.n_shared}x{wl.F_shared} score={wl.score} "
                        f"routing={wl.routing} cf={wl.capacity_factor or 'none'}",
            "T": wl.T, "d_model": wl.d, "E": wl.E, "k": wl.k, "d_ff": wl.F,
            "shared_d_ff": wl.F_sh, "capacity_factor": wl.capacity_factor or None,
            "l2": "inputs larger than L2 (expert weights "
                  f"{wl.E * 3 * wl.d * wl.F * 2 / 1e9:.2f} GB > 126 MB)",
            "parallelism": "replicas" if world == 1 else f"replicas x{world} (token shards)"}


def run_reference_arm(args, wl, config):
    """The oracle, as it stands, on the host cores: one bounded sample of the workload per
    step (the first S tokens as an independent batch)."""
    S = reference_sample_tokens(wl)
    hi, n_experts = reference_inputs(wl, S)
    for _ in range(max(args.warmup, 0)):
        oracle_sample(wl, hi, min(S, 8))
    times = [oracle_sample(wl, hi, S) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    val = S / (ms / 1e3)
    cores = cpu_cores()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"independent batch of the first {S} tokens per step "
                                   f"(plain C++ oracle, double accumulation; the {n_experts} "
                                   f"routed experts they select drawn on the host)"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def e2e_leg(m, pf, steps, barrier, max_over):
    """End to end through the public call with host buffers, copies inside the timed region:
    every step copies its tokens from pinned host memory to the device, runs moe_forward and
    copies the layer output and statistics back.  Like a serving loop, consecutive steps are
    pipelined on three streams with double buffers: step i's host-to-device copy and step
    i-1's device-to-host copy overlap step i's forward.  Returns (ms per step, h2d bytes, d2h
    bytes)."""
    import torch
    wl, inp, stream = pf.wl, pf.inp, pf.stream
    T, d, E = wl.T, wl.d, wl.E
    f32 = dict(dtype=torch.float32, device=pf.out.device)
    x_host = [inp["x"].cpu().pin_memory() for _ in range(2)]
    out_host = [torch.empty((T, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    stats_host = [torch.empty(E + 2, dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    out_dev = [torch.empty((T, d), **f32) for _ in range(2)]
    stats_dev = [torch.empty(E + 2, **f32) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_x = [torch.cuda.Event() for _ in range(2)]          # x copied in
    ev_y = [torch.cuda.Event() for _ in range(2)]          # forward done
    ev_xfree = [torch.cuda.Event() for _ in range(2)]      # forward no longer reads x
    ev_yfree = [torch.cuda.Event() for _ in range(2)]      # output copied out
    for b_ in range(2):
        for ev_ in (ev_xfree[b_], ev_yfree[b_]):
            ev_.record(stream)

    def e2e_step(i):
        b_ = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_xfree[b_])
            x_dev[b_].copy_(x_host[b_], non_blocking=True)
            ev_x[b_].record(s_in)
        stream.wait_event(ev_x[b_])
        stream.wait_event(ev_yfree[b_])
        m.moe_forward(pf.cfg, x_dev[b_], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"],
                      inp["ws13"], inp["ws2"], out_dev[b_], None, None, stats_dev[b_][:E], None,
                      stats_dev[b_][E:E + 1], stats_dev[b_][E + 1:E + 2], None, pf.ws, stream)
        ev_xfree[b_].record(stream)
        ev_y[b_].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_y[b_])
            out_host[b_].copy_(out_dev[b_], non_blocking=True)
            stats_host[b_].copy_(stats_dev[b_], non_blocking=True)
            ev_yfree[b_].record(s_out)

    for i in range(3):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        e2e_step(i)
    e1.record(s_out)
    barrier()
    ms = max_over(e0.elapsed_time(e1)) / steps
    # the pipelined copies must deliver the same output as a plain forward
    torch.cuda.synchronize()
    if not torch.equal(out_host[(steps - 1) % 2], pf.out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-timed forward")
    pf.check()
    h2d = x_host[0].numel() * x_host[0].element_size()
    d2h = out_host[0].numel() * out_host[0].element_size() + stats_host[0].numel() * 4
    return ms, h2d, d2h


def prefill_extra(m, name, steps, warmup, dev, stream, peaks, peak_kind):
    """One more prefill layer, timed like the headline (no end-to-end leg): its own weights,
    generated on the device and freed afterwards."""
    import torch
    import moe_inputs
    wl = moe_inputs.workload(name)
    inp = moe_inputs.make_inputs(wl, device="cuda")
    pf = Prefill(m, wl, inp, dev, stream)
    ms_total, gemm_ms, clocks = pf.timed(steps, warmup, torch.cuda.synchronize)
    ms_step = ms_total / steps
    res = {"workload": workload_config(wl, 1)["workload"], "value": wl.T / (ms_step / 1e3),
           "unit": "tokens/s", "steps": steps, "ms_per_step": ms_step,
           **prefill_figures(wl, ms_step, gemm_ms, clocks, peaks, peak_kind),
           "n_dropped": int(pf.nd.item()) if wl.routing == "token_choice" else None,
           "f_max": float(pf.f.max().item()), "l_balance": float(pf.lb.item()),
           "z_loss": float(pf.z.item()), "clocks": clocks}
    del pf, inp
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v3")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extras", default="mixtral,mixtral_collapsed,dsmoe16b,dsmoe16b_ec",
                    help="further prefill layers reported under per_config ('none': skip)")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--extra-decode", default="v3:1,8,64,256;mixtral:1,8,64,256",
                    help="decode batches reported under decode ('none': skip)")
    ap.add_argument("--extra-decode-steps", type=int, default=20)
    ap.add_argument("--decode-sweep", action="store_true",
                    help="decode-sized batches instead of the prefill step (one line per B)")
    ap.add_argument("--decode-workloads", default="v3,mixtral")
    ap.add_argument("--decode-batches", default="1,8,64,256")
    ap.add_argument("--decode-steps", type=int, default=100)
    ap.add_argument("--fp8", action="store_true",
                    help="decode sweep: E4M3 expert weights (moe_forward_fp8)")
    ap.add_argument("--no-graphs", action="store_true",
                    help="decode sweep: launch each forward directly instead of a CUDA graph")
    ap.add_argument("--router-backward", action="store_true",
                    help="time the router-side backward instead of the forward (one line per "
                         "workload)")
    ap.add_argument("--backward-workloads", default="mixtral,dsmoe16b,v3")
    ap.add_argument("--backward-steps", type=int, default=50)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (smaller cases for profiler captures; not a bench line)")
    args = ap.parse_args()

    if args.decode_sweep:
        decode_sweep(args)
        return
    if args.router_backward:
        router_backward_sweep(args)
        return

    import torch
    import moe_inputs

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = moe_inputs.workload(args.workload)
    if args.tokens:
        wl = wl.replace(T=args.tokens)
    if args.experts:
        wl = wl.replace(E=args.experts)
    peaks, peak_kind = load_peaks()
    config = workload_config(wl, world)

    if args.impl == "reference":
        if runs_reference_arm(rank):
            run_reference_arm(args, wl, config)
        return

    import top_routing_expert_scoring_b300 as m
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    inp = moe_inputs.make_inputs(wl, seed=rank, device="cuda")
    pf = Prefill(m, wl, inp, dev, stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def max_over(ms):
        return max_over_ranks(ms, dev)

    ms_local, gemm_ms, clocks = pf.timed(args.steps, args.warmup, barrier)
    ms_total = max_over(ms_local)
    ms_step = ms_total / args.steps
    value = job_tokens_per_s(world, wl.T, args.steps, ms_total)
    e2e_ms, h2d, d2h = e2e_leg(m, pf, args.steps, barrier, max_over)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded i.i.d. normal tokens and random-init expert weights)",
        "config": config,
        **prefill_figures(wl, ms_step, gemm_ms, clocks, peaks, peak_kind),
        "e2e": {"value": world * wl.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelining": "double-buffered H2D / forward / D2H on three streams"},
        "gpu_launches": launches_per_step(wl) * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        S, times = run_cpu_baseline(wl, inp)
        res["cpu_baseline"] = {"value": S * len(times) / sum(times), "unit": "tokens/s",
                               "cores": cpu_cores(), "kind": "oracle",
                               "sample": f"independent batch of the first {S} tokens, "
                                         f"{len(times)} pass(es), {sum(times):.1f} s of "
                                         f"plain C++ oracle work (double accumulation)"}
    # The extra keys run after the headline's timed regions (and only on a single GPU).
    if world == 1:
        hbm = float(peaks["hbm_gbs"])
        dec = {}
        plan = {}
        if args.extra_decode != "none":
            for part in args.extra_decode.split(";"):
                name, bs = part.split(":")
                plan[name] = [int(b) for b in bs.split(",")]
        if wl.name in plan:
            # the headline's expert weights serve its decode batches
            for B in plan.pop(wl.name):
                dec[f"{wl.name} B={B}"] = decode_case(m, wl, inp, B, args.extra_decode_steps,
                                                      hbm, peak_kind)
        del pf, inp
        torch.cuda.empty_cache()
        for name, bs in plan.items():
            wl0 = moe_inputs.workload(name)
            weights = moe_inputs.make_expert_weights(wl0, device="cuda")
            for B in bs:
                dec[f"{name} B={B}"] = decode_case(m, wl0, weights, B, args.extra_decode_steps,
                                                   hbm, peak_kind)
            del weights
            torch.cuda.empty_cache()
        if dec:
            res["decode"] = dec
        if args.extras != "none":
            res["per_config"] = {name: prefill_extra(m, name, args.extra_steps, args.warmup, dev,
                                                     stream, peaks, peak_kind)
                                 for name in args.extras.split(",")}
    print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
