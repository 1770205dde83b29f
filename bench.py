"""Benchmark of the single-GPU MoE layer forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixtral] [--no-cpu-baseline]

One step = one whole layer forward (router GEMM, scoring/Top-k, statistics, dispatch, grouped
SwiGLU expert GEMMs, shared experts, combine) over one batch of synthetic tokens already in HBM.
The timed step is moe_forward_timed: moe_forward's kernels, with two CUDA events recorded
around the expert GEMM launches so that the grouped GEMM's share is measured live.
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


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the grouped GEMM's two launches
# in one step, from an ncu capture of the bench command on the current kernel build
# (profiles/launches_mixtral_t4096_bench.md); None for a workload without a capture.
GEMM_TRAFFIC_BYTES = {("mixtral", 4096): (1946556672 + 224120832) + (1557085440 + 125510656)}


def workload_flops_bytes(wl):
    """Algorithmic FLOPs and bytes of one layer forward (per step).

    FLOPs = T * (2 d E  +  (k + shared) * 3 * 2 d F)  (router + SwiGLU experts)
    bytes = touched expert weights + router weights + x read + out write.
    """
    T, d, E, k, F, Fs = wl.T, wl.d, wl.E, wl.k, wl.F, wl.F_sh
    ffn = T * k * 3 * 2 * d * F + T * 3 * 2 * d * Fs
    router = T * 2 * d * E
    weights = (E * 3 * d * F + 3 * d * Fs + E * d) * 2
    act = 2 * T * d * 2
    return {"flops": ffn + router, "ffn_flops": ffn, "bytes": weights + act}


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
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
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
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(wl, inp_host, S):
    """The oracle (as it stands) on an independent batch of the first S tokens."""
    from oracle import moe_oracle as O
    h = dict(inp_host)
    h["x"] = h["x"][:S]
    sub = wl.replace(T=S)
    t0 = time.perf_counter()
    if wl.routing == "expert_choice":
        O.moe_forward_expert_choice(sub, h["x"], h["w_gate"], h["w13"], h["w2"], h["ws13"],
                                    h["ws2"])
    else:
        O.moe_forward(sub, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    return time.perf_counter() - t0


def host_inputs(inp):
    import moe_inputs
    return {k: moe_inputs.to_f64(v) for k, v in inp.items()}


def run_cpu_baseline(wl, inp, target_s=12.0, max_reps=8):
    """Sizes the oracle's sample so that it takes about target_s seconds (two probe sizes give
    the per-token cost) and times it; when even the whole batch is shorter, the batch is timed
    again until about target_s has passed (at most max_reps passes)."""
    hi = host_inputs(inp)
    s1, s2 = min(32, wl.T), min(256, wl.T)
    t1 = oracle_sample(wl, hi, s1)
    t2 = oracle_sample(wl, hi, s2) if s2 > s1 else t1
    per_tok = max((t2 - t1) / max(s2 - s1, 1), 1e-6)
    S = int(min(wl.T, max(s2, s1 + (target_s - t1) / per_tok)))
    times = [oracle_sample(wl, hi, S)]
    while sum(times) < target_s * 0.8 and len(times) < max_reps:
        times.append(oracle_sample(wl, hi, S))
    return S, times


def decode_sweep(args):
    """Decode-sized batches: B tokens per step, 100 seeded steps per B with fresh x and router
    weights (expert weights fixed), timed through moe_forward.  Reports tokens/s and the HBM
    bandwidth reached on the bytes a step must read: the experts it actually touches (counted
    from its own selection), the shared experts, the router, x and the output.  Also reports
    the distinct experts touched per step against E(1-(1-k/E)^B), as configured and with a
    zero selection bias (exchangeable experts, where the formula holds in expectation)."""
    import math
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
        if fp8:
            # one-byte E4M3 codes plus one fp32 scale per weight row, quantised once up front
            q = {key: (m.quantize_fp8(weights[key]) if weights[key] is not None else (None, None))
                 for key in ("w13", "w2", "ws13", "ws2")}
            torch.cuda.synchronize()
            del weights
            torch.cuda.empty_cache()
            per_expert = 3 * wl0.d * wl0.F + (2 * wl0.F + wl0.d) * 4
            shared_bytes = 3 * wl0.d * wl0.F_sh + ((2 * wl0.F_sh + wl0.d) * 4 if wl0.F_sh else 0)
        else:
            per_expert = 3 * wl0.d * wl0.F * 2
            shared_bytes = 3 * wl0.d * wl0.F_sh * 2
        for B in [int(b) for b in args.decode_batches.split(",")]:
            wl = wl0.replace(T=B)
            cfg = m.make_config(B, wl.d, wl.E, wl.k, wl.F, wl.F_sh, wl.score, wl.routing,
                                wl.n_groups, wl.topk_groups, wl.renormalize, wl.route_scale,
                                wl.capacity_factor, wl.dtype)
            steps = args.decode_steps
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
                    m.moe_forward(cfg, r["x"], r["w_gate"], r["bias"], weights["w13"],
                                  weights["w2"], weights["ws13"], weights["ws2"], out,
                                  topk_idx=idx_all[i], ws=ws)
            for i in range(min(5, steps)):
                fwd(i)
            torch.cuda.synchronize()
            graphs = []
            if not args.no_graphs:
                # one CUDA graph per step (its own inputs), captured outside the timed region
                for i in range(steps):
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr):
                        fwd(i)
                    graphs.append(gr)
                torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
            with ClockSampler(torch.cuda.current_device()) as clk:
                clk.start()
                ev[0].record()
                for i in range(steps):
                    if graphs:
                        graphs[i].replay()
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
            cfg0 = cfg
            logits = torch.empty((B, wl.E), dtype=torch.float32, device="cuda")
            w0 = torch.empty((B, wl.k), dtype=torch.float32, device="cuda")
            dz = []
            for i in range(steps):
                r = moe_inputs.make_router_inputs(zero, seed=5000 + i, device="cuda")
                m.moe_router_topk(cfg0, r["x"], r["w_gate"], None, logits, idx_all[i], w0, ws)
                dz.append(int(torch.unique(idx_all[i]).numel()))
            formula = wl.E * (1 - (1 - wl.k / wl.E) ** B)
            mean_z = sum(dz) / len(dz)
            se_z = (sum((v - mean_z) ** 2 for v in dz) / max(len(dz) - 1, 1)) ** 0.5 / math.sqrt(len(dz))
            print(json.dumps({
                "metric": "MoE layer fwd tokens/s, decode batch; % of HBM BW on touched expert "
                          "weights", "mode": "decode_fp8" if fp8 else "decode",
                "workload": f"{name} B={B}",
                "value": B * steps / total_s, "unit": "tokens/s", "steps": steps,
                "ms_per_step": sum(ms) / steps,
                "dtype": "e4m3 expert weights and activations, bf16 router" if fp8 else "bf16",
                "data": "synthetic",
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                             "frac": gbs / hbm, "peak_kind": f"{peak_kind} copy bandwidth"},
                "bytes_per_step_mean": sum(step_bytes) / steps,
                "distinct_experts": {"as_configured_mean": sum(distinct) / steps,
                                     "zero_bias_mean": mean_z, "zero_bias_se": se_z,
                                     "formula": formula},
                "clocks": clk.summary(), "cuda_graphs": bool(graphs),
                "l2": "each step reads >= 0.35 GB of expert weights (> 126 MB L2)"}))
            del routers, ws, graphs
            torch.cuda.empty_cache()
        if fp8:
            del q
        else:
            del weights
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
    """Router-side backward (dL/dg, dW_gate, dx) per workload: CUDA events around each call, L2
    flushed (256 MB write) between calls outside the events.  The routing inputs come from the
    forward's own router call."""
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
        reps = args.backward_steps
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.start()
            for a, b in ev:
                flush.fill_(1)
                a.record()
                call()
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
    flops = workload_flops_bytes(wl)
    peaks, peak_kind = load_peaks()
    config = {"workload": f"{wl.name}-shaped MoE layer: T={wl.T} d={wl.d} E={wl.E} k={wl.k} "
                          f"F={wl.F} shared={wl.n_shared}x{wl.F_shared} score={wl.score} "
                          f"routing={wl.routing} cf={wl.capacity_factor or 'none'}",
              "T": wl.T, "d_model": wl.d, "E": wl.E, "k": wl.k, "d_ff": wl.F,
              "shared_d_ff": wl.F_sh, "capacity_factor": wl.capacity_factor or None,
              "l2": "inputs larger than L2 (expert weights "
                    f"{wl.E * 3 * wl.d * wl.F * 2 / 1e9:.2f} GB > 126 MB)",
              "parallelism": "replicas" if world == 1 else f"replicas x{world} (token shards)"}

    if args.impl == "reference":
        if not runs_reference_arm(rank):
            return
        torch.manual_seed(0)
        inp = moe_inputs.make_inputs(wl, device="cpu")
        hi = host_inputs(inp)
        S = min(wl.T, 128)
        for _ in range(max(args.warmup, 0)):
            oracle_sample(wl, hi, min(S, 16))
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
                             "sample": f"independent batch of the first {S} tokens per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    import top_routing_expert_scoring_b300 as m
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = moe_inputs.make_inputs(wl, seed=rank, device="cuda")
    cfg = m.make_config(wl.T, wl.d, wl.E, wl.k, wl.F, wl.F_sh, wl.score, wl.routing, wl.n_groups,
                        wl.topk_groups, wl.renormalize, wl.route_scale, wl.capacity_factor,
                        wl.dtype)
    T, E, k, d = wl.T, wl.E, wl.k, wl.d
    ws = m.workspace(cfg, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    logits, idx, w = torch.empty((T, E), **f32), torch.empty((T, k), **i32), torch.empty((T, k), **f32)
    f, P, lb, z = (torch.empty(E, **f32), torch.empty(E, **f32), torch.empty(1, **f32),
                   torch.empty(1, **f32))
    nd = torch.empty(1, **i32)
    shared = wl.F_sh > 0
    out = torch.empty((T, d), **f32)      # fp32 layer output (out_dtype f32)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def step(gemm_events):
        m.moe_forward_timed(cfg, inp["x"], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"],
                            inp["ws13"], inp["ws2"], out, idx, w, f, P, lb, z, nd, ws, stream,
                            gemm_events[0], gemm_events[1])

    # our kernels per forward: router logits, Top-k (+statistics partials), dispatch (1 kernel
    # for T <= 256, else 4), 2 expert GEMMs, 2 shared-expert GEMMs, combine, statistics final.
    # A k <= 2 bf16 layer without shared experts and with a float32 output has no combine
    # kernel: the down GEMM adds the weighted rows into the output itself.
    combine_in_gemm = (wl.k <= 2 and not shared and wl.dtype == "bf16"
                       and os.environ.get("MOE_B300_COMBINE") != "separate")
    launches_per_step = (1 + 1 + (1 if T <= 256 else 4) + 2 + (2 if shared else 0)
                         + (0 if combine_in_gemm else 1) + 1)
    if wl.routing == "expert_choice":
        launches_per_step = 1 + 5 + 2 + 2 + (2 if shared else 0) + 1 + 2

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    warm_events = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for ev_ in warm_events:
        ev_.record(stream)              # torch creates the event handle on first record
    for _ in range(max(args.warmup, 3)):
        step(warm_events)
    barrier()
    st = m.sync_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st}: {m.status_string(st)}")

    gemm_pairs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                  for _ in range(args.steps)]
    for pair in gemm_pairs:
        for ev_ in pair:
            ev_.record(stream)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        clk.start()
        t_start.record(stream)
        for i in range(args.steps):
            step(gemm_pairs[i])
        t_end.record(stream)
        barrier()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), dev)
    gemm_ms = [a.elapsed_time(b) for a, b in gemm_pairs]
    ms_step = ms_total / args.steps
    value = job_tokens_per_s(world, T, args.steps, ms_total)

    # End to end through the public call with host buffers, copies inside the timed region:
    # every step copies its tokens from pinned host memory to the device, runs moe_forward and
    # copies the layer output and statistics back.  Like a serving loop, consecutive steps are
    # pipelined on three streams with double buffers: step i's host-to-device copy and step
    # i-1's device-to-host copy overlap step i's forward.
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
        m.moe_forward(cfg, x_dev[b_], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"],
                      inp["ws13"], inp["ws2"], out_dev[b_], None, None, stats_dev[b_][:E], None,
                      stats_dev[b_][E:E + 1], stats_dev[b_][E + 1:E + 2], None, ws, stream)
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
    for i in range(args.steps):
        e2e_step(i)
    e1.record(s_out)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
    # the pipelined copies must deliver the same output as a plain forward
    torch.cuda.synchronize()
    if not torch.equal(out_host[(args.steps - 1) % 2], out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-timed forward")
    st = m.sync_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st}: {m.status_string(st)}")

    if rank != 0:
        return
    gemm_avg = sum(gemm_ms) / len(gemm_ms)
    tflops = flops["ffn_flops"] / (gemm_avg / 1e3) / 1e12
    clocks = clk.summary()
    # burst peak while the GPU held its clock; the sustained (power-capped) peak only when the
    # median SM clock of the timed region sat materially below its maximum (a cap flag raised
    # now and then at full clock does not count)
    capped = bool(clocks.get("sm_mhz") and clocks.get("sm_max_mhz")
                  and clocks["sm_mhz"] < 0.95 * clocks["sm_max_mhz"])
    peak = float(peaks["bf16_tflops_sustained"] if capped and "bf16_tflops_sustained" in peaks
                 else peaks["bf16_tflops"])
    peak_name = ("bf16 sustained (timed region ran below 95% of the maximum SM clock)" if capped
                 else "bf16 burst")
    layer_roof_ms = max(flops["flops"] / (peak * 1e12), flops["bytes"] / (peaks["hbm_gbs"] * 1e9)) * 1e3
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded i.i.d. normal tokens and random-init expert weights)",
        "config": config,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak,
                     "traffic": GEMM_TRAFFIC_BYTES.get((wl.name, wl.T)),
                     "traffic_unit": "bytes per step (gate/up + down launches)",
                     "kernel": ("whole expert-choice forward" if wl.routing == "expert_choice"
                                else "grouped GEMM kernel (gate/up + down launches of one step)"),
                     "peak_kind": f"{peak_kind} {peak_name}"},
        "layer_roofline": {"roofline_ms": layer_roof_ms, "frac": layer_roof_ms / ms_step,
                           "flops_per_step": flops["flops"], "bytes_per_step": flops["bytes"]},
        "stage_ms": {"expert_ffn": gemm_avg, "rest": ms_step - gemm_avg},
        "e2e": {"value": world * T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host[0].numel() * x_host[0].element_size(),
                "d2h_bytes_per_step": out_host[0].numel() * out_host[0].element_size()
                + stats_host[0].numel() * 4,
                "ms_per_step": e2e_ms,
                "pipelining": "double-buffered H2D / forward / D2H on three streams"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        S, times = run_cpu_baseline(wl, inp)
        res["cpu_baseline"] = {"value": S * len(times) / sum(times), "unit": "tokens/s",
                               "cores": cpu_cores(), "kind": "oracle",
                               "sample": f"independent batch of the first {S} tokens, "
                                         f"{len(times)} pass(es), {sum(times):.1f} s of "
                                         f"float64 CPU work"}
    print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
