"""Benchmark of the routed-expert MoE layer on one GB300 (sm_103a).

Default workload: decode of one token through 40 stacked independent MoE layers
of 256 experts, top-8, d_model 2048, d_ff 768 (Qwen3.6-35B-A3B-shaped), int8
symmetric per-block-32 weights with fp16 scales, bf16 activations, Zipf(1.1)
router bias. One step = router GEMV + fp32 softmax + top-k + gathered gate/up +
SwiGLU + per-slot down + weighted combine + residual, for all 40 layers; the
last layer's output is fed back as the next step's input (a new token each
step). Inputs are seeded and synthetic (data="synthetic").

Prints ONE JSON line (rank 0). With --impl reference the CPU oracle is timed on
a bounded sample of the same workload instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "MoE-layer decode tokens/s and routed-expert HBM GB/s (% of GB300 peak), 1 GPU"
L2_BYTES = 129 * 1024 * 1024


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ decode

class DecodeStack:
    """40 layers resident in HBM, one token per step, residual chain."""

    def __init__(self, cfg: W.LayerConfig, dev, T: int = 1, layers: int = None):
        import moe_routed_expert_route_gb300 as M
        self.M = M
        self.cfg = cfg
        self.T = T
        self.L = layers or cfg.layers
        self.dev = dev
        self.layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(self.L)]
        self.routers = [M.Router(lw["Wr"], lw["bias"], cfg.k) for lw in self.layers]
        self.experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in self.layers]
        D = cfg.D
        self.X = [torch.empty(T, D, dtype=cfg.x_dtype, device=dev) for _ in range(self.L + 1)]
        self.X[0].copy_(W.make_tokens(cfg, T, 0, dev))
        self.idx = [torch.empty(T, cfg.k, dtype=torch.int32, device=dev) for _ in range(self.L)]
        self.w = [torch.empty(T, cfg.k, dtype=torch.float32, device=dev) for _ in range(self.L)]
        self.y = [torch.empty(T, D, dtype=torch.float32, device=dev) for _ in range(self.L)]
        self.ws = M.workspace(M.MOE_OP_LAYER, T, cfg.k, cfg.E, cfg.D, cfg.F, dev)
        self.graph = None

    def forward(self, feedback: bool = True):
        M = self.M
        for l in range(self.L):
            M.moe_layer(self.routers[l], self.experts[l], self.X[l], self.idx[l], self.w[l], None,
                        self.y[l], self.X[l + 1], self.ws)
        if feedback:
            self.X[0].copy_(self.X[self.L])

    def capture(self, stream):
        with torch.cuda.stream(stream):
            self.forward()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.forward()
        self.graph = g
        return g

    def kernels_per_step(self):
        return self.L  # one persistent layer launch per layer at T = 1

    def routed_bytes_per_step(self):
        """Algorithmic bytes: codes + scales of the distinct routed experts."""
        per_expert = W.routed_bytes_per_expert(self.cfg)
        total = 0
        for l in range(self.L):
            total += int(torch.unique(self.idx[l]).numel()) * per_expert
        return total


def time_graph(stack, stream, steps, warmup, world):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            stack.graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            stack.graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    if world > 1:
        t = torch.tensor([ms], device=stack.dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
        torch.distributed.barrier()
    return ms


def time_e2e(stack, stream, steps, warmup):
    """Host buffers: pinned x in, last layer's output back to the host, per step."""
    T, D = stack.T, stack.cfg.D
    n = max(1, min(steps, 256))
    xin = W.make_tokens(stack.cfg, T * n, 5, "cpu").reshape(n, T, D).pin_memory()
    xout = torch.empty(n, T, D, dtype=stack.cfg.x_dtype).pin_memory()

    def one(i):
        stack.X[0].copy_(xin[i % n], non_blocking=True)
        stack.graph.replay()
        xout[i % n].copy_(stack.X[stack.L], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    with torch.cuda.stream(stream):
        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            one(i)
        t1 = time.perf_counter()
    h2d = xin[0].numel() * xin.element_size()
    d2h = xout[0].numel() * xout.element_size()
    return (t1 - t0) * 1e3, h2d, d2h


def cpu_baseline_decode(stack, budget_s=15.0):
    """The oracle, as it stands, on the GB300 host's cores: tokens through all
    layers, as many as fit in about `budget_s` seconds (at least one)."""
    import oracle
    cfg = stack.cfg
    nth = os.cpu_count() or 1
    host = [(lw["Wr"].cpu(), lw["bias"].cpu() if lw["bias"] is not None else None) for lw in stack.layers]
    x = W.make_tokens(cfg, stack.T, 9, "cpu").double().numpy()
    tokens = 0
    t0 = time.perf_counter()
    while True:
        xl = x
        for l in range(stack.L):
            r = oracle.router(xl, host[l][0], host[l][1], cfg.k)
            y = oracle.moe(stack.layers[l], xl, r["idx"], r["w"], cfg.qbits, nthreads=nth)
            xl = torch.from_numpy(xl + y).to(torch.bfloat16).double().numpy()
        tokens += stack.T
        el = time.perf_counter() - t0
        if el >= budget_s or tokens >= 64:
            break
        x = xl
    return tokens / el, nth, f"{tokens} token(s) x {stack.L} layers (router + routed experts), {el:.1f} s"


def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    cfg = W.CONFIGS[1]
    stack = DecodeStack(cfg, dev, T=1, layers=args.layers)
    stream = torch.cuda.Stream(dev)
    stack.capture(stream)
    steps, warmup = args.steps, max(3, args.warmup)
    with ClockSampler(local) as clk:
        ms = time_graph(stack, stream, steps, warmup, world)
    status = stack.M.moe_check_status(stack.ws)
    assert status == 0, f"device status {status}"
    ms_step = ms / steps
    tok_s = world * stack.T * steps / (ms / 1e3)
    routed = stack.routed_bytes_per_step()
    hbm_peak, tf_peak, peak_kind = peaks()
    layer_us = ms_step * 1e3 / stack.L
    per_layer_bytes = routed / stack.L
    achieved = per_layer_bytes / (layer_us * 1e-6) / 1e9
    e2e_ms, h2d, d2h = time_e2e(stack, stream, min(steps, 2000), warmup)
    e2e = world * stack.T * min(steps, 2000) / (e2e_ms / 1e3)
    line = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 weights x bf16 activations, int32/fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": f"decode: 1 token x {stack.L} layers, E=256 top-8 D=2048 F=768, int8 sym "
                               "blk32 fp16 scales, bf16 x, Zipf(1.1) router bias",
                   "T": stack.T, "layers": stack.L, "E": cfg.E, "k": cfg.k, "D": cfg.D, "F": cfg.F,
                   "routed_bytes_per_token": routed // stack.T,
                   "routed_gbs": round(routed / (ms_step * 1e-3) / 1e9, 1),
                   "l2": f"no flush: {routed / 1e9:.2f} GB of distinct weights per step > "
                         f"{L2_BYTES / 2**20:.0f} MiB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "graph": "one CUDA graph per step, programmatic dependent launch between kernels"},
        "roofline": {"bound": "hbm", "kernel": "fused_layer_kernel (one launch = one whole layer)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                     "per_launch_bytes": int(per_layer_bytes), "per_launch_us": round(layer_us, 3),
                     "traffic": None},
        "e2e": {"value": round(e2e, 2), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": stack.kernels_per_step() * steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline_decode(stack, args.cpu_budget)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The CPU oracle on a bounded sample of the same workload."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = W.CONFIGS[1]
    L = cfg.layers
    nth = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(L)]
    host = [(lw["Wr"].cpu(), lw["bias"].cpu()) for lw in layers]
    x0 = W.make_tokens(cfg, 1, 0, "cpu").double().numpy()

    def step(x):
        for l in range(L):
            r = oracle.router(x, host[l][0], host[l][1], cfg.k)
            y = oracle.moe(layers[l], x, r["idx"], r["w"], cfg.qbits, nthreads=nth)
            x = torch.from_numpy(x + y).to(torch.bfloat16).double().numpy()
        return x

    x = x0
    for _ in range(max(0, min(args.warmup, 1))):
        x = step(x)
    steps = max(1, min(args.steps, 8))
    t0 = time.perf_counter()
    for _ in range(steps):
        x = step(x)
    el = time.perf_counter() - t0
    v = steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode: 1 token x 40 layers, E=256 top-8 D=2048 F=768, int8 sym "
                               "blk32 fp16 scales, bf16 x, Zipf(1.1) router bias"},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": nth, "kind": "oracle",
                         "sample": f"{steps} token(s) x {L} layers"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=None,
                    help="stacked layers (default: the workload's 40); fewer only for profiling captures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
