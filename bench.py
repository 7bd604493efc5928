"""Benchmark of the routed-expert MoE layer on one GB300 (sm_103a).

Default workload: decode of one token through 40 stacked independent MoE layers
of 256 experts, top-8, d_model 2048, d_ff 768 (Qwen3.6-35B-A3B-shaped), int8
symmetric per-block-32 weights with fp16 scales, bf16 activations, Zipf(1.1)
router bias. One step = router GEMV + fp32 softmax + top-k + gathered gate/up +
SwiGLU + per-slot down + weighted combine + residual, for all 40 layers. The
layers are independent: in each step every layer takes its own token, drawn
from a device-resident bank of distinct seeded tokens (data="synthetic").

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

# DRAM bytes (read + write) of one launch of the single-token layer kernel on
# the default workload: dram__bytes_read.sum + dram__bytes_write.sum from one
# ncu capture of that launch
LAYER_KERNEL_DRAM_BYTES = 41_244_928 + 5_120

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
                 "-lms", "500", "-i", str(self.index)],
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
    """40 layers resident in HBM; per step every layer decodes its own token."""

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
        self._buffers(T)
        self.graph = self.graph_e2e = None
        torch.cuda.synchronize()  # setup ran on the default stream; the steps run on another

    def _buffers(self, T):
        """Per-step buffers for T tokens. The layers are independent (each has
        its own weights): layer l of a step takes its own token batch, drawn
        from a bank of distinct synthetic tokens on the device, and writes
        x_next = x + y. (Feeding x_next of one layer into the next, without the
        normalisation a real model applies between layers, lets the residual
        stream of some tokens grow without bound through 40 random layers.)"""
        cfg, dev, M, L, D = self.cfg, self.dev, self.M, self.L, self.cfg.D
        self.T = T
        self.XIN = torch.empty(L, T, D, dtype=cfg.x_dtype, device=dev)
        self.XN = torch.empty(L, T, D, dtype=cfg.x_dtype, device=dev)
        self.idx = [torch.empty(T, cfg.k, dtype=torch.int32, device=dev) for _ in range(L)]
        self.w = [torch.empty(T, cfg.k, dtype=torch.float32, device=dev) for _ in range(L)]
        self.y = [torch.empty(T, D, dtype=torch.float32, device=dev) for _ in range(L)]
        self.ws = M.workspace(M.MOE_OP_LAYER, T, cfg.k, cfg.E, cfg.D, cfg.F, dev)
        # step i uses bank entry i mod NB: every step routes new tokens
        self.NB = 16 if T > 8 else 64
        self.bank = W.make_tokens(cfg, self.NB * L * T, 1, dev).reshape(self.NB, L, T, D)
        self.XIN.copy_(self.bank[0])
        self.ctr = torch.zeros(1, dtype=torch.long, device=dev)

    def forward(self, from_bank: bool = True):
        M = self.M
        if from_bank:
            torch.index_select(self.bank, 0, self.ctr, out=self.XIN.view(1, self.L, self.T, -1))
            self.ctr.add_(1).remainder_(self.NB)
        for l in range(self.L):
            M.moe_layer(self.routers[l], self.experts[l], self.XIN[l], self.idx[l], self.w[l], None,
                        self.y[l], self.XN[l], self.ws)

    def capture(self, stream):
        with torch.cuda.stream(stream):
            self.forward()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.forward()
        self.graph = g
        g2 = torch.cuda.CUDAGraph()  # the same layers without the bank: inputs come from the host
        with torch.cuda.graph(g2, stream=stream):
            self.forward(from_bank=False)
        self.graph_e2e = g2
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
        ms = max_over_ranks(ms, stack.dev)
    return ms


def max_over_ranks(ms: float, dev) -> float:
    """The slowest rank's time (replicas: the job ends when the last one does);
    every rank returns it. Needs an initialised process group."""
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput of N replicas: units all ranks processed / the
    slowest rank's time."""
    return world * units_per_rank / (ms / 1e3)


def time_e2e(stack, stream, steps, warmup):
    """Host buffers: each step's layer inputs copied in from pinned host memory,
    the last layer's x_next read back to the host."""
    T, D, L = stack.T, stack.cfg.D, stack.L
    n = max(1, min(steps, 16))
    xin = W.make_tokens(stack.cfg, n * L * T, 5, "cpu").reshape(n, L, T, D).pin_memory()
    xout = torch.empty(n, T, D, dtype=stack.cfg.x_dtype).pin_memory()

    def one(i):
        stack.XIN.copy_(xin[i % n], non_blocking=True)
        stack.graph_e2e.replay()
        xout[i % n].copy_(stack.XN[L - 1], non_blocking=True)
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
    xs = W.make_tokens(cfg, stack.T * stack.L, 9, "cpu").double().numpy().reshape(stack.L, stack.T, -1)
    tokens = 0
    t0 = time.perf_counter()
    while True:
        for l in range(stack.L):  # independent layers, each with its own token batch
            r = oracle.router(xs[l], host[l][0], host[l][1], cfg.k)
            oracle.moe(stack.layers[l], xs[l], r["idx"], r["w"], cfg.qbits, nthreads=nth)
        tokens += stack.T
        el = time.perf_counter() - t0
        if el >= budget_s or tokens >= 64:
            break
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
    tok_s = job_throughput(stack.T * steps, world, ms)
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
                   "inputs": "independent layers: each layer decodes its own bank token every step",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "graph": "one CUDA graph per step, programmatic dependent launch between kernels"},
        "roofline": {"bound": "hbm", "kernel": "fused_layer_kernel (one launch = one whole layer)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                     "per_launch_bytes": int(per_layer_bytes), "per_launch_us": round(layer_us, 3),
                     # measured DRAM bytes of one launch of this kernel, per launch like achieved
                     "traffic": LAYER_KERNEL_DRAM_BYTES, "traffic_unit": "bytes per launch"},
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


# ------------------------------------------------- secondary workloads
# (measured on request with --workload; the default line is the decode step)

def _time_graph_simple(g, stream, steps, warmup):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_batched(args, dev):
    """Batched decode over the 40-layer stack, T in {1,...,64}."""
    cfg = W.CONFIGS[2]
    per_expert = W.routed_bytes_per_expert(cfg)
    out = []
    stack = None
    for T in (1, 2, 4, 8, 16, 32, 64):
        if stack is None:
            stack = DecodeStack(cfg, dev, T=T, layers=args.layers)
        else:  # same weights, new token batch
            stack._buffers(T)
            torch.cuda.synchronize()
        stream = torch.cuda.Stream(dev)
        stack.capture(stream)
        ms = _time_graph_simple(stack.graph, stream, max(10, args.steps // 4), max(3, args.warmup))
        U = [int(torch.unique(stack.idx[l]).numel()) for l in range(stack.L)]
        routed = sum(U) * per_expert
        out.append({"T": T, "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
                    "union_experts_mean": round(sum(U) / len(U), 2), "union_min": min(U), "union_max": max(U),
                    "routed_gbs": round(routed / (ms * 1e-3) / 1e9, 1)})
        st = stack.M.moe_check_status(stack.ws)
        assert st == 0, f"T={T}: device status {st} ({stack.M.status_string(st)})"
    return {"workload": "batched decode sweep, 40 layers E=256 top-8 D=2048 F=768 int8", "points": out}


def run_substitution(args, dev):
    """Residency substitution (0.15 rule) + int4 decode, 512 experts top-10, 16 layers."""
    import moe_routed_expert_route_gb300 as M
    cfg = W.CONFIGS[3]
    L = args.layers or cfg.layers
    layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(L)]
    masks = [W.make_resident_mask(cfg, l, dev) for l in range(L)]
    per_expert = W.routed_bytes_per_expert(cfg)
    res = []
    for T in (1, 16):
        k = cfg.k
        # independent layers: each takes its own token batch from a device bank
        XIN = torch.empty(L, T, cfg.D, dtype=cfg.x_dtype, device=dev)
        XN = torch.empty(L, T, cfg.D, dtype=cfg.x_dtype, device=dev)
        bufs = [dict(idx=torch.empty(T, k, dtype=torch.int32, device=dev), w=torch.empty(T, k, device=dev),
                     probs=torch.empty(T, cfg.E, device=dev), idx2=torch.empty(T, k, dtype=torch.int32, device=dev),
                     w2=torch.empty(T, k, device=dev), flag=torch.empty(T, k, dtype=torch.uint8, device=dev),
                     mass=torch.empty(T, device=dev), y=torch.empty(T, cfg.D, device=dev)) for _ in range(L)]
        ws_r = M.workspace(M.MOE_OP_ROUTE, T, k, cfg.E, cfg.D, cfg.F, dev)
        ws_d = M.workspace(M.MOE_OP_DECODE, T, k, cfg.E, cfg.D, cfg.F, dev)
        routers = [M.Router(lw["Wr"], lw["bias"], k) for lw in layers]
        experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in layers]
        NB = 16 if T > 8 else 64
        bank = W.make_tokens(cfg, NB * L * T, 1, dev).reshape(NB, L, T, cfg.D)
        ctr = torch.zeros(1, dtype=torch.long, device=dev)
        torch.cuda.synchronize()  # setup ran on the default stream; the steps run on another

        def step():
            torch.index_select(bank, 0, ctr, out=XIN.view(1, L, T, -1))
            ctr.add_(1).remainder_(NB)
            for l in range(L):
                b = bufs[l]
                M.moe_route(routers[l], XIN[l], b["idx"], b["w"], b["probs"], ws_r)
                M.moe_substitute(b["probs"], b["idx"], b["w"], masks[l], cfg.threshold, b["idx2"], b["w2"],
                                 b["flag"], b["mass"])
                M.moe_decode(experts[l], XIN[l], b["idx2"], b["w2"], b["y"], XN[l], ws_d)

        stream = torch.cuda.Stream(dev)
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        ms = _time_graph_simple(g, stream, max(10, args.steps // 4), max(3, args.warmup))
        U = [int(torch.unique(bufs[l]["idx2"]).numel()) for l in range(L)]
        flags = torch.stack([b["flag"] for b in bufs]).cpu()
        mass = torch.stack([b["mass"] for b in bufs]).cpu()
        res.append({"T": T, "layers": L, "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
                    "us_per_layer": round(ms * 1e3 / L, 2), "distinct_experts_mean": round(sum(U) / L, 2),
                    "routed_gbs": round(sum(U) * per_expert / (ms * 1e-3) / 1e9, 1),
                    "substituted_frac": round(float((flags == 2).float().mean()), 4),
                    "fetched_miss_frac": round(float((flags == 1).float().mean()), 4),
                    "mass_mean": round(float(mass.mean()), 4), "mass_max": round(float(mass.max()), 4)})
        assert M.moe_check_status(ws_d) == 0
    return {"workload": "substitution 0.15 rule + int4 decode, E=512 top-10 D=2048 F=512, 25% resident",
            "points": res}


def run_prefill(args, dev, T=None):
    """Prefill of T tokens (default 2048), rotating over 4 layers (5 GB of weights)."""
    import moe_routed_expert_route_gb300 as M
    cfg = W.CONFIGS[4]
    T = T or cfg.T
    L = args.layers or 4
    layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(L)]
    routers = [M.Router(lw["Wr"], lw["bias"], cfg.k) for lw in layers]
    experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in layers]
    x = W.make_tokens(cfg, T, 0, dev)
    y = torch.empty(T, cfg.D, device=dev)
    idx = torch.empty(T, cfg.k, dtype=torch.int32, device=dev)
    w = torch.empty(T, cfg.k, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    ws = M.workspace(M.MOE_OP_PREFILL, T, cfg.k, cfg.E, cfg.D, cfg.F, dev)
    torch.cuda.synchronize()  # setup ran on the default stream; the steps run on another
    stream = torch.cuda.Stream(dev)

    def step(l):
        M.moe_prefill(routers[l], experts[l], x, y, idx, w, counts, None, ws)

    with torch.cuda.stream(stream):
        for l in range(L):
            step(l)
    torch.cuda.synchronize()
    U = int((counts > 0).sum())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l in range(L):
            step(l)
    ms = _time_graph_simple(g, stream, max(5, args.steps // 40), max(3, args.warmup)) / L
    flops = 2.0 * T * cfg.k * 3 * cfg.D * cfg.F
    wbytes = U * W.routed_bytes_per_expert(cfg)
    hbm, tf, kind = peaks()
    assert M.moe_check_status(ws) == 0
    return {"workload": f"prefill T={T} E=256 top-8 D=2048 F=768 int8 (fp16 tensor-core operands)",
            "T": T, "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_layer": round(ms, 4),
            "distinct_experts": U, "expert_weight_gb": round(wbytes / 1e9, 3),
            "expert_tflops": round(flops / (ms * 1e-3) / 1e12, 1), "tensor_frac_of_peak": round(flops / (ms * 1e-3) / 1e12 / tf, 4),
            "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1), "weight_frac_of_hbm_peak": round(wbytes / (ms * 1e-3) / 1e9 / hbm, 4)}


def run_workload(args):
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import __graft_entry__
    __graft_entry__.build()
    if args.workload == "batched":
        r = run_batched(args, dev)
    elif args.workload == "substitution":
        r = run_substitution(args, dev)
    else:
        r = run_prefill(args, dev)
        if args.prefill_extra:
            r["extra"] = run_prefill(args, dev, T=16384)
    print(json.dumps(r), flush=True)


def run_reference(args):
    """The CPU oracle on a bounded sample of the same workload."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = W.CONFIGS[1]
    L = args.layers or cfg.layers
    nth = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(L)]
    host = [(lw["Wr"].cpu(), lw["bias"].cpu()) for lw in layers]
    # independent layers, each with its own token, as in the GPU arm
    xs = W.make_tokens(cfg, L, 0, "cpu").double().numpy().reshape(L, 1, -1)

    def step(threads):
        for l in range(L):
            r = oracle.router(xs[l], host[l][0], host[l][1], cfg.k)
            oracle.moe(layers[l], xs[l], r["idx"], r["w"], cfg.qbits, nthreads=threads)

    for _ in range(max(0, min(args.warmup, 1))):
        step(nth)
    steps = max(1, min(args.steps, 8))
    t0 = time.perf_counter()
    for _ in range(steps):
        step(nth)
    el = time.perf_counter() - t0
    t1 = time.perf_counter()
    step(1)  # one step on one thread, for scale
    el1 = time.perf_counter() - t1
    v = steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"decode: 1 token x {L} layers, E=256 top-8 D=2048 F=768, int8 sym "
                               "blk32 fp16 scales, bf16 x, Zipf(1.1) router bias",
                   "inputs": "independent layers: each layer decodes its own token every step"},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": nth, "kind": "oracle",
                         "sample": f"{steps} token(s) x {L} layers",
                         "single_thread": {"value": round(1.0 / el1, 4), "unit": "tokens/s", "cores": 1,
                                           "sample": f"1 token x {L} layers"}},
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
    ap.add_argument("--workload", default="decode", choices=["decode", "batched", "substitution", "prefill"],
                    help="decode (default, the headline line) or a secondary workload")
    ap.add_argument("--prefill-extra", action="store_true", help="also time a 16384-token prefill")
    ap.add_argument("--layers", type=int, default=None,
                    help="stacked layers (default: the workload's 40); fewer only for profiling captures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "decode":
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
