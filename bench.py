"""Benchmark of the routed-expert MoE layer on one GB300 (sm_103a).

Headline workload: decode of one token through 40 stacked independent MoE
layers of 256 experts, top-8, d_model 2048, d_ff 768 (Qwen3.6-35B-A3B-shaped),
int8 symmetric per-block-32 weights with fp16 scales, bf16 activations,
Zipf(1.1) router bias. One step = router GEMV + fp32 softmax + top-k +
gathered gate/up + SwiGLU + per-slot down + weighted combine + residual, for
all 40 layers, in one launch of the stacked single-token layer kernel: layer
l+1 starts only after every CTA has finished layer l. Every layer takes its own
token, drawn from a device-resident bank of distinct seeded tokens
(data="synthetic").

The same run also measures, under "workloads", the other configurations on
the same resident weights: the batched decode sweep (T = 1..64), residency
substitution with int4 experts (T = 1, 16) and prefill (T = 2048, 16384), each
with its roofline, the CPU oracle's rate on a bounded sample, and the clocks
seen while it ran; then the shared expert with its unmerged LoRA and the
prerouter head (T = 1, 16), the expert cache with miss fetch and
background admission (512 experts, a quarter cached in HBM), and the
prerouter's prediction staged one token ahead through a slot table.

Prints ONE JSON line (rank 0). With --impl reference the CPU oracle is timed on
a bounded sample of the headline workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
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
# moe_layer runs up to this many tokens as one single-token layer launch per token
FUSED_TOKENS = 7
# tokens (each through every layer) in the oracle's timed sample: about 9 s of
# its arithmetic on 16 cores
CPU_SAMPLE_TOKENS = 64
# tokens per step of the reference arm
REF_TOKENS_PER_STEP = 8

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# single-token layer kernel on one layer of the headline workload, from the ncu
# capture summarised in the named file. Reported only while the kernel source
# is the one that capture measured (same sha256 prefix of csrc/fused.cu).
LAYER_KERNEL_TRAFFIC = {"fused_sha16": "cc38e7ab15a5af52", "bytes_per_layer": (82_411_008 + 1_299_200) // 2,
                        "source": "profiles/fused_layer_kernel_decode_E256_k8.md"}


def fused_sha16() -> str:
    p = os.path.join(ROOT, "moe_routed_expert_route_gb300", "csrc", "fused.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained") or 0) or None,
                "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


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
                 "-lms", "200", "-i", str(self.index)],
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


def roofline(bound, achieved, peak, unit, kernel, extra=None):
    d = {"bound": bound, "kernel": kernel, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4)}
    if extra:
        d.update(extra)
    return d


# ------------------------------------------------------------------ decode

class DecodeStack:
    """`layers` layers resident in HBM; per step every layer decodes its own
    token batch. T = 1 runs the whole stack in one launch of the stacked
    single-token layer kernel; T > 1 runs one moe_layer call per layer."""

    def __init__(self, cfg: W.LayerConfig, dev, T: int = 1, layers: int = None, layer_weights=None):
        import moe_routed_expert_route_gb300 as M
        self.M = M
        self.cfg = cfg
        self.L = layers or cfg.layers
        self.dev = dev
        self.layers = layer_weights or [W.make_layer(cfg, l, dev, chunk=64) for l in range(self.L)]
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
        if self.T == 1:
            M.moe_layer_stack(self.routers, self.experts, [self.XIN[l] for l in range(self.L)], False, self.idx,
                              self.w, self.y, [self.XN[l] for l in range(self.L)], self.ws)
            return
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
        if self.T == 1:
            return 1  # one launch of the stacked layer kernel
        if self.T <= FUSED_TOKENS:
            return self.L * self.T
        return self.L * 8  # router GEMM, top-k, grouping (3), gather, two grouped products, combine

    def unions(self):
        return [int(torch.unique(self.idx[l]).numel()) for l in range(self.L)]

    def routed_bytes_per_step(self):
        """Algorithmic bytes: codes + scales of the distinct routed experts."""
        return sum(self.unions()) * W.routed_bytes_per_expert(self.cfg)


def time_graph(graph, stream, steps, warmup, world=1, dev=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ms = start.elapsed_time(end)
    if world > 1:
        ms = max_over_ranks(ms, dev)
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


# ---------------------------------------------------- CPU oracle baselines
# The oracle as it stands, on this host's cores, on a bounded sample of each
# workload (the same seeded inputs as the GPU measurement).

def _host_layer(lw):
    return (lw["Wr"].cpu(), lw["bias"].cpu() if lw["bias"] is not None else None)


_EXPERT_TENSORS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def timed_oracle_moe(layer, x, idx, w, qbits, nthreads):
    """oracle.moe on host copies of the routed experts' rows; returns the
    seconds of the oracle call alone (the device-to-host copy is not timed:
    its speed depends on the host link, not on the oracle) and y."""
    import numpy as np
    import oracle
    idx = np.asarray(idx)
    used, remap = np.unique(idx, return_inverse=True)
    sel = torch.tensor(used.astype(np.int64), device=layer["gate_q"].device)
    sub = {n: layer[n][sel].cpu() for n in _EXPERT_TENSORS}
    idx_c = remap.reshape(idx.shape).astype(np.int32)
    t0 = time.perf_counter()
    y = oracle.moe(sub, x, idx_c, w, qbits, nthreads=nthreads, compact=False)
    return time.perf_counter() - t0, y


def oracle_decode_rate(cfg, layers, ntok: int, threads: int, warmup: int = 1):
    """Tokens/s of the oracle (router + routed experts) for ntok tokens, each
    through every layer, after `warmup` tokens. The device weights' rows of
    the experts a token routes to are copied to the host outside the timed
    region, so the figure is the oracle's arithmetic on host data (the copy's
    speed depends on the host link, not on the oracle)."""
    import oracle
    host = [_host_layer(lw) for lw in layers]
    L = len(layers)
    xs = W.make_tokens(cfg, (ntok + warmup) * L, 9, "cpu").double().numpy().reshape(ntok + warmup, L, 1, -1)

    def token(i):
        el = 0.0
        for l in range(L):
            t0 = time.perf_counter()
            r = oracle.router(xs[i, l], host[l][0], host[l][1], cfg.k)
            el += time.perf_counter() - t0
            el += timed_oracle_moe(layers[l], xs[i, l], r["idx"], r["w"], cfg.qbits, threads)[0]
        return el

    for i in range(warmup):
        token(i)
    el = sum(token(i) for i in range(warmup, warmup + ntok))
    return ntok / el, el


def cpu_baseline_decode(cfg, layers, ntok=8, single=True):
    nth = os.cpu_count() or 1
    v, el = oracle_decode_rate(cfg, layers, ntok, nth)
    out = {"value": round(v, 4), "unit": "tokens/s", "cores": nth, "kind": "oracle",
           "sample": f"{ntok} tokens x {len(layers)} layers (router + routed experts, fp64, on host copies "
                     f"of the routed experts' rows; the copies are not timed) after 1 warm-up token, {el:.1f} s"}
    if single:
        v1, el1 = oracle_decode_rate(cfg, layers, 1, 1, warmup=0)
        out["single_thread"] = {"value": round(v1, 4), "unit": "tokens/s", "cores": 1,
                                "sample": f"1 token x {len(layers)} layers, {el1:.1f} s"}
    return out


# ------------------------------------------------------------ workloads

def run_headline(args, dev, world, rank):
    cfg = W.CONFIGS[1]
    stack = DecodeStack(cfg, dev, T=1, layers=args.layers)
    stream = torch.cuda.Stream(dev)
    stack.capture(stream)
    steps, warmup = args.steps, max(3, args.warmup)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ms = time_graph(stack.graph, stream, steps, warmup, world, dev)
    status = stack.M.moe_check_status(stack.ws)
    assert status == 0, f"device status {status}"
    ms_step = ms / steps
    tok_s = job_throughput(stack.T * steps, world, ms)
    routed = stack.routed_bytes_per_step()
    hbm_peak, tf_peak, tf_sus, peak_kind = peaks()
    layer_us = ms_step * 1e3 / stack.L
    per_layer_bytes = routed / stack.L
    achieved = per_layer_bytes / (layer_us * 1e-6) / 1e9
    e2e_ms, h2d, d2h = time_e2e(stack, stream, min(steps, 2000), warmup)
    e2e = world * stack.T * min(steps, 2000) / (e2e_ms / 1e3)
    same = LAYER_KERNEL_TRAFFIC["fused_sha16"] == fused_sha16()
    traffic = LAYER_KERNEL_TRAFFIC["bytes_per_layer"] if same else None
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
        "dtype": "int8/fp16-scale weights x bf16 activations; dots on 16-bit block fixed-point activations "
                 "(int32 exact), fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": f"decode: 1 token x {stack.L} layers, E=256 top-8 D=2048 F=768, int8 sym "
                               "blk32 fp16 scales, bf16 x, Zipf(1.1) router bias",
                   "T": stack.T, "layers": stack.L, "E": cfg.E, "k": cfg.k, "D": cfg.D, "F": cfg.F,
                   "routed_bytes_per_token": routed // stack.T,
                   "routed_gbs": round(routed / (ms_step * 1e-3) / 1e9, 1),
                   "l2": f"no flush: {routed / 1e9:.2f} GB of distinct weights per step > "
                         f"{L2_BYTES / 2**20:.0f} MiB L2",
                   "inputs": "independent layers: each layer decodes its own bank token every step; layer l+1 "
                             "starts after every CTA finished layer l",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "graph": "one CUDA graph per step: token gather + one launch of the stacked layer kernel"},
        "roofline": roofline("hbm", achieved, hbm_peak, "GB/s",
                             "fused_layer_kernel (one launch = the whole 40-layer stack)",
                             {"peak_kind": peak_kind, "per_layer_bytes": int(per_layer_bytes),
                              "per_layer_us": round(layer_us, 3), "per_launch_bytes": int(routed),
                              "per_launch_us": round(ms_step * 1e3, 2),
                              "traffic": None if traffic is None else traffic * stack.L,
                              "traffic_unit": "DRAM bytes per launch",
                              "traffic_source": LAYER_KERNEL_TRAFFIC["source"] if same else
                              "no ncu capture of this kernel version"}),
        "e2e": {"value": round(e2e, 2), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": stack.kernels_per_step() * steps,
        "clocks": clk.summary(),
    }
    return line, stack, stream


def run_batched(args, dev, stack, cpu=None):
    """Batched decode over the same 40-layer stack, T in {1,...,64}."""
    cfg = W.CONFIGS[2]
    per_expert = W.routed_bytes_per_expert(cfg)
    hbm, _, _, kind = peaks()
    pts = []
    with ClockSampler(0) as clk:
        for T in (1, 2, 4, 8, 16, 32, 64):
            st = DecodeStack(cfg, dev, T=T, layers=stack.L, layer_weights=stack.layers)
            stream = torch.cuda.Stream(dev)
            st.capture(stream)
            steps = max(10, args.steps // 4)
            ms = time_graph(st.graph, stream, steps, max(3, args.warmup)) / steps
            U = st.unions()
            routed = sum(U) * per_expert
            gbs = routed / (ms * 1e-3) / 1e9
            pts.append({"T": T, "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
                        "union_experts_mean": round(sum(U) / len(U), 2), "union_min": min(U), "union_max": max(U),
                        "routed_gbs": round(gbs, 1),
                        "roofline": roofline("hbm", gbs, hbm, "GB/s",
                                             "stacked layer kernel" if T == 1 else
                                             ("single-token layer kernel per token" if T <= FUSED_TOKENS else
                                              "grouped tensor-core products"), {"peak_kind": kind})})
            s = st.M.moe_check_status(st.ws)
            assert s == 0, f"T={T}: device status {s}"
            del st
    torch.cuda.synchronize()
    if cpu is None:
        cpu = cpu_baseline_decode(cfg, stack.layers, ntok=8, single=False)
    cpu = dict(cpu, sample=cpu["sample"] + "; the oracle's cost per token does not depend on the batch")
    return {"workload": f"batched decode sweep, {stack.L} layers E=256 top-8 D=2048 F=768 int8, T = 1..64",
            "unit": "tokens/s", "points": pts, "cpu_baseline": cpu, "clocks": clk.summary()}


def run_substitution(args, dev):
    """Residency substitution (0.15 rule) + int4 experts, 512 experts top-10, 16 layers."""
    import moe_routed_expert_route_gb300 as M
    import oracle
    cfg = W.CONFIGS[3]
    L = cfg.layers if args.layers is None else min(args.layers, cfg.layers)
    layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(L)]
    masks = [W.make_resident_mask(cfg, l, dev) for l in range(L)]
    per_expert = W.routed_bytes_per_expert(cfg)
    hbm, _, _, kind = peaks()
    k = cfg.k
    routers = [M.Router(lw["Wr"], lw["bias"], k) for lw in layers]
    experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in layers]
    res = []
    with ClockSampler(0) as clk:
        for T in (1, 16):
            XIN = torch.empty(L, T, cfg.D, dtype=cfg.x_dtype, device=dev)
            XN = torch.empty(L, T, cfg.D, dtype=cfg.x_dtype, device=dev)
            bufs = [dict(idx=torch.empty(T, k, dtype=torch.int32, device=dev), w=torch.empty(T, k, device=dev),
                         used=torch.empty(T, k, dtype=torch.int32, device=dev),
                         flag=torch.empty(T, k, dtype=torch.uint8, device=dev),
                         mass=torch.empty(T, device=dev), y=torch.empty(T, cfg.D, device=dev)) for _ in range(L)]
            # one token: all layers in one launch of the stacked kernel
            ws = (M.workspace(M.MOE_OP_LAYER, 1, k, cfg.E, cfg.D, cfg.F, dev) if T == 1 else
                  M.workspace(M.MOE_OP_LAYER_RESIDENT, T, k, cfg.E, cfg.D, cfg.F, dev))
            NB = 16 if T > 8 else 64
            bank = W.make_tokens(cfg, NB * L * T, 1, dev).reshape(NB, L, T, cfg.D)
            ctr = torch.zeros(1, dtype=torch.long, device=dev)
            torch.cuda.synchronize()

            def step():
                torch.index_select(bank, 0, ctr, out=XIN.view(1, L, T, -1))
                ctr.add_(1).remainder_(NB)
                if T == 1:
                    M.moe_layer_stack_resident(routers, experts, [XIN[l] for l in range(L)], False, masks,
                                               cfg.threshold, *([b[n] for b in bufs] for n in
                                                                ("idx", "w", "used", "flag", "mass", "y")),
                                               [XN[l] for l in range(L)], ws)
                    return
                for l in range(L):
                    b = bufs[l]
                    M.moe_layer_resident(routers[l], experts[l], XIN[l], masks[l], cfg.threshold, b["idx"], b["w"],
                                         None, b["used"], b["flag"], b["mass"], b["y"], XN[l], ws)

            stream = torch.cuda.Stream(dev)
            with torch.cuda.stream(stream):
                step()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            steps = max(10, args.steps // 4)
            ms = time_graph(g, stream, steps, max(3, args.warmup)) / steps
            U = [int(torch.unique(bufs[l]["used"]).numel()) for l in range(L)]
            flags = torch.stack([b["flag"] for b in bufs]).cpu()
            mass = torch.stack([b["mass"] for b in bufs]).cpu()
            gbs = sum(U) * per_expert / (ms * 1e-3) / 1e9
            res.append({"T": T, "layers": L, "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
                        "us_per_layer": round(ms * 1e3 / L, 2), "distinct_experts_mean": round(sum(U) / L, 2),
                        "routed_gbs": round(gbs, 1),
                        "roofline": roofline("hbm", gbs, hbm, "GB/s",
                                             "stacked single-token layer kernel with substitution (one launch "
                                             "per step)" if T == 1 else
                                             "router GEMM + substitution + grouped tensor-core products",
                                             {"peak_kind": kind}),
                        "substituted_frac": round(float((flags == 2).float().mean()), 4),
                        "fetched_miss_frac": round(float((flags == 1).float().mean()), 4),
                        "mass_mean": round(float(mass.mean()), 4), "mass_max": round(float(mass.max()), 4)})
            assert M.moe_check_status(ws) == 0
            del g, bufs, bank
    # oracle: router + substitution + routed experts, a sample of tokens through all layers
    nth = os.cpu_count() or 1
    host = [_host_layer(lw) for lw in layers]
    hmask = [m.cpu() for m in masks]
    ntok = 4
    xs = W.make_tokens(cfg, (ntok + 1) * L, 9, "cpu").double().numpy().reshape(ntok + 1, L, 1, -1)

    def token(i, threads=nth):
        el = 0.0
        for l in range(L):
            t0 = time.perf_counter()
            r = oracle.router(xs[i, l], host[l][0], host[l][1], k)
            s = oracle.substitute(r["probs32"], r["idx"], r["w"], hmask[l], cfg.threshold)
            el += time.perf_counter() - t0
            el += timed_oracle_moe(layers[l], xs[i, l], s["idx"], s["w"], cfg.qbits, threads)[0]
        return el

    token(0)
    el = sum(token(i) for i in range(1, ntok + 1))
    el1 = token(1, threads=1)  # one token on one core
    t_layer = next(r["us_per_layer"] for r in res if r["T"] == 1)
    replay = run_replay(args, dev, cfg, routers, masks, t_layer)
    del layers, routers, experts
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return replay, {"workload": f"substitution 0.15 rule + int4 experts, E=512 top-10 D=2048 F=512, 25% resident, "
                        f"{L} layers", "unit": "tokens/s", "points": res,
            "cpu_baseline": {"value": round(ntok / el, 4), "unit": "tokens/s", "cores": nth, "kind": "oracle",
                             "sample": f"{ntok} tokens x {L} layers (router + substitution + routed experts, on host "
                                       f"copies of the routed experts' rows, copies not timed) after "
                                       f"1 warm-up token, {el:.1f} s",
                             "single_thread": {"value": round(1 / el1, 4), "unit": "tokens/s", "cores": 1,
                                               "sample": f"1 token x {L} layers, {el1:.1f} s"}},
            "clocks": clk.summary()}


def run_replay(args, dev, cfg, routers, masks, t_layer_us):
    """Router-logit replay: the GPU router logs the probabilities of N tokens
    through the layers, and the host simulator replays them under the page's
    policies, with a time model measured here: the one-token layer time of the
    substitution workload and the time to copy one expert from pinned host
    memory."""
    import numpy as np
    import moe_routed_expert_route_gb300 as M
    from oracle import replay as oracle_replay
    L, E, k = len(routers), cfg.E, cfg.k
    N = 512
    # the router's probabilities, per layer for the N tokens (on the GPU)
    x = W.make_tokens(cfg, N * L, 31, dev).view(L, N, cfg.D)
    probs = torch.empty(L, N, E, device=dev)
    idx = torch.empty(N, k, dtype=torch.int32, device=dev)
    w = torch.empty(N, k, device=dev)
    ws = M.workspace(M.MOE_OP_ROUTE, N, k, E, cfg.D, cfg.F, dev)
    for l in range(L):
        M.moe_route(routers[l], x[l], idx, w, probs[l], ws)
    assert M.moe_check_status(ws) == 0
    P = probs.transpose(0, 1).contiguous().cpu().numpy()  # [N][L][E]
    res0 = torch.stack(masks).cpu().numpy().astype(np.uint8)
    # one expert from pinned host memory to the device
    nb = W.routed_bytes_per_expert(cfg)
    host = torch.empty(nb, dtype=torch.uint8, pin_memory=True)
    devbuf = torch.empty(nb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for _ in range(5):
            devbuf.copy_(host, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(50):
            devbuf.copy_(host, non_blocking=True)
        b.record(stream)
    torch.cuda.synchronize()
    t_fetch = a.elapsed_time(b) * 1e3 / 50
    policies = [("fetch every miss", M.MOE_POLICY_FETCH_ALL, 0.0), ("0.15 rule", M.MOE_POLICY_THRESHOLD, 0.0),
                ("first-choice rule", M.MOE_POLICY_FIRST_CHOICE, 0.0),
                ("quality-first: 0.15 rule + admission at 0.5", M.MOE_POLICY_THRESHOLD, 0.5),
                ("speed-first: first-choice rule + admission at 0.5", M.MOE_POLICY_FIRST_CHOICE, 0.5)]
    out = []
    for name, pol, beta in policies:
        t0 = time.perf_counter()
        r = M.moe_replay(P, k, pol, 0.15, beta, t_layer_us, t_fetch, resident=res0.copy())
        el = time.perf_counter() - t0
        ms_tok = float(r["t_token_us"].mean()) / 1e3
        out.append({"policy": name, "est_ms_per_token": round(ms_tok, 4), "est_tokens_per_s": round(1e3 / ms_tok, 1),
                    "sync_fetches_per_token": round(float(r["fetches"].mean()), 3),
                    "substituted_frac": round(float(r["substituted"].sum()) / (N * L * k), 4),
                    "sub_mass_per_layer": round(float(r["sub_mass"].mean()) / L, 4),
                    "admissions_per_token": round(float(r["admissions"].mean()), 3),
                    "replay_tokens_per_s": round(N / el, 1)})
    # the oracle on the same tokens, quality-first policy
    ns = N
    t0 = time.perf_counter()
    oracle_replay.replay(P[:ns], k, oracle_replay.THRESHOLD, 0.15, 0.5, t_layer_us, t_fetch, resident=res0.tolist())
    el = time.perf_counter() - t0
    return {"workload": f"router-logit replay: {N} tokens x {L} layers of GPU-logged router probabilities, "
                        f"E={E} top-{k}, 25% resident; the simulator runs on the host",
            "unit": "tokens/s (replayed)", "t_layer_us": t_layer_us, "t_fetch_us": round(t_fetch, 2),
            "expert_bytes": nb, "policies": out,
            "roofline": None,
            "cpu_baseline": {"value": round(ns / el, 2), "unit": "tokens/s (replayed)", "cores": 1,
                             "kind": "oracle", "sample": f"{ns} tokens x {L} layers, quality-first policy, "
                                                         f"{el:.2f} s"}}


def run_prefill(args, dev, stack, T):
    """Prefill of T tokens on the decode layer shape, rotating over 4 layers
    of the resident stack (5 GB of weights)."""
    import moe_routed_expert_route_gb300 as M
    import oracle
    cfg = W.CONFIGS[4]
    L = min(4, stack.L)
    layers = stack.layers[:L]
    routers = stack.routers[:L]
    experts = stack.experts[:L]
    x = W.make_tokens(cfg, T, 0, dev)
    y = torch.empty(T, cfg.D, device=dev)
    idx = torch.empty(T, cfg.k, dtype=torch.int32, device=dev)
    w = torch.empty(T, cfg.k, device=dev)
    counts = torch.empty(L, cfg.E, dtype=torch.int32, device=dev)
    ws = M.workspace(M.MOE_OP_PREFILL, T, cfg.k, cfg.E, cfg.D, cfg.F, dev)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(dev)

    def step(l):
        M.moe_prefill(routers[l], experts[l], x, y, idx, w, counts[l], None, ws)

    with torch.cuda.stream(stream):
        for l in range(L):
            step(l)
    torch.cuda.synchronize()
    U = [int((counts[l] > 0).sum()) for l in range(L)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l in range(L):
            step(l)
    hbm, tf, tf_sus, kind = peaks()
    with ClockSampler(0) as clk:
        steps = max(5, args.steps // 40)
        ms = time_graph(g, stream, steps, max(3, args.warmup)) / steps / L
    flops = 2.0 * T * cfg.k * 3 * cfg.D * cfg.F
    wbytes = (sum(U) / L) * W.routed_bytes_per_expert(cfg)
    assert M.moe_check_status(ws) == 0
    tfs = flops / (ms * 1e-3) / 1e12
    gbs = wbytes / (ms * 1e-3) / 1e9
    tensor_frac, hbm_frac = tfs / tf, gbs / hbm
    # oracle on a sample of the same tokens (one layer)
    nth = os.cpu_count() or 1
    ns = 32
    xs = x[:ns].cpu()
    wr, br = layers[0]["Wr"].cpu(), layers[0]["bias"].cpu()
    t0 = time.perf_counter()
    r = oracle.router(xs, wr, br, cfg.k)
    el = time.perf_counter() - t0
    el += timed_oracle_moe(layers[0], xs, r["idx"], r["w"], cfg.qbits, nth)[0]
    # and 2 of those tokens on one core
    ns1 = 2
    t0 = time.perf_counter()
    r1 = oracle.router(xs[:ns1], wr, br, cfg.k)
    el1 = time.perf_counter() - t0
    el1 += timed_oracle_moe(layers[0], xs[:ns1], r1["idx"], r1["w"], cfg.qbits, 1)[0]
    del ws
    torch.cuda.empty_cache()
    return {"workload": f"prefill T={T} E=256 top-8 D=2048 F=768 int8 (fp16 tensor-core operands)",
            "T": T, "unit": "tokens/s", "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_layer": round(ms, 4),
            "distinct_experts_mean": round(sum(U) / L, 1), "expert_weight_gb": round(wbytes / 1e9, 3),
            "expert_tflops": round(tfs, 1), "weight_gbs": round(gbs, 1),
            "roofline": roofline("tensor" if tensor_frac >= hbm_frac else "hbm",
                                 tfs if tensor_frac >= hbm_frac else gbs,
                                 tf if tensor_frac >= hbm_frac else hbm,
                                 "TFLOP/s" if tensor_frac >= hbm_frac else "GB/s",
                                 "router GEMM + grouping + two grouped tensor-core products + combine",
                                 {"peak_kind": kind, "tensor_frac_of_bf16_peak": round(tensor_frac, 4),
                                  "hbm_frac_of_weights": round(hbm_frac, 4),
                                  "note": "fp16 operands: the bf16 peak applies (same nominal rate)"}),
            "cpu_baseline": {"value": round(ns / el, 4), "unit": "tokens/s", "cores": nth, "kind": "oracle",
                             "sample": f"{ns} of the {T} tokens through one layer (on host copies of the routed "
                                       f"experts' rows, copies not timed), {el:.1f} s",
                             "single_thread": {"value": round(ns1 / el1, 4), "unit": "tokens/s", "cores": 1,
                                               "sample": f"{ns1} of those tokens through one layer, {el1:.1f} s"}},
            "clocks": clk.summary()}


def _tensor_bytes(d: dict) -> int:
    return sum(v.numel() * v.element_size() for v in d.values() if isinstance(v, torch.Tensor))


def _time_calls(args, dev, calls, n_copies):
    """Captures one pass of `calls` (one call per copy) in a CUDA graph and
    returns the CUDA-event milliseconds of one call."""
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    steps = max(20, args.steps // 20)
    return time_graph(g, stream, steps, max(3, args.warmup)) / steps / n_copies


def run_edge0(args, dev):
    """The shared expert with its unmerged LoRA and the prerouter head (the
    xyznot.com Edge0 page, method section) at decode size. Each step calls
    every copy once: 80 shared experts (int4 base + rank-16 adapters, 1.9 MB
    each) and 40 heads (input 2048 + 2*256, hidden 512, bf16, 4.2 MB each), so
    more bytes than L2 pass per step."""
    import numpy as np
    import moe_routed_expert_route_gb300 as M
    import oracle
    hbm, _, _, kind = peaks()
    nth = os.cpu_count() or 1
    out = {}

    sc = W.SHARED_CONFIGS["decode"]
    n_sh = 80
    shared = [W.make_shared_expert(sc, l, dev) for l in range(n_sh)]
    objs = [M.Shared.from_dict(s) for s in shared]
    sh_bytes = _tensor_bytes(shared[0])
    host0 = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in shared[0].items()}
    for T in (1, 16):
        x = W.make_shared_tokens(sc, T, 0, dev)
        y = torch.empty(T, sc.D, device=dev)
        ws = M.workspace(M.MOE_OP_SHARED, T, 1, 1, sc.D, sc.F, dev)

        def calls():
            for o in objs:
                M.moe_shared_lora(o, x, y, False, ws)
        with ClockSampler(dev.index or 0) as clk:
            ms = _time_calls(args, dev, calls, n_sh)
        assert M.moe_check_status(ws) == 0
        gbs = sh_bytes / (ms * 1e-3) / 1e9
        xs = x.cpu()
        t0 = time.perf_counter()
        nrep = 3
        for _ in range(nrep):
            oracle.shared_lora(host0, xs)
        el = (time.perf_counter() - t0) / nrep
        out[f"shared_lora_T{T}"] = {
            "workload": f"shared expert D=2048 F=512 int4 blk32 fp16 scales + unmerged LoRA r=16 (bf16), "
                        f"T={T}, 80 copies", "T": T, "unit": "tokens/s",
            "tokens_per_s": round(T / (ms * 1e-3), 1), "us_per_call": round(ms * 1e3, 3),
            "bytes_per_call": sh_bytes, "weight_gbs": round(gbs, 1),
            "roofline": roofline("hbm", gbs, hbm, "GB/s", "lora_a + shared_gateup + lora_a + shared_down",
                                 {"peak_kind": kind}),
            "cpu_baseline": {"value": round(T / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{nrep} calls of one copy on T={T} tokens, {el * nrep:.2f} s"},
            "clocks": clk.summary()}
        del ws
    del shared, objs
    torch.cuda.empty_cache()

    cfg = W.CONFIGS[1]
    n_h = 40
    heads = [W.make_prerouter(cfg, l, H=512, device=dev) for l in range(n_h)]
    hobjs = [M.Prerouter.from_dict(h, cfg.k) for h in heads]
    h_bytes = _tensor_bytes(heads[0])
    hhost = {k: v.cpu() for k, v in heads[0].items()}
    for T in (1, 16):
        x = W.make_tokens(cfg, T, 7, dev)
        cur, prev = W.make_routing_history(cfg, T, stream=7, device=dev)
        idx = torch.empty(T, cfg.k, dtype=torch.int32, device=dev)
        w = torch.empty(T, cfg.k, device=dev)
        ws = M.workspace(M.MOE_OP_PREROUTE, T, cfg.k, cfg.E, cfg.D, 512, dev)

        def calls():
            for o in hobjs:
                M.moe_preroute(o, x, cur, prev, idx, w, None, ws)
        with ClockSampler(dev.index or 0) as clk:
            ms = _time_calls(args, dev, calls, n_h)
        assert M.moe_check_status(ws) == 0
        gbs = h_bytes / (ms * 1e-3) / 1e9
        xs, cs, ps = x.cpu(), cur.cpu(), prev.cpu()
        t0 = time.perf_counter()
        nrep = 3
        for _ in range(nrep):
            oracle.prerouter(hhost, xs, cs, ps, cfg.k)
        el = (time.perf_counter() - t0) / nrep
        out[f"prerouter_T{T}"] = {
            "workload": f"prerouter head D=2048 E=256 k=8 H=512 (input 2560, bf16), T={T}, 40 heads",
            "T": T, "unit": "tokens/s", "tokens_per_s": round(T / (ms * 1e-3), 1),
            "us_per_call": round(ms * 1e3, 3), "bytes_per_call": h_bytes, "weight_gbs": round(gbs, 1),
            "roofline": roofline("hbm", gbs, hbm, "GB/s", "preroute_hidden + preroute_logits + topk",
                                 {"peak_kind": kind}),
            "cpu_baseline": {"value": round(T / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{nrep} calls of one head on T={T} tokens, {el * nrep:.2f} s"},
            "clocks": clk.summary()}
        del ws
    del heads, hobjs
    torch.cuda.empty_cache()
    return out


def run_expert_cache(args, dev, n_tok: int = 96, warm: int = 16, L: int = 2):
    """Miss fetch and background admission (gist.science page, method
    section) on the 512-expert top-10 int4 layer: all experts in pinned host
    memory, a quarter of them (128) cached in an HBM pool per layer, the 0.15
    rule with admission at 0.5. One token at a time through L layers: router
    on the GPU, decisions on the host, kept misses copied in by the copy
    engines, decode from the pool, admissions on a copy stream. The path waits
    for the router once per layer, so the time is wall clock around the token
    loop (with a device synchronisation at its end)."""
    import numpy as np
    import moe_routed_expert_route_gb300 as M
    import oracle
    from oracle import replay as R
    cfg = W.CONFIGS[3]
    names = _EXPERT_TENSORS
    hbm, _, _, kind = peaks()
    per_expert = W.routed_bytes_per_expert(cfg)
    layers = []
    for l in range(L):
        lw = W.make_layer(cfg, l, dev)
        host = {n: lw[n].cpu().pin_memory() for n in names}
        pool = {n: torch.zeros((cfg.resident + cfg.k,) + tuple(lw[n].shape[1:]), dtype=lw[n].dtype, device=dev)
                for n in names}
        hx, px = M.Experts.from_layer(host, cfg.qbits), M.Experts.from_layer(pool, cfg.qbits)
        cached = torch.nonzero(W.make_resident_mask(cfg, l)).flatten().numpy()
        M.moe_pool_fetch(hx, px, cached, np.arange(cfg.resident))
        n, hb = M.moe_cache_workspace_bytes(cfg.E, cfg.resident, cfg.k, cfg.D, cfg.F)
        layers.append(dict(router=M.Router(lw["Wr"], lw["bias"], cfg.k), host=host, pool=pool, hx=hx, px=px,
                           cache=M.ExpertCache(cfg.E, cfg.k, cached), cached0=cached.copy(),
                           ws=torch.zeros(n, dtype=torch.uint8, device=dev),
                           scratch=torch.zeros(hb, dtype=torch.uint8).pin_memory(),
                           Wr=lw["Wr"].cpu(), bias=lw["bias"].cpu()))
        del lw
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    x = W.make_tokens(cfg, n_tok + warm, 11, dev)
    y = torch.empty(1, cfg.D, device=dev)
    cs = torch.cuda.Stream(dev)
    ev1, ev2 = torch.cuda.Event(), torch.cuda.Event()
    ev1.record()
    ev2.record()
    stats = dict(fetch=0, sub=0, adm=0, mass=0.0)

    def token(t, count):
        for ly in layers:
            d = M.moe_cached_layer(ly["router"], ly["hx"], ly["px"], ly["cache"], M.MOE_POLICY_THRESHOLD, 0.15, 0.5,
                                   x[t:t + 1], y, None, ly["scratch"], ly["ws"], None, cs, ev1, ev2)
            if count:
                stats["fetch"] += len(d["fetch_expert"])
                stats["sub"] += int((d["flag"] == 2).sum())
                stats["adm"] += len(d["admit_expert"])
                stats["mass"] += d["mass"]
    for t in range(warm):
        token(t, False)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        t0 = time.perf_counter()
        for t in range(warm, warm + n_tok):
            token(t, True)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
    for ly in layers:
        assert M.moe_check_status(ly["ws"]) == 0
    us_layer = el / (n_tok * L) * 1e6
    served = cfg.k * per_expert  # expert bytes the decode reads per token and layer
    fetched = (stats["fetch"] + stats["adm"]) * per_expert
    # the oracle on a sample: router, decisions, and the MoE on the served
    # experts, one layer, from the cache state the GPU run started with
    ns = 4
    ly0 = layers[0]
    xs = x[:ns].cpu()
    t1 = time.perf_counter()
    r = oracle.router(xs, ly0["Wr"], ly0["bias"], cfg.k)
    res = np.zeros((1, cfg.E), np.uint8)
    res[0, ly0["cached0"]] = 1
    rp = R.replay(r["probs32"][:, None, :], cfg.k, R.THRESHOLD, 0.15, 0.5, 0.0, 0.0, resident=res.tolist())
    for t in range(ns):
        used = np.asarray(rp["used"][t][0], np.int64)
        sub = {n: ly0["host"][n][torch.from_numpy(used)] for n in names}
        oracle.moe(sub, xs[t:t + 1], np.arange(cfg.k, dtype=np.int32)[None], r["w"][t:t + 1], cfg.qbits,
                   nthreads=os.cpu_count() or 1, compact=False)
    el_o = time.perf_counter() - t1
    out = {"workload": f"expert cache: 1 token x {L} layers, E=512 top-10 D=2048 F=512 int4, 128 of 512 experts "
                       "cached in HBM per layer, all in pinned host memory; 0.15 rule, admission at 0.5",
           "T": 1, "unit": "tokens/s", "tokens_per_s": round(n_tok / el, 2), "us_per_layer": round(us_layer, 2),
           "sync_fetches_per_token_layer": round(stats["fetch"] / (n_tok * L), 3),
           "substituted_per_token_layer": round(stats["sub"] / (n_tok * L), 3),
           "admissions_per_token_layer": round(stats["adm"] / (n_tok * L), 3),
           "substituted_mass_per_token_layer": round(stats["mass"] / (n_tok * L), 4),
           "host_to_device_gbs": round(fetched / el / 1e9, 2),
           "roofline": roofline("hbm", served / (us_layer * 1e-6) / 1e9, hbm, "GB/s",
                                "route + host decisions + copies + decode (wall clock per layer)",
                                {"peak_kind": kind, "note": "served expert bytes per layer over the wall-clock "
                                 "time of a layer, which includes the host round trip for the decisions"}),
           "cpu_baseline": {"value": round(ns / (el_o * L), 4), "unit": "tokens/s", "cores": os.cpu_count() or 1,
                            "kind": "oracle", "sample": f"router, replay decisions and MoE on the served experts "
                                                        f"for {ns} tokens of one layer, {el_o:.1f} s, scaled to {L} layers"},
           "timing": "wall clock (perf_counter) around the token loop, device synchronised at its end",
           "clocks": clk.summary()}
    del layers
    torch.cuda.empty_cache()
    return out


def run_staged(args, dev, n_tok: int = 64, warm: int = 8):
    """Prediction-as-routing through the staged slot table (xyznot.com Edge0
    page: prerouter; glossary: staged decode, incremental sticky-slot stack)
    on the 256-expert top-8 int8 layer: all experts in pinned host memory, a
    pool of 2k = 16 HBM slots. Per token t: the prerouter predicts token
    t+1's routing, the changed slots are loaded on a copy stream, and token
    t+1 is decoded from the pool once they are in. The staging waits for the
    prediction on the host, so the time is wall clock around the token loop."""
    import numpy as np
    import moe_routed_expert_route_gb300 as M
    import oracle
    cfg = W.CONFIGS[1]
    k, NS, H = cfg.k, 2 * cfg.k, 512
    names = _EXPERT_TENSORS
    hbm, _, _, kind = peaks()
    lw = W.make_layer(cfg, 1, dev)
    host = {n: lw[n].cpu().pin_memory() for n in names}
    del lw
    torch.cuda.empty_cache()
    pool = {n: torch.zeros((NS,) + tuple(host[n].shape[1:]), dtype=host[n].dtype, device=dev) for n in names}
    hx, px = M.Experts.from_layer(host, cfg.qbits), M.Experts.from_layer(pool, cfg.qbits)
    head = W.make_prerouter(cfg, 0, H=H, device=dev)
    pre = M.Prerouter.from_dict(head, k)
    T = n_tok + warm + 1
    x = W.make_tokens(cfg, T, 13, dev)
    cur, prev = W.make_routing_history(cfg, T, stream=13, device=dev)
    st = M.StageTable(cfg.E, NS, k)
    cs = torch.cuda.Stream(dev)
    ev = torch.cuda.Event()
    ev.record()
    scratch = torch.zeros(2 * k, dtype=torch.int32).pin_memory()
    slot_bufs = [torch.empty(k, dtype=torch.int32, device=dev) for _ in range(2)]
    idx_bufs = [torch.empty(1, k, dtype=torch.int32, device=dev) for _ in range(2)]
    w_bufs = [torch.empty(1, k, device=dev) for _ in range(2)]
    y = torch.empty(1, cfg.D, device=dev)
    ws_p = M.workspace(M.MOE_OP_PREROUTE, 1, k, cfg.E, cfg.D, H, dev)
    ws_d = M.workspace(M.MOE_OP_DECODE, 1, k, NS, cfg.D, cfg.F, dev)
    loads = [0]

    def token(t, count):
        b = t % 2
        M.moe_preroute(pre, x[t:t + 1], cur[t:t + 1], prev[t:t + 1], idx_bufs[b], w_bufs[b], None, ws_p)
        step = M.moe_stage_prediction(st, hx, px, idx_bufs[b][0], slot_bufs[b], scratch, None, cs, ev)
        torch.cuda.current_stream().wait_event(ev)
        M.moe_decode(px, x[t + 1:t + 2], slot_bufs[b].view(1, k), w_bufs[b], y, None, ws_d)
        if count:
            loads[0] += len(step["load_expert"])
    for t in range(warm):
        token(t, False)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        t0 = time.perf_counter()
        for t in range(warm, warm + n_tok):
            token(t, True)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
    assert M.moe_check_status(ws_p) == 0 and M.moe_check_status(ws_d) == 0
    per_expert = W.routed_bytes_per_expert(cfg)
    us_tok = el / n_tok * 1e6
    # the oracle on a sample: prerouter and the MoE on the predicted experts
    ns = 2
    hh = {n: v.cpu() for n, v in head.items()}
    t1 = time.perf_counter()
    r = oracle.prerouter(hh, x[:ns].cpu(), cur[:ns].cpu(), prev[:ns].cpu(), k)
    for t in range(ns):
        sub = {n: host[n][torch.from_numpy(r["idx"][t].astype("int64"))] for n in names}
        oracle.moe(sub, x[t + 1:t + 2].cpu(), np.arange(k, dtype=np.int32)[None], r["w"][t:t + 1],
                   cfg.qbits, nthreads=os.cpu_count() or 1, compact=False)
    el_o = time.perf_counter() - t1
    out = {"workload": "staged prediction: 1 token, E=256 top-8 D=2048 F=768 int8 layer in pinned host memory, "
                       "16 HBM slots; prerouter (input 2560, hidden 512) one token ahead, changed slots loaded "
                       "on a copy stream, decode from the pool",
           "T": 1, "unit": "tokens/s", "tokens_per_s": round(n_tok / el, 2), "us_per_token": round(us_tok, 2),
           "loads_per_token": round(loads[0] / n_tok, 3),
           "host_to_device_gbs": round(loads[0] * per_expert / el / 1e9, 2),
           "roofline": roofline("hbm", k * per_expert / (us_tok * 1e-6) / 1e9, hbm, "GB/s",
                                "preroute + host staging + copies + decode (wall clock per token)",
                                {"peak_kind": kind, "note": "decoded expert bytes per token over the wall-clock "
                                 "time of a token, which includes the host round trip for the staging"}),
           "cpu_baseline": {"value": round(ns / el_o, 4), "unit": "tokens/s", "cores": os.cpu_count() or 1,
                            "kind": "oracle", "sample": f"prerouter and MoE on the predicted experts for {ns} tokens, "
                                                        f"{el_o:.1f} s"},
           "timing": "wall clock (perf_counter) around the token loop, device synchronised at its end",
           "clocks": clk.summary()}
    del pool, host
    torch.cuda.empty_cache()
    return out


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
    line, stack, stream = run_headline(args, dev, world, rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(W.CONFIGS[1], stack.layers, ntok=CPU_SAMPLE_TOKENS)
    if world == 1 and not args.headline_only:
        extra = {}
        extra["batched_decode"] = run_batched(args, dev, stack, line.get("cpu_baseline"))
        extra["prefill_T2048"] = run_prefill(args, dev, stack, 2048)
        extra["prefill_T16384"] = run_prefill(args, dev, stack, 16384)
        del stack
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        extra["replay"], extra["substitution"] = run_substitution(args, dev)
        for key, fn in (("edge0", run_edge0), ("expert_cache", run_expert_cache), ("staged_prediction", run_staged)):
            try:
                extra[key] = fn(args, dev)
            except Exception as e:  # reported, never at the cost of the line above
                extra[key] = {"error": f"{type(e).__name__}: {e}"[:300]}
        line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The CPU oracle on a bounded sample of the headline workload: each step
    is 8 tokens through every layer, at most 8 steps (the GPU arm's
    cpu_baseline times the same 64-token sample)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = W.CONFIGS[1]
    L = args.layers or cfg.layers
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    layers = [W.make_layer(cfg, l, dev, chunk=64) for l in range(L)]
    steps = max(1, min(args.steps, CPU_SAMPLE_TOKENS // REF_TOKENS_PER_STEP))
    cb = cpu_baseline_decode(cfg, layers, ntok=steps * REF_TOKENS_PER_STEP)
    v = cb["value"]
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": steps, "warmup": 1, "ms_per_step": round(1e3 * REF_TOKENS_PER_STEP / v, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"decode: 1 token x {L} layers, E=256 top-8 D=2048 F=768, int8 sym "
                               "blk32 fp16 scales, bf16 x, Zipf(1.1) router bias",
                   "inputs": "independent layers: each layer decodes its own token every step"},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="only the 40-layer decode line (no batched / substitution / prefill workloads)")
    ap.add_argument("--layers", type=int, default=None,
                    help="stacked layers (default: the workload's 40); fewer only for profiling captures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
