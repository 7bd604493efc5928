"""Prefill (many tokens) through moe_prefill vs the CPU oracle.

Routing ids bit-exact except near ties (rules in tests/parity.py); expert counts
and the grouping permutation exactly equal to the oracle's (a stable counting
sort of the assignments by expert, unique given the routing); y within
2e-3 * max|y| of the oracle evaluated on the GPU's routing, for every token,
including all 2048 tokens of the full-size prefill.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import parity
import workloads as W

pytestmark = pytest.mark.gpu

M = None
if torch.cuda.is_available():
    import moe_routed_expert_route_gb300 as M  # noqa: F811

DEV = "cuda"
REL_TOL = parity.REL_TOL
NTH = parity.NTH


def run_prefill(cfg, layer, x):
    T = x.shape[0]
    router = M.Router(layer["Wr"], layer["bias"], cfg.k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    out = dict(y=torch.empty(T, cfg.D, device=DEV), idx=torch.empty(T, cfg.k, dtype=torch.int32, device=DEV),
               w=torch.empty(T, cfg.k, device=DEV), counts=torch.empty(cfg.E, dtype=torch.int32, device=DEV),
               perm=torch.empty(T * cfg.k, dtype=torch.int32, device=DEV))
    ws = M.workspace(M.MOE_OP_PREFILL, T, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_prefill(router, experts, x, out["y"], out["idx"], out["w"], out["counts"], out["perm"], ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    return {k_: v.cpu() for k_, v in out.items()}


def check_grouping(got, E):
    """Histogram, scan and stable permutation against the oracle's counting sort
    of the same routing."""
    idx = got["idx"].numpy()
    T, k = idx.shape
    ref = oracle.permute(idx, E)
    assert np.array_equal(got["counts"].numpy(), ref["cnt"])
    assert np.array_equal(np.concatenate([[0], np.cumsum(got["counts"].numpy())]), ref["off"])
    perm = got["perm"].numpy()
    assert np.array_equal(perm, ref["perm_tok"] * k + ref["perm_slot"])
    # the oracle's inverse maps every assignment back to its position
    assert np.array_equal(perm[ref["inv"].reshape(-1)], np.arange(T * k))


def check_routing(ref, got, k, max_skip_frac=0.1, label=""):
    return parity.check_routing(ref, dict(idx=got["idx"].numpy(), w=got["w"].numpy()), k, max_skip_frac,
                                label=label)


def check_y(layer, x, got, qbits, tokens=None):
    return parity.check_y(layer, x, got["idx"].numpy(), got["w"].double().numpy(), got["y"].double().numpy(),
                          qbits, tokens=tokens)


@pytest.mark.parametrize("E,k,D,F,T", [(16, 4, 256, 128, 300), (128, 4, 256, 192, 300), (256, 8, 512, 256, 700),
                                       (8, 2, 128, 64, 1), (128, 1, 128, 64, 5)])
@pytest.mark.parametrize("qbits", [8, 4])
def test_prefill_small(E, k, D, F, T, qbits):
    cfg = W.LayerConfig(f"prefill E{E}", E=E, k=k, D=D, F=F, T=T, qbits=qbits, scale_dtype=torch.float16,
                        x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.1, zipf=1.1,
                        layers=1, cfg_id=200 + qbits)
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, T, 1, DEV)
    got = run_prefill(cfg, layer, x)
    ref = oracle.router(x, layer["Wr"], layer["bias"], k)
    check_routing(ref, got, k, max_skip_frac=0.2, label=f"prefill E{E} k{k} D{D} F{F} T{T} q{qbits}")
    check_grouping(got, E)
    check_y(layer, x, got, qbits)


def test_prefill_fp32_activations_fall_back_to_cuda_core_router():
    cfg = W.CONFIGS[0]  # fp32 x, fp32 router, fp32 scales
    cfg = W.LayerConfig("fp32", E=8, k=2, D=128, F=64, T=37, qbits=8, scale_dtype=torch.float32,
                        x_dtype=torch.float32, router_dtype=torch.float32, router_sigma=0.1, zipf=None,
                        layers=1, cfg_id=210)
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, cfg.T, 0, DEV)
    got = run_prefill(cfg, layer, x)
    ref = oracle.router(x, layer["Wr"], None, cfg.k)
    check_routing(ref, got, cfg.k, max_skip_frac=0.2, label="prefill fp32 T37")
    check_grouping(got, cfg.E)
    check_y(layer, x, got, 8)


def test_prefill_2048_tokens_e256():
    """The 2048-token prefill on the 256-expert layer: routing and grouping of
    every token, and y of every token (the oracle on all host cores)."""
    cfg = W.CONFIGS[4]
    layer = W.make_layer(cfg, 0, DEV, chunk=64)
    x = W.make_tokens(cfg, cfg.T, 0, DEV)
    got = run_prefill(cfg, layer, x)
    ref = oracle.router(x, layer["Wr"], layer["bias"], cfg.k)
    check_routing(ref, got, cfg.k, max_skip_frac=0.05, label="prefill E256 T2048")
    check_grouping(got, cfg.E)
    check_y(layer, x.cpu(), got, cfg.qbits)


def test_prefill_deterministic():
    cfg = W.LayerConfig("det", E=128, k=4, D=256, F=128, T=500, qbits=8, scale_dtype=torch.float16,
                        x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.1, zipf=1.1,
                        layers=1, cfg_id=220)
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, cfg.T, 0, DEV)
    a = run_prefill(cfg, layer, x)
    for _ in range(3):
        b = run_prefill(cfg, layer, x)
        assert torch.equal(a["y"], b["y"]) and torch.equal(a["perm"], b["perm"])
