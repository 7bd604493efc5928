"""Prefill (many tokens) through moe_prefill vs the CPU oracle.

Routing ids bit-exact except near ties (as in test_parity_gpu); expert counts
and the grouping permutation exact (a stable sort of the assignments by expert,
unique given the routing); y within 2e-3 * max|y| of the oracle evaluated on
the GPU's routing, for every token of the small shapes and for a sample of
tokens at the full 2048-token shape.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

M = None
if torch.cuda.is_available():
    import moe_routed_expert_route_gb300 as M  # noqa: F811

DEV = "cuda"
REL_TOL = 2e-3
NTH = os.cpu_count() or 1


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
    idx = got["idx"].numpy().reshape(-1)
    assert np.array_equal(got["counts"].numpy(), np.bincount(idx, minlength=E))
    assert np.array_equal(got["perm"].numpy(), np.argsort(idx, kind="stable"))


def check_routing(ref, got, k, max_skip_frac=0.1):
    T = ref["idx"].shape[0]
    skip = set(oracle.near_tie_tokens(ref["probs32"], k).tolist())
    keep = np.array([t for t in range(T) if t not in skip], dtype=np.int64)
    assert len(skip) <= max(1, int(max_skip_frac * T)), f"{len(skip)} near-tie tokens of {T}"
    assert np.array_equal(got["idx"].numpy()[keep], ref["idx"][keep])
    np.testing.assert_allclose(got["w"].numpy()[keep], ref["w"][keep], rtol=0, atol=1e-5)


def check_y(layer, x, got, qbits, tokens=None):
    idx, w, y = got["idx"].numpy(), got["w"].double().numpy(), got["y"].double().numpy()
    xs = x
    if tokens is not None:
        idx, w, y, xs = idx[tokens], w[tokens], y[tokens], x[tokens]
    y_ref = oracle.moe(layer, xs, idx, w, qbits, nthreads=NTH)
    err = np.abs(y - y_ref).max()
    bound = REL_TOL * np.abs(y_ref).max()
    assert err <= bound, f"max|y - oracle| = {err:.3e} > {bound:.3e}"
    return err / np.abs(y_ref).max()


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
    check_routing(ref, got, k, max_skip_frac=0.2)
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
    check_routing(ref, got, cfg.k, max_skip_frac=0.2)
    check_grouping(got, cfg.E)
    check_y(layer, x, got, 8)


def test_prefill_2048_tokens_e256():
    """The 2048-token prefill on the 256-expert layer: routing and grouping of
    every token; y for a sample of 48 tokens (oracle one token at a time)."""
    cfg = W.CONFIGS[4]
    layer = W.make_layer(cfg, 0, DEV, chunk=64)
    x = W.make_tokens(cfg, cfg.T, 0, DEV)
    got = run_prefill(cfg, layer, x)
    ref = oracle.router(x, layer["Wr"], layer["bias"], cfg.k)
    check_routing(ref, got, cfg.k, max_skip_frac=0.05)
    check_grouping(got, cfg.E)
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(cfg.T, 48, replace=False))
    sample[0], sample[-1] = 0, cfg.T - 1
    check_y(layer, x.cpu(), got, cfg.qbits, tokens=sample)
    # the busiest expert has many 128-row tiles: its tokens must be right too
    busiest = int(np.argmax(got["counts"].numpy()))
    toks = np.unique(np.nonzero(got["idx"].numpy() == busiest)[0])[:16]
    check_y(layer, x.cpu(), got, cfg.qbits, tokens=toks)


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
