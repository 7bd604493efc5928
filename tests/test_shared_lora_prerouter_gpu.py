"""GPU parity of the shared expert with its unmerged LoRA (moe_shared_lora) and
of the prerouter head (moe_preroute) against the CPU oracle, through the C ABI
(xyznot.com "The Other Half of the Memory Wall", method section).

Criteria, as for the routed layer (tests/parity.py):
  * y (fp32): max |y_gpu - y_oracle| <= 2e-3 * max |y_oracle| per tensor;
  * predicted routing: ids bit-exact except near ties (two neighbours among the
    first k+1 sorted oracle fp32 probabilities within 1e-6), which must still
    be a valid top-k; weights within 1e-5; probabilities within 1e-6 + 1e-5 p.
Shapes: tiny ones with ragged token tiles (the kernels serve 8 tokens per pass
over a weight row), and the full 2048-wide shapes of the 256-expert decode
layer.
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


# Inputs are drawn on the CPU and moved to the device, so that they are the
# same wherever the test runs (and the near ties among them can be counted
# without a GPU: none at the shapes below).
def _to(d: dict, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def gpu_shared(se: dict, x: torch.Tensor, y0=None):
    T, D = x.shape
    F = se["gate_q"].shape[0]
    ws = M.workspace(M.MOE_OP_SHARED, T, 1, 1, D, F, DEV)
    y = torch.empty(T, D, dtype=torch.float32, device=DEV) if y0 is None else y0.clone()
    M.moe_shared_lora(M.Shared.from_dict(se), x, y, y0 is not None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    return y.cpu().numpy().astype(np.float64)


def _check_y(y, y_ref):
    err = np.abs(y - y_ref).max()
    bound = REL_TOL * np.abs(y_ref).max()
    assert err <= bound, f"max|y - oracle| = {err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("qbits", [8, 4])
@pytest.mark.parametrize("rank", [0, 4])
@pytest.mark.parametrize("T", [1, 3, 9, 17])
def test_shared_lora_tiny(qbits, rank, T):
    sc = W.SharedConfig("t", D=64, F=96, qbits=qbits, scale_dtype=torch.float32, rank=rank,
                        alpha=2.0 * max(rank, 1), lora_dtype=torch.float32, x_dtype=torch.float32,
                        weight_sigma=0.1, lora_a_sigma=0.2, lora_b_sigma=0.2, cfg_id=400 + rank)
    se = _to(W.make_shared_expert(sc, 0, "cpu"), DEV)
    x = W.make_shared_tokens(sc, T, 0, "cpu").to(DEV)
    _check_y(gpu_shared(se, x), oracle.shared_lora(se, x))


@pytest.mark.parametrize("T", [1, 16])
def test_shared_lora_decode_shape(T):
    # the shared expert of the 2048-wide decode layer: int4 base, fp16 scales,
    # rank-16 bf16 adapters, bf16 x
    sc = W.SHARED_CONFIGS["decode"]
    se = _to(W.make_shared_expert(sc, 0, "cpu"), DEV)
    x = W.make_shared_tokens(sc, T, 1, "cpu").to(DEV)
    y_ref = oracle.shared_lora(se, x)
    _check_y(gpu_shared(se, x), y_ref)
    # the adapter's contribution is resolved, not lost in the tolerance
    base = dict(se)
    for p in ("gate", "up", "down"):
        base[p + "_A"] = base[p + "_B"] = None
    y_base = oracle.shared_lora(base, x)
    y_gpu_base = gpu_shared(base, x)
    _check_y(y_gpu_base, y_base)
    delta_ref = y_ref - y_base
    delta_gpu = gpu_shared(se, x) - y_gpu_base
    assert np.abs(delta_ref).max() > 0
    np.testing.assert_allclose(delta_gpu, delta_ref, rtol=0, atol=0.05 * np.abs(delta_ref).max())


def test_shared_lora_accumulates_into_y_and_int8_bf16_adapters():
    sc = W.SharedConfig("t8", D=256, F=128, qbits=8, scale_dtype=torch.float16, rank=8, alpha=16.0,
                        lora_dtype=torch.bfloat16, x_dtype=torch.bfloat16, cfg_id=410)
    se = _to(W.make_shared_expert(sc, 0, "cpu"), DEV)
    x = W.make_shared_tokens(sc, 5, 0, "cpu").to(DEV)
    y0 = torch.randn(5, sc.D, device=DEV, generator=torch.Generator(DEV).manual_seed(3))
    y = gpu_shared(se, x, y0)
    _check_y(y, y0.cpu().numpy().astype(np.float64) + oracle.shared_lora(se, x))


# ------------------------------------------------------------ prerouter head

def gpu_preroute(cfg, head, x, cur, prev):
    T = x.shape[0]
    E = head["fc2"].shape[0]
    H = head["fc1"].shape[0]
    ws = M.workspace(M.MOE_OP_PREROUTE, T, cfg.k, E, cfg.D, H, DEV)
    out = dict(idx=torch.empty(T, cfg.k, dtype=torch.int32, device=DEV),
               w=torch.empty(T, cfg.k, dtype=torch.float32, device=DEV),
               probs=torch.empty(T, E, dtype=torch.float32, device=DEV))
    M.moe_preroute(M.Prerouter.from_dict(head, cfg.k), x, cur, prev, out["idx"], out["w"], out["probs"], ws)
    status = M.moe_check_status(ws)
    return {k: v.cpu().numpy() for k, v in out.items()}, status


def tiny_head_cfg(seed):
    return W.LayerConfig("t", E=12, k=3, D=32, F=32, T=4, qbits=8, scale_dtype=torch.float32,
                         x_dtype=torch.float32, router_dtype=torch.float32, router_sigma=0.3,
                         zipf=1.1, layers=2, cfg_id=420 + seed)


@pytest.mark.parametrize("T", [1, 5, 11])
def test_preroute_tiny(T):
    cfg = tiny_head_cfg(T)
    head = _to(W.make_prerouter(cfg, 0, H=32, device="cpu", sigma=0.3, hot_sigma=0.5), DEV)
    x = W.make_tokens(cfg, T, 0, "cpu").to(DEV)
    cur, prev = W.make_routing_history(cfg, T, stream=T, device=DEV)
    prev[0] = -1                  # the first token has no previous token
    if T > 1:
        cur[1, 2] = cur[1, 1]     # a repeated id counts once
    got, status = gpu_preroute(cfg, head, x, cur, prev)
    assert status == M.MOE_OK
    ref = oracle.prerouter(head, x, cur, prev, cfg.k)
    parity.check_routing(ref, got, cfg.k, label=f"prerouter tiny T={T}")


@pytest.mark.parametrize("T", [1, 16])
def test_preroute_decode_shape_feeds_decode(T):
    # the head of the 256-expert decode layer (input 2048 + 2*256, hidden 512)
    # predicts the next layer's routing, which is then used as that layer's
    # routing by moe_decode (prediction-as-routing)
    cfg = W.CONFIGS[1]
    head = _to(W.make_prerouter(cfg, 0, H=512, device="cpu"), DEV)
    x = W.make_tokens(cfg, T, 5, "cpu").to(DEV)
    cur, prev = W.make_routing_history(cfg, T, stream=5, device=DEV, absent_prev=(T == 1))
    got, status = gpu_preroute(cfg, head, x, cur, prev)
    assert status == M.MOE_OK
    ref = oracle.prerouter(head, x, cur, prev, cfg.k)
    parity.check_routing(ref, got, cfg.k, label=f"prerouter E256 T={T}")

    nxt = W.make_layer(cfg, 1, DEV)
    experts = M.Experts.from_layer(nxt, cfg.qbits)
    idx = torch.from_numpy(got["idx"]).to(DEV)
    w = torch.from_numpy(got["w"]).to(DEV)
    y = torch.empty(T, cfg.D, dtype=torch.float32, device=DEV)
    ws = M.workspace(M.MOE_OP_DECODE, T, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_decode(experts, x, idx, w, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    parity.check_y(nxt, x, got["idx"], got["w"], y.cpu().numpy(), cfg.qbits)


def test_preroute_records_an_out_of_range_id_and_skips_it():
    cfg = tiny_head_cfg(9)
    head = _to(W.make_prerouter(cfg, 0, H=32, device="cpu", sigma=0.3, hot_sigma=0.5), DEV)
    x = W.make_tokens(cfg, 2, 0, "cpu").to(DEV)
    cur, prev = W.make_routing_history(cfg, 2, stream=9, device=DEV)
    bad = cur.clone()
    bad[1, 0] = cfg.E + 5
    got, status = gpu_preroute(cfg, head, x, bad, prev)
    assert status == M.MOE_ERR_BAD_INDEX
    # the skipped entry acts as an absent one
    absent = cur.clone()
    absent[1, 0] = -1
    ref = oracle.prerouter(head, x, absent, prev, cfg.k)
    parity.check_routing(ref, got, cfg.k, label="prerouter bad id")
