"""Pins of the oracle's shared expert with an unmerged LoRA and of its prerouter
head (xyznot.com "The Other Half of the Memory Wall: Serving 35B MoEs from SSD
with Trained Routing Prediction", method section: "prerouter head architecture"
and "unmerged adapter execution").

Every pin checks ``oracle/`` against something other than itself: the NumPy
brute force in ``tests/brute.py`` (merged dense matrices, whole-matrix products,
SciPy's erf), textbook values of the normal distribution, and reductions to the
router and expert functions already pinned in ``test_oracle_pins.py``. The
planted-mistake tests rebuild the oracle with one plausible bug at a time and
require a pin to fail for each.
"""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from brute import (merged_dense_shared_lora, prerouter_dense, softmax, stable_topk, to_np)


# ------------------------------------------------------------------ inputs

def tiny_shared(D=64, F=96, qbits=8, rank=4, seed=0, lora_dtype=torch.float32):
    sc = W.SharedConfig("t", D=D, F=F, qbits=qbits, scale_dtype=torch.float32, rank=rank,
                        alpha=2.0 * max(rank, 1), lora_dtype=lora_dtype, x_dtype=torch.float32,
                        weight_sigma=0.1, lora_a_sigma=0.2, lora_b_sigma=0.2, cfg_id=200 + seed)
    return sc, W.make_shared_expert(sc, 0, "cpu")


def tiny_head_cfg(E=12, k=3, D=32, seed=0):
    return W.LayerConfig("t", E=E, k=k, D=D, F=32, T=4, qbits=8, scale_dtype=torch.float32,
                         x_dtype=torch.float32, router_dtype=torch.float32, router_sigma=0.3,
                         zipf=1.1, layers=2, cfg_id=300 + seed)


def tiny_head(E=12, k=3, D=32, H=16, seed=0):
    cfg = tiny_head_cfg(E, k, D, seed)
    head = W.make_prerouter(cfg, 0, H=H, device="cpu", sigma=0.3, hot_sigma=0.5)
    return cfg, head


def _x(T, D, seed):
    return np.random.default_rng(seed).standard_normal((T, D))


# ------------------------------------------------------- shared expert + LoRA

@pytest.mark.parametrize("qbits", [8, 4])
@pytest.mark.parametrize("rank", [1, 4, 16])
def test_shared_lora_equals_merged_dense_bruteforce(qbits, rank):
    sc, se = tiny_shared(qbits=qbits, rank=rank, seed=rank)
    x = _x(5, sc.D, rank)
    y = oracle.shared_lora(se, x)
    yd = merged_dense_shared_lora(se, x)
    np.testing.assert_allclose(y, yd, rtol=1e-11, atol=1e-12 * np.abs(yd).max())


def test_shared_lora_rank0_is_the_plain_expert():
    # without an adapter the shared expert is one routed expert with weight 1,
    # which the pinned routed-expert oracle computes
    for qbits in (8, 4):
        sc, se = tiny_shared(qbits=qbits, rank=0, seed=7)
        x = _x(3, sc.D, 7)
        y = oracle.shared_lora(se, x)
        layer = {n: se[n].unsqueeze(0) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")}
        y1 = oracle.moe(layer, x, np.zeros((3, 1), np.int32), np.ones((3, 1)), qbits, compact=False)
        np.testing.assert_allclose(y, y1, rtol=1e-14, atol=1e-15)


def test_shared_lora_zero_B_is_the_plain_expert_and_the_delta_matters():
    sc, se = tiny_shared(qbits=4, rank=4, seed=8)
    x = _x(3, sc.D, 8)
    base = dict(se)
    for p in ("gate", "up", "down"):
        base[p + "_A"] = base[p + "_B"] = None
    y0 = oracle.shared_lora(base, x)
    zb = dict(se)
    for p in ("gate", "up", "down"):
        zb[p + "_B"] = torch.zeros_like(se[p + "_B"])
    np.testing.assert_allclose(oracle.shared_lora(zb, x), y0, rtol=1e-14, atol=1e-15)
    # with the adapter the output moves, and only through the adapter's scale
    y = oracle.shared_lora(se, x)
    assert np.abs(y - y0).max() > 1e-3 * np.abs(y0).max()
    s0 = dict(se)
    s0["scale"] = 0.0
    np.testing.assert_allclose(oracle.shared_lora(s0, x), y0, rtol=1e-14, atol=1e-15)


def test_shared_lora_down_adapter_reads_the_gated_activation():
    # only the down adapter is non-zero and the base down matrix is zero: then
    # y = scale * B_d (A_d h) with h the SwiGLU of the base gate/up
    sc, se = tiny_shared(D=64, F=64, qbits=8, rank=2, seed=9)
    x = _x(2, sc.D, 9)
    s = dict(se)
    for p in ("gate", "up"):
        s[p + "_B"] = torch.zeros_like(se[p + "_B"])
    s["down_q"] = torch.zeros_like(se["down_q"])
    y = oracle.shared_lora(s, x)
    from brute import dequant
    G = dequant(to_np(se["gate_q"]), to_np(se["gate_s"]), 8)
    U = dequant(to_np(se["up_q"]), to_np(se["up_s"]), 8)
    g, u = x @ G.T, x @ U.T
    h = g / (1 + np.exp(-g)) * u
    exp_ = float(se["scale"]) * (h @ to_np(se["down_A"]).T) @ to_np(se["down_B"]).T
    np.testing.assert_allclose(y, exp_, rtol=1e-11, atol=1e-14)


# ------------------------------------------------------------- prerouter head

# Phi(1) and Phi(-1) of the standard normal distribution (textbook values):
# gelu(z) = z * Phi(z) in its erf form.
PHI_1 = 0.8413447460685429
PHI_M1 = 0.15865525393145707


def test_prerouter_gelu_is_the_erf_form():
    # D = 1, E = 2, H = 2: z = (1, -1), fc2 routes gelu(z_j) to logit j
    fc1 = np.zeros((2, 1 + 4))
    fc1[0, 0] = 1.0
    fc1[1, 0] = -1.0
    head = dict(fc1=fc1, b1=None, fc2=np.eye(2), L=np.zeros((2, 5)), bias=None)
    r = oracle.prerouter(head, np.ones((1, 1)), -np.ones((1, 1), np.int32), -np.ones((1, 1), np.int32), 1)
    np.testing.assert_allclose(r["logits"][0], [1.0 * PHI_1, -1.0 * PHI_M1], rtol=1e-15)


@pytest.mark.parametrize("norm_topk", [True, False])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prerouter_matches_numpy_bruteforce(norm_topk, seed):
    cfg, head = tiny_head(seed=seed)
    x = _x(6, cfg.D, 40 + seed)
    cur, prev = W.make_routing_history(cfg, 6, stream=seed)
    if seed == 2:
        prev[0] = -1  # the first token has no previous token
    r = oracle.prerouter(head, x, cur, prev, cfg.k, norm_topk)
    lg = prerouter_dense(head, x, cur.numpy(), prev.numpy())
    np.testing.assert_allclose(r["logits"], lg, rtol=1e-12, atol=1e-12)
    p = softmax(lg)
    np.testing.assert_allclose(r["probs"], p, rtol=1e-12)
    assert np.array_equal(r["idx"], stable_topk(p.astype(np.float32), cfg.k))
    sel = np.take_along_axis(p, r["idx"].astype(np.int64), axis=1)
    w = sel / sel.sum(axis=1, keepdims=True) if norm_topk else sel
    np.testing.assert_allclose(r["w"], w, rtol=1e-12)


def test_prerouter_without_head_is_the_next_layers_router():
    # fc2 = 0 and routing columns of L = 0: the prediction is the router of
    # layer N+1 (the linear path's warm start) applied to x, which the pinned
    # router oracle computes
    cfg, head = tiny_head(seed=3)
    h = dict(head)
    h["fc2"] = torch.zeros_like(head["fc2"])
    L = head["L"].clone()
    L[:, cfg.D:] = 0
    h["L"] = L
    x = _x(4, cfg.D, 3)
    cur, prev = W.make_routing_history(cfg, 4, stream=3)
    r = oracle.prerouter(h, x, cur, prev, cfg.k)
    Wr, bias = W.make_router(cfg, 1, "cpu")
    ref = oracle.router(x, Wr, bias, cfg.k)
    np.testing.assert_allclose(r["logits"], ref["logits"], rtol=1e-14, atol=1e-14)
    assert np.array_equal(r["idx"], ref["idx"])
    np.testing.assert_allclose(r["w"], ref["w"], rtol=1e-14)


def test_prerouter_khot_inputs():
    cfg, head = tiny_head(seed=4)
    x = _x(3, cfg.D, 4)
    cur, prev = W.make_routing_history(cfg, 3, stream=4)
    base = oracle.prerouter(head, x, cur, prev, cfg.k)
    # a repeated id is one hot entry: repeating it equals leaving the slot absent
    c2, c3 = cur.clone(), cur.clone()
    c2[:, 2] = c2[:, 1]
    c3[:, 2] = -1
    np.testing.assert_allclose(oracle.prerouter(head, x, c2, prev, cfg.k)["logits"],
                               oracle.prerouter(head, x, c3, prev, cfg.k)["logits"], rtol=1e-15)
    # the order of the ids does not matter
    np.testing.assert_allclose(oracle.prerouter(head, x, cur.flip(1), prev.flip(1), cfg.k)["logits"],
                               base["logits"], rtol=1e-13, atol=1e-13)
    # an absent previous token: its columns of fc1 and L are never read
    none = -torch.ones_like(prev)
    a = oracle.prerouter(head, x, cur, none, cfg.k)
    h2 = dict(head)
    E, D = cfg.E, cfg.D
    h2["fc1"] = head["fc1"].clone()
    h2["fc1"][:, D + E:] = 7.0
    h2["L"] = head["L"].clone()
    h2["L"][:, D + E:] = -3.0
    b = oracle.prerouter(h2, x, cur, none, cfg.k)
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=1e-15)
    # while a present previous token does move the prediction
    assert np.abs(base["logits"] - a["logits"]).max() > 1e-3
    with pytest.raises(ValueError):
        bad = cur.clone()
        bad[0, 0] = cfg.E
        oracle.prerouter(head, x, bad, prev, cfg.k)


# -------------------------------------------------------- planted mistakes

MUTANTS = {
    "lora_scale_dropped": ("out[n] = base + scale * delta;", "out[n] = base + delta;"),
    "lora_A_transposed": ("acc += A[j * K + kk] * v[kk];", "acc += A[kk * r + j] * v[kk];"),
    "lora_B_transposed": ("delta += B[n * r + j] * av[j];", "delta += B[j * N + n] * av[j];"),
    "shared_gate_up_swapped": ("h[n] = g[n] / (1.0 + exp(-g[n])) * u[n];",
                               "h[n] = u[n] / (1.0 + exp(-u[n])) * g[n];"),
    "down_adapter_on_base_input": (
        "lora_projection(D, F, r, qbits, down_q, down_s, down_A, down_B, scale, h, av, y + t * D);",
        "lora_projection(D, F, r, qbits, down_q, down_s, down_A, down_B, scale, g, av, y + t * D);"),
    "gelu_tanh_approximation": ("a[j] = 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
                                "a[j] = 0.5 * z * (1.0 + tanh(0.7978845608028654 * (z + 0.044715 * z * z * z)));"),
    "previous_token_dropped": ("if (prev[t * k + r] >= 0) f[D + E + prev[t * k + r]] = 1.0;", ""),
    "current_and_previous_swapped": ("if (cur[t * k + r] >= 0) f[D + cur[t * k + r]] = 1.0;",
                                     "if (cur[t * k + r] >= 0) f[D + E + cur[t * k + r]] = 1.0;",
                                     "if (prev[t * k + r] >= 0) f[D + E + prev[t * k + r]] = 1.0;",
                                     "if (prev[t * k + r] >= 0) f[D + prev[t * k + r]] = 1.0;"),
    "linear_path_dropped": ("lt[e] = head + lin + (bias ? bias[e] : 0.0);",
                            "lt[e] = head + (bias ? bias[e] : 0.0);"),
    "hidden_bias_dropped": ("double z = b1 ? b1[j] : 0.0;", "double z = 0.0;"),
    "hot_counts_repeats": ("f[D + cur[t * k + r]] = 1.0;", "f[D + cur[t * k + r]] += 1.0;"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")).read()
    subs = MUTANTS[name]
    for i in range(0, len(subs), 2):
        assert subs[i] in src, f"anchor for mutant {name} not found"
        src = src.replace(subs[i], subs[i + 1])
    c = tmp_path / f"{name}.c"
    c.write_text(src)
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c), "-lm"])
    return oracle.load_variant(str(so))


def _pins_pass(lib) -> bool:
    """A compact replay of the pins above against another oracle build."""
    try:
        for qbits, rank in ((8, 4), (4, 1)):
            sc, se = tiny_shared(qbits=qbits, rank=rank, seed=rank)
            x = _x(3, sc.D, rank)
            y = oracle.shared_lora(se, x, lib=lib)
            yd = merged_dense_shared_lora(se, x)
            if not np.allclose(y, yd, rtol=1e-11, atol=1e-12 * np.abs(yd).max()):
                return False
        fc1 = np.zeros((2, 5))
        fc1[0, 0], fc1[1, 0] = 1.0, -1.0
        head = dict(fc1=fc1, b1=None, fc2=np.eye(2), L=np.zeros((2, 5)), bias=None)
        r = oracle.prerouter(head, np.ones((1, 1)), -np.ones((1, 1), np.int32),
                             -np.ones((1, 1), np.int32), 1, lib=lib)
        if not np.allclose(r["logits"][0], [PHI_1, -PHI_M1], rtol=1e-15):
            return False
        for seed in (0, 1):
            cfg, head = tiny_head(seed=seed)
            x = _x(4, cfg.D, 40 + seed)
            cur, prev = W.make_routing_history(cfg, 4, stream=seed)
            cur[:, 2] = cur[:, 1]  # a repeated id
            r = oracle.prerouter(head, x, cur, prev, cfg.k, lib=lib)
            lg = prerouter_dense(head, x, cur.numpy(), prev.numpy())
            if not np.allclose(r["logits"], lg, rtol=1e-12, atol=1e-12):
                return False
        return True
    except ValueError:
        return False


def test_edge0_pins_pass_on_the_real_oracle():
    assert _pins_pass(oracle._load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_edge0_planted_mistake_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    assert not _pins_pass(lib), f"planted mistake {name} passed every pin"
