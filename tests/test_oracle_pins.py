"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks ``oracle/`` against a closed form, an invariant of the
mathematics, a special case that reduces to a simpler computation, or the
independent NumPy brute force in ``tests/brute.py``. The planted-mistake tests at
the end rebuild the oracle with one plausible bug at a time and check that at
least one of these pins fails for every such bug.
"""
from __future__ import annotations

import json
import math
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from brute import (dense_experts, dense_masked_moe, dequant, softmax, stable_topk,
                   substitute_bruteforce, to_np, unpack_codes)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s):
    return float(Fraction(s))


def tiny_layer(E=6, D=64, F=96, qbits=8, scale_dtype=torch.float32, seed=0, router_sigma=0.3,
               zipf=None):
    cfg = W.LayerConfig("t", E=E, k=2, D=D, F=F, T=4, qbits=qbits, scale_dtype=scale_dtype,
                        x_dtype=torch.float32, router_dtype=torch.float32,
                        router_sigma=router_sigma, zipf=zipf, layers=1, cfg_id=100 + seed,
                        weight_sigma=0.1)
    return cfg, W.make_layer(cfg, 0, "cpu")


def full_weights(T, E, idx, w):
    wf = np.zeros((T, E))
    for t in range(T):
        for r in range(idx.shape[1]):
            wf[t, idx[t, r]] += w[t, r]
    return wf


# ---------------------------------------------------------------- router

def test_router_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "router_ties.json")))
    c = np.array(g["c"], dtype=np.float64)
    Wr = np.log(c)[:, None]
    x = np.ones((1, 1))
    r = oracle.router(x, Wr, None, g["k"])
    np.testing.assert_allclose(r["probs"][0], [_frac(s) for s in g["probs"]], rtol=1e-14)
    assert r["idx"][0].tolist() == g["idx"]
    np.testing.assert_allclose(r["w"][0], [_frac(s) for s in g["w"]], rtol=1e-14)


def test_router_matches_numpy_softmax_and_full_sort():
    rng = np.random.default_rng(1)
    T, E, D, k = 7, 40, 96, 5
    x = rng.standard_normal((T, D))
    Wr = rng.standard_normal((E, D)) * 0.2
    b = rng.standard_normal(E)
    r = oracle.router(x, Wr, b, k)
    logits = x @ Wr.T + b
    np.testing.assert_allclose(r["logits"], logits, rtol=1e-12, atol=1e-12)
    p = softmax(logits)
    np.testing.assert_allclose(r["probs"], p, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["probs"].sum(1), 1.0, rtol=0, atol=1e-12)
    assert np.array_equal(r["probs32"], p.astype(np.float32))
    assert np.array_equal(r["idx"], stable_topk(r["probs32"], k))
    ws = p[np.arange(T)[:, None], r["idx"]]
    np.testing.assert_allclose(r["w"], ws / ws.sum(1, keepdims=True), rtol=1e-12)
    r0 = oracle.router(x, Wr, b, k, norm_topk=False)
    np.testing.assert_allclose(r0["w"], ws, rtol=1e-12)


def test_router_all_equal_logits_takes_lowest_indices():
    E, k = 16, 4
    r = oracle.router(np.zeros((2, 32)), np.ones((E, 32)), None, k)
    assert r["idx"].tolist() == [[0, 1, 2, 3]] * 2
    np.testing.assert_allclose(r["probs"], 1.0 / E, rtol=1e-15)
    np.testing.assert_allclose(r["w"], 1.0 / k, rtol=1e-15)


def test_one_hot_router():
    rng = np.random.default_rng(2)
    E, D = 32, 64
    for estar in (0, 17, 31):
        b = np.zeros(E)
        b[estar] = 30.0
        r = oracle.router(rng.standard_normal((3, D)) * 0.01, rng.standard_normal((E, D)) * 0.01,
                          b, 1)
        assert (r["idx"][:, 0] == estar).all()
        np.testing.assert_allclose(r["w"], 1.0, rtol=0, atol=0)


def test_router_k_equals_e_weights_are_probs():
    rng = np.random.default_rng(3)
    E = 12
    r = oracle.router(rng.standard_normal((4, 32)), rng.standard_normal((E, 32)), None, E)
    for t in range(4):
        np.testing.assert_allclose(r["w"][t], r["probs"][t][r["idx"][t]], rtol=1e-12)
        assert sorted(r["idx"][t].tolist()) == list(range(E))


# ------------------------------------------------------- expert arithmetic

def _structured_layer(qbits):
    """Permutation-structured experts whose output has a closed form.

    Expert e: Gate row n has a single code a at column (5n + 2 + e) % D, Up row n a
    single code b at column (3n + 1 + e) % D, Down row d a single code c at column
    (7d + 3 + e) % F. Then g_n = a*sg*x[pg(n)], u_n = b*su*x[pu(n)],
    o_d = c*sd*h[pd(d)]. A transposed operand or a mixed-up index changes which
    element is picked, so the closed form fails.
    """
    E, D, F = 3, 32, 32
    a, b, c = (-127, 113, -1) if qbits == 8 else (-7, 5, -1)
    sg, su, sd = 0.5, 0.25, 2.0
    gq = np.zeros((E, F, D), np.int64)
    uq = np.zeros((E, F, D), np.int64)
    dqc = np.zeros((E, D, F), np.int64)
    for e in range(E):
        for n in range(F):
            gq[e, n, (5 * n + 2 + e) % D] = a
            uq[e, n, (3 * n + 1 + e) % D] = b
        for d in range(D):
            dqc[e, d, (7 * d + 3 + e) % F] = c

    def enc(q):
        q8 = q.astype(np.int8)
        if qbits == 8:
            return q8
        return W.pack_int4(torch.from_numpy(q8)).numpy()
    layer = dict(gate_q=enc(gq), up_q=enc(uq), down_q=enc(dqc),
                 gate_s=np.full((E, F, D // 32), sg), up_s=np.full((E, F, D // 32), su),
                 down_s=np.full((E, D, F // 32), sd))
    return layer, (a, b, c, sg, su, sd), (E, D, F)


@pytest.mark.parametrize("qbits", [8, 4])
def test_structured_expert_closed_form(qbits):
    layer, (a, b, c, sg, su, sd), (E, D, F) = _structured_layer(qbits)
    x = np.array([[(i - 13.5) / 7.0 for i in range(D)], [math.sin(i) for i in range(D)]])
    idx = np.array([[2, 0], [1, 2]], np.int32)
    w = np.array([[0.7, 0.3], [0.45, 0.55]])
    y = oracle.moe(layer, x, idx, w, qbits, compact=False)
    expect = np.zeros((2, D))
    for t in range(2):
        for r in range(2):
            e = idx[t, r]
            for d in range(D):
                n = (7 * d + 3 + e) % F
                g = a * sg * x[t, (5 * n + 2 + e) % D]
                u = b * su * x[t, (3 * n + 1 + e) % D]
                h = g / (1.0 + math.exp(-g)) * u
                expect[t, d] += w[t, r] * c * sd * h
    np.testing.assert_allclose(y, expect, rtol=1e-13, atol=1e-15)


def test_int4_nibbles_golden():
    g = json.load(open(os.path.join(GOLDEN, "int4_nibbles.json")))
    nb = len(g["bytes"])
    K = 64  # one row of 64 codes: the fixture bytes, then zeros
    row = np.zeros(K // 2, np.uint8)
    row[:nb] = g["bytes"]
    # Gate = that row for every output n; x = one-hot e_k picks code k * scale.
    F, D = 32, K
    gq = np.tile(row, (1, F, 1))
    layer = dict(gate_q=gq, up_q=np.zeros_like(gq), down_q=np.zeros((1, D, F // 2), np.uint8),
                 gate_s=np.ones((1, F, D // 32)), up_s=np.ones((1, F, D // 32)),
                 down_s=np.ones((1, D, F // 32)))
    # the brute force's unpacking agrees with the hand-derived codes
    codes = unpack_codes(gq[0, 0], 4)
    assert codes[0:2 * nb:2].tolist() == g["even_codes"]
    assert codes[1:2 * nb:2].tolist() == g["odd_codes"]
    # the oracle's unpacking: up = gate, down = identity on the first F outputs,
    # x = e_k, so y[n] = silu(code_k) * code_k for every n < F
    layer["up_q"] = gq.copy()
    dq_row = np.zeros((D, F), np.int64)
    for d in range(D):
        dq_row[d, d % F] = 1 if d < F else 0
    layer["down_q"] = W.pack_int4(torch.from_numpy(dq_row.astype(np.int8)))[None].numpy()
    for kk in range(2 * nb):
        x = np.zeros((1, D))
        x[0, kk] = 1.0
        y = oracle.moe(layer, x, np.zeros((1, 1), np.int32), np.ones((1, 1)), 4, compact=False)
        q = (g["even_codes"] if kk % 2 == 0 else g["odd_codes"])[kk // 2]
        h = q / (1.0 + math.exp(-q)) * q
        np.testing.assert_allclose(y[0, :F], h, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("qbits,scale_dtype", [(8, torch.float32), (8, torch.float16),
                                                (4, torch.float16)])
def test_masked_dense_equals_gathered(qbits, scale_dtype):
    cfg, layer = tiny_layer(qbits=qbits, scale_dtype=scale_dtype, seed=qbits)
    rng = np.random.default_rng(4)
    T, k = 5, 3
    x = rng.standard_normal((T, cfg.D))
    r = oracle.router(x, layer["Wr"], None, k)
    y = oracle.moe(layer, x, r["idx"], r["w"], qbits)
    y_dense = dense_masked_moe(layer, x, full_weights(T, cfg.E, r["idx"], r["w"]), qbits)
    np.testing.assert_allclose(y, y_dense, rtol=1e-12, atol=1e-12 * np.abs(y_dense).max())


def test_k_equals_e_is_dense_moe():
    cfg, layer = tiny_layer(seed=5)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, cfg.D))
    r = oracle.layer_forward(layer, x, cfg.E, 8)
    p = softmax(x @ to_np(layer["Wr"]).T)
    y_dense = dense_masked_moe(layer, x, p, 8)
    np.testing.assert_allclose(r["y"], y_dense, rtol=1e-11, atol=1e-12 * np.abs(y_dense).max())


def test_one_hot_equals_selected_expert_mlp():
    cfg, layer = tiny_layer(seed=6)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, cfg.D))
    o = dense_experts(layer, x, 8)
    for e in range(cfg.E):
        y = oracle.moe(layer, x, np.full((2, 1), e, np.int32), np.ones((2, 1)), 8)
        np.testing.assert_allclose(y, o[:, e, :], rtol=1e-12, atol=1e-14)


def test_unrouted_experts_do_not_matter():
    cfg, layer = tiny_layer(seed=7)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((2, cfg.D))
    idx = np.array([[1, 4], [4, 0]], np.int32)
    w = np.array([[0.6, 0.4], [0.5, 0.5]])
    y = oracle.moe(layer, x, idx, w, 8, compact=False)
    poisoned = {n: to_np(v).copy() for n, v in layer.items() if n.endswith(("_q", "_s"))}
    for n in ("gate_s", "up_s", "down_s"):
        for e in (2, 3, 5):
            poisoned[n][e] = np.nan
    y2 = oracle.moe(poisoned, x, idx, w, 8, compact=False)
    assert np.array_equal(y, y2)


def test_down_takes_each_slots_own_activation():
    """Qiita gather_qmm section 7: feeding the shared x to down instead of the
    expert's own h corrupts the output silently (relative error of order 1)."""
    cfg, layer = tiny_layer(D=64, F=64, seed=8)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((4, cfg.D))
    r = oracle.layer_forward(layer, x, 2, 8)
    Dn = dequant(to_np(layer["down_q"]), to_np(layer["down_s"]), 8)
    wrong = np.zeros_like(r["y"])
    for t in range(4):
        for s in range(2):
            wrong[t] += r["w"][t, s] * (Dn[r["idx"][t, s]] @ x[t])
    rel = np.abs(wrong - r["y"]).max() / np.abs(r["y"]).max()
    assert rel > 0.5


def test_quantizer_round_trip():
    g = torch.Generator().manual_seed(9)
    w = torch.randn(4, 8, 128, generator=g) * 0.02
    for qbits, qmax in ((8, 127), (4, 7)):
        for sd in (torch.float32, torch.float16):
            q, s = W.quantize_sym_blk32(w, qbits, sd)
            codes = unpack_codes(q.numpy(), qbits)
            assert np.abs(codes).max() <= qmax
            sf = np.repeat(s.double().numpy(), 32, axis=-1)
            err = np.abs(w.double().numpy() - codes * sf)
            # half a step, plus the scale's own rounding when stored in fp16
            slack = 1e-7 if sd == torch.float32 else 2.0 ** -11 * qmax
            assert (err <= sf * (0.5 + slack) + 1e-12).all()


# ----------------------------------------------------------- substitution

def _sub_case(seed, T=6, E=24, k=5, n_res=7):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, 32))
    r = oracle.router(x, rng.standard_normal((E, 32)) * 0.6, None, k)
    res = np.zeros(E, np.uint8)
    res[rng.permutation(E)[:n_res]] = 1
    return r, res


@pytest.mark.parametrize("threshold", [0.0, 0.15, 0.3, float("inf")])
def test_substitution_matches_bruteforce(threshold):
    for seed in range(5):
        r, res = _sub_case(seed)
        s = oracle.substitute(r["probs32"], r["idx"], r["w"], res, threshold)
        idx2, flag, mass = substitute_bruteforce(r["probs32"], r["idx"], r["w"], res, threshold)
        assert np.array_equal(s["idx"], idx2)
        assert np.array_equal(s["flag"], flag)
        np.testing.assert_allclose(s["mass"], mass, rtol=1e-15, atol=0)
        np.testing.assert_array_equal(s["w"], r["w"])


def test_substitution_special_cases():
    r, res = _sub_case(11)
    T, k = r["idx"].shape
    s0 = oracle.substitute(r["probs32"], r["idx"], r["w"], res, 0.0)
    assert np.array_equal(s0["idx"], r["idx"]) and (s0["mass"] == 0).all()
    assert set(np.unique(s0["flag"])) <= {0, 1}
    sinf = oracle.substitute(r["probs32"], r["idx"], r["w"], res, float("inf"))
    miss = res[r["idx"]] == 0
    assert (sinf["flag"][:, 0] == np.where(miss[:, 0], 1, 0)).all()
    assert (sinf["flag"][:, 1:][miss[:, 1:]] == 2).all()
    assert (res[sinf["idx"][:, 1:]] == 1).all()
    np.testing.assert_array_less(sinf["mass"], 1.0 - r["w"][:, 0] + 1e-12)
    all_res = np.ones_like(res)
    sa = oracle.substitute(r["probs32"], r["idx"], r["w"], all_res, 0.15)
    assert np.array_equal(sa["idx"], r["idx"]) and (sa["flag"] == 0).all() and (sa["mass"] == 0).all()
    # replacements are distinct from each other and from the original routed set
    for t in range(T):
        assert len(set(sinf["idx"][t].tolist())) == k


def test_substitution_threshold_is_inclusive():
    """gist.science method section: a miss is fetched when its gate weight is >= 0.15."""
    E, k = 8, 3
    p = np.linspace(0.2, 0.05, E).astype(np.float32)[None]
    idx = np.array([[0, 1, 2]], np.int32)
    w = np.array([[0.6, float(np.float32(0.15)), 0.25 - 1e-9]])
    res = np.zeros(E, np.uint8)
    res[5:] = 1
    s = oracle.substitute(p, idx, w, res, 0.15)
    assert s["flag"][0].tolist() == [1, 1, 1]
    w2 = np.array([[0.6, float(np.nextafter(np.float32(0.15), np.float32(0))), 0.3]])
    s2 = oracle.substitute(p, idx, w2, res, 0.15)
    assert s2["flag"][0].tolist() == [1, 2, 1] and s2["idx"][0, 1] == 5


# ------------------------------------------------------------ permutation

def test_permutation_is_stable_counting_sort():
    rng = np.random.default_rng(12)
    for T, k, E in ((1, 8, 256), (37, 4, 9), (300, 8, 64)):
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
        p = oracle.permute(idx, E)
        flat = idx.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(p["perm_tok"], order // k)
        assert np.array_equal(p["perm_slot"], order % k)
        assert np.array_equal(p["cnt"], np.bincount(flat, minlength=E))
        assert p["off"][0] == 0 and np.array_equal(np.diff(p["off"]), p["cnt"])
        assert p["off"][-1] == T * k
        pos = np.empty(T * k, np.int64)
        pos[order] = np.arange(T * k)
        assert np.array_equal(p["inv"].reshape(-1), pos)


def test_cfg0_layer_against_bruteforce():
    cfg = W.CONFIGS[0]
    layer = W.make_layer(cfg, 0, "cpu")
    x = W.make_tokens(cfg, cfg.T, 0, "cpu")
    r = oracle.layer_forward(layer, x, cfg.k, cfg.qbits)
    xn = to_np(x)
    p = softmax(xn @ to_np(layer["Wr"]).T)
    np.testing.assert_allclose(r["probs"], p, rtol=1e-12)
    assert np.array_equal(r["idx"], stable_topk(p.astype(np.float32), cfg.k))
    yd = dense_masked_moe(layer, xn, full_weights(cfg.T, cfg.E, r["idx"], r["w"]), cfg.qbits)
    np.testing.assert_allclose(r["y"], yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())


# -------------------------------------------------------- planted mistakes

MUTANTS = {
    "down_reads_shared_x": ("acc += dq(dq_codes, ds, qbits, F, d, n) * h[n];",
                            "acc += dq(dq_codes, ds, qbits, F, d, n) * x[n];"),
    "no_int8_sign_extension": ("return (int)(int8_t)row[k];", "return (int)row[k];"),
    "int4_nibbles_swapped": ("int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);",
                             "int nib = (k & 1) ? (byte & 0xF) : (byte >> 4);"),
    "int4_no_sign_extension": ("return nib >= 8 ? nib - 16 : nib;", "return nib;"),
    "scale_of_wrong_row": ("scales[n * (K / BLK) + k / BLK]", "scales[k / BLK]"),
    "scale_of_wrong_block": ("scales[n * (K / BLK) + k / BLK]", "scales[n * (K / BLK)]"),
    "slot_weight_dropped": ("acc += w[t * k + r] * o[(t * k + r) * D + d];",
                            "acc += o[(t * k + r) * D + d];"),
    "gate_up_swapped": ("h[n] = g / (1.0 + exp(-g)) * u;", "h[n] = u / (1.0 + exp(-u)) * g;"),
    "tie_break_reversed": ("    return a < b;\n}", "    return a > b;\n}"),
    "no_renormalisation": ("norm_topk ? pt[order[r]] / norm : pt[order[r]]", "pt[order[r]]"),
    "first_choice_not_protected": ("if (r == 0 || (float)w[o] >= thr32)", "if ((float)w[o] >= thr32)"),
    "threshold_exclusive": ("(float)w[o] >= thr32", "(float)w[o] > thr32"),
    "replacement_may_repeat": ("            taken[best] = 1;\n", ""),
    "permutation_unstable": ("for (int t = 0; t < T; t++)\n        for (int r = 0; r < k; r++) {",
                             "for (int t = T - 1; t >= 0; t--)\n        for (int r = 0; r < k; r++) {"),
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
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c),
                           "-lm"])
    return oracle.load_variant(str(so))


def _pins_pass(lib) -> bool:
    """A compact replay of the pins above against another oracle build."""
    try:
        g = json.load(open(os.path.join(GOLDEN, "router_ties.json")))
        r = oracle.router(np.ones((1, 1)), np.log(np.array(g["c"], float))[:, None], None, g["k"],
                          lib=lib)
        if r["idx"][0].tolist() != g["idx"]:
            return False
        if not np.allclose(r["w"][0], [_frac(s) for s in g["w"]], rtol=1e-14):
            return False
        for qbits in (8, 4):
            layer, (a, b, c, sg, su, sd), (E, D, F) = _structured_layer(qbits)
            x = np.array([[(i - 13.5) / 7.0 for i in range(D)]])
            idx = np.array([[2, 0]], np.int32)
            w = np.array([[0.7, 0.3]])
            y = oracle.moe(layer, x, idx, w, qbits, compact=False, lib=lib)
            exp_ = np.zeros(D)
            for rr in range(2):
                e = idx[0, rr]
                for d in range(D):
                    n = (7 * d + 3 + e) % F
                    gg = a * sg * x[0, (5 * n + 2 + e) % D]
                    uu = b * su * x[0, (3 * n + 1 + e) % D]
                    exp_[d] += w[0, rr] * c * sd * gg / (1 + math.exp(-gg)) * uu
            if not np.allclose(y[0], exp_, rtol=1e-12, atol=1e-14):
                return False
        for qbits in (8, 4):
            cfg, layer = tiny_layer(D=64, F=64, qbits=qbits, scale_dtype=torch.float16, seed=20)
            x = np.random.default_rng(20).standard_normal((4, 64))
            rr = oracle.router(x, layer["Wr"], None, 3, lib=lib)
            y = oracle.moe(layer, x, rr["idx"], rr["w"], qbits, lib=lib)
            yd = dense_masked_moe(layer, x, full_weights(4, cfg.E, rr["idx"], rr["w"]), qbits)
            if not np.allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max()):
                return False
        for thr in (0.15, float("inf")):
            for seed in range(3):
                rs, res = _sub_case(seed)
                s = oracle.substitute(rs["probs32"], rs["idx"], rs["w"], res, thr, lib=lib)
                i2, f2, m2 = substitute_bruteforce(rs["probs32"], rs["idx"], rs["w"], res, thr)
                if not (np.array_equal(s["idx"], i2) and np.array_equal(s["flag"], f2)):
                    return False
        p = np.linspace(0.2, 0.05, 8).astype(np.float32)[None]
        res = np.zeros(8, np.uint8)
        res[5:] = 1
        s = oracle.substitute(p, np.array([[0, 1, 2]], np.int32),
                              np.array([[0.6, float(np.float32(0.15)), 0.25]]), res, 0.15, lib=lib)
        if s["flag"][0].tolist() != [1, 1, 1]:
            return False
        idx = np.random.default_rng(21).integers(0, 9, size=(37, 4)).astype(np.int32)
        pp = oracle.permute(idx, 9, lib=lib)
        if not np.array_equal(pp["perm_tok"], np.argsort(idx.reshape(-1), kind="stable") // 4):
            return False
        return True
    except ValueError:
        return False


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass(oracle._load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    assert not _pins_pass(lib), f"planted mistake {name} passed every pin"


# ------------------------------------------------- near-tie exclusion rules

def _exact(expr: str) -> float:
    """Value of a golden's arithmetic expression (numbers, + - * **), computed
    exactly with fractions and then rounded once to fp32."""
    import ast

    def ev(n):
        if isinstance(n, ast.Expression):
            return ev(n.body)
        if isinstance(n, ast.Constant) and isinstance(n.value, (int, float)):
            return Fraction(str(n.value))
        if isinstance(n, ast.UnaryOp) and isinstance(n.op, ast.USub):
            return -ev(n.operand)
        if isinstance(n, ast.BinOp):
            a, b = ev(n.left), ev(n.right)
            if isinstance(n.op, ast.Add):
                return a + b
            if isinstance(n.op, ast.Sub):
                return a - b
            if isinstance(n.op, ast.Mult):
                return a * b
            if isinstance(n.op, ast.Pow) and b.denominator == 1:
                return a ** int(b)
        raise ValueError(f"unsupported expression {expr!r}")

    v = ev(ast.parse(expr, mode="eval"))
    f32 = np.float32(float(v))
    assert Fraction(float(f32)) == v, f"{expr} is not exactly representable in fp32"
    return float(f32)


def test_near_tie_tokens_golden():
    g = json.load(open(os.path.join(GOLDEN, "near_ties.json")))
    for case in g["cases"]:
        p = np.array([[_exact(v) for v in row] for row in case["rows"]], dtype=np.float32)
        got = oracle.near_tie_tokens(p, case["k"]).tolist()
        assert got == case["excluded"], (case["why"], got)


def test_substitution_near_ties_golden():
    g = json.load(open(os.path.join(GOLDEN, "substitution_ties.json")))
    toks = g["tokens"]
    p = np.array([[_exact(v) for v in t["probs"]] for t in toks], dtype=np.float32)
    idx = np.array([t["idx"] for t in toks], dtype=np.int32)
    w = np.array([t["w"] for t in toks], dtype=np.float64)
    res = np.array(g["resident"], dtype=np.uint8)
    got = oracle.substitution_near_ties(p, idx, w, res, g["threshold"]).tolist()
    assert got == g["ambiguous"], got
    # the rule never fires for fetch-all (threshold 0) through the weight test,
    # nor for the first-choice rule (threshold +inf)
    assert 0 not in oracle.substitution_near_ties(p[:1], idx[:1], w[:1], res, float("inf")).tolist()
    assert oracle.substitution_near_ties(p[:2], idx[:2], w[:2], res, 0.0).tolist() == []
