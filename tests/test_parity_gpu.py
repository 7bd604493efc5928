"""GPU path vs the CPU oracle, element by element, through the C ABI.

Criteria (shared with the prefill tests, see tests/parity.py):
  * routing ids: bit-exact, except tokens whose sorted oracle probabilities have
    two neighbours among the first k+1 within 1e-6 (a near tie: another
    summation order may rank them differently); such a token must still get a
    valid top-k under the oracle's probabilities; the number excluded is
    asserted to be small and printed in the pytest summary;
  * routing weights: |gpu - oracle| <= 1e-5; probabilities: |gpu - oracle| <=
    1e-6 + 1e-5 * p (the 2048-term router dot is accumulated in fp32 in
    another order by the tensor-core router of the multi-token paths);
  * layer output y (fp32): max |y_gpu - y_oracle| <= 2e-3 * max |y_oracle| per
    tensor, where the oracle is evaluated on the routing the GPU chose (the
    routing itself is checked separately above), so near-tie tokens are checked
    too;
  * substitution: ids, flags bit-exact and mass within 1e-6 against the
    oracle's routing followed by the oracle's substitution, excluding routing
    near ties and ambiguous substitutions (a weight within 1e-6 of the
    threshold, near-tied replacement candidates), counted and printed.
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


def small_cfg(E, k, D, F, qbits=8, scale=torch.float16, x_dtype=torch.bfloat16,
              router_dtype=torch.bfloat16, zipf=1.1, sigma=0.035, cfg_id=50):
    return W.LayerConfig(f"E{E}k{k}D{D}F{F}q{qbits}", E=E, k=k, D=D, F=F, T=1, qbits=qbits,
                         scale_dtype=scale, x_dtype=x_dtype, router_dtype=router_dtype,
                         router_sigma=sigma, zipf=zipf, layers=1, cfg_id=cfg_id)


def gpu_layer(cfg, layer, x, probs=True, x_next=False):
    T = x.shape[0]
    router = M.Router(layer["Wr"], layer["bias"], cfg.k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    out = dict(idx=torch.empty(T, cfg.k, dtype=torch.int32, device=DEV),
               w=torch.empty(T, cfg.k, dtype=torch.float32, device=DEV),
               probs=torch.empty(T, cfg.E, dtype=torch.float32, device=DEV) if probs else None,
               y=torch.empty(T, cfg.D, dtype=torch.float32, device=DEV),
               x_next=torch.empty_like(x) if x_next else None)
    ws = M.workspace(M.MOE_OP_LAYER, T, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_layer(router, experts, x, out["idx"], out["w"], out["probs"], out["y"], out["x_next"], ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    return {k_: (v.cpu() if v is not None else None) for k_, v in out.items()}


def check_routing(ref, got, k, max_skip_frac=0.1, label=""):
    g = {n: (got[n].numpy() if got.get(n) is not None else None) for n in ("idx", "w", "probs")}
    return parity.check_routing(ref, g, k, max_skip_frac, label=label)


def check_y(layer, x, got, qbits, T=None):
    return parity.check_y(layer, x, got["idx"].numpy(), got["w"].double().numpy(), got["y"].double().numpy(),
                          qbits)


# ------------------------------------------------------------------ tiny

def test_tiny_layer_matches_oracle():
    cfg = W.CONFIGS[0]
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, cfg.T, 0, DEV)
    got = gpu_layer(cfg, layer, x)
    ref = oracle.layer_forward(layer, x, cfg.k, cfg.qbits)
    check_routing(ref, got, cfg.k, label="tiny E8 k2 T4")
    check_y(layer, x, got, cfg.qbits)
    # and against the oracle's own routing, token by token where routing agrees
    np.testing.assert_allclose(got["y"].double().numpy(), ref["y"], rtol=0,
                               atol=REL_TOL * np.abs(ref["y"]).max())


def test_route_then_decode_equals_layer():
    cfg = W.CONFIGS[0]
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, 9, 1, DEV)
    T = x.shape[0]
    router = M.Router(layer["Wr"], layer["bias"], cfg.k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    idx = torch.empty(T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, cfg.k, dtype=torch.float32, device=DEV)
    ws_r = M.workspace(M.MOE_OP_ROUTE, T, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_route(router, x, idx, w, None, ws_r)
    y = torch.empty(T, cfg.D, dtype=torch.float32, device=DEV)
    xn = torch.empty_like(x)
    ws = M.workspace(M.MOE_OP_DECODE, T, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_decode(experts, x, idx, w, y, xn, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    got = gpu_layer(cfg, layer, x)
    assert torch.equal(got["idx"], idx.cpu()) and torch.equal(got["w"], w.cpu())
    assert torch.equal(got["y"], y.cpu())
    assert torch.equal(xn.cpu(), (x.float() + y).to(x.dtype).cpu())


@pytest.mark.parametrize("qbits,scale,x_dtype,rdt", [
    (8, torch.float32, torch.float32, torch.float32),
    (8, torch.float16, torch.bfloat16, torch.bfloat16),
    (4, torch.float16, torch.bfloat16, torch.bfloat16),
    (4, torch.float32, torch.float32, torch.bfloat16),
])
@pytest.mark.parametrize("shape", [(13, 3, 96, 160, 7), (5, 5, 32, 32, 3), (40, 6, 512, 352, 11),
                                   (1, 1, 64, 64, 2)])
def test_ragged_shapes(qbits, scale, x_dtype, rdt, shape):
    E, k, D, F, T = shape
    cfg = small_cfg(E, k, D, F, qbits, scale, x_dtype, rdt, zipf=None, sigma=0.2, cfg_id=60 + qbits)
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, T, 3, DEV)
    got = gpu_layer(cfg, layer, x)
    ref = oracle.layer_forward(layer, x, cfg.k, cfg.qbits)
    check_routing(ref, got, cfg.k, max_skip_frac=0.5, label=f"ragged {shape} q{qbits}")
    check_y(layer, x, got, cfg.qbits)


@pytest.mark.parametrize("qbits,scale,x_dtype,rdt", [
    (8, torch.float32, torch.float32, torch.float32),
    (8, torch.float16, torch.bfloat16, torch.bfloat16),
    (4, torch.float16, torch.bfloat16, torch.bfloat16),
    (4, torch.float32, torch.float32, torch.float32),
])
@pytest.mark.parametrize("shape", [(8, 2, 64, 128), (13, 3, 96, 256), (300, 7, 1024, 512),
                                   (16, 16, 2048, 256), (1, 1, 32, 128), (256, 8, 2048, 768)])
def test_single_token_layer(qbits, scale, x_dtype, rdt, shape):
    """T = 1 runs the persistent one-launch layer kernel (grid barriers, bulk
    copies of the down rows) wherever its shape rules allow."""
    E, k, D, F = shape
    cfg = small_cfg(E, k, D, F, qbits, scale, x_dtype, rdt, zipf=1.1, sigma=0.1, cfg_id=80 + qbits)
    layer = W.make_layer(cfg, 0, DEV)
    for stream in range(3):
        x = W.make_tokens(cfg, 1, stream, DEV)
        got = gpu_layer(cfg, layer, x, x_next=True)
        ref = oracle.layer_forward(layer, x, cfg.k, cfg.qbits)
        check_routing(ref, got, cfg.k, max_skip_frac=1.0, label=f"single token {shape} q{qbits}")
        check_y(layer, x, got, cfg.qbits)
        assert torch.equal(got["x_next"], (x.cpu().float() + got["y"]).to(x.dtype))
        # the same routing through moe_decode (no router phase)
        experts = M.Experts.from_layer(layer, cfg.qbits)
        y2 = torch.empty(1, D, dtype=torch.float32, device=DEV)
        ws = M.workspace(M.MOE_OP_DECODE, 1, k, E, D, F, DEV)
        M.moe_decode(experts, x, got["idx"].to(DEV), got["w"].to(DEV), y2, None, ws)
        assert M.moe_check_status(ws) == M.MOE_OK
        check_y(layer, x, dict(idx=got["idx"], w=got["w"], y=y2.cpu()), cfg.qbits)


def test_single_token_repeated_launches_reuse_workspace():
    """Back-to-back persistent launches on one workspace: every launch tags
    its exchanges with a new sequence number and leaves no counter behind."""
    cfg = small_cfg(64, 4, 512, 256, cfg_id=90)
    layer = W.make_layer(cfg, 0, DEV)
    router = M.Router(layer["Wr"], layer["bias"], cfg.k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    ws = M.workspace(M.MOE_OP_LAYER, 1, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    xs = [W.make_tokens(cfg, 1, s, DEV) for s in range(20)]
    outs = []
    for x in xs:
        idx = torch.empty(1, cfg.k, dtype=torch.int32, device=DEV)
        w = torch.empty(1, cfg.k, device=DEV)
        y = torch.empty(1, cfg.D, device=DEV)
        M.moe_layer(router, experts, x, idx, w, None, y, None, ws)
        outs.append((x, idx, w, y))
    assert M.moe_check_status(ws) == M.MOE_OK
    hdr = ws[:16].view(torch.int32).cpu().tolist()
    assert hdr[1] == 0 and hdr[3] == 0, f"counters not reset: {hdr}"
    for x, idx, w, y in outs[::5]:
        check_y(layer, x, dict(idx=idx.cpu(), w=w.cpu(), y=y.cpu()), cfg.qbits)


def test_k_equals_e_and_one_hot():
    cfg = small_cfg(8, 8, 64, 96, zipf=None, sigma=0.2, cfg_id=70)
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, 6, 0, DEV)
    got = gpu_layer(cfg, layer, x)
    ref = oracle.layer_forward(layer, x, cfg.k, cfg.qbits)
    check_routing(ref, got, cfg.k, label="k = E = 8")
    check_y(layer, x, got, cfg.qbits)
    np.testing.assert_allclose(got["w"].numpy().sum(1), 1.0, atol=1e-6)
    # one-hot router: bias +30 on expert 5, k = 1 -> y = that expert's MLP
    cfg1 = small_cfg(8, 1, 64, 96, zipf=None, sigma=0.01, cfg_id=71)
    layer1 = W.make_layer(cfg1, 0, DEV)
    layer1["bias"] = torch.zeros(8, device=DEV)
    layer1["bias"][5] = 30.0
    got1 = gpu_layer(cfg1, layer1, x)
    assert (got1["idx"] == 5).all() and torch.allclose(got1["w"], torch.ones_like(got1["w"]))
    y_ref = oracle.moe(layer1, x, np.full((6, 1), 5, np.int32), np.ones((6, 1)), 8)
    assert np.abs(got1["y"].double().numpy() - y_ref).max() <= REL_TOL * np.abs(y_ref).max()


# -------------------------------------------------- decode (256 experts)

@pytest.fixture(scope="module")
def cfg1_layers():
    cfg = W.CONFIGS[1]
    return cfg, [W.make_layer(cfg, l, DEV, chunk=64) for l in range(3)]


def test_decode_e256_chain_matches_oracle(cfg1_layers):
    """Three chained layers at T=1: each GPU layer is fed the oracle's input so
    a near tie in one layer cannot carry into the next."""
    cfg, layers = cfg1_layers
    x = W.make_tokens(cfg, 1, 0, DEV)
    skipped = 0
    for l, layer in enumerate(layers):
        got = gpu_layer(cfg, layer, x, x_next=True)
        ref = oracle.layer_forward(layer, x, cfg.k, cfg.qbits)
        skipped += check_routing(ref, got, cfg.k, max_skip_frac=1.0, label="decode E256 chain")
        check_y(layer, x, got, cfg.qbits)
        # x_{l+1} = bf16(x_l + y_l), built from the oracle's y
        x = (x.cpu().double() + torch.from_numpy(ref["y"])).to(torch.bfloat16).to(DEV)
    assert skipped <= 1


@pytest.mark.parametrize("T", [1, 2, 4, 7, 8, 16, 32, 64])
def test_batched_decode_sweep(cfg1_layers, T):
    cfg, layers = cfg1_layers
    layer = layers[0]
    x = W.make_tokens(cfg, T, 7, DEV)
    got = gpu_layer(cfg, layer, x)
    ref = oracle.router(x, layer["Wr"], layer["bias"], cfg.k)
    check_routing(ref, got, cfg.k, label=f"batched decode E256 T={T}")
    check_y(layer, x, got, cfg.qbits)


def test_deterministic_reruns(cfg1_layers):
    cfg, layers = cfg1_layers
    x = W.make_tokens(cfg, 4, 9, DEV)
    a = gpu_layer(cfg, layers[1], x)
    for _ in range(5):
        b = gpu_layer(cfg, layers[1], x)
        assert torch.equal(a["y"], b["y"]) and torch.equal(a["idx"], b["idx"])


def test_cuda_graph_replay_matches_eager(cfg1_layers):
    cfg, layers = cfg1_layers
    T = 2
    x = W.make_tokens(cfg, T, 11, DEV)
    router = M.Router(layers[2]["Wr"], layers[2]["bias"], cfg.k)
    experts = M.Experts.from_layer(layers[2], cfg.qbits)
    idx = torch.empty(T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, cfg.k, dtype=torch.float32, device=DEV)
    y = torch.empty(T, cfg.D, dtype=torch.float32, device=DEV)
    ws = M.workspace(M.MOE_OP_LAYER, T, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        M.moe_layer(router, experts, x, idx, w, None, y, None, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        M.moe_layer(router, experts, x, idx, w, None, y, None, ws)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    eager = gpu_layer(cfg, layers[2], x)
    assert torch.equal(y.cpu(), eager["y"])


# ------------------------------------------------------ substitution (int4)

@pytest.fixture(scope="module")
def cfg3_layer():
    cfg = W.CONFIGS[3]
    return cfg, W.make_layer(cfg, 0, DEV, chunk=64), W.make_resident_mask(cfg, 0, DEV)


@pytest.mark.parametrize("T", [1, 16])
@pytest.mark.parametrize("threshold", [0.15, 0.0, float("inf")])
def test_substitution_and_int4_decode(cfg3_layer, T, threshold):
    cfg, layer, mask = cfg3_layer
    x = W.make_tokens(cfg, T, 2, DEV)
    router = M.Router(layer["Wr"], layer["bias"], cfg.k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    k = cfg.k
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    probs = torch.empty(T, cfg.E, dtype=torch.float32, device=DEV)
    ws_r = M.workspace(M.MOE_OP_ROUTE, T, k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_route(router, x, idx, w, probs, ws_r)
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    flag = torch.empty(T, k, dtype=torch.uint8, device=DEV)
    mass = torch.empty(T, dtype=torch.float32, device=DEV)
    M.moe_substitute(probs, idx, w, mask, threshold, idx2, w2, flag, mass)
    y = torch.empty(T, cfg.D, dtype=torch.float32, device=DEV)
    ws = M.workspace(M.MOE_OP_DECODE, T, k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_decode(experts, x, idx2, w2, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    got = dict(idx=idx.cpu(), w=w.cpu(), probs=probs.cpu())
    ref = oracle.router(x, layer["Wr"], layer["bias"], k)
    check_routing(ref, got, k, max_skip_frac=0.2, label=f"substitution E512 T={T} thr={threshold}")
    # the kernel alone: the oracle's rule on the GPU's own probabilities (decisions in fp32)
    sref = oracle.substitute(probs.cpu().numpy(), idx.cpu(), w.cpu().double(), mask.cpu(), threshold)
    assert np.array_equal(flag.cpu().numpy(), sref["flag"])
    assert np.array_equal(idx2.cpu().numpy(), sref["idx"])
    np.testing.assert_allclose(mass.cpu().numpy(), sref["mass"], rtol=0, atol=1e-6)
    assert torch.equal(w2.cpu(), w.cpu())
    # end to end: the oracle's own routing followed by its substitution rule
    parity.check_substitution(ref, mask.cpu().numpy(), threshold,
                              dict(idx_used=idx2.cpu().numpy(), flag=flag.cpu().numpy(), mass=mass.cpu().numpy()),
                              label=f"substitution E512 T={T} thr={threshold}")
    check_y(layer, x, dict(idx=idx2.cpu(), w=w2.cpu(), y=y.cpu()), cfg.qbits)
    n_sub = int((flag == 2).sum())
    print(f"T={T} thr={threshold}: substituted {n_sub}/{T * k}, mass mean {mass.mean().item():.4f}")


@pytest.mark.parametrize("T", [1, 2, 7, 16])
@pytest.mark.parametrize("threshold", [0.15, 0.0, float("inf")])
def test_layer_resident_matches_oracle(cfg3_layer, T, threshold):
    """moe_layer_resident: routing, substitution and int4 experts in one call
    (one launch per token for T <= 7)."""
    cfg, layer, mask = cfg3_layer
    k = cfg.k
    x = W.make_tokens(cfg, T, 12, DEV)
    router = M.Router(layer["Wr"], layer["bias"], k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    out = dict(idx=torch.empty(T, k, dtype=torch.int32, device=DEV), w=torch.empty(T, k, device=DEV),
               probs=torch.empty(T, cfg.E, device=DEV), idx_used=torch.full((T, k), -9, dtype=torch.int32,
                                                                            device=DEV),
               flag=torch.full((T, k), 9, dtype=torch.uint8, device=DEV), mass=torch.empty(T, device=DEV),
               y=torch.empty(T, cfg.D, device=DEV), xn=torch.empty_like(x))
    ws = M.workspace(M.MOE_OP_LAYER_RESIDENT, T, k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_layer_resident(router, experts, x, mask, threshold, out["idx"], out["w"], out["probs"], out["idx_used"],
                         out["flag"], out["mass"], out["y"], out["xn"], ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    got = {n: v.cpu() for n, v in out.items()}
    ref = oracle.router(x, layer["Wr"], layer["bias"], k)
    label = f"layer_resident E512 T={T} thr={threshold}"
    check_routing(ref, got, k, max_skip_frac=0.2, label=label)
    # the rule on the GPU's own probabilities and routing: exact
    sref = oracle.substitute(got["probs"].numpy(), got["idx"], got["w"].double(), mask.cpu(), threshold)
    assert np.array_equal(got["flag"].numpy(), sref["flag"])
    assert np.array_equal(got["idx_used"].numpy(), sref["idx"])
    np.testing.assert_allclose(got["mass"].numpy(), sref["mass"], rtol=0, atol=1e-6)
    # and end to end against the oracle's routing
    parity.check_substitution(ref, mask.cpu().numpy(), threshold,
                              dict(idx_used=got["idx_used"].numpy(), flag=got["flag"].numpy(),
                                   mass=got["mass"].numpy()), label=label)
    check_y(layer, x, dict(idx=got["idx_used"], w=got["w"], y=got["y"]), cfg.qbits)
    assert torch.equal(got["xn"], (x.cpu().float() + got["y"]).to(x.dtype))


# ------------------------------------------------------- stacked layers

@pytest.mark.parametrize("cfg_id", [1, 3])
def test_layer_stack_chain_matches_oracle(cfg_id):
    """Three layers in one launch, chained through x_next: each layer is
    checked against the oracle evaluated on the input that layer actually
    received (the previous layer's x_next), and y against the oracle on the
    GPU's routing."""
    cfg = W.CONFIGS[cfg_id]
    L = 3
    layers = [W.make_layer(cfg, l, DEV, chunk=64) for l in range(L)]
    routers = [M.Router(lw["Wr"], lw["bias"], cfg.k) for lw in layers]
    experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in layers]
    x0 = W.make_tokens(cfg, 1, 31, DEV)
    idx = [torch.empty(1, cfg.k, dtype=torch.int32, device=DEV) for _ in range(L)]
    w = [torch.empty(1, cfg.k, device=DEV) for _ in range(L)]
    y = [torch.empty(1, cfg.D, device=DEV) for _ in range(L)]
    xn = [torch.empty_like(x0) for _ in range(L)]
    ws = M.workspace(M.MOE_OP_LAYER, 1, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    xs = [x0] + [None] * (L - 1)
    M.moe_layer_stack(routers, experts, [x0] * L, True, idx, w, y, xn, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    x_in = x0
    for l in range(L):
        ref = oracle.router(x_in, layers[l]["Wr"], layers[l]["bias"], cfg.k)
        got = dict(idx=idx[l].cpu(), w=w[l].cpu(), y=y[l].cpu())
        check_routing(ref, got, cfg.k, max_skip_frac=1.0, label=f"stack chain cfg{cfg_id} layer {l}")
        check_y(layers[l], x_in, got, cfg.qbits)
        assert torch.equal(xn[l].cpu(), (x_in.cpu().float() + got["y"]).to(x0.dtype))
        x_in = xn[l]
    del xs


def test_layer_stack_independent_equals_single_layers(cfg1_layers):
    """Independent inputs: a stack launch gives bit-identical results to one
    moe_layer call per layer."""
    cfg, layers = cfg1_layers
    L = len(layers)
    routers = [M.Router(lw["Wr"], lw["bias"], cfg.k) for lw in layers]
    experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in layers]
    xs = [W.make_tokens(cfg, 1, 40 + l, DEV) for l in range(L)]
    idx = [torch.empty(1, cfg.k, dtype=torch.int32, device=DEV) for _ in range(L)]
    w = [torch.empty(1, cfg.k, device=DEV) for _ in range(L)]
    y = [torch.empty(1, cfg.D, device=DEV) for _ in range(L)]
    ws = M.workspace(M.MOE_OP_LAYER, 1, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_layer_stack(routers, experts, xs, False, idx, w, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    for l in range(L):
        one = gpu_layer(cfg, layers[l], xs[l], probs=False)
        assert torch.equal(one["idx"], idx[l].cpu()) and torch.equal(one["w"], w[l].cpu())
        assert torch.equal(one["y"], y[l].cpu())


@pytest.mark.parametrize("threshold", [0.15, 0.0])
def test_layer_stack_resident_matches_single_layers_and_oracle(cfg3_layer, threshold):
    """moe_layer_stack_resident: four layers (the cfg3 layer with four masks and
    four tokens) in one launch give bit-identical outputs to one
    moe_layer_resident call per layer, and each layer's substitution matches
    the oracle's routing followed by the oracle's rule."""
    cfg, layer, mask0 = cfg3_layer
    L, k = 4, cfg.k
    masks = [mask0] + [W.make_resident_mask(cfg, l, DEV) for l in range(1, L)]
    router = M.Router(layer["Wr"], layer["bias"], k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    xs = [W.make_tokens(cfg, 1, 60 + l, DEV) for l in range(L)]

    def outs():
        return dict(idx=[torch.empty(1, k, dtype=torch.int32, device=DEV) for _ in range(L)],
                    w=[torch.empty(1, k, device=DEV) for _ in range(L)],
                    used=[torch.full((1, k), -9, dtype=torch.int32, device=DEV) for _ in range(L)],
                    flag=[torch.full((1, k), 9, dtype=torch.uint8, device=DEV) for _ in range(L)],
                    mass=[torch.empty(1, device=DEV) for _ in range(L)],
                    y=[torch.empty(1, cfg.D, device=DEV) for _ in range(L)],
                    xn=[torch.empty_like(xs[0]) for _ in range(L)])
    st = outs()
    ws = M.workspace(M.MOE_OP_LAYER, 1, k, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_layer_stack_resident([router] * L, [experts] * L, xs, False, masks, threshold, st["idx"], st["w"],
                               st["used"], st["flag"], st["mass"], st["y"], st["xn"], ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    one = outs()
    ws1 = M.workspace(M.MOE_OP_LAYER_RESIDENT, 1, k, cfg.E, cfg.D, cfg.F, DEV)
    for l in range(L):
        M.moe_layer_resident(router, experts, xs[l], masks[l], threshold, one["idx"][l], one["w"][l], None,
                             one["used"][l], one["flag"][l], one["mass"][l], one["y"][l], one["xn"][l], ws1)
    assert M.moe_check_status(ws1) == M.MOE_OK
    for l in range(L):
        for n in ("idx", "w", "used", "flag", "mass", "y", "xn"):
            assert torch.equal(st[n][l], one[n][l]), f"layer {l}: {n} differs from the single-layer call"
        ref = oracle.router(xs[l], layer["Wr"], layer["bias"], k)
        label = f"stack_resident E512 thr={threshold} layer {l}"
        check_routing(ref, dict(idx=st["idx"][l].cpu(), w=st["w"][l].cpu()), k, max_skip_frac=1.0, label=label)
        parity.check_substitution(ref, masks[l].cpu().numpy(), threshold,
                                  dict(idx_used=st["used"][l].cpu().numpy(), flag=st["flag"][l].cpu().numpy(),
                                       mass=st["mass"][l].cpu().numpy()), label=label)
        check_y(layer, xs[l], dict(idx=st["used"][l].cpu(), w=st["w"][l].cpu(), y=st["y"][l].cpu()), cfg.qbits)


# ------------------------------------------------------ bounded waits

def test_wait_limit_runs_out_and_the_workspace_recovers(cfg1_layers):
    """A wait limit of a few cycles makes the layer kernel's cross-CTA waits run
    out: a three-layer stack waits, at every layer boundary, for the slowest
    CTA's output, which never arrives within 16 cycles. The call must finish,
    record MOE_ERR_DEVICE_TIMEOUT, and the same workspace must give correct
    results once the limit is restored."""
    cfg, layers = cfg1_layers
    L = len(layers)
    routers = [M.Router(lw["Wr"], lw["bias"], cfg.k) for lw in layers]
    experts = [M.Experts.from_layer(lw, cfg.qbits) for lw in layers]
    ws = M.workspace(M.MOE_OP_LAYER, 1, cfg.k, cfg.E, cfg.D, cfg.F, DEV)
    xs = [W.make_tokens(cfg, 1, 50 + l, DEV) for l in range(L)]
    idx = [torch.empty(1, cfg.k, dtype=torch.int32, device=DEV) for _ in range(L)]
    w = [torch.empty(1, cfg.k, device=DEV) for _ in range(L)]
    y = [torch.empty(1, cfg.D, device=DEV) for _ in range(L)]
    M.moe_set_wait_limit(ws, 16)
    M.moe_layer_stack(routers, experts, xs, False, idx, w, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_ERR_DEVICE_TIMEOUT
    assert M.moe_check_status(ws) == M.MOE_OK  # cleared by the read
    M.moe_set_wait_limit(ws, 0)
    M.moe_layer_stack(routers, experts, xs, False, idx, w, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    for l in range(L):
        one = gpu_layer(cfg, layers[l], xs[l], probs=False)
        assert torch.equal(one["idx"], idx[l].cpu()) and torch.equal(one["y"], y[l].cpu())
        ref = oracle.router(xs[l], layers[l]["Wr"], layers[l]["bias"], cfg.k)
        check_routing(ref, dict(idx=idx[l].cpu(), w=w[l].cpu()), cfg.k, max_skip_frac=1.0, label="after a timeout")
        check_y(layers[l], xs[l], dict(idx=idx[l].cpu(), w=w[l].cpu(), y=y[l].cpu()), cfg.qbits)


# ------------------------------------------------------------- edge cases

def test_bad_expert_id_is_reported_and_skipped():
    cfg = W.CONFIGS[0]
    layer = W.make_layer(cfg, 0, DEV)
    x = W.make_tokens(cfg, 3, 4, DEV)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    idx = torch.tensor([[1, 2], [cfg.E + 5, 0], [3, -1]], dtype=torch.int32, device=DEV)
    w = torch.full((3, 2), 0.5, device=DEV)
    y = torch.empty(3, cfg.D, device=DEV)
    ws = M.workspace(M.MOE_OP_DECODE, 3, 2, cfg.E, cfg.D, cfg.F, DEV)
    M.moe_decode(experts, x, idx, w, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_ERR_BAD_INDEX
    assert M.moe_check_status(ws) == M.MOE_OK  # reset by the read
    # the valid slots are still computed: token 0 fully, tokens 1/2 their valid slot
    ic = idx.cpu().numpy().copy()
    wc = w.cpu().double().numpy().copy()
    bad = (ic < 0) | (ic >= cfg.E)
    wc[bad] = 0.0
    ic[bad] = 0
    y_ref = oracle.moe(layer, x, ic, wc, cfg.qbits)
    assert np.abs(y.cpu().double().numpy() - y_ref).max() <= REL_TOL * np.abs(y_ref).max()
    # the library keeps working after a reported error
    idx.fill_(1)
    M.moe_decode(experts, x, idx, w, y, None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK


# ------------------------------------------------------------ exact ties
def _tied_router(E, D, n_distinct, seed):
    """Router rows drawn from only n_distinct rows, scattered over the experts,
    so that many experts get bit-identical logits: the top-k is then decided by
    the lowest-index rule alone."""
    g = torch.Generator().manual_seed(seed)
    base = torch.randn(n_distinct, D, generator=g) * 0.1
    pick = (torch.arange(E) * 37 + 11) % n_distinct
    return base[pick].to(torch.bfloat16)


@pytest.mark.parametrize("E,k,n_distinct", [(256, 8, 16), (512, 10, 24), (64, 4, 3), (128, 1, 5)])
def test_exact_ties_take_lowest_ids(E, k, n_distinct):
    """Exact ties in fp32 probabilities: ids must equal the oracle's (lowest id
    first) in the single-token layer kernel, the multi-token router kernel and
    the prefill top-k; no near-tie exclusion applies to exact ties."""
    D, F = 256, 64
    cfg = small_cfg(E, k, D, F, zipf=None, sigma=0.1, cfg_id=90 + k)
    layer = W.make_layer(cfg, 0, DEV)
    layer["Wr"] = _tied_router(E, D, n_distinct, seed=E + k).to(DEV)
    layer["bias"] = None
    x = W.make_tokens(cfg, 5, 0, DEV)
    ref = oracle.router(x.cpu(), layer["Wr"].cpu(), None, k)
    # the fixture really has ties inside the top k + 1
    srt = np.sort(ref["probs32"], axis=1)[:, ::-1]
    assert (srt[:, :k + 1][:, 1:] == srt[:, :k + 1][:, :-1]).any()
    router = M.Router(layer["Wr"], None, k)
    # single token, fused layer kernel
    for t in range(2):
        got = gpu_layer(cfg, layer, x[t:t + 1].contiguous())
        assert np.array_equal(got["idx"].numpy()[0], ref["idx"][t])
        np.testing.assert_allclose(got["w"].numpy()[0], ref["w"][t], rtol=0, atol=1e-5)
    # several tokens, router kernel
    idx = torch.empty(5, k, dtype=torch.int32, device=DEV)
    w = torch.empty(5, k, device=DEV)
    ws = M.workspace(M.MOE_OP_ROUTE, 5, k, E, D, F, DEV)
    M.moe_route(router, x, idx, w, None, ws)
    assert M.moe_check_status(ws) == M.MOE_OK
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    # prefill (tensor-core router + warp top-k)
    T = 5
    experts = M.Experts.from_layer(layer, cfg.qbits)
    out = dict(y=torch.empty(T, D, device=DEV), idx=torch.empty(T, k, dtype=torch.int32, device=DEV),
               w=torch.empty(T, k, device=DEV), counts=torch.empty(E, dtype=torch.int32, device=DEV),
               perm=torch.empty(T * k, dtype=torch.int32, device=DEV))
    wsp = M.workspace(M.MOE_OP_PREFILL, T, k, E, D, F, DEV)
    M.moe_prefill(router, experts, x, out["y"], out["idx"], out["w"], out["counts"], out["perm"], wsp)
    assert M.moe_check_status(wsp) == M.MOE_OK
    assert np.array_equal(out["idx"].cpu().numpy(), ref["idx"])
