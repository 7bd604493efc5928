"""GPU run of the expert cache (moe_pool_fetch, moe_cached_layer) against the
oracles, through the C ABI.

gist.science "Which expert misses are worth waiting for?", method section: the
experts live in host memory, a device pool caches some of them; per token a
kept miss (first choice or gate weight >= 0.15) is fetched, any other miss is
served by a cached stand-in, and the substituted gate weight admits experts in
the background (here at 0.5, the page's value). Checked per token:
  * the router's probabilities against the oracle router (1e-6 + 1e-5 p);
  * every decision (serving expert, flag, admissions) equal to the replay
    oracle's on the same fp32 probabilities;
  * y against the oracle's MoE on the served experts and weights
    (max |y - y_oracle| <= 2e-3 max |y_oracle|);
and at the end every cached slot of the pool holds its expert's bytes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import parity
import workloads as W
from oracle import replay as R

pytestmark = pytest.mark.gpu

M = None
if torch.cuda.is_available():
    import moe_routed_expert_route_gb300 as M  # noqa: F811

DEV = "cuda"
NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def _setup(S=8, seed=0):
    # a router dominated by its Zipf bias, so that the same low-weight experts
    # come back and their substituted weight reaches the admission threshold
    cfg = W.LayerConfig("cache E32 k4 D256 F128", E=32, k=4, D=256, F=128, T=1, qbits=8,
                        scale_dtype=torch.float16, x_dtype=torch.bfloat16, router_dtype=torch.bfloat16,
                        router_sigma=0.02, zipf=1.1, layers=1, cfg_id=500 + seed)
    layer = W.make_layer(cfg, 0, "cpu")
    host = {n: layer[n].pin_memory() for n in NAMES}
    pool = {n: torch.zeros((S + cfg.k,) + tuple(layer[n].shape[1:]), dtype=layer[n].dtype, device=DEV)
            for n in NAMES}
    hx = M.Experts.from_layer(host, cfg.qbits)
    px = M.Experts.from_layer(pool, cfg.qbits)
    cached = np.random.default_rng(seed).permutation(cfg.E)[:S]
    M.moe_pool_fetch(hx, px, cached, np.arange(S))
    router = M.Router(layer["Wr"].to(DEV), layer["bias"].to(DEV), cfg.k)
    return cfg, layer, host, pool, hx, px, cached, router


def _run(cfg, hx, px, router, cache, x, copy_stream, beta=0.5):
    n, hb = M.moe_cache_workspace_bytes(cfg.E, cache.S, cfg.k, cfg.D, cfg.F)
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    scratch = torch.zeros(hb, dtype=torch.uint8).pin_memory()
    ev1, ev2 = torch.cuda.Event(), torch.cuda.Event()
    ev1.record()
    ev2.record()  # the events exist from here on
    ys, probs, dec = [], [], []
    for t in range(x.shape[0]):
        y = torch.empty(1, cfg.D, dtype=torch.float32, device=DEV)
        d = M.moe_cached_layer(router, hx, px, cache, M.MOE_POLICY_THRESHOLD, 0.15, beta, x[t:t + 1], y, None,
                               scratch, ws, None, copy_stream, ev1 if copy_stream else None,
                               ev2 if copy_stream else None)
        probs.append(scratch[: 4 * cfg.E].view(torch.float32).numpy().copy())
        dec.append(d)
        ys.append(y)
    torch.cuda.synchronize()
    return np.stack(probs), dec, [y.cpu().numpy()[0] for y in ys]


# (copy stream, cache slots, tokens, what the case must exercise): with 8
# slots the token's routed experts and stand-ins never use every slot, so misses
# enter the cache and substituted weight admits experts (3 and 1 admissions on
# the oracle's routing of these tokens); with 3 slots fetched misses often find
# every cached expert in use and go to their transient slot. Every routing
# weight of these tokens is at least 1e-3 away from the 0.15 threshold.
CASES = [(True, 8, 64, "admission"), (False, 8, 32, "admission"), (True, 3, 16, "transient")]


@pytest.mark.parametrize("use_copy_stream,S,N,what", CASES)
def test_cached_layer_against_the_oracles(use_copy_stream, S, N, what):
    cfg, layer, host, pool, hx, px, cached, router = _setup(S=S, seed=5)
    x = W.make_tokens(cfg, N, 3, "cpu").to(DEV)
    cache = M.ExpertCache(cfg.E, cfg.k, cached)
    cs = torch.cuda.Stream() if use_copy_stream else None
    probs, dec, ys = _run(cfg, hx, px, router, cache, x, cs)

    # the router against the oracle router
    ref = oracle.router(x, layer["Wr"], layer["bias"], cfg.k)
    np.testing.assert_allclose(probs, ref["probs"], rtol=1e-5, atol=1e-6)
    # every decision against the replay oracle on the same probabilities
    res = np.zeros((1, cfg.E), np.uint8)
    res[0, cached] = 1
    rp = R.replay(probs[:, None, :], cfg.k, R.THRESHOLD, 0.15, 0.5, 0.0, 0.0, resident=res.tolist())
    n_fetch = n_sub = n_adm = n_transient = 0
    for t, d in enumerate(dec):
        assert d["expert"].tolist() == rp["used"][t][0], t
        assert d["flag"].tolist() == rp["flags"][t][0], t
        assert d["admit_expert"].tolist() == rp["admitted"][t][0], t
        n_fetch += len(d["fetch_expert"])
        n_sub += int((d["flag"] == 2).sum())
        n_adm += len(d["admit_expert"])
        n_transient += int((d["flag"] == 4).sum())
        # y from the served experts and weights
        parity.check_y(layer, x[t:t + 1], d["expert"][None], d["w"][None], ys[t][None], cfg.qbits)
    assert n_fetch > 0 and n_sub > 0, (n_fetch, n_sub)
    assert (n_adm if what == "admission" else n_transient) > 0, (n_adm, n_transient)
    assert (cache.slot_of >= 0).astype(int).tolist() == rp["resident"][0]
    # the pool's cached slots hold their experts' bytes
    for s_, e in enumerate(cache.expert_of):
        for n in NAMES:
            assert torch.equal(pool[n][s_].cpu(), host[n][e]), (s_, int(e), n)


def test_prediction_staged_one_token_ahead_through_the_slot_table():
    """Prediction-as-routing with a staged slot table (xyznot.com "The Other
    Half of the Memory Wall": prerouter; glossary: staged decode, incremental
    sticky-slot stack): at token t the prerouter predicts the routing of token
    t+1, the predicted experts are staged from host memory into a pool of 2k
    slots on a copy stream (only changed slots are loaded), and token t+1 is
    decoded from the pool with the predicted ids and weights. Checked: the
    predicted routing against the oracle prerouter, every slot and load
    against the staging oracle, y against the oracle's MoE on the predicted
    experts, and the pool's bytes."""
    from oracle import staging as S
    cfg = W.LayerConfig("stage E32 k4 D256 F128", E=32, k=4, D=256, F=128, T=1, qbits=8,
                        scale_dtype=torch.float16, x_dtype=torch.bfloat16, router_dtype=torch.bfloat16,
                        router_sigma=0.035, zipf=1.1, layers=2, cfg_id=520)
    k, NS = cfg.k, 2 * cfg.k
    layer = W.make_layer(cfg, 1, "cpu")  # the layer whose routing the head predicts
    head_cpu = W.make_prerouter(cfg, 0, H=32, device="cpu")
    head = {n: v.to(DEV) for n, v in head_cpu.items()}
    host = {n: layer[n].pin_memory() for n in NAMES}
    pool = {n: torch.zeros((NS,) + tuple(layer[n].shape[1:]), dtype=layer[n].dtype, device=DEV) for n in NAMES}
    hx, px = M.Experts.from_layer(host, cfg.qbits), M.Experts.from_layer(pool, cfg.qbits)
    N = 13
    x = W.make_tokens(cfg, N, 4, "cpu").to(DEV)
    cur, prev = W.make_routing_history(cfg, N, stream=4, device=DEV)
    st = M.StageTable(cfg.E, NS, k)
    cs = torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record()
    scratch = torch.zeros(2 * k, dtype=torch.int32).pin_memory()
    slot_bufs = [torch.empty(k, dtype=torch.int32, device=DEV) for _ in range(2)]
    ws_p = M.workspace(M.MOE_OP_PREROUTE, 1, k, cfg.E, cfg.D, 32, DEV)
    ws_d = M.workspace(M.MOE_OP_DECODE, 1, k, NS, cfg.D, cfg.F, DEV)
    pre = M.Prerouter.from_dict(head, k)
    preds, wts, steps, ys = [], [], [], []
    for t in range(N - 1):
        idx = torch.empty(1, k, dtype=torch.int32, device=DEV)
        w = torch.empty(1, k, dtype=torch.float32, device=DEV)
        M.moe_preroute(pre, x[t:t + 1], cur[t:t + 1], prev[t:t + 1], idx, w, None, ws_p)
        sb = slot_bufs[t % 2]
        steps.append(M.moe_stage_prediction(st, hx, px, idx[0], sb, scratch, None, cs, ev))
        torch.cuda.current_stream().wait_event(ev)
        y = torch.empty(1, cfg.D, dtype=torch.float32, device=DEV)
        M.moe_decode(px, x[t + 1:t + 2], sb.view(1, k), w, y, None, ws_d)
        preds.append(idx.cpu().numpy()[0])
        wts.append(w.cpu().numpy()[0])
        ys.append(y)
    torch.cuda.synchronize()
    assert M.moe_check_status(ws_p) == M.MOE_OK and M.moe_check_status(ws_d) == M.MOE_OK
    preds, wts = np.stack(preds), np.stack(wts)
    ref = oracle.prerouter(head_cpu, x[:N - 1], cur[:N - 1], prev[:N - 1], k)
    parity.check_routing(ref, {"idx": preds, "w": wts}, k, label="staged prediction")
    so = S.stage(preds.tolist(), NS)
    n_loads = 0
    for t in range(N - 1):
        assert steps[t]["slot"].tolist() == so["slots"][t], t
        assert list(zip(steps[t]["load_expert"].tolist(), steps[t]["load_slot"].tolist())) == so["loads"][t], t
        n_loads += len(so["loads"][t])
        parity.check_y(layer, x[t + 1:t + 2], preds[t][None], wts[t][None], ys[t].cpu().numpy(), cfg.qbits)
    assert n_loads < (N - 1) * k  # sticky slots: some predicted experts were staged already
    for s_, e in enumerate(st.expert_of):
        if e >= 0:
            for n in NAMES:
                assert torch.equal(pool[n][s_].cpu(), host[n][e]), (s_, int(e), n)
