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
