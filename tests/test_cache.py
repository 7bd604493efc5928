"""The expert cache's host planning (moe_cache_plan) against the replay oracle,
decision by decision, and the argument checks of the cache calls (no GPU).

gist.science "Which expert misses are worth waiting for?", method section: a
kept miss (first choice, or gate weight >= 0.15) is fetched into the cache,
any other miss is served by a resident stand-in, the substituted gate weight
admits an expert in the background at a threshold, eviction goes by routing
frequency. The oracle (``oracle/replay.py``, plain Python, pinned in
``test_replay.py``) decides on the same probabilities; the plan must agree on
every slot, every count, the final cache and its counters, and must keep its
slot table a one-to-one map whose slots hold exactly the served experts.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest

import moe_routed_expert_route_gb300 as M
from moe_routed_expert_route_gb300 import _lib as L
from oracle import replay as R

POLICIES = {M.MOE_POLICY_FETCH_ALL: R.FETCH_ALL, M.MOE_POLICY_THRESHOLD: R.THRESHOLD,
            M.MOE_POLICY_FIRST_CHOICE: R.FIRST_CHOICE}


def _case(rng, N, E, ties=False):
    lg = rng.standard_normal((N, E)) * rng.uniform(0.5, 3.0)
    p = (np.exp(lg) / np.exp(lg).sum(-1, keepdims=True)).astype(np.float32)
    if ties:
        p[:, 1:4] = p[:, :1]
    return p


def _check_slots(cache: M.ExpertCache, d: dict):
    S, k = cache.S, cache.k
    # one-to-one slot table
    assert sorted(cache.expert_of.tolist()) == sorted(np.nonzero(cache.slot_of >= 0)[0].tolist())
    for s_, e in enumerate(cache.expert_of):
        assert cache.slot_of[e] == s_
    fetched = []
    for r in range(k):
        if d["flag"][r] == 4:
            assert d["slot"][r] == S + r
        else:
            # served from the cache: the slot holds the serving expert
            assert 0 <= d["slot"][r] < S
            assert cache.expert_of[d["slot"][r]] == d["expert"][r]
        assert d["flag"][r] in (0, 1, 2, 4)
        if d["flag"][r] in (1, 4):
            fetched.append((int(d["expert"][r]), int(d["slot"][r])))
    assert list(zip(d["fetch_expert"].tolist(), d["fetch_slot"].tolist())) == fetched
    for e, s_ in zip(d["admit_expert"], d["admit_slot"]):
        assert cache.slot_of[e] == s_ and e not in d["expert"]


@pytest.mark.parametrize("seed", range(12))
def test_plan_matches_the_replay_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(1, 40))
    E = int(rng.integers(4, 64))
    k = int(rng.integers(1, min(E - 1, 10) + 1))
    S = int(rng.integers(1, E + 1))
    p = _case(rng, N, E, ties=seed % 4 == 0)
    pol = [M.MOE_POLICY_FETCH_ALL, M.MOE_POLICY_THRESHOLD, M.MOE_POLICY_FIRST_CHOICE][seed % 3]
    thr = float(rng.choice([0.0, 0.15, 0.3, math.inf]))
    beta = float(rng.choice([0.0, 0.2, 0.5]))
    cached = rng.permutation(E)[:S]
    cache = M.ExpertCache(E, k, cached)
    res = np.zeros((1, E), np.uint8)
    res[0, cached] = 1
    ref = R.replay(p[:, None, :], k, POLICIES[pol], thr, beta, 0.0, 0.0, resident=res.tolist())
    for t in range(N):
        d = M.moe_cache_plan(cache, p[t], pol, thr, beta)
        _check_slots(cache, d)
        assert d["expert"].tolist() == ref["used"][t][0], t
        assert d["flag"].tolist() == ref["flags"][t][0], t
        assert d["admit_expert"].tolist() == ref["admitted"][t][0], t
        assert len(d["fetch_expert"]) == ref["fetches"][t]
        assert int((d["flag"] == 2).sum()) == ref["substituted"][t]
        assert d["mass"] == ref["sub_mass"][t]
        # weights: the k probabilities over their sum, in double, then fp32
        top = np.argsort(-p[t].astype(np.float64), kind="stable")[:k]
        w = p[t][top].astype(np.float64) / p[t][top].astype(np.float64).sum()
        assert np.array_equal(d["w"], w.astype(np.float32))
    assert (cache.slot_of >= 0).astype(int).tolist() == ref["resident"][0]
    assert cache.freq.tolist() == ref["freq"][0]
    assert cache.acc.tolist() == ref["acc"][0]


def test_plan_at_the_substitution_shape():
    # the 512-expert top-10 layer, a quarter cached, 0.15 rule with admission
    # at 0.5 (the page's quality-first policy), 60 tokens
    rng = np.random.default_rng(7)
    p = _case(rng, 60, 512)
    cached = rng.choice(512, 128, replace=False)
    cache = M.ExpertCache(512, 10, cached)
    res = np.zeros((1, 512), np.uint8)
    res[0, cached] = 1
    ref = R.replay(p[:, None, :], 10, R.THRESHOLD, 0.15, 0.5, 0.0, 0.0, resident=res.tolist())
    for t in range(60):
        d = M.moe_cache_plan(cache, p[t], M.MOE_POLICY_THRESHOLD, 0.15, 0.5)
        _check_slots(cache, d)
        assert d["expert"].tolist() == ref["used"][t][0]
        assert d["flag"].tolist() == ref["flags"][t][0]
        assert d["admit_expert"].tolist() == ref["admitted"][t][0]
    assert (cache.slot_of >= 0).astype(int).tolist() == ref["resident"][0]


def test_plan_uses_the_transient_slot_when_nothing_can_be_evicted():
    # E=4, k=3, cache of 2 holding experts 0 and 1, both routed: the third
    # choice is fetched into transient slot S + 2 and not cached
    cache = M.ExpertCache(4, 3, [1, 0])
    d = M.moe_cache_plan(cache, np.array([0.4, 0.3, 0.2, 0.1], np.float32), M.MOE_POLICY_THRESHOLD, 0.15)
    assert d["expert"].tolist() == [0, 1, 2]
    assert d["slot"].tolist() == [1, 0, 4]
    assert d["flag"].tolist() == [0, 0, 4]
    assert d["fetch_expert"].tolist() == [2] and d["fetch_slot"].tolist() == [4]
    assert cache.slot_of.tolist() == [1, 0, -1, -1]


def test_plan_worked_example_golden_in_slots():
    # the hand-worked example of the replay golden (E=6, k=2, experts 0-2
    # cached in slots 0-2, 0.15 rule, admission at 0.15), followed slot by slot:
    # token 0 fetches e3 into e0's slot 0 and e4 into e1's slot 1; token 1
    # serves e5 by e2 (slot 2); token 2 serves e5 by e4 (slot 1) and admits e5
    # into e2's slot 2
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    probs = [[0.10, 0.05, 0.05, 0.50, 0.25, 0.05], [0.02, 0.03, 0.05, 0.80, 0.03, 0.07],
             [0.02, 0.03, 0.02, 0.80, 0.04, 0.09]]
    cache = M.ExpertCache(6, 2, [0, 1, 2])
    want = [([3, 4], [0, 1], [1, 1], [], []), ([3, 2], [0, 2], [0, 2], [], []), ([3, 4], [0, 1], [0, 2], [5], [2])]
    for t, (ex, sl, fl, ae, as_) in enumerate(want):
        d = M.moe_cache_plan(cache, np.array([f32(v) for v in probs[t]], np.float32), M.MOE_POLICY_THRESHOLD,
                             0.15, 0.15)
        assert d["expert"].tolist() == ex and d["slot"].tolist() == sl and d["flag"].tolist() == fl, t
        assert d["admit_expert"].tolist() == ae and d["admit_slot"].tolist() == as_, t
    assert cache.expert_of.tolist() == [3, 4, 5]


def test_cache_calls_reject_bad_arguments():
    lib = L._lib
    cache = M.ExpertCache(8, 2, [0, 1, 2])
    p = np.full(8, 0.125, np.float32)
    pol = L._policy(M.MOE_POLICY_THRESHOLD, 0.15, 0.5)
    # an inconsistent slot table
    cache.expert_of[1] = 0
    assert lib.moe_cache_plan(ctypes.byref(cache._c), p.ctypes.data, ctypes.byref(pol),
                              ctypes.byref(cache._st)) == M.MOE_ERR_INVALID_ARG
    cache.expert_of[1] = 1
    assert lib.moe_cache_plan(ctypes.byref(cache._c), p.ctypes.data, ctypes.byref(pol),
                              ctypes.byref(cache._st)) == M.MOE_OK
    bad = L._ReplayPolicy(7, 0.15, 0.5, 0.0, 0.0)
    assert lib.moe_cache_plan(ctypes.byref(cache._c), p.ctypes.data, ctypes.byref(bad),
                              ctypes.byref(cache._st)) == M.MOE_ERR_INVALID_ARG
    nan = L._ReplayPolicy(1, float("nan"), 0.5, 0.0, 0.0)
    assert lib.moe_cache_plan(ctypes.byref(cache._c), p.ctypes.data, ctypes.byref(nan),
                              ctypes.byref(cache._st)) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_cache_plan(ctypes.byref(cache._c), None, ctypes.byref(pol),
                              ctypes.byref(cache._st)) == M.MOE_ERR_INVALID_ARG
    # workspace sizes
    n, hb = M.moe_cache_workspace_bytes(256, 64, 8, 2048, 768)
    assert n > 0 and hb == 4 * 256 + 8 * 8
    assert M.moe_cache_workspace_bytes(256, 300, 8, 2048, 768)[0] == 0   # S > E
    assert M.moe_cache_workspace_bytes(256, 64, 33, 2048, 768)[0] == 0   # k > 32
    # pool fetch: slot outside the pool, expert outside the store, format mismatch
    host = L._Experts(8, 64, 64, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)
    pool = L._Experts(5, 64, 64, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)
    ex = np.array([3], np.int32)
    assert lib.moe_pool_fetch(ctypes.byref(host), ctypes.byref(pool), 1, ex.ctypes.data,
                              np.array([5], np.int32).ctypes.data, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_pool_fetch(ctypes.byref(host), ctypes.byref(pool), 1, np.array([8], np.int32).ctypes.data,
                              np.array([0], np.int32).ctypes.data, None) == M.MOE_ERR_INVALID_ARG
    pool4 = L._Experts(5, 64, 64, L.MOE_Q_INT4_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)
    assert lib.moe_pool_fetch(ctypes.byref(host), ctypes.byref(pool4), 1, ex.ctypes.data,
                              np.array([0], np.int32).ctypes.data, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_pool_fetch(ctypes.byref(host), ctypes.byref(pool), 0, None, None, None) == M.MOE_OK
    # cached layer: the pool must have S + k slots, a copy stream needs events
    r = L._Router(8, 64, 2, L.MOE_BF16, 16, None, 1)
    scratch = np.zeros(64, np.uint8)

    def call(pool_, cs=None, ev=None):
        return lib.moe_cached_layer(ctypes.byref(r), ctypes.byref(host), ctypes.byref(pool_), ctypes.byref(cache._c),
                                    ctypes.byref(pol), 16, L.MOE_BF16, 16, None, ctypes.byref(cache._st),
                                    scratch.ctypes.data, 256, 10 ** 7, None, cs, ev, ev)
    assert call(L._Experts(6, 64, 64, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)) == \
        M.MOE_ERR_INVALID_ARG
    assert call(pool, cs=16, ev=None) == M.MOE_ERR_INVALID_ARG
