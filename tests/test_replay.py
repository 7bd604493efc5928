"""Router-logit replay simulator (host code): the oracle pinned by a hand-worked
example and by invariants of the policies, then the library's moe_replay
compared with the oracle exactly. No GPU is needed: both run on the host."""
import json
import math
import os
import struct

import numpy as np
import pytest

import moe_routed_expert_route_gb300 as M
import oracle
from oracle import replay as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "replay_worked.json")
OUTS = ("t_token_us", "fetches", "substituted", "sub_mass", "admissions")


def f32(v):
    return struct.unpack("f", struct.pack("f", float(v)))[0]


def random_case(rng, N, L, E, k, resident_frac=0.35, ties=False):
    lg = rng.standard_normal((N, L, E)) * rng.uniform(0.5, 3.0)
    p = np.exp(lg) / np.exp(lg).sum(-1, keepdims=True)
    p = p.astype(np.float32)
    if ties:
        p[:, :, 1:4] = p[:, :, :1]
    res = (rng.random((L, E)) < resident_frac).astype(np.uint8)
    return p, res


def run_oracle(p, k, policy, thr, beta, tl, tf, res, freq=None, acc=None):
    return R.replay(p, k, policy, thr, beta, tl, tf, resident=res.tolist(),
                    freq=None if freq is None else freq.tolist(), acc=None if acc is None else acc.tolist())


# ------------------------------------------------------------ oracle pins

def test_worked_example_golden():
    g = json.load(open(GOLDEN))
    probs = [[[f32(v) for v in row] for row in tok] for tok in g["probs"]]
    o = R.replay(probs, g["k"], R.THRESHOLD, g["threshold"], g["admit_mass"], g["t_layer_us"],
                 g["t_fetch_us"], resident=g["resident"])
    ex = g["expect"]
    for n in ("t_token_us", "fetches", "substituted", "admissions", "resident", "freq", "acc",
              "used", "flags", "admitted"):
        assert o[n] == ex[n], n
    for t, terms in enumerate(ex["sub_mass_terms"]):
        m = 0.0
        for a, b in terms:
            pa, pb = probs[t][0][a], probs[t][0][b]
            m += pa / (pb + pa)
        assert math.isclose(o["sub_mass"][t], m, rel_tol=0, abs_tol=1e-15)


def test_oracle_miss_with_nothing_evictable_is_used_without_entering():
    # E=4, k=3, experts 0 and 1 resident, both routed: the third choice e2
    # (weight 0.2/0.9 >= 0.15) is fetched, but every resident is in use, so it
    # serves its slot without entering the cache (flag 4)
    p = [[[f32(0.4), f32(0.3), f32(0.2), f32(0.1)]]]
    o = R.replay(p, 3, R.THRESHOLD, 0.15, 0.0, 1.0, 1.0, resident=[[1, 1, 0, 0]])
    assert o["used"] == [[[0, 1, 2]]]
    assert o["flags"] == [[[0, 0, 4]]]
    assert o["fetches"] == [1]
    assert o["resident"] == [[1, 1, 0, 0]]


@pytest.mark.parametrize("seed", range(6))
def test_oracle_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    N, L, E, k = 25, 3, 24, 4
    p, res = random_case(rng, N, L, E, k, ties=seed % 3 == 0)
    tl, tf = 12.5, 80.0
    cap = res.sum(axis=1).tolist()
    every = {}
    for pol in (R.FETCH_ALL, R.THRESHOLD, R.FIRST_CHOICE):
        for beta in (0.0, 0.5):
            o = run_oracle(p, k, pol, 0.15, beta, tl, tf, res)
            every[(pol, beta)] = o
            # the cache keeps its size
            assert [sum(r) for r in o["resident"]] == cap
            for t in range(N):
                # each slot is a hit, a fetch or a substitution
                assert o["fetches"][t] + o["substituted"][t] <= L * k
                assert o["t_token_us"][t] == pytest.approx(L * tl + o["fetches"][t] * tf, abs=1e-9)
                assert 0.0 <= o["sub_mass"][t] <= L + 1e-12
                assert o["admissions"][t] <= o["substituted"][t]
                if pol == R.FIRST_CHOICE:
                    assert o["fetches"][t] <= L
            # the frequencies count every routed expert once per token and layer
            assert [sum(r) for r in o["freq"]] == [N * k] * L
            if beta == 0.0:
                assert sum(o["admissions"]) == 0
    fa = every[(R.FETCH_ALL, 0.0)]
    assert sum(fa["substituted"]) == 0 and sum(fa["sub_mass"]) == 0.0
    # threshold 0 fetches every miss; +inf keeps only the first choice
    assert run_oracle(p, k, R.THRESHOLD, 0.0, 0.0, tl, tf, res) == fa
    assert run_oracle(p, k, R.THRESHOLD, math.inf, 0.0, tl, tf, res) == every[(R.FIRST_CHOICE, 0.0)]
    # an unreachable admission threshold admits nothing
    assert run_oracle(p, k, R.THRESHOLD, 0.15, 1e9, tl, tf, res) == every[(R.THRESHOLD, 0.0)]


def test_oracle_everything_resident_means_no_miss():
    rng = np.random.default_rng(7)
    p, _ = random_case(rng, 10, 2, 12, 3)
    res = np.ones((2, 12), np.uint8)
    o = run_oracle(p, 3, R.THRESHOLD, 0.15, 0.5, 5.0, 50.0, res)
    assert o["fetches"] == [0] * 10 and o["substituted"] == [0] * 10 and o["t_token_us"] == [10.0] * 10


def test_oracle_replay_resumes_from_its_state():
    rng = np.random.default_rng(8)
    p, res = random_case(rng, 30, 2, 20, 3)
    whole = run_oracle(p, 3, R.THRESHOLD, 0.15, 0.4, 1.0, 9.0, res)
    a = run_oracle(p[:13], 3, R.THRESHOLD, 0.15, 0.4, 1.0, 9.0, res)
    b = R.replay(p[13:], 3, R.THRESHOLD, 0.15, 0.4, 1.0, 9.0, resident=a["resident"], freq=a["freq"], acc=a["acc"])
    for n in OUTS:
        assert a[n] + b[n] == whole[n], n
    assert b["resident"] == whole["resident"] and b["freq"] == whole["freq"] and b["acc"] == whole["acc"]


def test_oracle_stand_in_is_the_most_probable_unused_resident():
    # one token, one layer: e0 routed first (resident), e1 second (missed, weight
    # below 0.15); residents e0, e2, e3 with p(e3) > p(e2): the stand-in is e3,
    # then admission at a tiny threshold evicts the least frequent unused
    # resident, e2 (e0 is routed, e3 stands in)
    p = np.array([[[0.80, 0.10, 0.02, 0.08]]], np.float32)
    res = np.array([[1, 0, 1, 1]], np.uint8)
    o = R.replay(p, 2, R.THRESHOLD, 0.15, 1e-3, 0.0, 0.0, resident=res.tolist())
    assert o["substituted"] == [1] and o["admissions"] == [1]
    assert o["resident"] == [[1, 1, 0, 1]]


# ------------------------------------------------- library against oracle

@pytest.mark.parametrize("seed", range(12))
def test_moe_replay_matches_the_oracle(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 30))
    L = int(rng.integers(1, 5))
    E = int(rng.integers(3, 48))
    k = int(rng.integers(1, min(E, 8) + 1))
    p, res = random_case(rng, N, L, E, k, resident_frac=float(rng.uniform(0.1, 0.9)), ties=seed % 4 == 0)
    pol = int(rng.integers(0, 3))
    thr = float(rng.choice([0.0, 0.15, 0.3, math.inf]))
    beta = float(rng.choice([0.0, 0.2, 0.5]))
    tl, tf = float(rng.uniform(1, 30)), float(rng.uniform(10, 300))
    got = M.moe_replay(p, k, pol, thr, beta, tl, tf, resident=res.copy())
    ref = run_oracle(p, k, pol, thr, beta, tl, tf, res)
    for n in OUTS:
        assert got[n].tolist() == ref[n], n
    assert got["resident"].tolist() == ref["resident"]
    assert got["freq"].tolist() == ref["freq"]
    assert got["acc"].tolist() == ref["acc"]


def test_moe_replay_at_the_substitution_shape():
    # the 512-expert top-10 layer with a quarter resident, 0.15 rule and
    # admission at 0.5 (the page's quality-first policy), 4 layers x 40 tokens
    rng = np.random.default_rng(21)
    p, _ = random_case(rng, 40, 4, 512, 10)
    res = np.zeros((4, 512), np.uint8)
    for l in range(4):
        res[l, rng.choice(512, 128, replace=False)] = 1
    got = M.moe_replay(p, 10, M.MOE_POLICY_THRESHOLD, 0.15, 0.5, 20.0, 500.0, resident=res.copy())
    ref = run_oracle(p, 10, R.THRESHOLD, 0.15, 0.5, 20.0, 500.0, res)
    for n in OUTS:
        assert got[n].tolist() == ref[n], n
    assert got["resident"].tolist() == ref["resident"]


def test_moe_replay_rejects_bad_arguments():
    p = np.full((2, 1, 4), 0.25, np.float32)
    res = np.zeros((1, 4), np.uint8)
    with pytest.raises(M.MoeError):
        M.moe_replay(p, 5, M.MOE_POLICY_THRESHOLD, resident=res.copy())  # k > E
    with pytest.raises(M.MoeError):
        M.moe_replay(p, 2, 7, resident=res.copy())  # no such policy
    with pytest.raises(M.MoeError):
        M.moe_replay(p, 2, M.MOE_POLICY_THRESHOLD, threshold=float("nan"), resident=res.copy())
    with pytest.raises(M.MoeError):
        M.moe_replay(p, 2, M.MOE_POLICY_THRESHOLD, t_fetch_us=-1.0, resident=res.copy())


def test_oracle_top_k_ties_take_the_lower_ids():
    p = np.array([[[0.3, 0.3, 0.3, 0.1]]], np.float32)
    o = R.replay(p, 2, R.FETCH_ALL, resident=[[1, 1, 1, 1]])
    assert o["freq"] == [[1, 1, 0, 0]]


def test_oracle_eviction_ties_take_the_lower_id():
    # residents e0, e1 never routed (frequency 0): a fetched first choice evicts e0
    p = np.array([[[0.1, 0.1, 0.7, 0.1]]], np.float32)
    o = R.replay(p, 1, R.THRESHOLD, resident=[[1, 1, 0, 0]])
    assert o["fetches"] == [1] and o["resident"] == [[0, 1, 1, 0]]


def test_oracle_threshold_rule_splits_at_the_threshold():
    # second slot weight 0.25 (>= 0.15): fetched; 0.10: substituted
    res = [[1, 0, 0, 1]]
    hi = R.replay(np.array([[[0.60, 0.20, 0.05, 0.15]]], np.float32), 2, R.THRESHOLD, resident=res)
    lo = R.replay(np.array([[[0.72, 0.08, 0.05, 0.06]]], np.float32), 2, R.THRESHOLD, resident=res)
    assert hi["fetches"] == [1] and hi["substituted"] == [0]
    assert lo["fetches"] == [0] and lo["substituted"] == [1]


# ------------------------------------------------------ planted mistakes

MUTANTS = [
    ("(count[l][c], c)", "(count[l][c], -c)"),                       # eviction tie-break
    ("stand_in = max(pool,", "stand_in = min(pool,"),                # stand-in choice
    ("mass_of[l][e] = 0.0\n", "pass\n"),                            # admission does not restart
    ("want = r == 0\n", "want = r <= 1\n"),                          # first-choice rule
    ("for e in chosen:\n                count[l][e] += 1", "for e in chosen[:1]:\n                count[l][e] += 1"),
    ("fetched_here * t_fetch_us", "n_fetch * t_fetch_us"),           # time uses the running count
    ("key=lambda e: (-p[e], e))", "key=lambda e: (-p[e], -e))"),     # top-k tie-break
    ("weights[r] >= threshold", "weights[r] > 2 * threshold"),       # threshold rule
    ("if e in cache[l]:\n                    continue", "if e in cache[l] and r > 0:\n                    continue"),
]


def _pins_pass(mod) -> bool:
    global R
    saved = R
    R = mod
    try:
        test_worked_example_golden()
        test_oracle_stand_in_is_the_most_probable_unused_resident()
        test_oracle_top_k_ties_take_the_lower_ids()
        test_oracle_eviction_ties_take_the_lower_id()
        test_oracle_threshold_rule_splits_at_the_threshold()
        test_oracle_invariants(0)
        test_oracle_everything_resident_means_no_miss()
        return True
    except AssertionError:
        return False
    finally:
        R = saved


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_pins_catch_planted_mistakes(i):
    import types
    src = open(R.__file__).read()
    old, new = MUTANTS[i]
    assert src.count(old) == 1, old
    mod = types.ModuleType(f"replay_mutant_{i}")
    exec(compile(src.replace(old, new), f"replay_mutant_{i}", "exec"), mod.__dict__)
    assert _pins_pass(R)
    assert not _pins_pass(mod), f"planted mistake not caught: {new!r}"
