"""The staged slot table: the oracle (``oracle/staging.py``) pinned by a
hand-worked example and by the invariants the glossary of the xyznot.com Edge0
page fixes (staged decode: fixed slots reached through a slot table, double
buffering; incremental sticky-slot stack: only changed slots are rewritten),
and the library's moe_stage_plan matched to it step by step (no GPU)."""
from __future__ import annotations

import ctypes
import json
import os
import types

import numpy as np
import pytest

import moe_routed_expert_route_gb300 as M
from moe_routed_expert_route_gb300 import _lib as L
from oracle import staging as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "staging_worked.json")


def _random_pred(rng, N, E, k, sticky=0.6):
    """Predicted id lists that often repeat experts of the previous step."""
    out, prev = [], list(rng.choice(E, k, replace=False))
    for _ in range(N):
        keep = [e for e in prev if rng.random() < sticky]
        rest = [e for e in rng.permutation(E) if e not in keep][: k - len(keep)]
        ids = list(rng.permutation(keep + rest))
        out.append([int(e) for e in ids])
        prev = ids
    return out


def _pins_hold(stage_fn) -> bool:
    g = json.load(open(GOLDEN))
    o = stage_fn(g["pred"], g["n_slots"])
    if o["slots"] != g["expect"]["slots"]:
        return False
    if [[list(p) for p in ld] for ld in o["loads"]] != g["expect"]["loads"]:
        return False
    if o["expert_of"] != g["expect"]["expert_of"]:
        return False
    rng = np.random.default_rng(3)
    for case in range(20):
        E = int(rng.integers(4, 40))
        k = int(rng.integers(1, min(E // 2, 8) + 1))
        pred = _random_pred(rng, 30, E, k)
        o = stage_fn(pred, 2 * k)
        staged = {}
        in_flight = []
        for t, ids in enumerate(pred):
            slots, loads = o["slots"][t], o["loads"][t]
            # the loads are exactly the predicted experts not staged before, each once
            if sorted(e for e, _ in loads) != sorted(set(e for e in ids if e not in staged)):
                return False
            for e, s in loads:
                if s in in_flight or not 0 <= s < 2 * k:  # never into a slot the step in flight reads
                    return False
                for e2 in [x for x, y in staged.items() if y == s]:
                    del staged[e2]
                staged[e] = s
            for e, s in zip(ids, slots):
                if staged.get(e) != s:  # each predicted expert is read from its own slot
                    return False
            in_flight = slots
    return True


def test_staging_oracle_pins():
    assert _pins_hold(S.stage)


def test_fewer_than_2k_slots_can_run_out():
    with pytest.raises(ValueError):
        S.stage([[0, 1], [2, 3]], 3)


MUTANTS = {
    "in_flight_not_locked": ("locked = set(in_flight) | {", "locked = set() | {"),
    "highest_free_slot": ("s = free[0]", "s = free[-1]"),
    "not_sticky": ("            if e in slot_of:\n                slots.append(slot_of[e])\n                continue\n",
                   "            if e in slot_of and e in ids[:ids.index(e)]:\n                slots.append(slot_of[e])\n"
                   "                continue\n"),
    "eviction_not_recorded": ("            if old >= 0:\n                del slot_of[old]\n", ""),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_staging_planted_mistake_is_caught(name):
    src = open(S.__file__).read()
    a, b = MUTANTS[name]
    assert a in src, name
    mod = types.ModuleType("staging_" + name)
    exec(compile(src.replace(a, b), S.__file__, "exec"), mod.__dict__)
    try:
        held = _pins_hold(mod.stage)
    except (ValueError, KeyError):
        held = False
    assert not held, f"planted mistake {name} passed every pin"


@pytest.mark.parametrize("seed", range(8))
def test_stage_plan_matches_the_oracle(seed):
    rng = np.random.default_rng(50 + seed)
    E = int(rng.integers(4, 300))
    k = int(rng.integers(1, min(E // 2, 16) + 1))
    n_slots = 2 * k + int(rng.integers(0, 5))
    pred = _random_pred(rng, 40, E, k, sticky=float(rng.uniform(0.2, 0.9)))
    if seed % 3 == 0:
        pred[5][1 % k] = pred[5][0]  # a repeated id maps to one slot
    ref = S.stage(pred, n_slots)
    st = M.StageTable(E, n_slots, k)
    for t, ids in enumerate(pred):
        got = M.moe_stage_plan(st, ids)
        assert got["slot"].tolist() == ref["slots"][t], t
        assert list(zip(got["load_expert"].tolist(), got["load_slot"].tolist())) == ref["loads"][t], t
    assert st.expert_of.tolist() == ref["expert_of"]
    assert st.in_flight.tolist() == ref["in_flight"]


def test_stage_plan_rejects_bad_arguments():
    lib = L._lib
    st = M.StageTable(8, 4, 2)
    ids = np.array([1, 9], np.int32)  # 9 >= E
    out = st._out
    assert lib.moe_stage_plan(ctypes.byref(st._c), ids.ctypes.data, *out) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_stage_plan(ctypes.byref(st._c), None, *out) == M.MOE_ERR_INVALID_ARG
    bad = M.StageTable(8, 3, 2)  # fewer than 2k slots
    ids = np.array([1, 2], np.int32)
    assert lib.moe_stage_plan(ctypes.byref(bad._c), ids.ctypes.data, *bad._out) == M.MOE_ERR_INVALID_ARG
