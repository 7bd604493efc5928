"""Oracle of the staged slot table -- TEST INFRASTRUCTURE ONLY.

xyznot.com "The Other Half of the Memory Wall" (glossary: "staged decode",
"incremental sticky-slot stack"; method: "prediction-as-routing"): the
prerouter's prediction for the next token is staged before that token runs,
into a fixed set of expert slots reached through a slot table (no allocation
per step, double buffering), and a step rewrites only the slots whose expert
changed. The page leaves the slot choice open; it is read as follows:
- a predicted expert that is already staged keeps its slot (sticky);
- any other takes the lowest-numbered slot that holds neither one of this
  step's predicted experts nor one read by the step in flight (the previous
  step's slots, whose decode may still run), and is loaded into it;
- with 2k slots such a slot always exists (the two steps lock at most 2k
  slots, and every staged expert of this step already holds its own).
Plain Python with dictionaries; ids within a step are processed in order, and
a repeated id maps to the slot its first occurrence got.
"""
from __future__ import annotations


def stage(pred, n_slots, slot_of=None, expert_of=None, in_flight=None):
    """pred: [N][k] predicted expert ids per step. Returns per-step slot lists
    and load lists [(expert, slot)], and the final state (slot_of as a dict,
    expert_of as a list with -1 for an empty slot, in_flight as a list)."""
    slot_of = dict(slot_of or {})
    expert_of = list(expert_of) if expert_of is not None else [-1] * n_slots
    in_flight = list(in_flight or [])
    out = dict(slots=[], loads=[])
    for ids in pred:
        ids = [int(e) for e in ids]
        locked = set(in_flight) | {slot_of[e] for e in ids if e in slot_of}
        slots, loads = [], []
        for e in ids:
            if e in slot_of:
                slots.append(slot_of[e])
                continue
            free = [s for s in range(n_slots) if s not in locked]
            if not free:
                raise ValueError("no free slot: fewer than 2k slots")
            s = free[0]
            old = expert_of[s]
            if old >= 0:
                del slot_of[old]
            expert_of[s] = e
            slot_of[e] = s
            locked.add(s)
            slots.append(s)
            loads.append((e, s))
        out["slots"].append(slots)
        out["loads"].append(loads)
        in_flight = slots
    out["slot_of"] = slot_of
    out["expert_of"] = expert_of
    out["in_flight"] = in_flight
    return out
