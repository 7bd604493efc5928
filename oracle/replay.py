"""Oracle of the router-logit replay simulator -- TEST INFRASTRUCTURE ONLY.

gist.science "Which expert misses are worth waiting for?", method section: a
tool that replays router outputs to compare fetch/substitution policies,
estimating the time per token and the cache state. The policies follow the
page: fetch every miss; the 0.15 rule (a miss is fetched when it is the
router's first choice or its gate weight is at least the threshold, else a
resident expert stands in); the first-choice rule; background admission (the
gate mass substituted for an expert accumulates, and at the threshold -- 0.5
on the page -- the expert is admitted to the cache); frequency-based eviction.

Plain Python loops over tokens, layers and slots, in that order, with sets
and dictionaries for the cache. Besides the per-token totals it reports, per
token and layer, the expert that serves each slot, how it was obtained and
which experts were admitted, so that a cache that really moves experts can be
checked decision by decision. The open points are read as follows:
- the ranking is by fp32 probability, descending, lower id on equal values;
  weights are the k probabilities over their sum, in double, summed in rank
  order;
- the frequency of an expert is how often the layer's router chose it so far,
  counting the current token before any eviction;
- an expert that is fetched synchronously, or admitted, enters the cache,
  evicting the least frequent resident expert (lower id on ties) that the
  current token does not use in that layer (routed or chosen as a stand-in);
  when there is none, the expert is used without entering;
- the stand-in for a substituted miss is the resident expert of highest
  probability that is neither routed nor already a stand-in (lower id on
  ties); a miss with no stand-in left is fetched;
- the accumulated mass of an admitted expert restarts at zero; admission
  happens as soon as a substitution brings it to the threshold;
- the time of a token is, per layer, the layer's compute time plus its
  synchronous fetches times the fetch time; background admissions cost none.
"""
from __future__ import annotations

import math
import struct

FETCH_ALL, THRESHOLD, FIRST_CHOICE = 0, 1, 2


def _f32(v: float) -> float:
    return struct.unpack("f", struct.pack("f", float(v)))[0]


def replay(probs, k, policy, threshold=0.15, admit_mass=0.0, t_layer_us=0.0, t_fetch_us=0.0,
           resident=None, freq=None, acc=None):
    """probs: [N][L][E] (nested sequences or an array) of fp32 probabilities.
    resident: [L][E] of 0/1 (required); freq: [L][E] ints; acc: [L][E] floats.
    Returns per-token lists and the final state (as new lists)."""
    N = len(probs)
    L = len(resident)
    E = len(resident[0])
    cache = [set(e for e in range(E) if resident[l][e]) for l in range(L)]
    count = [[int(freq[l][e]) if freq is not None else 0 for e in range(E)] for l in range(L)]
    mass_of = [[float(acc[l][e]) if acc is not None else 0.0 for e in range(E)] for l in range(L)]
    # the policy's thresholds are fp32 values
    threshold = _f32(threshold)
    admit_mass = _f32(admit_mass)
    admit = admit_mass > 0 and math.isfinite(admit_mass)
    out = dict(t_token_us=[], fetches=[], substituted=[], sub_mass=[], admissions=[],
               used=[], flags=[], admitted=[])

    def insert(l, e, busy):
        candidates = [c for c in cache[l] if c not in busy]
        if not candidates:
            return False
        out_e = min(candidates, key=lambda c: (count[l][c], c))
        cache[l].remove(out_e)
        cache[l].add(e)
        return True

    for t in range(N):
        time_us, mass, n_fetch, n_sub, n_adm = 0.0, 0.0, 0, 0, 0
        used_t, flags_t, admitted_t = [], [], []
        for l in range(L):
            p = [float(v) for v in probs[t][l]]
            order = sorted(range(E), key=lambda e: (-p[e], e))
            chosen = order[:k]
            total = 0.0
            for e in chosen:
                total += p[e]
            weights = [(p[e] / total if total > 0 else 0.0) for e in chosen]
            for e in chosen:
                count[l][e] += 1
            busy = set(chosen)
            fetched_here = 0
            # per slot: the expert that serves it, and how (0 hit; 1 fetched
            # and cached; 2 substituted; 4 fetched, not cached: nothing
            # evictable). Stand-ins and evictions are drawn from the same
            # experts (cached, not used by the token), so a miss fetched for
            # want of a stand-in always takes 4.
            used = list(chosen)
            flags = [0] * k
            admitted = []
            for r, e in enumerate(chosen):
                if e in cache[l]:
                    continue
                if policy == FETCH_ALL:
                    want = True
                elif policy == FIRST_CHOICE:
                    want = r == 0
                else:
                    want = r == 0 or weights[r] >= threshold
                stand_in = None
                if not want:
                    pool = [c for c in cache[l] if c not in busy]
                    if pool:
                        stand_in = max(pool, key=lambda c: (p[c], -c))
                if stand_in is None:
                    fetched_here += 1
                    flags[r] = 1 if insert(l, e, busy) else 4
                    continue
                busy.add(stand_in)
                used[r] = stand_in
                flags[r] = 2
                n_sub += 1
                mass += weights[r]
                mass_of[l][e] += weights[r]
                if admit and mass_of[l][e] >= admit_mass and e not in cache[l]:
                    if insert(l, e, busy):
                        n_adm += 1
                        mass_of[l][e] = 0.0
                        admitted.append(e)
            used_t.append(used)
            flags_t.append(flags)
            admitted_t.append(admitted)
            n_fetch += fetched_here
            time_us += t_layer_us + fetched_here * t_fetch_us
        out["t_token_us"].append(time_us)
        out["fetches"].append(n_fetch)
        out["substituted"].append(n_sub)
        out["sub_mass"].append(mass)
        out["admissions"].append(n_adm)
        out["used"].append(used_t)
        out["flags"].append(flags_t)
        out["admitted"].append(admitted_t)
    out["resident"] = [[1 if e in cache[l] else 0 for e in range(E)] for l in range(L)]
    out["freq"] = count
    out["acc"] = mass_of
    return out
