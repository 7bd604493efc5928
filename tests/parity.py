"""Comparison rules shared by the GPU parity tests (CUDA path vs the oracle).

Routing ids are compared bit-exactly except on tokens whose sorted oracle fp32
probabilities have two neighbours among the first k+1 within 1e-6 (a near tie:
another summation order may legitimately rank them differently). Such a token
is still checked: the GPU's ids must be *a* valid top-k under the oracle's
probabilities (every chosen probability >= every unchosen one - 1e-6, in
descending order within 1e-6, ids distinct), and its weights must be the
oracle probabilities of those ids renormalised. Every exclusion is counted per
test case and printed in the pytest summary.
"""
from __future__ import annotations

import os
from collections import OrderedDict

import numpy as np

import oracle

REL_TOL = 2e-3       # max |y - y_oracle| <= REL_TOL * max |y_oracle| (fp32-accumulated outputs)
TIE_EPS = 1e-6       # near-tie band on fp32 probabilities
W_ATOL = 1e-5        # routing weights
NTH = os.cpu_count() or 1

# label -> [excluded, total] for routing ties and substitution ambiguities
TIES: "OrderedDict[str, list]" = OrderedDict()


def record(label: str, kind: str, excluded: int, total: int):
    key = f"{label} [{kind}]"
    e = TIES.setdefault(key, [0, 0])
    e[0] += int(excluded)
    e[1] += int(total)


def check_valid_topk(p32_row: np.ndarray, ids: np.ndarray, k: int, eps: float = TIE_EPS):
    """ids must be a valid top-k of the probabilities p32_row within eps."""
    p = np.asarray(p32_row, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    assert ids.shape == (k,)
    assert ((ids >= 0) & (ids < p.shape[0])).all(), f"ids out of range: {ids}"
    assert len(set(ids.tolist())) == k, f"repeated ids: {ids}"
    chosen = p[ids]
    assert (np.diff(chosen) <= eps).all(), f"not descending within {eps}: {chosen}"
    rest = np.delete(p, ids)
    if rest.size:
        assert chosen.min() >= rest.max() - eps, f"an unchosen expert beats a chosen one by > {eps}"


def check_routing(ref: dict, got: dict, k: int, max_skip_frac: float = 0.1, label: str = "",
                  probs_rtol: float = 1e-5, probs_atol: float = 1e-6) -> int:
    """Compare the GPU routing (idx, w, optional probs) with the oracle's."""
    T = ref["idx"].shape[0]
    skip = set(oracle.near_tie_tokens(ref["probs32"], k).tolist())
    keep = np.array([t for t in range(T) if t not in skip], dtype=np.int64)
    assert len(skip) <= max(1, int(max_skip_frac * T)), f"{len(skip)} near-tie tokens of {T}"
    gi = np.asarray(got["idx"])
    gw = np.asarray(got["w"], dtype=np.float64)
    assert np.array_equal(gi[keep], ref["idx"][keep]), "routing ids differ from the oracle"
    np.testing.assert_allclose(gw[keep], ref["w"][keep], rtol=0, atol=W_ATOL)
    for t in sorted(skip):
        check_valid_topk(ref["probs32"][t], gi[t], k)
        pt = ref["probs32"][t].astype(np.float64)[gi[t]]
        np.testing.assert_allclose(gw[t], pt / pt.sum(), rtol=0, atol=W_ATOL)
    if got.get("probs") is not None:
        np.testing.assert_allclose(np.asarray(got["probs"]), ref["probs"], rtol=probs_rtol, atol=probs_atol)
    record(label or "routing", "near-tie tokens", len(skip), T)
    return len(skip)


def check_y(layer: dict, x, idx, w, y, qbits: int, tokens=None) -> float:
    """y against the oracle evaluated on the given routing (idx, w)."""
    idx = np.asarray(idx)
    w = np.asarray(w, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    xs = x
    if tokens is not None:
        idx, w, y = idx[tokens], w[tokens], y[tokens]
        xs = x[tokens]
    y_ref = oracle.moe(layer, xs, idx, w, qbits, nthreads=NTH)
    err = np.abs(y - y_ref).max()
    bound = REL_TOL * np.abs(y_ref).max()
    assert err <= bound, f"max|y - oracle| = {err:.3e} > {bound:.3e}"
    return float(err / max(np.abs(y_ref).max(), 1e-300))


def check_substitution(ref: dict, resident, threshold: float, got: dict, label: str = "") -> int:
    """End to end: the GPU's substitution decisions against the oracle's own
    routing followed by the oracle's substitution rule. Tokens excluded: routing
    near ties, and the substitution ambiguities of oracle.substitution_near_ties
    (a missed non-first slot with |w - threshold| <= 1e-6, or near-tied
    replacement candidates). Everything else must agree exactly; the mass, a sum
    of up to k-1 routing weights, within k times the weight tolerance."""
    T, k = ref["idx"].shape
    sref = oracle.substitute(ref["probs32"], ref["idx"], ref["w"], resident, threshold)
    tie_tok = set(oracle.near_tie_tokens(ref["probs32"], k).tolist())
    amb_tok = set(oracle.substitution_near_ties(ref["probs32"], ref["idx"], ref["w"], resident, threshold).tolist())
    keep = np.array([t for t in range(T) if t not in tie_tok and t not in amb_tok], dtype=np.int64)
    assert np.array_equal(np.asarray(got["idx_used"])[keep], sref["idx"][keep]), "substituted ids differ"
    assert np.array_equal(np.asarray(got["flag"])[keep], sref["flag"][keep]), "substitution flags differ"
    # mass sums up to k-1 weights, each within the routing-weight tolerance
    np.testing.assert_allclose(np.asarray(got["mass"], dtype=np.float64)[keep], sref["mass"][keep], rtol=0,
                               atol=W_ATOL * k)
    record(label or "substitution", "ambiguous substitution tokens", len(amb_tok - tie_tok), T)
    return len(amb_tok - tie_tok)
