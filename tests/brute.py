"""Independent NumPy brute force used to pin the C oracle (CPU only).

Written separately from ``oracle/moe_oracle.c``: it dequantises every expert in
full with vectorised NumPy, evaluates *all* E experts densely for every token, and
only then masks to the routed ones. The identity "dense over all experts, masked
to the top k == gathered over the routed experts" is the one the Qiita gather_qmm
write-up relies on (section 4: unrouted experts contribute nothing, so skipping
their reads changes nothing; section 6: the gather equals the dequantised
reference).
"""
from __future__ import annotations

import numpy as np


def unpack_codes(codes: np.ndarray, qbits: int) -> np.ndarray:
    """Codes [..., K] (int8) or packed [..., K/2] (int4) -> int64 [..., K]."""
    c = np.asarray(codes)
    if qbits == 8:
        return c.view(np.int8).astype(np.int64)
    b = c.view(np.uint8).astype(np.int64)
    lo = b & 0xF
    hi = (b >> 4) & 0xF
    out = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return np.where(out >= 8, out - 16, out)


def dequant(codes: np.ndarray, scales: np.ndarray, qbits: int) -> np.ndarray:
    q = unpack_codes(codes, qbits).astype(np.float64)
    s = np.asarray(scales, dtype=np.float64)
    return q * np.repeat(s, 32, axis=-1)


def to_np(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch
        t = a.detach().cpu()
        if t.dtype in (torch.int8, torch.uint8):
            return t.numpy()
        return t.double().numpy()
    return np.asarray(a)


def dense_experts(layer: dict, x: np.ndarray, qbits: int) -> np.ndarray:
    """o[t][e][d] = Down_e( silu(Gate_e x_t) * (Up_e x_t) ) for every expert e."""
    G = dequant(to_np(layer["gate_q"]), to_np(layer["gate_s"]), qbits)   # [E][F][D]
    U = dequant(to_np(layer["up_q"]), to_np(layer["up_s"]), qbits)
    Dn = dequant(to_np(layer["down_q"]), to_np(layer["down_s"]), qbits)  # [E][D][F]
    x = np.asarray(x, dtype=np.float64)
    g = np.einsum("efd,td->tef", G, x)
    u = np.einsum("efd,td->tef", U, x)
    h = g * (1.0 / (1.0 + np.exp(-g))) * u
    return np.einsum("edf,tef->ted", Dn, h)


def dense_masked_moe(layer: dict, x, weights_full: np.ndarray, qbits: int) -> np.ndarray:
    """y[t] = sum_e weights_full[t][e] * o[t][e]; weights_full is zero off the route."""
    o = dense_experts(layer, np.asarray(x, np.float64), qbits)
    return np.einsum("te,ted->td", weights_full, o)


def softmax(logits: np.ndarray) -> np.ndarray:
    z = logits - logits.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def stable_topk(p32: np.ndarray, k: int) -> np.ndarray:
    """Full sort by (fp32 prob descending, expert index ascending), first k."""
    T, E = p32.shape
    out = np.empty((T, k), np.int64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -p32[t].astype(np.float64)))
        out[t] = order[:k]
    return out


def substitute_bruteforce(p32, idx, w, resident, threshold):
    """Python loops over the substitution rule, for tiny cases."""
    T, k = idx.shape
    E = p32.shape[1]
    idx2 = idx.copy()
    flag = np.zeros((T, k), np.uint8)
    mass = np.zeros(T)
    for t in range(T):
        chosen = set(int(e) for e in idx[t])
        for r in range(k):
            e = int(idx[t][r])
            if resident[e]:
                continue
            if r == 0 or np.float32(w[t][r]) >= np.float32(threshold):
                flag[t][r] = 1
                continue
            cands = [c for c in range(E) if resident[c] and c not in chosen]
            if not cands:
                flag[t][r] = 3
                continue
            best = sorted(cands, key=lambda c: (-float(p32[t][c]), c))[0]
            chosen.add(best)
            idx2[t][r] = best
            flag[t][r] = 2
            mass[t] += w[t][r]
    return idx2, flag, mass


def merged_dense_shared_lora(se: dict, x: np.ndarray) -> np.ndarray:
    """Shared expert with its adapter computed the other way round from the
    oracle: each projection's adapter is first merged, in fp64, into the
    dequantised weight (W' = dq(W) + scale * B A, a dense matrix), and the
    SwiGLU MLP then runs on the merged matrices with NumPy products. Merging is
    exact in fp64 (no re-quantisation), so it equals the unmerged form up to
    rounding: the distributive law behind the xyznot.com Edge0 page's parallel
    delta y = W(x) + (alpha/r) B A x."""
    qb = int(se["qbits"])

    def merged(p):
        W_ = dequant(to_np(se[p + "_q"]), to_np(se[p + "_s"]), qb)
        if se.get(p + "_A") is None:
            return W_
        return W_ + float(se["scale"]) * (to_np(se[p + "_B"]) @ to_np(se[p + "_A"]))

    G, U, Dn = merged("gate"), merged("up"), merged("down")
    x = np.asarray(x, np.float64)
    g = x @ G.T
    u = x @ U.T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ Dn.T


def khot_features(x: np.ndarray, cur: np.ndarray, prev: np.ndarray, E: int) -> np.ndarray:
    """[x ; hot(cur) ; hot(prev)] per token, negative ids absent."""
    T, D = x.shape
    f = np.zeros((T, D + 2 * E))
    f[:, :D] = x
    for t in range(T):
        for e in cur[t]:
            if e >= 0:
                f[t, D + e] = 1.0
        for e in prev[t]:
            if e >= 0:
                f[t, D + E + e] = 1.0
    return f


def prerouter_dense(head: dict, x, cur, prev) -> np.ndarray:
    """Prerouter logits with whole-matrix NumPy products and SciPy's erf."""
    from scipy.special import erf
    fc1, fc2, L = to_np(head["fc1"]), to_np(head["fc2"]), to_np(head["L"])
    E = fc2.shape[0]
    f = khot_features(np.asarray(x, np.float64), np.asarray(cur), np.asarray(prev), E)
    z = f @ fc1.T
    if head.get("b1") is not None:
        z = z + to_np(head["b1"])
    a = 0.5 * z * (1.0 + erf(z / np.sqrt(2.0)))
    logits = a @ fc2.T + f @ L.T
    if head.get("bias") is not None:
        logits = logits + to_np(head["bias"])
    return logits
