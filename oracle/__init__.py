"""CPU oracle of the routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. It wraps ``moe_oracle.c`` (plain C, double precision,
straight loops) through ctypes, and shares nothing with the CUDA library.

Inputs are torch tensors or numpy arrays on any device; they are converted to
float64 on the host exactly (fp16/bf16/fp32 -> fp64 is exact), so the oracle sees
the same codes, scales and activations as the GPU path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (gcc, -O2, IEEE arithmetic, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_router.argtypes = [i, i, i, i, i, P, P, P, P, P, P, P, P]
    lib.oracle_substitute.argtypes = [i, i, i, P, P, P, P, ctypes.c_double, P, P, P, P]
    lib.oracle_moe.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, P, i]
    lib.oracle_permute.argtypes = [i, i, i, P, P, P, P, P, P]
    lib.oracle_max_threads.argtypes = []
    lib.oracle_shared_lora.argtypes = [i, i, i, i, i] + [P] * 12 + [ctypes.c_double, P, P]
    lib.oracle_prerouter.argtypes = [i, i, i, i, i, i] + [P] * 13
    for f in ("oracle_router", "oracle_substitute", "oracle_moe", "oracle_permute",
              "oracle_max_threads", "oracle_shared_lora", "oracle_prerouter"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def load_variant(so_path: str):
    """Load another build of moe_oracle.c (used by the tests' planted-mistake checks)."""
    return _bind(ctypes.CDLL(so_path))


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _u8(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu").contiguous().view(torch.uint8).numpy()
    return np.ascontiguousarray(a).view(np.uint8)


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().oracle_max_threads()


def router(x, Wr, bias, k: int, norm_topk: bool = True, lib=None) -> dict:
    """logits, probs (fp64), probs32 (the fp32 decision values), idx, w."""
    x, Wr = _f64(x), _f64(Wr)
    T, D = x.shape
    E = Wr.shape[0]
    b = None if bias is None else _f64(bias)
    out = dict(logits=np.empty((T, E)), probs=np.empty((T, E)),
               probs32=np.empty((T, E), np.float32), idx=np.empty((T, k), np.int32),
               w=np.empty((T, k)))
    rc = _load(lib).oracle_router(T, E, D, k, int(norm_topk), _p(x), _p(Wr),
                               None if b is None else _p(b), _p(out["logits"]),
                               _p(out["probs"]), _p(out["probs32"]), _p(out["idx"]), _p(out["w"]))
    if rc != 0:
        raise ValueError(f"oracle_router rc={rc}")
    return out


def substitute(probs32, idx, w, resident, threshold: float, lib=None) -> dict:
    """idx, w after residency substitution, flag (0 hit, 1 fetched, 2 substituted,
    3 no candidate) and per-token substituted mass."""
    p = np.ascontiguousarray(probs32, dtype=np.float32)
    idx, w, res = _i32(idx), _f64(w), _u8(resident)
    T, E = p.shape
    k = idx.shape[1]
    out = dict(idx=np.empty((T, k), np.int32), w=np.empty((T, k)),
               flag=np.empty((T, k), np.uint8), mass=np.empty(T))
    rc = _load(lib).oracle_substitute(T, E, k, _p(p), _p(idx), _p(w), _p(res), float(threshold),
                                   _p(out["idx"]), _p(out["w"]), _p(out["flag"]), _p(out["mass"]))
    if rc != 0:
        raise ValueError(f"oracle_substitute rc={rc}")
    return out


def moe(layer: dict, x, idx, w, qbits: int, nthreads: int = 1, compact: bool = True,
        lib=None) -> np.ndarray:
    """y[t] = sum_r w[t][r] * expert_mlp(idx[t][r], x[t]) in fp64.

    ``layer`` holds gate_q/gate_s/up_q/up_s/down_q/down_s (torch or numpy, any
    device). With ``compact`` only the routed experts' rows are copied to the host.
    """
    x = _f64(x)
    idx = _i32(idx)
    w = _f64(w)
    T, D = x.shape
    k = idx.shape[1]
    gq = layer["gate_q"]
    E = gq.shape[0]
    F = gq.shape[1]
    if compact:
        used, remap = np.unique(idx, return_inverse=True)
        sel = list(int(e) for e in used)
        idx_c = remap.reshape(idx.shape).astype(np.int32)

        def take(a):
            if hasattr(a, "detach"):
                import torch
                return a[torch.tensor(sel, dtype=torch.long, device=a.device)]
            return a[sel]
        parts = {n: take(layer[n]) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")}
        Ec = len(sel)
    else:
        parts, idx_c, Ec = layer, idx, E
    arrs = dict(gate_q=_u8(parts["gate_q"]), up_q=_u8(parts["up_q"]), down_q=_u8(parts["down_q"]),
                gate_s=_f64(parts["gate_s"]), up_s=_f64(parts["up_s"]), down_s=_f64(parts["down_s"]))
    y = np.empty((T, D))
    rc = _load(lib).oracle_moe(T, Ec, k, D, F, qbits, _p(arrs["gate_q"]), _p(arrs["gate_s"]),
                            _p(arrs["up_q"]), _p(arrs["up_s"]), _p(arrs["down_q"]),
                            _p(arrs["down_s"]), _p(x), _p(idx_c), _p(w), _p(y), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_moe rc={rc}")
    return y


def permute(idx, E: int, lib=None) -> dict:
    """cnt [E], off [E+1], perm_tok/perm_slot [T*k], inv [T][k]."""
    idx = _i32(idx)
    T, k = idx.shape
    out = dict(cnt=np.empty(E, np.int32), off=np.empty(E + 1, np.int32),
               perm_tok=np.empty(T * k, np.int32), perm_slot=np.empty(T * k, np.int32),
               inv=np.empty((T, k), np.int32))
    rc = _load(lib).oracle_permute(T, k, E, _p(idx), _p(out["cnt"]), _p(out["off"]),
                                _p(out["perm_tok"]), _p(out["perm_slot"]), _p(out["inv"]))
    if rc != 0:
        raise ValueError(f"oracle_permute rc={rc}")
    return out


def layer_forward(layer: dict, x, k: int, qbits: int, norm_topk: bool = True,
                  nthreads: int = 1, lib=None) -> dict:
    """Router then routed experts: the whole layer for tokens x."""
    r = router(x, layer["Wr"], layer.get("bias"), k, norm_topk, lib=lib)
    r["y"] = moe(layer, x, r["idx"], r["w"], qbits, nthreads, lib=lib)
    return r


def shared_lora(se: dict, x, lib=None) -> np.ndarray:
    """Shared expert with its unmerged recovery LoRA, y [T][D] in fp64.

    ``se`` holds gate_q/gate_s/up_q/up_s ([F][D] codes, [F][D/32] scales),
    down_q/down_s ([D][F], [D][F/32]), qbits, and the adapters gate_A/up_A
    ([r][D]), down_A ([r][F]), gate_B/up_B ([F][r]), down_B ([D][r]) with
    ``scale`` = alpha / r; r = 0 (or adapters None) is the base expert alone.
    """
    x = _f64(x)
    T, D = x.shape
    F = se["gate_q"].shape[0]
    qbits = int(se["qbits"])
    r = 0 if se.get("gate_A") is None else int(se["gate_A"].shape[0])
    q = {n: _u8(se[n]) for n in ("gate_q", "up_q", "down_q")}
    s = {n: _f64(se[n]) for n in ("gate_s", "up_s", "down_s")}
    empty = np.zeros(1)
    ad = {n: (_f64(se[n]) if r > 0 else empty)
          for n in ("gate_A", "gate_B", "up_A", "up_B", "down_A", "down_B")}
    y = np.empty((T, D))
    rc = _load(lib).oracle_shared_lora(
        T, D, F, r, qbits, _p(q["gate_q"]), _p(s["gate_s"]), _p(q["up_q"]), _p(s["up_s"]),
        _p(q["down_q"]), _p(s["down_s"]), _p(ad["gate_A"]), _p(ad["gate_B"]), _p(ad["up_A"]),
        _p(ad["up_B"]), _p(ad["down_A"]), _p(ad["down_B"]), float(se.get("scale", 0.0)), _p(x),
        _p(y))
    if rc != 0:
        raise ValueError(f"oracle_shared_lora rc={rc}")
    return y


def prerouter(head: dict, x, cur, prev, k: int, norm_topk: bool = True, lib=None) -> dict:
    """Prerouter head on tokens x with the current and previous tokens' routing
    ids ``cur``/``prev`` [T][k] (negative = absent): logits, probs (fp64),
    probs32, and the predicted idx / w used as the next layer's routing.

    ``head`` holds fc1 [H][D+2E], b1 [H] or None, fc2 [E][H], L [E][D+2E],
    bias [E] or None.
    """
    x = _f64(x)
    T, D = x.shape
    fc1, fc2, Lw = _f64(head["fc1"]), _f64(head["fc2"]), _f64(head["L"])
    H = fc1.shape[0]
    E = fc2.shape[0]
    b1 = None if head.get("b1") is None else _f64(head["b1"])
    bias = None if head.get("bias") is None else _f64(head["bias"])
    cur, prev = _i32(cur), _i32(prev)
    out = dict(logits=np.empty((T, E)), probs=np.empty((T, E)),
               probs32=np.empty((T, E), np.float32), idx=np.empty((T, k), np.int32),
               w=np.empty((T, k)))
    rc = _load(lib).oracle_prerouter(
        T, D, E, H, k, int(norm_topk), _p(x), _p(cur), _p(prev), _p(fc1),
        None if b1 is None else _p(b1), _p(fc2), _p(Lw), None if bias is None else _p(bias),
        _p(out["logits"]), _p(out["probs"]), _p(out["probs32"]), _p(out["idx"]), _p(out["w"]))
    if rc != 0:
        raise ValueError(f"oracle_prerouter rc={rc}")
    return out


def near_tie_tokens(probs32: np.ndarray, k: int, eps: float = 1e-6) -> np.ndarray:
    """Tokens whose ranking among the first k+1 sorted probabilities has two
    neighbours within ``eps``: their top-k set or order may legitimately differ
    under another summation order, so exact index comparison skips them."""
    p = np.sort(np.asarray(probs32, dtype=np.float64), axis=1)[:, ::-1]
    kk = min(k + 1, p.shape[1])
    gaps = p[:, : kk - 1] - p[:, 1:kk]
    return np.nonzero((gaps <= eps).any(axis=1))[0]


def substitution_near_ties(probs32, idx, w, resident, threshold: float, eps: float = 1e-6) -> np.ndarray:
    """Tokens whose residency substitution (gist.science, method section: keep
    a missed expert that is the first choice or has weight >= threshold, else
    replace it by the best resident expert outside the token's k) could
    legitimately come out differently under another summation order of the
    same arithmetic:

      * a missed slot r >= 1 whose weight lies within ``eps`` of a positive
        threshold (the keep-or-replace decision could flip), or
      * m >= 1 slots are replaced and two neighbours among the first m+1
        replacement candidates (resident experts outside the token's k, sorted
        by fp32 probability) lie within ``eps`` (which candidate goes to which
        slot could change).
    """
    p = np.asarray(probs32, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    w = np.asarray(w, dtype=np.float64)
    res = np.asarray(resident).astype(bool)
    T, k = idx.shape
    out = []
    for t in range(T):
        own = set(idx[t].tolist())
        ambiguous = False
        m = 0
        for r in range(1, k):
            if res[idx[t, r]]:
                continue
            if threshold > 0 and abs(w[t, r] - threshold) <= eps:
                ambiguous = True
            elif w[t, r] < threshold:
                m += 1
        if not ambiguous and m >= 1:
            cand = np.array([p[t, e] for e in range(p.shape[1]) if res[e] and e not in own])
            cand = np.sort(cand)[::-1][: m + 1]
            if cand.size >= 2 and ((cand[:-1] - cand[1:]) <= eps).any():
                ambiguous = True
        if ambiguous:
            out.append(t)
    return np.asarray(out, dtype=np.int64)
