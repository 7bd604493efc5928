"""Thin Python binding of libmoe_route.so (argument marshalling only).

Every function here converts torch tensors into device pointers, checks their
dtype, shape, device and contiguity, calls the C entry point of the same name
on the current torch stream, and raises ``MoeError`` on a non-OK status. No
computation of the layer happens in Python, and there is no fallback: if the
CUDA library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_route.so")

# moe_status_t
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_BAD_INDEX, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_WORKSPACE = 4, 5, 6
# moe_dtype_t / moe_qfmt_t / op ids
MOE_F32, MOE_BF16, MOE_F16 = 0, 1, 2
MOE_Q_INT8_SYM_B32, MOE_Q_INT4_SYM_B32 = 0, 1
MOE_OP_ROUTE, MOE_OP_DECODE, MOE_OP_LAYER, MOE_OP_PREFILL, MOE_OP_LAYER_RESIDENT = 0, 1, 2, 3, 4
MOE_OP_SHARED, MOE_OP_PREROUTE = 5, 6

EXPORTED = ("moe_workspace_bytes", "moe_route", "moe_substitute", "moe_decode", "moe_layer",
            "moe_layer_resident", "moe_layer_stack", "moe_layer_stack_resident", "moe_prefill", "moe_layer_noalloc",
            "moe_replay", "moe_shared_lora", "moe_preroute", "moe_cache_plan", "moe_pool_fetch",
            "moe_cache_workspace_bytes", "moe_cached_layer", "moe_stage_plan", "moe_stage_prediction",
            "moe_check_status", "moe_set_wait_limit", "moe_status_string")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


class _Router(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("D", ctypes.c_int), ("k", ctypes.c_int),
                ("w_dtype", ctypes.c_int), ("W", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("norm_topk", ctypes.c_int)]


class _ReplayPolicy(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int), ("threshold", ctypes.c_float), ("admit_mass", ctypes.c_float),
                ("t_layer_us", ctypes.c_double), ("t_fetch_us", ctypes.c_double)]


MOE_POLICY_FETCH_ALL, MOE_POLICY_THRESHOLD, MOE_POLICY_FIRST_CHOICE = 0, 1, 2


class _Experts(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("D", ctypes.c_int), ("F", ctypes.c_int),
                ("q", ctypes.c_int), ("s_dtype", ctypes.c_int),
                ("gate_q", ctypes.c_void_p), ("gate_s", ctypes.c_void_p),
                ("up_q", ctypes.c_void_p), ("up_s", ctypes.c_void_p),
                ("down_q", ctypes.c_void_p), ("down_s", ctypes.c_void_p)]


class _Shared(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("F", ctypes.c_int), ("r", ctypes.c_int),
                ("q", ctypes.c_int), ("s_dtype", ctypes.c_int),
                ("gate_q", ctypes.c_void_p), ("gate_s", ctypes.c_void_p),
                ("up_q", ctypes.c_void_p), ("up_s", ctypes.c_void_p),
                ("down_q", ctypes.c_void_p), ("down_s", ctypes.c_void_p),
                ("lora_dtype", ctypes.c_int),
                ("gate_A", ctypes.c_void_p), ("gate_B", ctypes.c_void_p),
                ("up_A", ctypes.c_void_p), ("up_B", ctypes.c_void_p),
                ("down_A", ctypes.c_void_p), ("down_B", ctypes.c_void_p),
                ("lora_scale", ctypes.c_float)]


class _Prerouter(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("E", ctypes.c_int), ("H", ctypes.c_int), ("k", ctypes.c_int),
                ("w_dtype", ctypes.c_int), ("fc1", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("fc2", ctypes.c_void_p), ("L", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("norm_topk", ctypes.c_int)]


class _Cache(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("S", ctypes.c_int), ("k", ctypes.c_int),
                ("slot_of", ctypes.c_void_p), ("expert_of", ctypes.c_void_p),
                ("freq", ctypes.c_void_p), ("acc", ctypes.c_void_p)]


class _CacheStep(ctypes.Structure):
    _fields_ = [("expert", ctypes.c_void_p), ("slot", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("flag", ctypes.c_void_p), ("fetch_expert", ctypes.c_void_p), ("fetch_slot", ctypes.c_void_p),
                ("admit_expert", ctypes.c_void_p), ("admit_slot", ctypes.c_void_p),
                ("n_fetch", ctypes.c_int), ("n_admit", ctypes.c_int), ("mass", ctypes.c_double)]


class _Stage(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("n_slots", ctypes.c_int), ("k", ctypes.c_int),
                ("slot_of", ctypes.c_void_p), ("expert_of", ctypes.c_void_p), ("in_flight", ctypes.c_void_p)]


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with moe_routed_expert_route_gb300/build.py "
                          "(nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.moe_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.moe_workspace_bytes.restype = S
    lib.moe_route.argtypes = [P, P, I, I, P, P, P, P, S, P]
    lib.moe_substitute.argtypes = [I, I, I, P, P, P, P, ctypes.c_float, P, P, P, P, P]
    lib.moe_decode.argtypes = [P, P, I, I, I, P, P, P, P, P, S, P]
    lib.moe_layer.argtypes = [P, P, P, I, I, P, P, P, P, P, P, S, P]
    lib.moe_prefill.argtypes = [P, P, P, I, I, P, P, P, P, P, P, S, P]
    lib.moe_layer_noalloc.argtypes = [P, P, P, I, P, P, P, P, P, P]
    lib.moe_layer_resident.argtypes = [P, P, P, I, I, P, ctypes.c_float, P, P, P, P, P, P, P, P, P, S, P]
    lib.moe_layer_stack.argtypes = [I, P, P, P, I, I, P, P, P, P, P, S, P]
    lib.moe_replay.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P]
    lib.moe_layer_stack_resident.argtypes = [I, P, P, P, I, I, P, ctypes.c_float, P, P, P, P, P, P, P, P, S, P]
    lib.moe_shared_lora.argtypes = [P, P, I, I, P, I, P, S, P]
    lib.moe_preroute.argtypes = [P, P, I, I, P, P, P, P, P, P, S, P]
    lib.moe_cache_plan.argtypes = [P, P, P, P]
    lib.moe_pool_fetch.argtypes = [P, P, I, P, P, P]
    lib.moe_cache_workspace_bytes.argtypes = [I, I, I, I, I, P]
    lib.moe_cache_workspace_bytes.restype = S
    lib.moe_cached_layer.argtypes = [P, P, P, P, P, P, I, P, P, P, P, P, S, P, P, P, P]
    lib.moe_stage_plan.argtypes = [P, P, P, P, P, P]
    lib.moe_stage_prediction.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.moe_check_status.argtypes = [P, P]
    lib.moe_set_wait_limit.argtypes = [P, ctypes.c_ulonglong, P]
    lib.moe_status_string.argtypes = [I]
    lib.moe_status_string.restype = ctypes.c_char_p
    for f in ("moe_route", "moe_substitute", "moe_decode", "moe_layer", "moe_prefill",
              "moe_layer_noalloc", "moe_layer_resident", "moe_layer_stack", "moe_check_status",
              "moe_set_wait_limit", "moe_shared_lora", "moe_preroute", "moe_cache_plan", "moe_pool_fetch",
              "moe_cached_layer", "moe_stage_plan", "moe_stage_prediction"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


_lib = load()


def status_string(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _host(t: torch.Tensor, name: str, dtype=None, shape=None):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _act_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise ValueError(f"activations must be float32 or bfloat16, got {t.dtype}")


@dataclass
class Router:
    """Router weights of one layer: W [E][D] (fp32/bf16), bias [E] fp32 or None."""
    W: torch.Tensor
    bias: Optional[torch.Tensor]
    k: int
    norm_topk: bool = True

    def struct(self) -> _Router:
        _dev(self.W, "W", (torch.float32, torch.bfloat16))
        if self.bias is not None:
            _dev(self.bias, "bias", torch.float32, (self.W.shape[0],))
        E, D = self.W.shape
        return _Router(E, D, self.k, MOE_F32 if self.W.dtype == torch.float32 else MOE_BF16,
                       self.W.data_ptr(), None if self.bias is None else self.bias.data_ptr(),
                       1 if self.norm_topk else 0)


@dataclass
class Experts:
    """Quantised experts of one layer ([E][rows][cols], cols contiguous)."""
    gate_q: torch.Tensor
    gate_s: torch.Tensor
    up_q: torch.Tensor
    up_s: torch.Tensor
    down_q: torch.Tensor
    down_s: torch.Tensor
    qbits: int = 8

    @property
    def E(self):
        return self.gate_q.shape[0]

    @property
    def F(self):
        return self.gate_q.shape[1]

    @property
    def D(self):
        return self.down_q.shape[1]

    @classmethod
    def from_layer(cls, layer: dict, qbits: int) -> "Experts":
        return cls(layer["gate_q"], layer["gate_s"], layer["up_q"], layer["up_s"],
                   layer["down_q"], layer["down_s"], qbits)

    def struct(self, host: bool = False) -> _Experts:
        """host: the tensors are in host memory (an expert store for
        moe_pool_fetch / moe_cached_layer), else on the device."""
        E, F = self.gate_q.shape[:2]
        D = self.down_q.shape[1]
        cb = 1 if self.qbits == 8 else 2
        qd = (torch.int8, torch.uint8)
        sd = (torch.float32, torch.float16)
        chk = _host if host else _dev
        chk(self.gate_q, "gate_q", qd, (E, F, D // cb))
        chk(self.up_q, "up_q", qd, (E, F, D // cb))
        chk(self.down_q, "down_q", qd, (E, D, F // cb))
        chk(self.gate_s, "gate_s", sd, (E, F, D // 32))
        chk(self.up_s, "up_s", self.gate_s.dtype, (E, F, D // 32))
        chk(self.down_s, "down_s", self.gate_s.dtype, (E, D, F // 32))
        return _Experts(E, D, F, MOE_Q_INT8_SYM_B32 if self.qbits == 8 else MOE_Q_INT4_SYM_B32,
                        MOE_F32 if self.gate_s.dtype == torch.float32 else MOE_F16,
                        self.gate_q.data_ptr(), self.gate_s.data_ptr(), self.up_q.data_ptr(),
                        self.up_s.data_ptr(), self.down_q.data_ptr(), self.down_s.data_ptr())


@dataclass
class Shared:
    """A shared expert ([F][D] gate/up, [D][F] down, quantised as the routed
    experts, no E dimension) and its unmerged adapters: A [r][in], B [out][r]
    in bf16/fp32 (None for r = 0), scale = alpha / r."""
    gate_q: torch.Tensor
    gate_s: torch.Tensor
    up_q: torch.Tensor
    up_s: torch.Tensor
    down_q: torch.Tensor
    down_s: torch.Tensor
    qbits: int = 8
    gate_A: Optional[torch.Tensor] = None
    gate_B: Optional[torch.Tensor] = None
    up_A: Optional[torch.Tensor] = None
    up_B: Optional[torch.Tensor] = None
    down_A: Optional[torch.Tensor] = None
    down_B: Optional[torch.Tensor] = None
    scale: float = 0.0

    @classmethod
    def from_dict(cls, se: dict) -> "Shared":
        return cls(**{k: se[k] for k in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
                                         "qbits", "gate_A", "gate_B", "up_A", "up_B", "down_A",
                                         "down_B", "scale")})

    @property
    def D(self):
        return self.down_q.shape[0]

    @property
    def F(self):
        return self.gate_q.shape[0]

    def struct(self) -> _Shared:
        F, D = self.F, self.D
        cb = 1 if self.qbits == 8 else 2
        qd = (torch.int8, torch.uint8)
        sd = (torch.float32, torch.float16)
        _dev(self.gate_q, "gate_q", qd, (F, D // cb))
        _dev(self.up_q, "up_q", qd, (F, D // cb))
        _dev(self.down_q, "down_q", qd, (D, F // cb))
        _dev(self.gate_s, "gate_s", sd, (F, D // 32))
        _dev(self.up_s, "up_s", self.gate_s.dtype, (F, D // 32))
        _dev(self.down_s, "down_s", self.gate_s.dtype, (D, F // 32))
        r = 0 if self.gate_A is None else self.gate_A.shape[0]
        lt = (torch.float32, torch.bfloat16)
        if r > 0:
            _dev(self.gate_A, "gate_A", lt, (r, D))
            _dev(self.up_A, "up_A", self.gate_A.dtype, (r, D))
            _dev(self.down_A, "down_A", self.gate_A.dtype, (r, F))
            _dev(self.gate_B, "gate_B", self.gate_A.dtype, (F, r))
            _dev(self.up_B, "up_B", self.gate_A.dtype, (F, r))
            _dev(self.down_B, "down_B", self.gate_A.dtype, (D, r))
        ld = MOE_BF16 if r > 0 and self.gate_A.dtype == torch.bfloat16 else MOE_F32
        return _Shared(D, F, r, MOE_Q_INT8_SYM_B32 if self.qbits == 8 else MOE_Q_INT4_SYM_B32,
                       MOE_F32 if self.gate_s.dtype == torch.float32 else MOE_F16,
                       self.gate_q.data_ptr(), self.gate_s.data_ptr(), self.up_q.data_ptr(),
                       self.up_s.data_ptr(), self.down_q.data_ptr(), self.down_s.data_ptr(), ld,
                       *[(None if t is None or r == 0 else t.data_ptr())
                         for t in (self.gate_A, self.gate_B, self.up_A, self.up_B, self.down_A,
                                   self.down_B)],
                       float(self.scale) if r > 0 else 0.0)


@dataclass
class Prerouter:
    """Prerouter head: fc1 [H][D+2E], b1 [H] fp32 or None, fc2 [E][H],
    L [E][D+2E] (fc1/fc2/L all fp32 or all bf16), bias [E] fp32 or None."""
    fc1: torch.Tensor
    b1: Optional[torch.Tensor]
    fc2: torch.Tensor
    L: torch.Tensor
    bias: Optional[torch.Tensor]
    k: int
    norm_topk: bool = True

    @classmethod
    def from_dict(cls, head: dict, k: int, norm_topk: bool = True) -> "Prerouter":
        return cls(head["fc1"], head.get("b1"), head["fc2"], head["L"], head.get("bias"), k, norm_topk)

    def struct(self) -> _Prerouter:
        E, H = self.fc2.shape
        D = self.fc1.shape[1] - 2 * E
        _dev(self.fc1, "fc1", (torch.float32, torch.bfloat16), (H, D + 2 * E))
        _dev(self.fc2, "fc2", self.fc1.dtype, (E, H))
        _dev(self.L, "L", self.fc1.dtype, (E, D + 2 * E))
        if self.b1 is not None:
            _dev(self.b1, "b1", torch.float32, (H,))
        if self.bias is not None:
            _dev(self.bias, "bias", torch.float32, (E,))
        return _Prerouter(D, E, H, self.k, MOE_F32 if self.fc1.dtype == torch.float32 else MOE_BF16,
                          self.fc1.data_ptr(), None if self.b1 is None else self.b1.data_ptr(),
                          self.fc2.data_ptr(), self.L.data_ptr(),
                          None if self.bias is None else self.bias.data_ptr(),
                          1 if self.norm_topk else 0)


class ExpertCache:
    """Host state of one layer's expert cache (slot table, routing counts,
    accumulated substituted weight) and the arrays of one token's decisions,
    all numpy arrays handed to the C calls by address."""

    def __init__(self, E: int, k: int, cached):
        import numpy as np
        cached = [int(e) for e in cached]
        self.E, self.S, self.k = E, len(cached), k
        self.slot_of = np.full(E, -1, np.int32)
        self.expert_of = np.asarray(cached, np.int32).copy()
        for s_, e in enumerate(cached):
            self.slot_of[e] = s_
        self.freq = np.zeros(E, np.int32)
        self.acc = np.zeros(E, np.float64)
        self.step = {n: np.zeros(k, t) for n, t in (
            ("expert", np.int32), ("slot", np.int32), ("w", np.float32), ("flag", np.uint8),
            ("fetch_expert", np.int32), ("fetch_slot", np.int32), ("admit_expert", np.int32),
            ("admit_slot", np.int32))}
        self._c = _Cache(E, self.S, k, *(a.ctypes.data for a in (self.slot_of, self.expert_of, self.freq,
                                                                  self.acc)))
        self._st = _CacheStep(*(self.step[n].ctypes.data for n in (
            "expert", "slot", "w", "flag", "fetch_expert", "fetch_slot", "admit_expert", "admit_slot")), 0, 0, 0.0)

    def decisions(self) -> dict:
        d = {n: a.copy() for n, a in self.step.items()}
        d["fetch_expert"] = d["fetch_expert"][: self._st.n_fetch]
        d["fetch_slot"] = d["fetch_slot"][: self._st.n_fetch]
        d["admit_expert"] = d["admit_expert"][: self._st.n_admit]
        d["admit_slot"] = d["admit_slot"][: self._st.n_admit]
        d["mass"] = self._st.mass
        return d


class StageTable:
    """Host state of a staged slot table (slot of each expert, expert of each
    slot, the slots of the step in flight) and one step's outputs, numpy arrays
    handed to the C calls by address. All slots start empty."""

    def __init__(self, E: int, n_slots: int, k: int):
        import numpy as np
        self.E, self.n_slots, self.k = E, n_slots, k
        self.slot_of = np.full(E, -1, np.int32)
        self.expert_of = np.full(n_slots, -1, np.int32)
        self.in_flight = np.full(k, -1, np.int32)
        self.slot = np.zeros(k, np.int32)
        self.load_expert = np.zeros(k, np.int32)
        self.load_slot = np.zeros(k, np.int32)
        self.n_load = ctypes.c_int(0)
        self._c = _Stage(E, n_slots, k, self.slot_of.ctypes.data, self.expert_of.ctypes.data,
                         self.in_flight.ctypes.data)
        self._out = (self.slot.ctypes.data, self.load_expert.ctypes.data, self.load_slot.ctypes.data,
                     ctypes.byref(self.n_load))

    def step(self) -> dict:
        n = self.n_load.value
        return dict(slot=self.slot.copy(), load_expert=self.load_expert[:n].copy(),
                    load_slot=self.load_slot[:n].copy())


def moe_stage_plan(stage: StageTable, ids) -> dict:
    import numpy as np
    a = np.ascontiguousarray(ids, dtype=np.int32)
    if a.shape != (stage.k,):
        raise ValueError(f"ids has shape {a.shape}, expected ({stage.k},)")
    _check("moe_stage_plan", _lib.moe_stage_plan(ctypes.byref(stage._c), a.ctypes.data, *stage._out))
    return stage.step()


def moe_stage_prediction(stage: StageTable, host: "Experts", pool: "Experts", pred_idx: torch.Tensor,
                         slot_idx: torch.Tensor, host_scratch: torch.Tensor, stream=None, copy_stream=None,
                         ev_staged=None) -> dict:
    """Stages one predicted id list [k] (device); slot_idx [k] int32 (device)
    receives the slot ids for the decode, once ev_staged has been reached."""
    k = stage.k
    _dev(pred_idx, "pred_idx", torch.int32, (k,))
    _dev(slot_idx, "slot_idx", torch.int32, (k,))
    _host(host_scratch, "host_scratch", torch.int32, (2 * k,))
    h, d = host.struct(host=True), pool.struct()
    cs = None if copy_stream is None else ctypes.c_void_p(copy_stream.cuda_stream)
    ev = None if ev_staged is None else ctypes.c_void_p(ev_staged.cuda_event)
    _check("moe_stage_prediction", _lib.moe_stage_prediction(
        ctypes.byref(stage._c), ctypes.byref(h), ctypes.byref(d), _ptr(pred_idx), _ptr(slot_idx),
        _ptr(host_scratch), *stage._out, _stream(stream), cs, ev))
    return stage.step()


def _policy(policy: int, threshold: float, admit_mass: float) -> _ReplayPolicy:
    return _ReplayPolicy(policy, threshold, admit_mass, 0.0, 0.0)


def moe_cache_plan(cache: ExpertCache, probs, policy: int, threshold: float = 0.15,
                   admit_mass: float = 0.0) -> dict:
    """One token's decisions at one layer from its fp32 probabilities [E] (host)."""
    import numpy as np
    p = np.ascontiguousarray(probs, dtype=np.float32)
    if p.shape != (cache.E,):
        raise ValueError(f"probs has shape {p.shape}, expected ({cache.E},)")
    pol = _policy(policy, threshold, admit_mass)
    _check("moe_cache_plan", _lib.moe_cache_plan(ctypes.byref(cache._c), p.ctypes.data, ctypes.byref(pol),
                                                 ctypes.byref(cache._st)))
    return cache.decisions()


def moe_pool_fetch(host: "Experts", pool: "Experts", experts, slots, stream=None):
    import numpy as np
    ex = np.ascontiguousarray(experts, dtype=np.int32)
    sl = np.ascontiguousarray(slots, dtype=np.int32)
    if ex.shape != sl.shape or ex.ndim != 1:
        raise ValueError("experts and slots must be 1-D of the same length")
    h, d = host.struct(host=True), pool.struct()
    _check("moe_pool_fetch", _lib.moe_pool_fetch(ctypes.byref(h), ctypes.byref(d), int(ex.size), ex.ctypes.data,
                                                 sl.ctypes.data, _stream(stream)))


def moe_cache_workspace_bytes(E: int, S: int, k: int, D: int, F: int):
    hb = ctypes.c_size_t(0)
    n = int(_lib.moe_cache_workspace_bytes(E, S, k, D, F, ctypes.byref(hb)))
    return n, int(hb.value)


def moe_cached_layer(router: "Router", host: "Experts", pool: "Experts", cache: ExpertCache, policy: int,
                     threshold: float, admit_mass: float, x: torch.Tensor, y: torch.Tensor,
                     x_next: Optional[torch.Tensor], host_scratch: torch.Tensor, ws: torch.Tensor,
                     stream=None, copy_stream=None, ev_issued=None, ev_copied=None) -> dict:
    """One token through a cached layer; returns the token's decisions.
    ev_issued / ev_copied are torch.cuda.Event objects that have been recorded
    once (so that they exist)."""
    r = router.struct()
    _dev(x, "x", (torch.float32, torch.bfloat16), (1, r.D))
    _dev(y, "y", torch.float32, (1, r.D))
    if x_next is not None:
        _dev(x_next, "x_next", x.dtype, (1, r.D))
    _host(host_scratch, "host_scratch", torch.uint8)
    h, d = host.struct(host=True), pool.struct()
    pol = _policy(policy, threshold, admit_mass)
    cs = None if copy_stream is None else ctypes.c_void_p(copy_stream.cuda_stream)
    e1 = None if ev_issued is None else ctypes.c_void_p(ev_issued.cuda_event)
    e2 = None if ev_copied is None else ctypes.c_void_p(ev_copied.cuda_event)
    _check("moe_cached_layer", _lib.moe_cached_layer(
        ctypes.byref(r), ctypes.byref(h), ctypes.byref(d), ctypes.byref(cache._c), ctypes.byref(pol), _ptr(x),
        _act_dtype(x), _ptr(y), _ptr(x_next), ctypes.byref(cache._st), _ptr(host_scratch), _ptr(ws), ws.numel(),
        _stream(stream), cs, e1, e2))
    return cache.decisions()


def moe_workspace_bytes(op: int, T: int, k: int, E: int, D: int, F: int) -> int:
    return int(_lib.moe_workspace_bytes(op, T, k, E, D, F))


def workspace(op: int, T: int, k: int, E: int, D: int, F: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for `op` (torch allocations are 256-byte aligned)."""
    n = moe_workspace_bytes(op, T, k, E, D, F)
    if n == 0:
        raise ValueError("invalid workspace request")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def moe_route(router: Router, x: torch.Tensor, idx: torch.Tensor, w: torch.Tensor,
              probs: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    r = router.struct()
    T = x.shape[0]
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, r.D))
    _dev(idx, "idx", torch.int32, (T, r.k))
    _dev(w, "w", torch.float32, (T, r.k))
    if probs is not None:
        _dev(probs, "probs", torch.float32, (T, r.E))
    _check("moe_route", _lib.moe_route(ctypes.byref(r), _ptr(x), _act_dtype(x), T, _ptr(idx),
                                       _ptr(w), _ptr(probs), _ptr(ws), ws.numel(), _stream(stream)))


def moe_shared_lora(shared: Shared, x: torch.Tensor, y: torch.Tensor, accumulate: bool,
                    ws: torch.Tensor, stream=None):
    s = shared.struct()
    T = x.shape[0]
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, s.D))
    _dev(y, "y", torch.float32, (T, s.D))
    _check("moe_shared_lora", _lib.moe_shared_lora(ctypes.byref(s), _ptr(x), _act_dtype(x), T, _ptr(y),
                                                   1 if accumulate else 0, _ptr(ws), ws.numel(),
                                                   _stream(stream)))


def moe_preroute(head: Prerouter, x: torch.Tensor, cur: torch.Tensor, prev: torch.Tensor,
                 idx: torch.Tensor, w: torch.Tensor, probs: Optional[torch.Tensor], ws: torch.Tensor,
                 stream=None):
    h = head.struct()
    T = x.shape[0]
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, h.D))
    _dev(cur, "cur", torch.int32, (T, h.k))
    _dev(prev, "prev", torch.int32, (T, h.k))
    _dev(idx, "idx", torch.int32, (T, h.k))
    _dev(w, "w", torch.float32, (T, h.k))
    if probs is not None:
        _dev(probs, "probs", torch.float32, (T, h.E))
    _check("moe_preroute", _lib.moe_preroute(ctypes.byref(h), _ptr(x), _act_dtype(x), T, _ptr(cur),
                                             _ptr(prev), _ptr(idx), _ptr(w), _ptr(probs), _ptr(ws),
                                             ws.numel(), _stream(stream)))


def moe_substitute(probs, idx_in, w_in, resident, threshold: float, idx_out, w_out, sub_flag,
                   sub_mass, stream=None):
    T, E = probs.shape
    k = idx_in.shape[1]
    _dev(probs, "probs", torch.float32)
    _dev(idx_in, "idx_in", torch.int32, (T, k))
    _dev(w_in, "w_in", torch.float32, (T, k))
    _dev(resident, "resident", torch.uint8, (E,))
    _dev(idx_out, "idx_out", torch.int32, (T, k))
    _dev(w_out, "w_out", torch.float32, (T, k))
    _dev(sub_flag, "sub_flag", torch.uint8, (T, k))
    _dev(sub_mass, "sub_mass", torch.float32, (T,))
    thr = float(threshold)
    if math.isinf(thr):
        thr = float("inf")
    _check("moe_substitute", _lib.moe_substitute(T, E, k, _ptr(probs), _ptr(idx_in), _ptr(w_in),
                                                 _ptr(resident), ctypes.c_float(thr), _ptr(idx_out),
                                                 _ptr(w_out), _ptr(sub_flag), _ptr(sub_mass),
                                                 _stream(stream)))


def moe_decode(experts: Experts, x, idx, w, y, x_next, ws, stream=None):
    e = experts.struct()
    T, k = idx.shape
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, e.D))
    _dev(idx, "idx", torch.int32)
    _dev(w, "w", torch.float32, (T, k))
    _dev(y, "y", torch.float32, (T, e.D))
    if x_next is not None:
        _dev(x_next, "x_next", x.dtype, (T, e.D))
    _check("moe_decode", _lib.moe_decode(ctypes.byref(e), _ptr(x), _act_dtype(x), T, k, _ptr(idx),
                                         _ptr(w), _ptr(y), _ptr(x_next), _ptr(ws), ws.numel(),
                                         _stream(stream)))


def moe_layer(router: Router, experts: Experts, x, idx, w, probs, y, x_next, ws, stream=None):
    r = router.struct()
    e = experts.struct()
    T = x.shape[0]
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, e.D))
    _dev(idx, "idx", torch.int32, (T, r.k))
    _dev(w, "w", torch.float32, (T, r.k))
    if probs is not None:
        _dev(probs, "probs", torch.float32, (T, r.E))
    _dev(y, "y", torch.float32, (T, e.D))
    if x_next is not None:
        _dev(x_next, "x_next", x.dtype, (T, e.D))
    _check("moe_layer", _lib.moe_layer(ctypes.byref(r), ctypes.byref(e), _ptr(x), _act_dtype(x), T,
                                       _ptr(idx), _ptr(w), _ptr(probs), _ptr(y), _ptr(x_next),
                                       _ptr(ws), ws.numel(), _stream(stream)))


def moe_prefill(router: Router, experts: Experts, x, y, idx, w, counts, perm, ws, stream=None):
    r = router.struct()
    e = experts.struct()
    T = x.shape[0]
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, e.D))
    _dev(y, "y", torch.float32, (T, e.D))
    for t, n, shp, dt in ((idx, "idx", (T, r.k), torch.int32), (w, "w", (T, r.k), torch.float32),
                          (counts, "counts", (r.E,), torch.int32), (perm, "perm", (T * r.k,), torch.int32)):
        if t is not None:
            _dev(t, n, dt, shp)
    _check("moe_prefill", _lib.moe_prefill(ctypes.byref(r), ctypes.byref(e), _ptr(x), _act_dtype(x), T,
                                           _ptr(y), _ptr(idx), _ptr(w), _ptr(counts), _ptr(perm),
                                           _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_noalloc(router: Router, experts: Experts, x, idx, w, probs, y, x_next, stream=None):
    """One token through the layer with the library's static scratch (no workspace)."""
    r = router.struct()
    e = experts.struct()
    _dev(x, "x", (torch.float32, torch.bfloat16), (1, e.D))
    _dev(idx, "idx", torch.int32, (1, r.k))
    _dev(w, "w", torch.float32, (1, r.k))
    if probs is not None:
        _dev(probs, "probs", torch.float32, (1, r.E))
    _dev(y, "y", torch.float32, (1, e.D))
    if x_next is not None:
        _dev(x_next, "x_next", x.dtype, (1, e.D))
    _check("moe_layer_noalloc", _lib.moe_layer_noalloc(ctypes.byref(r), ctypes.byref(e), _ptr(x),
                                                       _act_dtype(x), _ptr(idx), _ptr(w), _ptr(probs),
                                                       _ptr(y), _ptr(x_next), _stream(stream)))


def moe_layer_resident(router: Router, experts: Experts, x, resident, threshold: float, idx, w, probs,
                       idx_used, sub_flag, sub_mass, y, x_next, ws, stream=None):
    """One layer with residency substitution between the router and the experts."""
    r = router.struct()
    e = experts.struct()
    T = x.shape[0]
    _dev(x, "x", (torch.float32, torch.bfloat16), (T, e.D))
    _dev(resident, "resident", torch.uint8, (r.E,))
    _dev(idx, "idx", torch.int32, (T, r.k))
    _dev(w, "w", torch.float32, (T, r.k))
    if probs is not None:
        _dev(probs, "probs", torch.float32, (T, r.E))
    _dev(idx_used, "idx_used", torch.int32, (T, r.k))
    _dev(sub_flag, "sub_flag", torch.uint8, (T, r.k))
    _dev(sub_mass, "sub_mass", torch.float32, (T,))
    _dev(y, "y", torch.float32, (T, e.D))
    if x_next is not None:
        _dev(x_next, "x_next", x.dtype, (T, e.D))
    thr = float(threshold)
    _check("moe_layer_resident", _lib.moe_layer_resident(
        ctypes.byref(r), ctypes.byref(e), _ptr(x), _act_dtype(x), T, _ptr(resident), ctypes.c_float(thr),
        _ptr(idx), _ptr(w), _ptr(probs), _ptr(idx_used), _ptr(sub_flag), _ptr(sub_mass), _ptr(y),
        _ptr(x_next), _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_stack(routers, experts, x, chain: bool, idx, w, y, x_next, ws, stream=None):
    """One token through a stack of layers in one launch.

    routers, experts: lists of Router / Experts (one per layer). x, idx, w, y,
    x_next: lists of per-layer tensors ([1][D], [1][k], [1][k], [1][D], [1][D])
    or stacked tensors whose first dimension is the layer; x_next may be None
    when ``chain`` is false."""
    _layer_stack(routers, experts, x, chain, idx, w, y, x_next, ws, stream)


def moe_layer_stack_resident(routers, experts, x, chain: bool, resident, threshold: float, idx, w, idx_used,
                             sub_flag, sub_mass, y, x_next, ws, stream=None):
    """moe_layer_stack with residency substitution in every layer: resident is a
    list of [E] uint8 masks; idx_used [1][k] int32, sub_flag [1][k] uint8 and
    sub_mass [1] fp32 per layer are outputs."""
    _layer_stack(routers, experts, x, chain, idx, w, y, x_next, ws, stream,
                 res=(resident, float(threshold), idx_used, sub_flag, sub_mass))


def _layer_stack(routers, experts, x, chain, idx, w, y, x_next, ws, stream, res=None):
    L = len(routers)
    if len(experts) != L:
        raise ValueError("one Experts per Router")
    rs = (_Router * L)(*[r.struct() for r in routers])
    es = (_Experts * L)(*[e.struct() for e in experts])
    D, k = es[0].D, rs[0].k

    def ptrs(ts, name, dtype, shape, optional=False):
        arr = (ctypes.c_void_p * L)()
        for l in range(L):
            t = None if ts is None else ts[l]
            if t is None:
                if not optional:
                    raise ValueError(f"{name}[{l}] is required")
                arr[l] = None
                continue
            _dev(t, f"{name}[{l}]", dtype, shape)
            arr[l] = t.data_ptr()
        return arr

    xd = x[0].dtype
    xs = ptrs(x, "x", xd, (1, D))
    _act_dtype(x[0])
    ia = ptrs(idx, "idx", torch.int32, (1, k))
    wa = ptrs(w, "w", torch.float32, (1, k))
    ya = ptrs(y, "y", torch.float32, (1, D))
    xn = None if x_next is None else ptrs(x_next, "x_next", xd, (1, D), optional=True)
    if res is None:
        _check("moe_layer_stack", _lib.moe_layer_stack(L, rs, es, xs, _act_dtype(x[0]), 1 if chain else 0, ia,
                                                       wa, ya, xn, _ptr(ws), ws.numel(), _stream(stream)))
        return
    resident, thr, idx_used, sub_flag, sub_mass = res
    E = rs[0].E
    ra = ptrs(resident, "resident", torch.uint8, (E,))
    ua = ptrs(idx_used, "idx_used", torch.int32, (1, k))
    fa = ptrs(sub_flag, "sub_flag", torch.uint8, (1, k))
    ma = ptrs(sub_mass, "sub_mass", torch.float32, (1,))
    _check("moe_layer_stack_resident", _lib.moe_layer_stack_resident(
        L, rs, es, xs, _act_dtype(x[0]), 1 if chain else 0, ra, ctypes.c_float(thr), ia, wa, ua, fa, ma, ya, xn,
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_check_status(ws: torch.Tensor, stream=None) -> int:
    return int(_lib.moe_check_status(_ptr(ws), _stream(stream)))


def moe_set_wait_limit(ws: torch.Tensor, cycles: int, stream=None):
    """Longest spin of any device wait on this workspace (clock64 cycles; 0 = default)."""
    _check("moe_set_wait_limit", _lib.moe_set_wait_limit(_ptr(ws), int(cycles), _stream(stream)))


def moe_replay(probs, k: int, policy: int, threshold: float = 0.15, admit_mass: float = 0.0,
               t_layer_us: float = 0.0, t_fetch_us: float = 0.0, resident=None, freq=None, acc=None) -> dict:
    """Router-logit replay on the host (see moe_replay in the header).

    probs: numpy float32 [N][L][E]. resident [L][E] uint8, freq [L][E] int32 and
    acc [L][E] float64 are the cache state, updated in place (freq and acc start
    at zero when not given). Returns the per-token outputs and the state."""
    import numpy as np
    probs = np.ascontiguousarray(probs, dtype=np.float32)
    if probs.ndim != 3:
        raise ValueError("probs must be [N][L][E]")
    N, L, E = probs.shape
    if resident is None:
        raise ValueError("resident [L][E] is required")
    for name, a, dt in (("resident", resident, np.uint8), ("freq", freq, np.int32), ("acc", acc, np.float64)):
        if a is not None and (a.dtype != dt or a.shape != (L, E) or not a.flags["C_CONTIGUOUS"]):
            raise ValueError(f"{name} must be a contiguous {np.dtype(dt).name} array of shape {(L, E)}")
    freq = np.zeros((L, E), np.int32) if freq is None else freq
    acc = np.zeros((L, E), np.float64) if acc is None else acc
    out = dict(t_token_us=np.zeros(N, np.float64), fetches=np.zeros(N, np.int32),
               substituted=np.zeros(N, np.int32), sub_mass=np.zeros(N, np.float64),
               admissions=np.zeros(N, np.int32))
    pol = _ReplayPolicy(int(policy), float(threshold), float(admit_mass), float(t_layer_us), float(t_fetch_us))

    def p(a):
        return ctypes.c_void_p(a.ctypes.data)
    _check("moe_replay", _lib.moe_replay(N, L, E, int(k), p(probs), ctypes.byref(pol), p(resident), p(freq), p(acc),
                                         p(out["t_token_us"]), p(out["fetches"]), p(out["substituted"]),
                                         p(out["sub_mass"]), p(out["admissions"])))
    out.update(resident=resident, freq=freq, acc=acc)
    return out
