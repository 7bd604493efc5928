"""C ABI checks that need no GPU: the library loads, exports every function the
header declares, sizes workspaces, and rejects bad arguments before launching."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import moe_routed_expert_route_gb300 as M
from moe_routed_expert_route_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z_]+)\s*\(",
                                src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "moe_route" in names and "moe_decode" in names and "moe_prefill" in names
    lib = ctypes.CDLL(M.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(L.EXPORTED)


def test_status_strings():
    for s in range(7):
        assert M.status_string(s) and M.status_string(s) != "unknown status"
    assert M.status_string(99) == "unknown status"


def test_workspace_sizes():
    a = M.moe_workspace_bytes(M.MOE_OP_LAYER, 1, 8, 256, 2048, 768)
    b = M.moe_workspace_bytes(M.MOE_OP_LAYER, 64, 8, 256, 2048, 768)
    assert 0 < a < b
    # h alone needs T*k*F floats
    assert b >= 64 * 8 * 768 * 4
    assert M.moe_workspace_bytes(M.MOE_OP_DECODE, 1, 8, 256, 2048, 768) > 0
    assert M.moe_workspace_bytes(M.MOE_OP_ROUTE, 4, 2, 8, 64, 0) > 0
    assert M.moe_workspace_bytes(M.MOE_OP_LAYER, 0, 8, 256, 2048, 768) == 0
    assert M.moe_workspace_bytes(M.MOE_OP_LAYER, 1, 8, 256, 2047, 768) == 0
    assert M.moe_workspace_bytes(M.MOE_OP_DECODE, 1, 8, 256, 2048, 100) == 0


def test_several_token_workspace_covers_the_grouped_products():
    # from 2 tokens on, a layer/decode workspace must also hold everything the
    # grouped products use (the prefill layout of the same T)
    for T in (2, 4, 64, 256):
        p = M.moe_workspace_bytes(M.MOE_OP_PREFILL, T, 8, 256, 2048, 768)
        assert p > 0
        assert M.moe_workspace_bytes(M.MOE_OP_LAYER, T, 8, 256, 2048, 768) >= p
        assert M.moe_workspace_bytes(M.MOE_OP_DECODE, T, 8, 256, 2048, 768) >= p
    # shapes outside the grouped products keep the smaller CUDA-core layout
    assert M.moe_workspace_bytes(M.MOE_OP_PREFILL, 8, 3, 13, 96, 160) == 0
    assert M.moe_workspace_bytes(M.MOE_OP_LAYER, 8, 3, 13, 96, 160) > 0


def _router(E=8, D=64, k=2, W=16):
    return L._Router(E, D, k, L.MOE_BF16, W, None, 1)


def test_invalid_arguments_rejected_before_launch():
    lib = L._lib
    r = _router()
    null = None
    # null x / outputs
    assert lib.moe_route(ctypes.byref(r), null, L.MOE_BF16, 1, 16, 16, null, 256, 10 ** 6, null) == \
        M.MOE_ERR_INVALID_ARG
    # k > E
    bad = _router(E=4, k=5)
    assert lib.moe_route(ctypes.byref(bad), 16, L.MOE_BF16, 1, 16, 16, null, 256, 10 ** 6, null) == \
        M.MOE_ERR_INVALID_ARG
    # D not a multiple of 32
    bad = _router(D=48)
    assert lib.moe_route(ctypes.byref(bad), 16, L.MOE_BF16, 1, 16, 16, null, 256, 10 ** 6, null) == \
        M.MOE_ERR_INVALID_ARG
    # misaligned router weights
    bad = _router(W=18)
    assert lib.moe_route(ctypes.byref(bad), 16, L.MOE_BF16, 1, 16, 16, null, 256, 10 ** 6, null) == \
        M.MOE_ERR_INVALID_ARG
    # unsupported activation dtype
    assert lib.moe_route(ctypes.byref(r), 16, L.MOE_F16, 1, 16, 16, null, 256, 10 ** 6, null) == \
        M.MOE_ERR_UNSUPPORTED
    # workspace too small / misaligned / missing
    assert lib.moe_route(ctypes.byref(r), 16, L.MOE_BF16, 1, 16, 16, null, 256, 8, null) == \
        M.MOE_ERR_WORKSPACE
    assert lib.moe_route(ctypes.byref(r), 16, L.MOE_BF16, 1, 16, 16, null, 272, 10 ** 6, null) == \
        M.MOE_ERR_WORKSPACE
    assert lib.moe_route(ctypes.byref(r), 16, L.MOE_BF16, 1, 16, 16, null, null, 10 ** 6, null) == \
        M.MOE_ERR_WORKSPACE
    # experts: F not a multiple of 32, null scale, k > E
    ex = L._Experts(8, 64, 48, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)
    assert lib.moe_decode(ctypes.byref(ex), 16, L.MOE_BF16, 1, 2, 16, 16, 16, null, 256, 10 ** 6,
                          null) == M.MOE_ERR_INVALID_ARG
    ex = L._Experts(8, 64, 64, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, null, 16, 16, 16, 16)
    assert lib.moe_decode(ctypes.byref(ex), 16, L.MOE_BF16, 1, 2, 16, 16, 16, null, 256, 10 ** 6,
                          null) == M.MOE_ERR_INVALID_ARG
    ex = L._Experts(8, 64, 64, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)
    assert lib.moe_decode(ctypes.byref(ex), 16, L.MOE_BF16, 1, 9, 16, 16, 16, null, 256, 10 ** 6,
                          null) == M.MOE_ERR_INVALID_ARG
    # T = 0
    assert lib.moe_decode(ctypes.byref(ex), 16, L.MOE_BF16, 0, 2, 16, 16, 16, null, 256, 10 ** 6,
                          null) == M.MOE_ERR_INVALID_ARG
    # substitution: negative / NaN threshold, k > E
    assert lib.moe_substitute(1, 8, 2, 16, 16, 16, 16, ctypes.c_float(-1.0), 16, 16, 16, 16, null) == \
        M.MOE_ERR_INVALID_ARG
    assert lib.moe_substitute(1, 8, 2, 16, 16, 16, 16, ctypes.c_float(float("nan")), 16, 16, 16, 16,
                              null) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_substitute(1, 8, 9, 16, 16, 16, 16, ctypes.c_float(0.15), 16, 16, 16, 16, null) == \
        M.MOE_ERR_INVALID_ARG
    # check_status without workspace
    assert lib.moe_check_status(null, null) == M.MOE_ERR_WORKSPACE


def test_binding_requires_cuda_tensors():
    import torch
    W = torch.zeros(8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        M.Router(W, None, 2).struct()


def _shared(D=64, F=64, r=4, q=L.MOE_Q_INT8_SYM_B32, s=L.MOE_F16, ld=L.MOE_BF16, A=16, scale=2.0):
    return L._Shared(D, F, r, q, s, 16, 16, 16, 16, 16, 16, ld, A, 16, 16, 16, 16, 16, scale)


def test_shared_lora_rejects_bad_arguments_before_launch():
    lib = L._lib
    null = None
    ws = M.moe_workspace_bytes(M.MOE_OP_SHARED, 4, 1, 1, 64, 64)
    assert ws > M.moe_workspace_bytes(M.MOE_OP_SHARED, 1, 1, 1, 64, 64) > 0
    assert M.moe_workspace_bytes(M.MOE_OP_SHARED, 1, 1, 1, 64, 48) == 0

    def call(s, x=16, xd=L.MOE_BF16, T=4, y=16, w=256, n=ws):
        return lib.moe_shared_lora(ctypes.byref(s), x, xd, T, y, 0, w, n, null)
    assert call(_shared(F=48)) == M.MOE_ERR_INVALID_ARG          # F not a multiple of 32
    assert call(_shared(r=65)) == M.MOE_ERR_INVALID_ARG          # rank above 64
    assert call(_shared(r=-1)) == M.MOE_ERR_INVALID_ARG
    assert call(_shared(A=18)) == M.MOE_ERR_INVALID_ARG          # misaligned adapter
    assert call(_shared(A=None)) == M.MOE_ERR_INVALID_ARG        # missing adapter with r > 0
    assert call(_shared(scale=float("inf"))) == M.MOE_ERR_INVALID_ARG
    assert call(_shared(ld=L.MOE_F16)) == M.MOE_ERR_UNSUPPORTED  # fp16 adapters
    assert call(_shared(s=L.MOE_BF16)) == M.MOE_ERR_UNSUPPORTED  # bf16 scales
    assert call(_shared(), xd=L.MOE_F16) == M.MOE_ERR_UNSUPPORTED
    assert call(_shared(), T=0) == M.MOE_ERR_INVALID_ARG
    assert call(_shared(), y=null) == M.MOE_ERR_INVALID_ARG
    assert call(_shared(), n=ws - 1) == M.MOE_ERR_WORKSPACE
    assert call(_shared(), w=272) == M.MOE_ERR_WORKSPACE
    assert lib.moe_shared_lora(null, 16, L.MOE_BF16, 1, 16, 0, 256, ws, null) == M.MOE_ERR_INVALID_ARG


def test_preroute_rejects_bad_arguments_before_launch():
    lib = L._lib
    null = None
    ws = M.moe_workspace_bytes(M.MOE_OP_PREROUTE, 2, 2, 8, 64, 32)
    assert ws > 0

    def head(D=64, E=8, H=32, k=2, wd=L.MOE_BF16, fc1=16, b1=None):
        return L._Prerouter(D, E, H, k, wd, fc1, b1, 16, 16, None, 1)

    def call(h, T=2, xd=L.MOE_BF16, cur=16, n=ws):
        return lib.moe_preroute(ctypes.byref(h), 16, xd, T, cur, 16, 16, 16, null, 256, n, null)
    assert call(head(E=6)) == M.MOE_ERR_INVALID_ARG      # E not a multiple of 4
    assert call(head(E=2048)) == M.MOE_ERR_INVALID_ARG   # E above 1024
    assert call(head(k=9)) == M.MOE_ERR_INVALID_ARG      # k > E
    assert call(head(H=40)) == M.MOE_ERR_INVALID_ARG     # H not a multiple of 32
    assert call(head(D=48)) == M.MOE_ERR_INVALID_ARG
    assert call(head(fc1=24)) == M.MOE_ERR_INVALID_ARG   # misaligned weights
    assert call(head(b1=18)) == M.MOE_ERR_INVALID_ARG    # misaligned bias
    assert call(head(wd=L.MOE_F16)) == M.MOE_ERR_UNSUPPORTED
    assert call(head(), xd=L.MOE_F16) == M.MOE_ERR_UNSUPPORTED
    assert call(head(), cur=null) == M.MOE_ERR_INVALID_ARG
    assert call(head(), T=0) == M.MOE_ERR_INVALID_ARG
    assert call(head(), n=ws - 1) == M.MOE_ERR_WORKSPACE


def test_noalloc_size_limits_rejected_before_launch():
    # moe_layer_noalloc keeps its scratch in a fixed array: E <= 1024 and
    # k*F <= 32768; beyond either it reports MOE_ERR_WORKSPACE before any
    # device work (fake, aligned pointers: nothing is dereferenced)
    lib = L._lib

    def call(E, k, D, F):
        r = L._Router(E, D, k, L.MOE_BF16, 16, None, 1)
        ex = L._Experts(E, D, F, L.MOE_Q_INT8_SYM_B32, L.MOE_F16, 16, 16, 16, 16, 16, 16)
        return lib.moe_layer_noalloc(ctypes.byref(r), ctypes.byref(ex), 16, L.MOE_BF16, 16, 16, None, 16, None,
                                     None)
    assert call(1025, 2, 64, 64) == M.MOE_ERR_WORKSPACE
    assert call(8, 8, 64, 8192) == M.MOE_ERR_WORKSPACE       # k*F = 65536
    assert call(1025, 2, 48, 64) == M.MOE_ERR_INVALID_ARG     # shape errors come first
