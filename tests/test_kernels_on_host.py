"""The shared-expert/prerouter kernels (csrc/edge0.cu) and the expert cache
and staging host code (csrc/cache.cu), compiled from their own source as
plain C++ and run on the CPU against the oracles (no GPU).

edge0.cu is built against ``host_emulation/kernels.h``: the few CUDA builtins
it uses, with every warp's 32 lanes run as fibers that meet at each shuffle.
cache.cu is built against ``host_emulation/cuda_runtime.h`` (copies as host
copies) and ``host_emulation/stubs.cpp`` (plain definitions of the router and
the expert MLP in place of the library's moe_route / moe_decode). Both are
built with AddressSanitizer when the compiler has it, so an access outside a
buffer fails the test; an unaligned 16-byte load aborts, as it would fault on
the GPU. This runs the kernels' own index arithmetic, code unpacking, token
tiling and host orchestration on the shapes of the GPU tests; the GPU tests
(test_shared_lora_prerouter_gpu.py, test_streamed_expert_cache_gpu.py) remain
the parity tests of the CUDA path.

Sources: xyznot.com "The Other Half of the Memory Wall" (method: prerouter,
unmerged adapter execution; glossary: staged decode, incremental sticky-slot
stack); gist.science "Which expert misses are worth waiting for?" (method).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import parity
import workloads as W
import moe_routed_expert_route_gb300 as M
from moe_routed_expert_route_gb300 import _lib as L
from oracle import replay as R
from oracle import staging as S

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "moe_routed_expert_route_gb300", "csrc")
EMU = os.path.join(HERE, "host_emulation")
NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")
P, I, Sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


def _asan_flags():
    # AddressSanitizer needs its runtime loaded first; inside an ordinary
    # Python process only the flags for bounds checks of stack and globals
    # would apply, so it is used only when the process was started with it
    return ["-fsanitize=address"] if "libasan" in os.environ.get("LD_PRELOAD", "") else []


def _gxx():
    g = shutil.which("g++")
    if not g:
        pytest.skip("g++ not available")
    return g


@pytest.fixture(scope="module")
def edge0_lib(tmp_path_factory):
    d = tmp_path_factory.mktemp("edge0")
    # the quoted include resolves next to the source: build a copy of
    # edge0.cu beside the emulation header
    shutil.copy(os.path.join(CSRC, "edge0.cu"), d / "edge0.cu")
    shutil.copy(os.path.join(EMU, "kernels.h"), d / "kernels.h")
    so = d / "libedge0_host.so"
    subprocess.check_call([_gxx(), "-std=c++20", "-O2", "-fPIC", "-shared", *_asan_flags(),
                           "-I", os.path.join(ROOT, "include"), "-x", "c++", str(d / "edge0.cu"), "-o", str(so)])
    lib = ctypes.CDLL(str(so))
    lib.moe_shared_lora.argtypes = [P, P, I, I, P, I, P, Sz, P]
    lib.moe_preroute.argtypes = [P, P, I, I, P, P, P, P, P, P, Sz, P]
    return lib


@pytest.fixture(scope="module")
def cache_lib(tmp_path_factory):
    d = tmp_path_factory.mktemp("cache")
    so = d / "libcache_host.so"
    subprocess.check_call([_gxx(), "-std=c++20", "-O2", "-fPIC", "-shared", *_asan_flags(), "-I", EMU,
                           "-I", os.path.join(ROOT, "include"), "-x", "c++", os.path.join(CSRC, "cache.cu"),
                           "-x", "c++", os.path.join(EMU, "stubs.cpp"), "-o", str(so)])
    lib = ctypes.CDLL(str(so))
    lib.moe_pool_fetch.argtypes = [P, P, I, P, P, P]
    lib.moe_cache_workspace_bytes.argtypes = [I, I, I, I, I, P]
    lib.moe_cache_workspace_bytes.restype = Sz
    lib.moe_cached_layer.argtypes = [P] * 6 + [I] + [P] * 5 + [Sz] + [P] * 4
    lib.moe_stage_prediction.argtypes = [P] * 13
    return lib


def _aligned(nbytes):
    buf = torch.zeros(nbytes + 256, dtype=torch.uint8)
    return buf, buf.data_ptr() + (-buf.data_ptr()) % 256


def _act(t):
    return L.MOE_BF16 if t.dtype == torch.bfloat16 else L.MOE_F32


def _check_y(y, y_ref):
    err = np.abs(y - y_ref).max()
    assert err <= parity.REL_TOL * np.abs(y_ref).max(), f"max|y - oracle| = {err:.3e}"


# ------------------------------------------------- shared expert + LoRA

def _shared_struct(se):
    r = 0 if se.get("gate_A") is None else se["gate_A"].shape[0]
    F, D = se["gate_q"].shape[0], se["down_q"].shape[0]

    def ptr(t):
        return None if t is None or r == 0 else t.data_ptr()
    return L._Shared(D, F, r, L.MOE_Q_INT8_SYM_B32 if se["qbits"] == 8 else L.MOE_Q_INT4_SYM_B32,
                     L.MOE_F32 if se["gate_s"].dtype == torch.float32 else L.MOE_F16,
                     *[se[n].data_ptr() for n in NAMES],
                     L.MOE_BF16 if r and se["gate_A"].dtype == torch.bfloat16 else L.MOE_F32,
                     *[ptr(se.get(n)) for n in ("gate_A", "gate_B", "up_A", "up_B", "down_A", "down_B")],
                     float(se["scale"]) if r else 0.0)


def _run_shared(lib, se, x, y0=None):
    T, D = x.shape
    n = M.moe_workspace_bytes(M.MOE_OP_SHARED, T, 1, 1, D, se["gate_q"].shape[0])
    keep, ws = _aligned(n)
    y = torch.zeros(T, D) if y0 is None else y0.clone()
    s = _shared_struct(se)
    assert lib.moe_shared_lora(ctypes.byref(s), x.data_ptr(), _act(x), T, y.data_ptr(), int(y0 is not None),
                               ws, n, None) == 0
    return y.double().numpy()


@pytest.mark.parametrize("qbits", [8, 4])
@pytest.mark.parametrize("rank", [0, 4])
@pytest.mark.parametrize("T", [1, 9, 17])
def test_shared_lora_tiny_on_host(edge0_lib, qbits, rank, T):
    sc = W.SharedConfig("t", D=64, F=96, qbits=qbits, scale_dtype=torch.float32, rank=rank,
                        alpha=2.0 * max(rank, 1), lora_dtype=torch.float32, x_dtype=torch.float32,
                        weight_sigma=0.1, lora_a_sigma=0.2, lora_b_sigma=0.2, cfg_id=400 + rank)
    se = W.make_shared_expert(sc, 0, "cpu")
    x = W.make_shared_tokens(sc, T, 0, "cpu")
    _check_y(_run_shared(edge0_lib, se, x), oracle.shared_lora(se, x))


@pytest.mark.parametrize("T", [1, 16])
def test_shared_lora_decode_shape_on_host(edge0_lib, T):
    sc = W.SHARED_CONFIGS["decode"]
    se = W.make_shared_expert(sc, 0, "cpu")
    x = W.make_shared_tokens(sc, T, 1, "cpu")
    _check_y(_run_shared(edge0_lib, se, x), oracle.shared_lora(se, x))


def test_shared_lora_accumulates_on_host(edge0_lib):
    sc = W.SharedConfig("t8", D=256, F=128, qbits=8, scale_dtype=torch.float16, rank=8, alpha=16.0,
                        lora_dtype=torch.bfloat16, x_dtype=torch.bfloat16, cfg_id=410)
    se = W.make_shared_expert(sc, 0, "cpu")
    x = W.make_shared_tokens(sc, 5, 0, "cpu")
    y0 = torch.randn(5, sc.D, generator=torch.Generator().manual_seed(3))
    _check_y(_run_shared(edge0_lib, se, x, y0), y0.double().numpy() + oracle.shared_lora(se, x))


# ---------------------------------------------------------- prerouter head

def _run_preroute(lib, k, head, x, cur, prev):
    T, D = x.shape
    E, H = head["fc2"].shape[0], head["fc1"].shape[0]
    n = M.moe_workspace_bytes(M.MOE_OP_PREROUTE, T, k, E, D, H)
    keep, ws = _aligned(n)
    idx, w = torch.zeros(T, k, dtype=torch.int32), torch.zeros(T, k)
    h = L._Prerouter(D, E, H, k, L.MOE_F32 if head["fc1"].dtype == torch.float32 else L.MOE_BF16,
                     head["fc1"].data_ptr(), head["b1"].data_ptr(), head["fc2"].data_ptr(), head["L"].data_ptr(),
                     head["bias"].data_ptr(), 1)
    assert lib.moe_preroute(ctypes.byref(h), x.data_ptr(), _act(x), T, cur.data_ptr(), prev.data_ptr(),
                            idx.data_ptr(), w.data_ptr(), None, ws, n, None) == 0
    # the head's logits, in the workspace after the header and the hidden activations
    off = 256 + (4 * T * H + 255) // 256 * 256
    logits = np.ctypeslib.as_array((ctypes.c_float * (T * E)).from_address(ws + off)).reshape(T, E)
    return logits.astype(np.float64), ctypes.c_int.from_address(ws).value


def _tiny_head_cfg(seed):
    return W.LayerConfig("t", E=12, k=3, D=32, F=32, T=4, qbits=8, scale_dtype=torch.float32,
                         x_dtype=torch.float32, router_dtype=torch.float32, router_sigma=0.3,
                         zipf=1.1, layers=2, cfg_id=420 + seed)


@pytest.mark.parametrize("T", [1, 5, 11])
def test_prerouter_tiny_on_host(edge0_lib, T):
    cfg = _tiny_head_cfg(T)
    head = W.make_prerouter(cfg, 0, H=32, device="cpu", sigma=0.3, hot_sigma=0.5)
    x = W.make_tokens(cfg, T, 0, "cpu")
    cur, prev = W.make_routing_history(cfg, T, stream=T)
    prev[0] = -1
    if T > 1:
        cur[1, 2] = cur[1, 1]
    lg, status = _run_preroute(edge0_lib, cfg.k, head, x, cur, prev)
    assert status == 0
    np.testing.assert_allclose(lg, oracle.prerouter(head, x, cur, prev, cfg.k)["logits"], rtol=0, atol=1e-5)


@pytest.mark.parametrize("T", [1, 16])
def test_prerouter_decode_shape_on_host(edge0_lib, T):
    cfg = W.CONFIGS[1]
    head = W.make_prerouter(cfg, 0, H=512, device="cpu")
    x = W.make_tokens(cfg, T, 5, "cpu")
    cur, prev = W.make_routing_history(cfg, T, stream=5, absent_prev=(T == 1))
    lg, status = _run_preroute(edge0_lib, cfg.k, head, x, cur, prev)
    assert status == 0
    np.testing.assert_allclose(lg, oracle.prerouter(head, x, cur, prev, cfg.k)["logits"], rtol=0, atol=1e-5)


def test_prerouter_bad_id_on_host(edge0_lib):
    cfg = _tiny_head_cfg(9)
    head = W.make_prerouter(cfg, 0, H=32, device="cpu", sigma=0.3, hot_sigma=0.5)
    x = W.make_tokens(cfg, 2, 0, "cpu")
    cur, prev = W.make_routing_history(cfg, 2, stream=9)
    bad = cur.clone()
    bad[1, 0] = cfg.E + 5
    lg, status = _run_preroute(edge0_lib, cfg.k, head, x, bad, prev)
    assert status == M.MOE_ERR_BAD_INDEX
    absent = cur.clone()
    absent[1, 0] = -1
    np.testing.assert_allclose(lg, oracle.prerouter(head, x, absent, prev, cfg.k)["logits"], rtol=0, atol=1e-5)


# ----------------------------------------------- expert cache and staging

def _ex_struct(d, qbits):
    E, F = d["gate_q"].shape[:2]
    D = d["down_q"].shape[1]
    return L._Experts(E, D, F, L.MOE_Q_INT8_SYM_B32 if qbits == 8 else L.MOE_Q_INT4_SYM_B32,
                      L.MOE_F32 if d["gate_s"].dtype == torch.float32 else L.MOE_F16,
                      *[d[n].data_ptr() for n in NAMES])


@pytest.mark.parametrize("copy_stream,S_,N,what,qbits,scale", [
    (True, 8, 64, "admission", 8, torch.float16), (False, 8, 32, "admission", 8, torch.float16),
    (True, 3, 16, "transient", 8, torch.float16), (True, 8, 24, "any", 4, torch.float32)])
def test_cached_layer_on_host(cache_lib, copy_stream, S_, N, what, qbits, scale):
    lib = cache_lib
    cfg = W.LayerConfig("cache", E=32, k=4, D=256, F=128, T=1, qbits=qbits, scale_dtype=scale,
                        x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.02, zipf=1.1,
                        layers=1, cfg_id=505)
    layer = W.make_layer(cfg, 0, "cpu")
    host = {n: layer[n].contiguous() for n in NAMES}
    pool = {n: torch.zeros((S_ + cfg.k,) + tuple(layer[n].shape[1:]), dtype=layer[n].dtype) for n in NAMES}
    cached = np.random.default_rng(5).permutation(cfg.E)[:S_]
    h, p = _ex_struct(host, qbits), _ex_struct(pool, qbits)
    ex, sl = np.ascontiguousarray(cached, np.int32), np.arange(S_, dtype=np.int32)
    assert lib.moe_pool_fetch(ctypes.byref(h), ctypes.byref(p), S_, ex.ctypes.data, sl.ctypes.data, None) == 0
    r = L._Router(cfg.E, cfg.D, cfg.k, L.MOE_BF16, layer["Wr"].data_ptr(), layer["bias"].data_ptr(), 1)
    x = W.make_tokens(cfg, N, 3, "cpu")
    cache = M.ExpertCache(cfg.E, cfg.k, cached)
    hb = ctypes.c_size_t(0)
    n = lib.moe_cache_workspace_bytes(cfg.E, S_, cfg.k, cfg.D, cfg.F, ctypes.byref(hb))
    keep, ws = _aligned(n)
    scratch = torch.zeros(hb.value, dtype=torch.uint8)
    pol = L._policy(M.MOE_POLICY_THRESHOLD, 0.15, 0.5)
    fake = (16, 32, 48) if copy_stream else (None, None, None)  # stream and event handles: unused on the host
    probs, dec, ys = [], [], []
    for t in range(N):
        y = torch.zeros(1, cfg.D)
        assert lib.moe_cached_layer(ctypes.byref(r), ctypes.byref(h), ctypes.byref(p), ctypes.byref(cache._c),
                                    ctypes.byref(pol), x[t:t + 1].data_ptr(), L.MOE_BF16, y.data_ptr(), None,
                                    ctypes.byref(cache._st), scratch.data_ptr(), ws, n, None, *fake) == 0
        probs.append(scratch[:4 * cfg.E].view(torch.float32).numpy().copy())
        dec.append(cache.decisions())
        ys.append(y.numpy()[0].copy())
    probs = np.stack(probs)
    res = np.zeros((1, cfg.E), np.uint8)
    res[0, cached] = 1
    rp = R.replay(probs[:, None, :], cfg.k, R.THRESHOLD, 0.15, 0.5, 0.0, 0.0, resident=res.tolist())
    n_adm = n_tr = 0
    for t, d in enumerate(dec):
        assert d["expert"].tolist() == rp["used"][t][0], t
        assert d["flag"].tolist() == rp["flags"][t][0], t
        assert d["admit_expert"].tolist() == rp["admitted"][t][0], t
        n_adm += len(d["admit_expert"])
        n_tr += int((d["flag"] == 4).sum())
        parity.check_y(layer, x[t:t + 1], d["expert"][None], d["w"][None], ys[t][None], cfg.qbits)
    assert what == "any" or (n_adm if what == "admission" else n_tr) > 0
    for s_, e in enumerate(cache.expert_of):
        for nm in NAMES:
            assert torch.equal(pool[nm][s_], host[nm][e]), (s_, int(e), nm)


def test_stage_prediction_on_host(cache_lib):
    lib = cache_lib
    cfg = W.LayerConfig("stage", E=32, k=4, D=256, F=128, T=1, qbits=8, scale_dtype=torch.float16,
                        x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.035, zipf=1.1,
                        layers=2, cfg_id=520)
    k, NS, N = cfg.k, 2 * cfg.k, 13
    layer = W.make_layer(cfg, 1, "cpu")
    head = W.make_prerouter(cfg, 0, H=32, device="cpu")
    host = {n: layer[n].contiguous() for n in NAMES}
    pool = {n: torch.zeros((NS,) + tuple(layer[n].shape[1:]), dtype=layer[n].dtype) for n in NAMES}
    h, p = _ex_struct(host, 8), _ex_struct(pool, 8)
    x = W.make_tokens(cfg, N, 4, "cpu")
    cur, prev = W.make_routing_history(cfg, N, stream=4)
    ref = oracle.prerouter(head, x[:N - 1], cur[:N - 1], prev[:N - 1], k)
    st = M.StageTable(cfg.E, NS, k)
    scratch = torch.zeros(2 * k, dtype=torch.int32)
    bufs = [torch.zeros(k, dtype=torch.int32) for _ in range(2)]
    steps = []
    for t in range(N - 1):
        pred = torch.from_numpy(ref["idx"][t].copy())
        sb = bufs[t % 2]
        assert lib.moe_stage_prediction(ctypes.byref(st._c), ctypes.byref(h), ctypes.byref(p), pred.data_ptr(),
                                        sb.data_ptr(), scratch.data_ptr(), *st._out, None, 16, 32) == 0
        steps.append(st.step())
        assert sb.tolist() == steps[-1]["slot"].tolist()
        for r_, s_ in enumerate(sb.tolist()):  # the named slots hold the predicted experts
            for nm in NAMES:
                assert torch.equal(pool[nm][s_], host[nm][int(pred[r_])])
    so = S.stage(ref["idx"].tolist(), NS)
    for t in range(N - 1):
        assert steps[t]["slot"].tolist() == so["slots"][t]
        assert list(zip(steps[t]["load_expert"].tolist(), steps[t]["load_slot"].tolist())) == so["loads"][t]
