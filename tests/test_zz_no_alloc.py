"""moe_layer_noalloc: the single-token layer for callers that cannot allocate
device memory where they run it (a frozen or captured pool, an allocator that
is out of reach, an embedding that hands over only input and output buffers).
Its scratch is a static device array inside the library instead of a
caller-provided workspace; its results must equal the workspace entry point's.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3


def _run_pair(cfg, layer, stream_ids):
    import moe_routed_expert_route_gb300 as M
    router = M.Router(layer["Wr"], layer["bias"], cfg.k)
    experts = M.Experts.from_layer(layer, cfg.qbits)
    ws = M.workspace(M.MOE_OP_LAYER, 1, cfg.k, cfg.E, cfg.D, cfg.F, "cuda")
    for s in stream_ids:  # two calls in a row
        x = W.make_tokens(cfg, 1, s, "cuda")
        ref = dict(idx=torch.empty(1, cfg.k, dtype=torch.int32, device="cuda"),
                   w=torch.empty(1, cfg.k, device="cuda"), y=torch.empty(1, cfg.D, device="cuda"),
                   xn=torch.empty_like(x))
        got = {k_: torch.full_like(v, -7) for k_, v in ref.items()}
        M.moe_layer(router, experts, x, ref["idx"], ref["w"], None, ref["y"], ref["xn"], ws)
        M.moe_layer_noalloc(router, experts, x, got["idx"], got["w"], None, got["y"], got["xn"])
        torch.cuda.synchronize()
        assert M.moe_check_status(ws) == M.MOE_OK
        assert torch.equal(got["idx"], ref["idx"])
        torch.testing.assert_close(got["w"], ref["w"], rtol=0, atol=1e-6)
        y_ref = ref["y"].double().cpu().numpy()
        err = np.abs(got["y"].double().cpu().numpy() - y_ref).max()
        assert err <= REL_TOL * np.abs(y_ref).max(), f"max |y_noalloc - y| = {err:.3e}"
        assert torch.equal(got["xn"], (x.float() + got["y"]).to(x.dtype))
        # and directly against the oracle, on the routing this entry point chose
        y_or = oracle.moe(layer, x, got["idx"].cpu(), got["w"].cpu().double(), cfg.qbits)
        err_or = np.abs(got["y"].double().cpu().numpy() - y_or).max()
        assert err_or <= REL_TOL * np.abs(y_or).max(), f"max |y_noalloc - oracle| = {err_or:.3e}"


def test_noalloc_matches_workspace_layer_e256():
    cfg = W.CONFIGS[1]
    _run_pair(cfg, W.make_layer(cfg, 0, "cuda", chunk=64), [21, 22])


def test_noalloc_matches_workspace_layer_int4_e512():
    cfg = W.CONFIGS[3]
    _run_pair(cfg, W.make_layer(cfg, 0, "cuda", chunk=64), [23, 24])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """k*F beyond the static scratch is refused before anything is launched."""
    import moe_routed_expert_route_gb300 as M
    cfg = W.LayerConfig("big", E=8, k=8, D=64, F=8192, T=1, qbits=8, scale_dtype=torch.float16,
                        x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.1,
                        zipf=None, layers=1, cfg_id=99)
    layer = W.make_layer(cfg, 0, "cuda")
    x = W.make_tokens(cfg, 1, 0, "cuda")
    with pytest.raises(M.MoeError) as ei:
        M.moe_layer_noalloc(M.Router(layer["Wr"], layer["bias"], cfg.k), M.Experts.from_layer(layer, 8), x,
                            torch.empty(1, 8, dtype=torch.int32, device="cuda"), torch.empty(1, 8, device="cuda"),
                            None, torch.empty(1, 64, device="cuda"), None)
    assert ei.value.status == M.MOE_ERR_WORKSPACE
