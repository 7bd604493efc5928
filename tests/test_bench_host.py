"""Host-side check of the benchmark's CPU baseline (no GPU): the timed oracle
call runs on host copies of only the routed experts' rows, and must compute
exactly what the oracle computes on the whole layer."""
import dataclasses

import numpy as np
import torch

import bench
import oracle
import workloads as W


def _check(cfg, T):
    layer = W.make_layer(cfg, 0, "cpu")
    x = W.make_tokens(cfg, T, 3, "cpu")
    r = oracle.router(x, layer["Wr"], layer["bias"], cfg.k)
    el, y = bench.timed_oracle_moe(layer, x, r["idx"], r["w"], cfg.qbits, 2)
    assert el >= 0.0
    y_ref = oracle.moe(layer, x, r["idx"], r["w"], cfg.qbits, nthreads=2, compact=False)
    assert np.array_equal(y, y_ref)


def test_timed_oracle_moe_equals_the_oracle_int8():
    _check(W.CONFIGS[0], 5)


def test_timed_oracle_moe_equals_the_oracle_int4():
    # a small int4 layer with the substitution workload's formats
    cfg = dataclasses.replace(W.CONFIGS[3], E=16, k=3, D=128, F=64, cfg_id=90)
    _check(cfg, 4)
