"""Host-side checks of the seeded synthetic inputs (no GPU): the shapes and
formats the layer consumes, the documented distributions, and determinism."""
import dataclasses

import numpy as np
import torch

import workloads as W


def test_configs_match_the_documented_shapes():
    c0, c1, c2, c3, c4 = (W.CONFIGS[i] for i in range(5))
    assert (c0.E, c0.k, c0.D, c0.F, c0.T, c0.qbits) == (8, 2, 64, 128, 4, 8)
    assert (c1.E, c1.k, c1.D, c1.F, c1.T, c1.qbits, c1.layers) == (256, 8, 2048, 768, 1, 8, 40)
    assert (c2.E, c2.k, c2.D, c2.F) == (256, 8, 2048, 768)
    assert (c3.E, c3.k, c3.D, c3.F, c3.qbits, c3.resident) == (512, 10, 2048, 512, 4, 128)
    assert abs(c3.threshold - 0.15) < 1e-12
    assert (c4.E, c4.k, c4.D, c4.F, c4.T) == (256, 8, 2048, 768, 2048)


def test_routed_bytes_per_expert():
    # cfg1: G+U codes 3,145,728 + fp16 scales 196,608, D codes 1,572,864 + 98,304
    assert W.routed_bytes_per_expert(W.CONFIGS[1]) == 5_013_504
    # cfg3 (int4): G+U 1,048,576 + 131,072, D 524,288 + 65,536
    assert W.routed_bytes_per_expert(W.CONFIGS[3]) == 1_769_472


def test_resident_mask_has_exactly_the_configured_count_and_is_seeded():
    cfg = W.CONFIGS[3]
    for layer in range(4):
        m = W.make_resident_mask(cfg, layer)
        assert m.dtype == torch.uint8 and m.shape == (cfg.E,)
        assert int(m.sum()) == cfg.resident
        assert torch.equal(m, W.make_resident_mask(cfg, layer))
    assert not torch.equal(W.make_resident_mask(cfg, 0), W.make_resident_mask(cfg, 1))


def test_layers_and_tokens_are_deterministic_and_distinct():
    cfg = W.CONFIGS[0]
    a, b = W.make_layer(cfg, 0), W.make_layer(cfg, 0)
    for key in ("Wr", "gate_q", "gate_s", "up_q", "down_q", "down_s"):
        assert torch.equal(a[key], b[key]), key
    c = W.make_layer(cfg, 1)
    assert not torch.equal(a["gate_q"], c["gate_q"])
    assert torch.equal(W.make_tokens(cfg, 4, 0), W.make_tokens(cfg, 4, 0))
    assert not torch.equal(W.make_tokens(cfg, 4, 0), W.make_tokens(cfg, 4, 1))


def test_zipf_bias_is_a_shuffled_log_rank_law():
    cfg = W.LayerConfig("zipf", E=64, k=4, D=64, F=64, T=1, qbits=8, scale_dtype=torch.float16,
                        x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.035,
                        zipf=1.1, layers=1, cfg_id=77)
    bias = W.make_layer(cfg, 0)["bias"].double().numpy()
    ranks = np.sort(np.exp(-bias / 1.1))  # = rank(e) for bias = -1.1 ln(rank)
    np.testing.assert_allclose(ranks, np.arange(1, 65), rtol=1e-5)
    assert not np.all(np.diff(bias) <= 0)  # shuffled, not in id order


def test_quantised_codes_stay_in_range():
    for cfg, qmax in ((W.CONFIGS[0], 127), ):
        L = W.make_layer(cfg, 0)
        for key in ("gate_q", "up_q", "down_q"):
            q = L[key]
            assert q.dtype == torch.int8
            assert int(q.abs().max()) <= qmax
    cfg4 = W.LayerConfig("q4", E=4, k=2, D=64, F=64, T=1, qbits=4, scale_dtype=torch.float16,
                         x_dtype=torch.bfloat16, router_dtype=torch.bfloat16, router_sigma=0.035,
                         zipf=None, layers=1, cfg_id=78)
    L = W.make_layer(cfg4, 0)
    packed = L["gate_q"].view(torch.uint8).numpy().astype(np.int32)
    lo = ((packed & 0xF) ^ 8) - 8
    hi = (((packed >> 4) & 0xF) ^ 8) - 8
    assert lo.min() >= -7 and lo.max() <= 7 and hi.min() >= -7 and hi.max() <= 7
    assert L["gate_q"].shape[-1] == cfg4.D // 2


def test_shared_expert_generator():
    sc = W.SHARED_CONFIGS["decode"]
    a = W.make_shared_expert(sc, 0)
    b = W.make_shared_expert(sc, 0)
    D, F, r = sc.D, sc.F, sc.rank
    assert a["gate_q"].shape == (F, D // 2) and a["down_q"].shape == (D, F // 2)  # int4, packed
    assert a["gate_s"].shape == (F, D // 32) and a["gate_s"].dtype == torch.float16
    assert a["gate_A"].shape == (r, D) and a["down_A"].shape == (r, F)
    assert a["gate_B"].shape == (F, r) and a["down_B"].shape == (D, r)
    assert a["gate_A"].dtype == torch.bfloat16 and a["scale"] == sc.alpha / r
    for n in ("gate_q", "gate_s", "down_q", "gate_A", "up_B", "down_B"):
        assert torch.equal(a[n], b[n])  # seeded
    assert not torch.equal(a["gate_A"], W.make_shared_expert(sc, 1)["gate_A"])
    # the adapters' delta (alpha/r) B A has an RMS of about 1e-3, the size the
    # Edge0 page gives for its recovery LoRA (below one 4-bit step)
    for p in ("gate", "up", "down"):
        delta = a["scale"] * (a[p + "_B"].double() @ a[p + "_A"].double())
        rms = float(delta.pow(2).mean().sqrt())
        assert 0.8e-3 < rms < 1.25e-3, (p, rms)
    z = W.make_shared_expert(dataclasses.replace(sc, rank=0), 0)
    assert z["gate_A"] is None and z["scale"] == 0.0


def test_prerouter_generator_warm_starts_from_the_next_router():
    cfg = W.CONFIGS[1]
    h = W.make_prerouter(cfg, 3, H=512)
    E, D = cfg.E, cfg.D
    assert h["fc1"].shape == (512, D + 2 * E) and h["fc2"].shape == (E, 512) and h["L"].shape == (E, D + 2 * E)
    Wr, bias = W.make_router(cfg, 4)
    assert torch.equal(h["L"][:, :D], Wr) and torch.equal(h["bias"], bias)
    assert torch.equal(W.make_layer(W.CONFIGS[0], 0)["Wr"], W.make_router(W.CONFIGS[0], 0)[0])
    assert torch.equal(h["fc1"], W.make_prerouter(cfg, 3, H=512)["fc1"])


def test_routing_history_generator():
    cfg = W.CONFIGS[1]
    cur, prev = W.make_routing_history(cfg, 20, stream=2)
    assert cur.shape == (20, cfg.k) and cur.dtype == torch.int32
    for row in torch.cat([cur, prev]).tolist():
        assert len(set(row)) == cfg.k and all(0 <= e < cfg.E for e in row)
    _, none = W.make_routing_history(cfg, 5, absent_prev=True)
    assert (none == -1).all()
