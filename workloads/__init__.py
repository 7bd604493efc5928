"""Seeded synthetic inputs for the routed-expert MoE layer.

This module draws random numbers and lays them out in the formats the layer
consumes. It holds none of the layer's arithmetic: no routing, no softmax, no
dequantisation, no matrix product. The CPU oracle (``oracle/``) and the CUDA
library (``moe_routed_expert_route_gb300``) both read what it produces, and
neither of them imports the other.

Weight format ("sym8" / "sym4", symmetric linear, one scale per block of 32
consecutive input elements, as named in the Qiita gather_qmm write-up, section 6
"quality"): for each row n of an expert matrix and each block b of 32 elements
along the input (K) dimension,

    s[n][b] = cast(max_k |w[n][k]| / qmax)          (qmax = 127 for int8, 7 for int4)
    q[n][k] = clamp(round_half_even(w[n][k] / s[n][b]), -qmax, qmax)

with an all-zero block giving s = 0 and q = 0. Quantisation happens here, once,
so both implementations see identical codes and scales. Layout follows the MLX
stacked-expert array ``(num_experts, output_dims, input_dims)`` from the
lilting.ch router article (section "warm-up vs mmap cache"): codes are
``[E][N][K]`` with K contiguous, scales ``[E][N][K/32]``. int4 codes are packed
two per byte: byte j of a row holds element 2j in the low nibble and element
2j+1 in the high nibble, two's complement.

Router: logits = x . Wr^T + bias. The bias gives a Zipf(1.1) expert popularity:
bias[e] = -1.1 * ln(rank(e)), rank a seeded permutation of 1..E, so that
softmax(bias) is the Zipf law over a shuffled expert order.

Every tensor has its own seed, derived from (config seed, config id, layer,
tensor name) by a stable hash, so any layer can be regenerated on its own.
Generation uses torch's generator on the requested device; the bytes are the
same for every consumer within one process because they are produced once and
shared.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, Optional

import torch

__all__ = [
    "LayerConfig", "CONFIGS", "seed_for", "quantize_sym_blk32", "pack_int4",
    "make_layer", "make_router", "make_tokens", "make_resident_mask", "routed_bytes_per_expert",
    "SharedConfig", "SHARED_CONFIGS", "make_shared_expert", "make_shared_tokens",
    "make_prerouter", "make_routing_history",
]

BLOCK = 32


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape and distributions of one MoE layer workload."""
    name: str
    E: int                 # experts
    k: int                 # routed experts per token
    D: int                 # d_model (input of gate/up, output of down)
    F: int                 # d_ff (output of gate/up, input of down)
    T: int                 # default tokens per call
    qbits: int             # 8 or 4
    scale_dtype: torch.dtype
    x_dtype: torch.dtype
    router_dtype: torch.dtype
    router_sigma: float
    zipf: Optional[float]  # Zipf exponent of the router bias, None = no bias
    layers: int            # independent stacked layers
    weight_sigma: float = 0.02
    resident: int = 0      # experts marked resident (substitution workload)
    threshold: float = 0.15
    cfg_id: int = 0
    seed: int = 0


CONFIGS: Dict[int, LayerConfig] = {
    # Tiny layer for exhaustive comparison.
    0: LayerConfig("tiny E8 k2 D64 F128 int8", E=8, k=2, D=64, F=128, T=4, qbits=8,
                   scale_dtype=torch.float32, x_dtype=torch.float32,
                   router_dtype=torch.float32, router_sigma=0.05, zipf=None,
                   layers=1, cfg_id=0),
    # 256 experts, top-8, d_model 2048, d_ff 768 (Qwen3.6-35B-A3B-shaped), 40 layers.
    1: LayerConfig("decode E256 k8 D2048 F768 int8 x40 layers", E=256, k=8, D=2048,
                   F=768, T=1, qbits=8, scale_dtype=torch.float16,
                   x_dtype=torch.bfloat16, router_dtype=torch.bfloat16,
                   router_sigma=0.035, zipf=1.1, layers=40, cfg_id=1),
    # Batched decode sweep over the same layer stack (T in 1..64).
    2: LayerConfig("batched decode E256 k8 D2048 F768 int8 x40 layers", E=256, k=8,
                   D=2048, F=768, T=64, qbits=8, scale_dtype=torch.float16,
                   x_dtype=torch.bfloat16, router_dtype=torch.bfloat16,
                   router_sigma=0.035, zipf=1.1, layers=40, cfg_id=1),
    # 512 experts, top-10, d_ff 512, int4 (Qwen3-Next-80B-A3B-shaped), 25% resident.
    3: LayerConfig("substitution E512 k10 D2048 F512 int4 x16 layers", E=512, k=10,
                   D=2048, F=512, T=1, qbits=4, scale_dtype=torch.float16,
                   x_dtype=torch.bfloat16, router_dtype=torch.bfloat16,
                   router_sigma=0.035, zipf=1.1, layers=16, resident=128,
                   threshold=0.15, cfg_id=3),
    # Prefill of 2048 tokens on the decode layer shape.
    4: LayerConfig("prefill T2048 E256 k8 D2048 F768 int8", E=256, k=8, D=2048, F=768,
                   T=2048, qbits=8, scale_dtype=torch.float16,
                   x_dtype=torch.bfloat16, router_dtype=torch.bfloat16,
                   router_sigma=0.035, zipf=1.1, layers=1, cfg_id=1),
}


def seed_for(*parts) -> int:
    """Stable 63-bit seed from any tuple of ints/strings."""
    h = hashlib.sha256(repr(tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def pack_int4(q: torch.Tensor) -> torch.Tensor:
    """Pack int4 codes in [-8, 7] along the last dim: even index -> low nibble."""
    assert q.shape[-1] % 2 == 0
    u = (q.to(torch.int16) & 0xF).to(torch.uint8)
    lo = u[..., 0::2]
    hi = u[..., 1::2]
    return (lo | (hi << 4)).contiguous()


def quantize_sym_blk32(w: torch.Tensor, qbits: int, scale_dtype: torch.dtype):
    """Symmetric per-block-32 quantisation of float weights ``[..., K]``.

    Returns (codes, scales): int8 codes ``[..., K]`` (int4: packed uint8
    ``[..., K/2]``) and scales ``[..., K/32]`` in ``scale_dtype``.
    """
    qmax = 127 if qbits == 8 else 7
    K = w.shape[-1]
    assert K % BLOCK == 0
    wb = w.float().reshape(*w.shape[:-1], K // BLOCK, BLOCK)
    s = (wb.abs().amax(dim=-1) / qmax).to(scale_dtype)
    sf = s.float().unsqueeze(-1)
    safe = torch.where(sf == 0, torch.ones_like(sf), sf)
    q = torch.round(wb / safe)
    q = torch.where(sf == 0, torch.zeros_like(q), q)
    q = q.clamp(-qmax, qmax).to(torch.int8).reshape(w.shape)
    if qbits == 4:
        q = pack_int4(q)
    return q.contiguous(), s.contiguous()


def _quantized_matrix(cfg: LayerConfig, layer: int, name: str, rows: int, cols: int,
                      device, chunk: int):
    qcols = cols if cfg.qbits == 8 else cols // 2
    qdtype = torch.int8 if cfg.qbits == 8 else torch.uint8
    codes = torch.empty((cfg.E, rows, qcols), dtype=qdtype, device=device)
    scales = torch.empty((cfg.E, rows, cols // BLOCK), dtype=cfg.scale_dtype, device=device)
    g = _gen(device, seed_for(cfg.seed, cfg.cfg_id, layer, name))
    for e0 in range(0, cfg.E, chunk):
        e1 = min(cfg.E, e0 + chunk)
        w = torch.randn((e1 - e0, rows, cols), generator=g, device=device) * cfg.weight_sigma
        q, s = quantize_sym_blk32(w, cfg.qbits, cfg.scale_dtype)
        codes[e0:e1].copy_(q)
        scales[e0:e1].copy_(s)
        del w, q, s
    return codes, scales


def make_router(cfg: LayerConfig, layer: int = 0, device="cpu"):
    """Router weights of one layer: ``Wr`` [E][D] (router_dtype) and ``bias`` [E]
    fp32 (the Zipf log-popularity over a seeded expert order) or None."""
    g = _gen(device, seed_for(cfg.seed, cfg.cfg_id, layer, "router"))
    Wr = (torch.randn((cfg.E, cfg.D), generator=g, device=device) * cfg.router_sigma).to(cfg.router_dtype)
    bias = None
    if cfg.zipf is not None:
        gp = _gen("cpu", seed_for(cfg.seed, cfg.cfg_id, layer, "bias_perm"))
        rank = torch.randperm(cfg.E, generator=gp).to(torch.float64) + 1.0
        bias = (-cfg.zipf * torch.log(rank)).to(torch.float32).to(device)
    return Wr.contiguous(), bias


def make_layer(cfg: LayerConfig, layer: int = 0, device="cpu", chunk: int = 16) -> dict:
    """All weights of one layer.

    Keys: ``Wr`` [E][D] (router_dtype), ``bias`` [E] fp32 or None,
    ``gate_q``/``up_q`` [E][F][D or D/2], ``gate_s``/``up_s`` [E][F][D/32],
    ``down_q`` [E][D][F or F/2], ``down_s`` [E][D][F/32].
    """
    E, D, F = cfg.E, cfg.D, cfg.F
    Wr, bias = make_router(cfg, layer, device)
    gate_q, gate_s = _quantized_matrix(cfg, layer, "gate", F, D, device, chunk)
    up_q, up_s = _quantized_matrix(cfg, layer, "up", F, D, device, chunk)
    down_q, down_s = _quantized_matrix(cfg, layer, "down", D, F, device, chunk)
    return dict(Wr=Wr, bias=bias, gate_q=gate_q, gate_s=gate_s,
                up_q=up_q, up_s=up_s, down_q=down_q, down_s=down_s)


def make_tokens(cfg: LayerConfig, T: int, stream: int = 0, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1) of shape [T][D] in the config's activation dtype."""
    g = _gen(device, seed_for(cfg.seed, cfg.cfg_id, "x", stream, T))
    return torch.randn((T, cfg.D), generator=g, device=device).to(cfg.x_dtype).contiguous()


def make_resident_mask(cfg: LayerConfig, layer: int = 0, device="cpu") -> torch.Tensor:
    """uint8 [E]: exactly ``cfg.resident`` experts set to 1, chosen uniformly."""
    g = _gen("cpu", seed_for(cfg.seed, cfg.cfg_id, layer, "mask"))
    perm = torch.randperm(cfg.E, generator=g)
    m = torch.zeros(cfg.E, dtype=torch.uint8)
    m[perm[: cfg.resident]] = 1
    return m.to(device)


def routed_bytes_per_expert(cfg: LayerConfig) -> int:
    """Weight + scale bytes of one expert's gate, up and down matrices."""
    code_bytes = 1 if cfg.qbits == 8 else 0.5
    sb = torch.tensor([], dtype=cfg.scale_dtype).element_size()
    n = 3 * cfg.F * cfg.D
    return int(n * code_bytes + (n // BLOCK) * sb)



# ------------------------------------------------ shared expert with its LoRA

@dataclasses.dataclass(frozen=True)
class SharedConfig:
    """Shape of a MoE block's shared expert and of its recovery LoRA."""
    name: str
    D: int                 # d_model
    F: int                 # the shared expert's d_ff
    qbits: int             # base weights: 8 or 4
    scale_dtype: torch.dtype
    rank: int              # LoRA rank r (0 = no adapter)
    alpha: float           # the adapter is scaled by alpha / r
    lora_dtype: torch.dtype
    x_dtype: torch.dtype
    weight_sigma: float = 0.02
    lora_a_sigma: float = 0.01
    lora_b_sigma: float = 0.0125
    cfg_id: int = 10
    seed: int = 0


# The shared expert of the 256-expert decode layer served as the Edge0 page
# serves it: 4-bit base, rank-16 adapter with alpha = 32. sigma_A * sigma_B is
# chosen so that the delta (alpha/r) B A has an RMS of about 1e-3, the size the
# page gives for its adapters (below one 4-bit quantisation step).
SHARED_CONFIGS: Dict[str, SharedConfig] = {
    "decode": SharedConfig("shared expert D2048 F512 int4 + LoRA r16", D=2048, F=512, qbits=4,
                           scale_dtype=torch.float16, rank=16, alpha=32.0,
                           lora_dtype=torch.bfloat16, x_dtype=torch.bfloat16),
}


def _quantized_single(sc: SharedConfig, layer: int, name: str, rows: int, cols: int, device):
    g = _gen(device, seed_for(sc.seed, sc.cfg_id, layer, name))
    w = torch.randn((rows, cols), generator=g, device=device) * sc.weight_sigma
    return quantize_sym_blk32(w, sc.qbits, sc.scale_dtype)


def make_shared_expert(sc: SharedConfig, layer: int = 0, device="cpu") -> dict:
    """A shared expert and its unmerged adapters.

    Keys: ``gate_q``/``up_q`` [F][D or D/2], ``gate_s``/``up_s`` [F][D/32],
    ``down_q`` [D][F or F/2], ``down_s`` [D][F/32]; ``gate_A``/``up_A`` [r][D],
    ``down_A`` [r][F], ``gate_B``/``up_B`` [F][r], ``down_B`` [D][r] in
    lora_dtype (None when r = 0); ``scale`` = alpha / r; ``qbits``.
    """
    D, F, r = sc.D, sc.F, sc.rank
    out = dict(qbits=sc.qbits, scale=(sc.alpha / r) if r > 0 else 0.0)
    out["gate_q"], out["gate_s"] = _quantized_single(sc, layer, "shared_gate", F, D, device)
    out["up_q"], out["up_s"] = _quantized_single(sc, layer, "shared_up", F, D, device)
    out["down_q"], out["down_s"] = _quantized_single(sc, layer, "shared_down", D, F, device)
    for proj, n_in, n_out in (("gate", D, F), ("up", D, F), ("down", F, D)):
        if r == 0:
            out[proj + "_A"] = out[proj + "_B"] = None
            continue
        ga = _gen(device, seed_for(sc.seed, sc.cfg_id, layer, proj + "_lora_A"))
        gb = _gen(device, seed_for(sc.seed, sc.cfg_id, layer, proj + "_lora_B"))
        out[proj + "_A"] = (torch.randn((r, n_in), generator=ga, device=device) *
                            sc.lora_a_sigma).to(sc.lora_dtype).contiguous()
        out[proj + "_B"] = (torch.randn((n_out, r), generator=gb, device=device) *
                            sc.lora_b_sigma).to(sc.lora_dtype).contiguous()
    return out


def make_shared_tokens(sc: SharedConfig, T: int, stream: int = 0, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1) of shape [T][D] in the config's activation dtype."""
    g = _gen(device, seed_for(sc.seed, sc.cfg_id, "x", stream, T))
    return torch.randn((T, sc.D), generator=g, device=device).to(sc.x_dtype).contiguous()


# ------------------------------------------------------------ prerouter head

def make_prerouter(cfg: LayerConfig, layer: int = 0, H: int = 512, device="cpu",
                   sigma: float = 0.02, hot_sigma: float = 0.1) -> dict:
    """Prerouter head held by layer ``layer`` that predicts layer ``layer + 1``'s
    routing. Input width D + 2E (hidden state, k-hot routing of the current and
    of the previous token).

    Keys: ``fc1`` [H][D+2E] and ``fc2`` [E][H] ~ N(0, sigma) in the router dtype,
    ``b1`` [H] fp32 ~ N(0, sigma); ``L`` [E][D+2E]: its first D columns are the
    next layer's router weights (the warm start) and its 2E routing columns
    ~ N(0, hot_sigma); ``bias`` = the next layer's router bias.
    """
    E, D = cfg.E, cfg.D
    nf = D + 2 * E
    Wr_next, bias_next = make_router(cfg, layer + 1, device)
    g = _gen(device, seed_for(cfg.seed, cfg.cfg_id, layer, "prerouter"))
    fc1 = (torch.randn((H, nf), generator=g, device=device) * sigma).to(cfg.router_dtype)
    b1 = (torch.randn((H,), generator=g, device=device) * sigma).to(torch.float32)
    fc2 = (torch.randn((E, H), generator=g, device=device) * sigma).to(cfg.router_dtype)
    hot = (torch.randn((E, 2 * E), generator=g, device=device) * hot_sigma).to(cfg.router_dtype)
    L = torch.cat([Wr_next.to(cfg.router_dtype), hot], dim=1)
    return dict(fc1=fc1.contiguous(), b1=b1.contiguous(), fc2=fc2.contiguous(),
                L=L.contiguous(), bias=bias_next)


def make_routing_history(cfg: LayerConfig, T: int, stream: int = 0, device="cpu",
                         absent_prev: bool = False):
    """Seeded k-expert id lists (distinct ids per token) standing in for the
    current and previous tokens' routing: ``cur``, ``prev`` int32 [T][k]; with
    ``absent_prev`` the previous token is missing (ids -1)."""
    g = _gen("cpu", seed_for(cfg.seed, cfg.cfg_id, "history", stream, T))
    cur = torch.stack([torch.randperm(cfg.E, generator=g)[: cfg.k] for _ in range(T)])
    prev = torch.stack([torch.randperm(cfg.E, generator=g)[: cfg.k] for _ in range(T)])
    if absent_prev:
        prev = torch.full_like(prev, -1)
    return cur.to(torch.int32).to(device).contiguous(), prev.to(torch.int32).to(device).contiguous()
