"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors; it holds none of the layer's
arithmetic.  The same tensors are fed to the CUDA library and to the CPU
oracle, so neither side regenerates anything on its own.

Workloads (shapes from the Qwen3-30B-A3B config quoted on the vLLM page,
"An expert is a small SwiGLU MLP"; the 256-expert top-8 64-layer stack from
the MoE execution analysis page; the 60-expert top-4 K=1408 shape from the
SGLang issue page):

  toy       M=3,   E=4,   k=2, H=128,  I=64,   B=16, seed 0
  decode    M in {1,8,32,64},        E=128, k=8, H=2048, I=768
  prefill   M in {512,4096,16384},   E=128, k=8, H=2048, I=768, Zipf(1.1) router offset
  stack     M in {1,16,128}, 64 layers, E=256, k=8, H=2048, I=512, residual chaining
  tail      M in {1,64,8192},        E=60,  k=4, H=2048, I=1408, logits ~ N(0,1) given

Distributions: weights W_r, W13, W2 ~ N(0, 0.02), x ~ N(0, 1), given logits
~ N(0, 1); each drawn in fp32 and rounded to bf16.  FP8 expert weights
(layer_weights_fp8) are drawn as codes directly: E4M3 codes of N(0, 64^2)
values (torch's float8_e4m3fn cast of a clamped fp32 draw) with one fp32 row
scale 0.02/64 * U(0.8, 1.2), so the weights they stand for have about the
bf16 weights' spread.  Seeds: s = 1_000_003 * cfg + 1_009 * layer +
tensor_idx (W_r:0, W13:1, W2:2, x:3, logits:4, W13 scales:5, W2 scales:6;
the toy config uses s = tensor_idx).  Timing repetitions draw x with
seed s + 100 * rep so that the routed expert set changes between reps.
"""
from __future__ import annotations

import dataclasses

import torch

TENSOR_IDX = {"w_router": 0, "w13": 1, "w2": 2, "x": 3, "logits": 4, "w13_scale": 5,
              "w2_scale": 6}


@dataclasses.dataclass(frozen=True)
class Workload:
    cfg: int
    name: str
    E: int
    top_k: int
    H: int
    I: int
    Ms: tuple
    renormalize: bool = True
    block_size_m: int = 0          # 0 = the library's automatic choice
    zipf_s: float = 0.0            # > 0: per-expert router offset -s*ln(rank)
    logits_given: bool = False     # router logits drawn directly, no W_r
    layers: int = 1
    residual: bool = False         # layer l+1 input = y_l computed with residual x_l


WORKLOADS = {
    1: Workload(1, "toy_e4_k2_h128_i64", E=4, top_k=2, H=128, I=64, Ms=(3,), block_size_m=16),
    2: Workload(2, "qwen3_30b_a3b_decode", E=128, top_k=8, H=2048, I=768, Ms=(1, 8, 32, 64)),
    3: Workload(3, "qwen3_30b_a3b_prefill_zipf", E=128, top_k=8, H=2048, I=768,
                Ms=(512, 4096, 16384), zipf_s=1.1),
    4: Workload(4, "e256_k8_i512_decode_stack64", E=256, top_k=8, H=2048, I=512,
                Ms=(1, 16, 128), layers=64, residual=True),
    5: Workload(5, "e60_k4_i1408_tail", E=60, top_k=4, H=2048, I=1408,
                Ms=(1, 64, 8192), logits_given=True),
}


def seed_of(cfg: int, layer: int, tensor: str, rep: int = 0) -> int:
    idx = TENSOR_IDX[tensor]
    base = idx if cfg == 1 else 1_000_003 * cfg + 1_009 * layer + idx
    return base + 100 * rep


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 with a seeded generator on `device`, rounded to bf16."""
    g = _gen(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def zipf_router_bias(E: int, s: float, seed: int = 1) -> torch.Tensor:
    """Per-expert offset -s*ln(rank_e), rank = 1 + a seeded permutation of 0..E-1 (fp32 [E]).

    Added to the router logits, it tilts the softmax by rank^-s, a Zipf(s)
    skew of the expert loads.
    """
    g = _gen(seed, "cpu")
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-s * torch.log(rank)).to(torch.float32)


def router_weights(w: Workload, layer: int = 0, device="cpu") -> dict:
    """W_r [E,H] bf16 (None when logits are given) and the router bias [E] (or None)."""
    out = {"w_router": None, "router_bias": None}
    if not w.logits_given:
        out["w_router"] = normal_bf16((w.E, w.H), 0.02, seed_of(w.cfg, layer, "w_router"), device)
    if w.zipf_s > 0:
        out["router_bias"] = zipf_router_bias(w.E, w.zipf_s).to(device)
    return out


def layer_weights(w: Workload, layer: int = 0, device="cpu") -> dict:
    """W_r [E,H] (unless logits are given), W13 [E,2I,H], W2 [E,H,I] (bf16), bias [E] or None."""
    out = {
        "w13": normal_bf16((w.E, 2 * w.I, w.H), 0.02, seed_of(w.cfg, layer, "w13"), device),
        "w2": normal_bf16((w.E, w.H, w.I), 0.02, seed_of(w.cfg, layer, "w2"), device),
    }
    out.update(router_weights(w, layer, device))
    return out


def fp8_codes(shape, seed: int, device="cpu") -> torch.Tensor:
    """uint8 E4M3 bit patterns of N(0, 64^2) draws (clamped to +-448 before the cast)."""
    g = _gen(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32).mul_(64.0)
    return t.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def row_scales(shape, seed: int, device="cpu") -> torch.Tensor:
    """fp32 per-row scales 0.02/64 * U(0.8, 1.2)."""
    g = _gen(seed, device)
    u = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    return u.mul_(0.4).add_(0.8).mul_(0.02 / 64.0)


def layer_weights_fp8(w: Workload, layer: int = 0, device="cpu") -> dict:
    """E4M3 expert weights: W13 codes [E,2I,H] + scales [E,2I], W2 codes [E,H,I] + scales [E,H]
    (uint8 / fp32); W_r and the bias as layer_weights draws them."""
    out = router_weights(w, layer, device)
    out["w13"] = fp8_codes((w.E, 2 * w.I, w.H), seed_of(w.cfg, layer, "w13"), device)
    out["w13_scale"] = row_scales((w.E, 2 * w.I), seed_of(w.cfg, layer, "w13_scale"), device)
    out["w2"] = fp8_codes((w.E, w.H, w.I), seed_of(w.cfg, layer, "w2"), device)
    out["w2_scale"] = row_scales((w.E, w.H), seed_of(w.cfg, layer, "w2_scale"), device)
    return out


def layer_input(w: Workload, M: int, rep: int = 0, device="cpu") -> dict:
    """x [M,H] bf16, and logits [M,E] bf16 when the workload gives logits directly."""
    out = {"x": normal_bf16((M, w.H), 1.0, seed_of(w.cfg, 0, "x", rep), device), "router_logits": None}
    if w.logits_given:
        out["router_logits"] = normal_bf16((M, w.E), 1.0, seed_of(w.cfg, 0, "logits", rep), device)
    return out


def random_shape_case(seed: int, *, max_M=40, max_E=48, max_H=256, max_I=192):
    """A small random (M, E, k, H, I) with H and I multiples of 16, for property tests."""
    g = _gen(seed, "cpu")

    def r(lo, hi):
        return int(torch.randint(lo, hi + 1, (1,), generator=g).item())

    E = r(1, max_E)
    k = r(1, min(E, 8))
    return dict(M=r(1, max_M), E=E, top_k=k, H=16 * r(1, max_H // 16), I=16 * r(1, max_I // 16))


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor as its numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def from_bits(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bf16 bit patterns -> torch bf16 tensor."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
