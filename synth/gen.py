"""Seeded generators (torch RNG; CPU or CUDA device).

A stream is identified by (seed, *key). The key is hashed with a fixed
64-bit mixer into a torch Generator seed, so tensor i of a workload does not
depend on how many tensors were drawn before it.
"""
from __future__ import annotations

import torch

_MASK64 = (1 << 64) - 1


def _mix64(z: int) -> int:
    # splitmix64 finaliser (Steele, Lea, Flood 2014)
    z = (z + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_seed(seed: int, *key) -> int:
    """Deterministic 63-bit seed for the stream (seed, *key)."""
    h = _mix64(int(seed) & _MASK64)
    for k in key:
        if isinstance(k, str):
            for ch in k.encode():
                h = _mix64(h ^ ch)
        else:
            h = _mix64(h ^ (int(k) & _MASK64))
    return h & ((1 << 63) - 1)


def _gen(device, seed, *key) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(seed, *key))
    return g


def weight_fp32(shape, seed: int = 0, index: int = 0, std: float = 0.02,
                device="cpu") -> torch.Tensor:
    """W ~ N(0, std) in FP32, stream ('w', index)."""
    g = _gen(device, seed, "w", index)
    w = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return w.mul_(std)


def activation_bf16(n: int, d: int, seed: int = 0, index: int = 0,
                    std: float = 1.0, device="cpu") -> torch.Tensor:
    """x ~ N(0, std) rounded to BF16, shape [n, d], stream ('x', index)."""
    g = _gen(device, seed, "x", index)
    x = torch.randn((n, d), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def expert_ids(n: int, topk: int, n_experts: int, seed: int = 0,
               layer: int = 0) -> torch.Tensor:
    """[n, topk] int32: per token, topk distinct experts drawn uniformly
    without replacement from [0, n_experts). CPU tensor."""
    g = _gen("cpu", seed, "ids", layer)
    u = torch.rand((n, n_experts), generator=g, dtype=torch.float64)
    return torch.argsort(u, dim=1)[:, :topk].to(torch.int32).contiguous()


def route_weights(n: int, topk: int, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """[n, topk] FP32 combine weights: U(0,1) normalised to sum 1 per token.
    CPU tensor."""
    g = _gen("cpu", seed, "route", layer)
    u = torch.rand((n, topk), generator=g, dtype=torch.float64) + 1e-3
    return (u / u.sum(dim=1, keepdim=True)).to(torch.float32).contiguous()
