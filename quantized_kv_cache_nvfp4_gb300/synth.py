"""Seeded synthetic inputs shaped like the pages' KV workloads.

This module holds no codec arithmetic: it only draws random numbers (torch's
seeded generators), narrows them to bf16 with torch's own cast, and samples slot
ids, block tables and position maps.  Both the CUDA path and the CPU oracle are
fed from here, so they see identical bytes.

Recipe (each stream has its own generator, seeded ``seed * 1000 + stream``):
  values     N(0, 1) in fp32; a Bernoulli(p) mask multiplies entries by a factor
             (the outliers); then an RNE cast to bf16.
  slots      a seeded sample without replacement from the pool's slots.
  tables     a seeded permutation of the pool's physical blocks.
  positions  a sorted seeded sample of P of the T token rows (int32).
"""

from __future__ import annotations

import numpy as np
import torch

STREAM_K, STREAM_V, STREAM_SLOTS, STREAM_TABLE, STREAM_POS, STREAM_STEP = 1, 2, 3, 4, 5, 6


def gen(seed: int, stream: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + stream)
    return g


def normal_bf16(shape, seed: int, stream: int, outlier_frac: float = 0.0,
                outlier_scale: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """bf16 tensor of N(0,1) values with a fraction of entries scaled (outliers)."""
    g = gen(seed, stream, device)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if outlier_frac > 0.0:
        mask = torch.rand(shape, generator=g, dtype=torch.float32, device=device) < outlier_frac
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def sample_slots(n: int, num_slots: int, seed: int) -> torch.Tensor:
    """n distinct slot ids (int64) from a pool of num_slots."""
    g = gen(seed, STREAM_SLOTS)
    return torch.randperm(num_slots, generator=g)[:n].to(torch.int64)


def block_permutation(num_blocks: int, seed: int) -> torch.Tensor:
    g = gen(seed, STREAM_TABLE)
    return torch.randperm(num_blocks, generator=g).to(torch.int32)


def sorted_positions(T: int, P: int, seed: int, stream: int = STREAM_POS) -> torch.Tensor:
    g = gen(seed, stream)
    return torch.sort(torch.randperm(T, generator=g)[:P]).values.to(torch.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bf16 bit patterns -> CPU bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
def layer_kv(T: int, H: int, D: int, seed: int, outlier_frac: float = 0.0,
             outlier_scale: float = 1.0, device: str = "cpu"):
    """K and V [T, H, D] bf16."""
    k = normal_bf16((T, H, D), seed, STREAM_K, outlier_frac, outlier_scale, device)
    v = normal_bf16((T, H, D), seed, STREAM_V, outlier_frac, outlier_scale, device)
    return k, v


def one_layer_case(seed: int = 0):
    """K, V [256, 8, 128], N(0,1) with 1% x20 outliers; contiguous slots 0..255."""
    k, v = layer_kv(256, 8, 128, seed, 0.01, 20.0)
    return k, v, torch.arange(256, dtype=torch.int64)


def decode_step_case(seed: int = 2, T: int = 256, H: int = 8, D: int = 128,
                     qkv_width: int = 1152, num_slots: int = 65536):
    """256 requests appending one token each.

    K is a strided view of a fused qkv tensor [T, qkv_width] (row pitch qkv_width);
    V is a separate contiguous tensor whose row pitch (H*D) differs from K's.
    """
    qkv = normal_bf16((T, qkv_width), seed, STREAM_K)
    k = qkv[:, : H * D].unflatten(1, (H, D))
    v = normal_bf16((T, H, D), seed, STREAM_V)
    slots = sample_slots(T, num_slots, seed)
    return qkv, k, v, slots


def residual_loops(T: int = 4096, H: int = 8, D: int = 128, loops: int = 4, seed: int = 4,
                   step: float = 0.1, stream: int = STREAM_K):
    """loop 0 ~ N(0,1); loop i = bf16(loop i-1 + step * N(0,1)).  One chain per
    stream (K and V draw from different generators)."""
    out = []
    prev = normal_bf16((T, H, D), seed, stream)
    out.append(prev)
    g = gen(seed, STREAM_STEP + 10 * stream)
    for _ in range(1, loops):
        noise = torch.randn((T, H, D), generator=g, dtype=torch.float32)
        prev = (prev.float() + step * noise).to(torch.bfloat16)
        out.append(prev)
    return out
