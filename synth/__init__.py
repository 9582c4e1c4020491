"""Seeded synthetic inputs for the CSA2 global-attention layer.

This module is shared by the CPU oracle side and the CUDA side of the tests and
the benchmark.  It only draws random numbers and shapes them into the value
distributions the workloads name; it performs none of the layer's own
arithmetic (no compression, normalisation of cache latents, RoPE, quantisation,
scoring, selection or attention).

Distributions (one seed per workload):
  * latents            N(0,1) float32 rounded to bf16 (round-to-nearest-even)
  * compressor weights softplus(N(0,1)) per channel, float32
  * index projection   N(0, 1/512) rounded to bf16, shape [128, 512]
  * index queries      N(0,1) bf16, [.., 32 heads, 128]
  * head weights       N(0,1) float32, [.., 32]
  * main queries       N(0,1) bf16, [.., 64 heads, 512]
  * SWA rows           N(0,1) rows scaled to unit root-mean-square, then bf16
  * index-key bytes    for tests that need a long index cache without the
                       cache write: uniform code bytes (every E2M1 nibble
                       equally likely) and E8M0 scale bytes uniform in 121..127

All bf16 tensors are returned as ``uint16`` bit patterns so that both sides
consume byte-identical inputs.
"""
from __future__ import annotations

import numpy as np

D_LATENT = 512
N_INDEX_HEADS = 32
D_INDEX = 128
N_HEADS = 64


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def latents(g: np.random.Generator, *shape: int) -> np.ndarray:
    """N(0,1) latents ``[..., 512]`` as bf16 bits."""
    return f32_to_bf16_bits(g.standard_normal((*shape, D_LATENT), dtype=np.float32))


def compressor_weights(g: np.random.Generator) -> tuple[np.ndarray, np.ndarray]:
    """Two positive per-channel weight vectors softplus(N(0,1)), float32 [512]."""
    z = g.standard_normal((2, D_LATENT))
    w = np.log1p(np.exp(z)).astype(np.float32)
    return np.ascontiguousarray(w[0]), np.ascontiguousarray(w[1])


def index_projection(g: np.random.Generator) -> np.ndarray:
    """Index-K projection matrix N(0, 1/512), bf16 bits [128, 512]."""
    w = g.standard_normal((D_INDEX, D_LATENT)) / np.sqrt(D_LATENT)
    return f32_to_bf16_bits(w.astype(np.float32))


def index_queries(g: np.random.Generator, *shape: int) -> np.ndarray:
    """Indexer queries N(0,1), bf16 bits [..., 32, 128]."""
    return f32_to_bf16_bits(
        g.standard_normal((*shape, N_INDEX_HEADS, D_INDEX), dtype=np.float32))


def head_weights(g: np.random.Generator, *shape: int) -> np.ndarray:
    """Per-head indexer weights N(0,1), float32 [..., 32]."""
    return g.standard_normal((*shape, N_INDEX_HEADS), dtype=np.float32)


def main_queries(g: np.random.Generator, *shape: int) -> np.ndarray:
    """Main attention queries N(0,1), bf16 bits [..., 64, 512]."""
    return f32_to_bf16_bits(
        g.standard_normal((*shape, N_HEADS, D_LATENT), dtype=np.float32))


def swa_rows(g: np.random.Generator, *shape: int) -> np.ndarray:
    """Sliding-window rows: N(0,1) scaled to unit RMS per row, bf16 bits [..., 512]."""
    z = g.standard_normal((*shape, D_LATENT))
    z = z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True))
    return f32_to_bf16_bits(z.astype(np.float32))


def index_key_bytes(g: np.random.Generator, *shape: int) -> tuple[np.ndarray, np.ndarray]:
    """Random MXFP4 index keys as stored bytes: codes uint8 [..., 64] and
    scales uint8 [..., 4]."""
    codes = g.integers(0, 256, size=(*shape, D_INDEX // 2), dtype=np.uint8)
    scales = g.integers(121, 128, size=(*shape, D_INDEX // 32), dtype=np.uint8)
    return codes, scales


# ---------------------------------------------------------------- device side
# Large workloads (hundreds of MB to GB of latents) are drawn on the GPU with a
# seeded torch generator; the host copies back only the rows a sampled check
# needs.  These helpers return torch tensors and are imported lazily so that the
# CPU-only oracle tests never need torch.

def torch_latents(seed: int, shape: tuple[int, ...], device: str = "cuda"):
    """N(0,1) bf16 latents drawn with a seeded torch generator on ``device``."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn(*shape, D_LATENT, generator=gen, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def torch_normal(seed: int, shape: tuple[int, ...], dtype, device: str = "cuda"):
    """N(0,1) tensor of ``shape`` drawn with a seeded torch generator."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn(*shape, generator=gen, device=device,
                       dtype=torch.float32).to(dtype)


def torch_swa_rows(seed: int, shape: tuple[int, ...], device: str = "cuda"):
    """Unit-RMS N(0,1) rows, bf16, drawn with a seeded torch generator."""
    import torch
    z = torch_normal(seed, (*shape, D_LATENT), torch.float32, device)
    z = z * torch.rsqrt(torch.mean(z * z, dim=-1, keepdim=True))
    return z.to(torch.bfloat16)
