"""Seeded synthetic inputs for block-quantized matmul and QMoE.

This module only draws random numbers and fixes shapes; it holds none of the
method's arithmetic (no packing, decoding, scaling or accumulation).  Both the
CUDA parity tests and the oracle consume what it returns, and bench.py uses it
for its workloads.

Distributions follow the workload descriptions: activations ~N(0,1); per-block
scales ~U[0.005, 0.02]; packed weights are uniform random bytes, so every code
of every width is uniform over [0, 2^bits) (padding bits of a partial last
block are random too, which the consumers must ignore); zero points are
uniform random bytes of the packed zero-point stream; router logits ~N(0,1),
optionally with +3.0 added to experts 0-7 for every tenth token (t % 10 == 0).

Half-precision values are returned as uint16 bit patterns (IEEE binary16 from
numpy's round-to-nearest-even cast; bfloat16 by round-to-nearest-even of the
float32 pattern), fp32 values as float32.
"""
from __future__ import annotations

import numpy as np

# Shapes of one Qwen3-1.7B decoder layer's projections (K -> N) and the vocabulary head.
QWEN3_1P7B_PROJECTIONS = [
    ("qkv", 2048, 4096),      # output columns split [2048, 1024, 1024]
    ("o_proj", 2048, 2048),
    ("gate", 2048, 6144),
    ("up", 2048, 6144),
    ("down", 6144, 2048),
]
QWEN3_1P7B_LM_HEAD = ("lm_head", 2048, 151936)
QWEN3_1P7B_LAYERS = 28
QKV_SPLIT = (2048, 1024, 1024)

# One Qwen3-30B-A3B-shaped MoE layer.
QWEN3_30B_A3B_MOE = dict(H=2048, I=768, E=128, k=8)

# The tiny MatMulNBits case.
TINY = dict(M=1, K=256, N=128, bits=4, bs=32)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def cast(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> storage of `dtype` ("f32" | "f16" | "bf16")."""
    if dtype == "f32":
        return np.asarray(x, np.float32)
    if dtype == "f16":
        return to_f16_bits(x)
    if dtype == "bf16":
        return to_bf16_bits(x)
    raise ValueError(dtype)


def normal(g: np.random.Generator, shape, dtype: str = "f32") -> np.ndarray:
    return cast(g.standard_normal(shape, dtype=np.float32), dtype)


def uniform(g: np.random.Generator, shape, lo: float, hi: float, dtype: str = "f32") -> np.ndarray:
    return cast(g.uniform(lo, hi, size=shape).astype(np.float32), dtype)


def random_bytes(g: np.random.Generator, shape) -> np.ndarray:
    return g.integers(0, 256, size=shape, dtype=np.uint8)


def n_blocks(K: int, bs: int) -> int:
    return (K + bs - 1) // bs


def packed_row_bytes(K: int, bits: int, bs: int) -> int:
    """Bytes of one packed weight row: ceil(K/bs) blobs of bs*bits/8 bytes."""
    return n_blocks(K, bs) * bs * bits // 8


def zp_row_bytes(K: int, bits: int, bs: int) -> int:
    return (n_blocks(K, bs) * bits + 7) // 8


def quantized_weight(g: np.random.Generator, N: int, K: int, bits: int, bs: int,
                     scale_dtype: str = "f32", with_zp: bool = False, lead=()):
    """Packed weights [*lead, N, nb*blob] (as [..., N, row_bytes] uint8), scales
    [*lead, N, nb] and optional packed zero points [*lead, N, zp_row_bytes]."""
    lead = tuple(lead)
    nb = n_blocks(K, bs)
    packed = random_bytes(g, lead + (N, packed_row_bytes(K, bits, bs)))
    scales = uniform(g, lead + (N, nb), 0.005, 0.02, scale_dtype)
    zp = random_bytes(g, lead + (N, zp_row_bytes(K, bits, bs))) if with_zp else None
    return packed, scales, zp


def router_logits(g: np.random.Generator, T: int, E: int, skew: bool = False) -> np.ndarray:
    x = g.standard_normal((T, E), dtype=np.float32)
    if skew:
        x[::10, :8] += np.float32(3.0)
    return x


def moe_layer(g: np.random.Generator, T: int, H: int, I: int, E: int, fc1_bits: int,
              fc2_bits: int, bs: int, act_dtype: str, with_zp: bool = False, skew: bool = False):
    """Inputs of one QMoE layer: X [T,H], logits [T,E], FC1 [E,2I,...] and FC2 [E,H,...]."""
    X = normal(g, (T, H), act_dtype)
    logits = router_logits(g, T, E, skew)
    w1, s1, z1 = quantized_weight(g, 2 * I, H, fc1_bits, bs, act_dtype, with_zp, lead=(E,))
    w2, s2, z2 = quantized_weight(g, H, I, fc2_bits, bs, act_dtype, with_zp, lead=(E,))
    return dict(X=X, logits=logits, fc1_w=w1, fc1_scales=s1, fc1_zp=z1, fc2_w=w2,
                fc2_scales=s2, fc2_zp=z2)
