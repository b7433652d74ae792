"""Seeded synthetic BF16 workloads shared by the tests, the bench and the oracle.

This module holds input generation only -- none of the codec's arithmetic.
Random numbers come from numpy's PCG64 (``numpy.random.default_rng``); the
fp32 -> BF16 conversion of generated values is torch's own CPU cast (round to
nearest even), i.e. library plumbing, not the codec's rounding.

The page measured on real training tensors (activations, gradients,
parameters) that are not available; following its observation that those are
near-Gaussian (ZipCCL technical summary 2.A), seeded Gaussians with the
stated shapes stand in for them.  All arrays are uint16 BF16 bit patterns.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


def f32_to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of float32 values, via torch's CPU cast."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def gaussian(n: int, sigma: float, seed: int = 0) -> np.ndarray:
    """n i.i.d. N(0, sigma^2) values as BF16 (weights / all-gather payload)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(n, dtype=np.float32)
    return f32_to_bf16_bits(z * np.float32(sigma))


def activation_mix(rows: int = 8192, cols: int = 4096, seed: int = 0) -> np.ndarray:
    """Activation-like payload: 2% exact +0, 0.1% outliers N(0, 50^2), the
    rest N(0, 1).  Draw order: first u ~ U[0,1) for all n, then z ~ N(0,1)."""
    n = rows * cols
    rng = np.random.default_rng(seed)
    u = rng.random(n)
    z = rng.standard_normal(n, dtype=np.float32)
    v = z.copy()
    outl = (u >= 0.02) & (u < 0.021)
    v[outl] = z[outl] * np.float32(50.0)
    v[u < 0.02] = np.float32(0.0)
    return f32_to_bf16_bits(v)


@dataclass
class MoEPayload:
    payload: np.ndarray          # uint16 [rows * hidden], expert-sorted rows
    hidden: int
    counts: np.ndarray           # tokens per expert
    capacity: int                # static rows per expert
    segments: list               # [(row_start, rows)] : 2e = static, 2e+1 = dynamic


def moe_routing_counts(tokens: int, top_k: int, experts: int, zipf_s: float,
                       rng: np.random.Generator) -> np.ndarray:
    """Tokens routed to each expert: top-k of `experts` per token without
    replacement, expert probabilities p_e ~ (e+1)^-s, drawn by Gumbel-top-k
    (equivalent to sequential multinomial sampling without replacement)."""
    p = (np.arange(experts, dtype=np.float64) + 1.0) ** (-zipf_s)
    logp = np.log(p / p.sum())
    g = rng.gumbel(size=(tokens, experts))
    top = np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :top_k]
    return np.bincount(top.ravel(), minlength=experts)


def moe_payload(tokens: int = 16384, top_k: int = 8, experts: int = 64, hidden: int = 2048,
                zipf_s: float = 1.2, seed: int = 0, with_payload: bool = True) -> MoEPayload:
    """MoE all-to-all payload split into per-expert static and dynamic parts
    (ZipCCL technical summary 2.D): the static part of expert e is its first
    min(count_e, capacity) rows, capacity = ceil(mean count); the dynamic
    part is the rest (possibly empty)."""
    rng = np.random.default_rng(seed)
    counts = moe_routing_counts(tokens, top_k, experts, zipf_s, rng)
    rows = int(counts.sum())
    cap = int(math.ceil(rows / experts))
    segments = []
    start = 0
    for e in range(experts):
        c = int(counts[e])
        st = min(c, cap)
        segments.append((start, st))
        segments.append((start + st, c - st))
        start += c
    payload = np.zeros(0, np.uint16)
    if with_payload:
        z = rng.standard_normal(rows * hidden, dtype=np.float32)
        payload = f32_to_bf16_bits(z)
    return MoEPayload(payload, hidden, counts, cap, segments)


def reduce_shards(S: int = 8, n: int = 16777216, sigma: float = 1e-3, seed: int = 0):
    """S gradient shards of n values each, N(0, sigma^2), drawn from one seeded
    stream in shard order."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(S):
        z = rng.standard_normal(n, dtype=np.float32)
        out.append(f32_to_bf16_bits(z * np.float32(sigma)))
    return out


def random_bits(n: int, seed: int = 0) -> np.ndarray:
    """Uniformly random 16-bit patterns (every exponent, NaN/Inf/subnormals)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 65536, size=n, dtype=np.uint16)


SPECIALS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81, 0x0001,
                     0x8001, 0x007F, 0x807F, 0x0080, 0x7F7F, 0xFF7F], dtype=np.uint16)


def special_values(n: int, seed: int = 0, frac: float = 0.3) -> np.ndarray:
    """N(0,1) values with a fraction replaced by +-0, +-Inf, NaNs,
    subnormals and +-max-finite."""
    rng = np.random.default_rng(seed + 1)
    base = gaussian(n, 1.0, seed)
    pick = rng.random(n) < frac
    base[pick] = SPECIALS[rng.integers(0, SPECIALS.size, size=int(pick.sum()))]
    return base


# Workload table: sizes and value recipes of the five standard configurations.
CONFIGS = {
    "gauss1m": dict(n=1_048_576, sigma=0.02, desc="1,048,576 BF16 N(0, 0.02^2), seed 0"),
    "gauss268m": dict(n=1 << 28, sigma=0.02,
                      desc="268,435,456 BF16 N(0, 0.02^2), seed 0: one large stream (a 512 MB all-gather bucket)"),
    "llama3_8b_allgather": dict(n=4096 * 14336, sigma=0.02,
                                desc="4096x14336 BF16 N(0, 0.02^2), seed 0"),
    "activation_mix": dict(n=8192 * 4096, sigma=1.0,
                           desc="8192x4096 BF16: 97.9% N(0,1), 0.1% N(0,50^2), 2% +0"),
    "moe_a2a": dict(tokens=16384, top_k=8, experts=64, hidden=2048, sigma=1.0,
                    desc="16384 tokens x top-8 of 64 experts (Zipf 1.2), hidden 2048, N(0,1)"),
    "rs_local": dict(S=8, n=16_777_216, sigma=1e-3,
                     desc="8 shards x 16,777,216 BF16 N(0, 1e-3^2)"),
    # the same shards as one rank (position 3) sees them: its own shard stays uncompressed
    "rs_local_own": dict(S=8, n=16_777_216, sigma=1e-3, local_pos=3,
                         desc="8 shards x 16,777,216 BF16 N(0, 1e-3^2); shard 3 is the rank's own, plain BF16"),
    # the activation payload again, for the measured-LUT statistics pass
    "activation_mix_lut": dict(n=8192 * 4096, sigma=1.0,
                               desc="exponent histogram + LUT of 8192x4096 BF16: 97.9% N(0,1), "
                                    "0.1% N(0,50^2), 2% +0"),
}
