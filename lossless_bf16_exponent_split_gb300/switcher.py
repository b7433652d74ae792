"""Reduce-scatter switcher: profile the codec on this GPU, then choose the
native reduce-scatter or the zipped all-to-all + local decompress-and-reduce
per call ("ZipCCL: Efficient Lossless Data Compression of Communication
Collectives for Accelerating LLM Training", technical summary 2.D).

The link's bandwidth and latency are the caller's (this library runs no
collective); the codec's fixed cost and rate, and the compression ratio, are
measured here with the library's own kernels on a sample of the payload.
The decision itself is ``zccl_rs_plan`` in the C library.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (OP_DECOMPRESS_REDUCE, check, zccl_decompress_reduce_local, zccl_rs_plan,
               zccl_workspace_bytes)
from .codec import Codec


@dataclass
class CodecProfile:
    ratio: float              # compressed bytes / BF16 bytes of the sample
    compress_gbs: float       # GB/s of BF16 input
    compress_fixed_us: float
    reduce_gbs: float         # decompress-reduce, GB/s of BF16 input (all shards)
    reduce_fixed_us: float


def _time_us(fn, reps: int) -> float:
    """Mean CUDA-event time of fn() on the current stream, after one warm-up."""
    fn()
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(reps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) * 1e3 / reps


def _fit(x_small: float, t_small: float, x_large: float, t_large: float):
    """t = fixed + x / rate through two points (fixed clamped at 0)."""
    slope = (t_large - t_small) / (x_large - x_small)  # us per byte
    if slope <= 0:
        return x_large / (t_large * 1e3), 0.0
    fixed = max(t_small - slope * x_small, 0.0)
    return 1.0 / (slope * 1e3), fixed


def profile_codec(sample: torch.Tensor, lut: bytes, ranks: int, reps: int = 10) -> CodecProfile:
    """Measure compress and decompress-reduce on `sample` (a contiguous
    16-bit CUDA tensor of BF16 bits, one shard's worth of the payload) and on
    its first half, and fit fixed cost + rate for each.  The codec's time is
    not linear in size (small calls are bound by launch and latency), so the
    fit is local: profile with a shard of the size the plans will be for."""
    if ranks < 2:
        raise ValueError("profiling needs at least two ranks' worth of shards")
    codec = Codec(sample.device)
    n = sample.numel()
    points = []
    for m in (max(n // 2, 4096), n):
        x = sample[:m]
        out, nbytes = codec.compress(x, lut)
        t_c = _time_us(lambda: codec.compress(x, lut, out=out, out_bytes=nbytes), reps)
        size = int(nbytes.item())
        # the own shard first, plain BF16; the other ranks' shards compressed
        ptrs = torch.tensor([0] + [out.data_ptr()] * (ranks - 1), dtype=torch.int64, device=sample.device)
        in_bytes = torch.tensor([0] + [size] * (ranks - 1), dtype=torch.int64, device=sample.device)
        y = torch.empty(m, dtype=torch.int16, device=sample.device)
        ws, wsb = codec.workspace(zccl_workspace_bytes(OP_DECOMPRESS_REDUCE, m, ranks))
        handle = torch.cuda.current_stream().cuda_stream

        def reduce():
            check(zccl_decompress_reduce_local(ptrs.data_ptr(), in_bytes.data_ptr(), ranks, x.data_ptr(), 0, 0,
                                               y.data_ptr(), m, ws, wsb, codec.status.data_ptr(), handle),
                  "zccl_decompress_reduce_local")
        t_r = _time_us(reduce, reps)
        codec.check_status("profile")
        points.append((m, t_c, t_r, size))
    (m0, c0, r0, _), (m1, c1, r1, size1) = points
    compress_gbs, compress_fixed = _fit(2 * m0, c0, 2 * m1, c1)
    reduce_gbs, reduce_fixed = _fit(2 * m0 * ranks, r0, 2 * m1 * ranks, r1)
    return CodecProfile(size1 / (2 * m1), compress_gbs, compress_fixed, reduce_gbs, reduce_fixed)


class RsSwitcher:
    """Profiles once at construction; `plan(nbytes)` then gives the choice
    and both paths' modelled times for a reduce-scatter of nbytes per rank."""

    def __init__(self, ranks: int, link_gbs: float, link_latency_us: float, sample: torch.Tensor, lut: bytes):
        self.ranks = ranks
        self.link_gbs = link_gbs
        self.link_latency_us = link_latency_us
        self.profile = profile_codec(sample, lut, ranks)

    def plan(self, nbytes: int, ratio: float | None = None) -> dict:
        p = self.profile
        return zccl_rs_plan(self.ranks, nbytes, p.ratio if ratio is None else ratio, self.link_gbs,
                            self.link_latency_us, p.compress_gbs, p.compress_fixed_us, p.reduce_gbs,
                            p.reduce_fixed_us)
