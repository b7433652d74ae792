"""Oracle of the reduce-scatter switcher's cost model (test infrastructure:
only tests, the smoke check and the bench's CPU legs use it).

ZipCCL technical summary 2.D: at start-up the switcher profiles link
bandwidth, latency and the compression ratio, and then runs either the
native reduce-scatter or a zipped all-to-all followed by a local
decompress-and-reduce, whichever is faster.  The pages give no formula; the
plainest time model under that description [R17], in fp64:

  P ranks, each holding `bytes` of BF16 = P shards of s = bytes / P;
  link: bandwidth beta (bytes/s), per-message latency alpha (s);
  codec: t(x) = fixed + x / rate for x bytes of BF16 input.

  native ring reduce-scatter:  (P - 1) * (alpha + s / beta)
      (P - 1 steps of one shard each; the reduction is fused into the
      receive and hidden under the link)
  zipped: compress the P - 1 outgoing shards, exchange them,
      decompress-reduce all P shards (the own one uncompressed):
      t_c((P - 1) * s) + (P - 1) * (alpha + r * s / beta) + t_r(P * s)

  zipped iff its time is strictly smaller; P = 1 has nothing to exchange
  (native, both times 0).  Break-even bandwidth: the latency terms cancel,
  so zipped wins iff beta < (P - 1) * s * (1 - r) / (t_c + t_r)  (0 if r >= 1).
"""
from __future__ import annotations


def rs_plan(ranks: int, nbytes: int, ratio: float, link_gbs: float, link_latency_us: float,
            compress_gbs: float, compress_fixed_us: float, reduce_gbs: float, reduce_fixed_us: float) -> dict:
    """Times in microseconds, rates in GB/s (1e9 bytes/s)."""
    P = int(ranks)
    if P < 1:
        raise ValueError("ranks >= 1")
    if P == 1:
        return {"zipped": False, "native_us": 0.0, "zipped_us": 0.0, "breakeven_link_gbs": 0.0}
    s = nbytes / P                                   # shard bytes
    us = lambda x, gbs: x / (gbs * 1e3)              # bytes at GB/s -> microseconds
    native = (P - 1) * (link_latency_us + us(s, link_gbs))
    codec = (compress_fixed_us + us((P - 1) * s, compress_gbs)) + (reduce_fixed_us + us(P * s, reduce_gbs))
    zipped = codec + (P - 1) * (link_latency_us + us(ratio * s, link_gbs))
    saved_bytes = (P - 1) * s * (1 - ratio)          # bytes the link no longer carries
    breakeven = saved_bytes / (codec * 1e3) if ratio < 1 and codec > 0 else (float("inf") if ratio < 1 else 0.0)
    return {"zipped": zipped < native, "native_us": native, "zipped_us": zipped, "breakeven_link_gbs": breakeven}
