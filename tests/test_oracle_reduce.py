"""Pins of the oracle's local reduction (ZipCCL technical summary 2.D:
zipped all-to-all + local reduction) and of its fp32 -> BF16 rounding.

Independent pins: torch's fp32 -> bf16 cast (a library round-to-nearest-even)
on random bit patterns, hand-worked rounding midpoints, numpy float32 sums in
shard order, and an order-sensitive case.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_exponent_split_gb300 import workloads


def f32(bits):
    return np.array([bits], np.uint32).view(np.float32)[0]


def torch_bf16_bits(f):
    t = torch.from_numpy(np.ascontiguousarray(f, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_rounding_matches_library_cast_on_random_patterns():
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2 ** 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[~np.isnan(f)]
    assert np.array_equal(oracle.round_bf16_array(f), torch_bf16_bits(f))


def _nearest_bf16_by_distance(u):
    """The definition itself, for finite fp32 bit patterns u: of the two BF16
    values around |x| (truncation and the next one up, the next up past the
    largest finite being 2^128, i.e. infinity), the one at the smaller exact
    distance (computed in double, where every difference of these values is
    exact), ties to the even mantissa; the sign is kept."""
    mag = u & np.uint32(0x7FFFFFFF)
    lo = mag >> np.uint32(16)
    hi = lo + np.uint32(1)
    v = mag.view(np.float32).astype(np.float64)
    vlo = (lo << np.uint32(16)).view(np.float32).astype(np.float64)
    vhi = np.where(hi == 0x7F80, 2.0 ** 128, (hi << np.uint32(16)).view(np.float32).astype(np.float64))
    dlo, dhi = v - vlo, vhi - v
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (pick | ((u >> np.uint32(16)) & np.uint32(0x8000))).astype(np.uint16)


def test_rounding_matches_exact_distance_on_1e8_patterns():
    """10^8 random finite fp32 patterns against the exact-distance definition
    (independent of the oracle's bit trick and of any library cast)."""
    rng = np.random.default_rng(12)
    total = 0
    while total < 100_000_000:
        u = rng.integers(0, 2 ** 32, size=10_000_000, dtype=np.uint64).astype(np.uint32)
        u = u[(u & np.uint32(0x7F800000)) != np.uint32(0x7F800000)]  # finite only (NaN, Inf: hand cases)
        got = oracle.round_bf16_array(u.view(np.float32))
        assert np.array_equal(got, _nearest_bf16_by_distance(u))
        total += u.size


def test_rounding_near_every_bf16_midpoint():
    """For every BF16 magnitude b: the exact midpoint above it and its two fp32
    neighbours."""
    b = np.arange(0, 0x7F80, dtype=np.uint32)
    mid = (b << 16) | 0x8000
    pats = np.concatenate([mid, mid - 1, mid + 1, mid | 0x80000000])
    f = pats.view(np.float32)
    assert np.array_equal(oracle.round_bf16_array(f), torch_bf16_bits(f))


@pytest.mark.parametrize("bits,expect", [
    (0x3F808000, 0x3F80),   # 1 + 2^-8: tie between 0x3F80 (even) and 0x3F81 -> even
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: tie between 0x3F81 and 0x3F82 (even)
    (0x3F808001, 0x3F81),   # just above the tie
    (0x7F7F7FFF, 0x7F7F),   # just below the overflow midpoint -> max finite
    (0x7F7F8000, 0x7F80),   # overflow midpoint ties to even (0x7F80 = +Inf)
    (0xFF7F8000, 0xFF80),   # negative overflow -> -Inf
    (0x00008000, 0x0000),   # subnormal tie -> even (zero)
    (0x00018000, 0x0002),   # subnormal tie -> even
    (0x80000000, 0x8000),   # -0 stays -0
    (0x7F800000, 0x7F80),   # +Inf
    (0x7FC00001, 0x7FC0),   # NaN -> canonical
    (0xFFFFFFFF, 0x7FC0),   # negative NaN -> canonical
])
def test_rounding_hand_cases(bits, expect):
    assert oracle.round_bf16(f32(bits)) == expect


def bits_to_f32(x):
    return (x.astype(np.uint32) << 16).view(np.float32)


def test_reduce_equals_in_order_float32_sum():
    n = 3 * 4096 + 77
    S = 5
    shards = [workloads.special_values(n, seed=s, frac=0.05) for s in range(S)]
    luts = [oracle.lut_from_sigma(1.0), oracle.lut_from_sigma(0.5)]
    streams = [oracle.compress(x, luts[s % 2]) for s, x in enumerate(shards)]
    got = oracle.decompress_reduce(streams, n)
    with np.errstate(all="ignore"):
        acc = bits_to_f32(shards[0])
        for x in shards[1:]:
            acc = (acc + bits_to_f32(x)).astype(np.float32)
    want = torch_bf16_bits(acc).copy()
    want[np.isnan(acc)] = 0x7FC0
    assert np.array_equal(got, want)


def test_reduce_single_shard_is_decode_with_canonical_nan():
    x = workloads.special_values(9000, seed=2)
    s = oracle.compress(x, oracle.lut_from_sigma(1.0))
    got = oracle.decompress_reduce([s], x.size)
    want = x.copy()
    want[np.isnan(bits_to_f32(x))] = 0x7FC0
    assert np.array_equal(got, want)


def test_reduce_order_is_fixed():
    """(2^27 + -2^27) + 1 = 1, while 2^27 + (-2^27 + 1) = 0 in fp32."""
    lut = oracle.lut_from_sigma(1.0)
    a = np.full(10, 0x4D00, np.uint16)   # 2^27
    b = np.full(10, 0xCD00, np.uint16)   # -2^27
    c = np.full(10, 0x3F80, np.uint16)   # 1
    streams = [oracle.compress(v, lut) for v in (a, b, c)]
    assert (oracle.decompress_reduce(streams, 10) == 0x3F80).all()
    streams = [oracle.compress(v, lut) for v in (b, c, a)]
    assert (oracle.decompress_reduce(streams, 10) == 0x0000).all()


def test_reduce_signed_zero_and_overflow():
    lut = oracle.lut_from_sigma(1.0)
    negz = np.full(4, 0x8000, np.uint16)
    big = np.full(4, 0x7F7F, np.uint16)   # max finite
    s = [oracle.compress(v, lut) for v in (negz, negz)]
    assert (oracle.decompress_reduce(s, 4) == 0x8000).all()
    s = [oracle.compress(v, lut) for v in (big, big)]
    assert (oracle.decompress_reduce(s, 4) == 0x7F80).all()


def test_reduce_rejects_mismatched_n():
    lut = oracle.lut_from_sigma(1.0)
    s1 = oracle.compress(np.zeros(100, np.uint16), lut)
    s2 = oracle.compress(np.zeros(101, np.uint16), lut)
    with pytest.raises(oracle.OracleError) as e:
        oracle.decompress_reduce([s1, s2], 100)
    assert e.value.status == oracle.CORRUPT


def _numpy_fold(parts):
    """In-order float32 left fold of BF16 bit arrays, rounded by torch's
    cast (NaN -> 0x7FC0): the definition the oracle must meet."""
    with np.errstate(all="ignore"):
        acc = bits_to_f32(parts[0])
        for x in parts[1:]:
            acc = (acc + bits_to_f32(x)).astype(np.float32)
    want = torch_bf16_bits(acc).copy()
    want[np.isnan(acc)] = 0x7FC0
    return want


@pytest.mark.parametrize("local_pos", [0, 2, 4])
def test_reduce_local_shard_at_each_position(local_pos):
    """ZipCCL 2.D from one rank's view: the rank's own shard enters the fold
    uncompressed, at its rank position."""
    n = 2 * 4096 + 301
    S = 5
    shards = [workloads.special_values(n, seed=10 + s, frac=0.05) for s in range(S)]
    lut = oracle.lut_from_sigma(1.0)
    streams = [None if s == local_pos else oracle.compress(x, lut) for s, x in enumerate(shards)]
    got = oracle.decompress_reduce_local(streams, n, local=shards[local_pos], local_pos=local_pos)
    assert np.array_equal(got, _numpy_fold(shards))


def test_reduce_accumulates_into_existing_output():
    n = 4096 + 9
    S = 3
    shards = [workloads.special_values(n, seed=30 + s, frac=0.05) for s in range(S)]
    initial = workloads.special_values(n, seed=99, frac=0.05)
    lut = oracle.lut_from_sigma(1.0)
    streams = [oracle.compress(x, lut) for x in shards]
    got = oracle.decompress_reduce_local(streams, n, initial=initial)
    assert np.array_equal(got, _numpy_fold([initial] + shards))
    # both at once: the existing output first, then the shards with the local one in place
    streams[1] = None
    got = oracle.decompress_reduce_local(streams, n, local=shards[1], local_pos=1, initial=initial)
    assert np.array_equal(got, _numpy_fold([initial] + shards))


def test_reduce_single_local_shard_is_canonical_copy():
    x = workloads.special_values(5000, seed=7, frac=0.3)
    got = oracle.decompress_reduce_local([None], x.size, local=x, local_pos=0)
    want = x.copy()
    want[((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)] = 0x7FC0  # every NaN becomes the canonical one
    assert np.array_equal(got, want)
