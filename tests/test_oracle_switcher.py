"""Pins of the reduce-scatter switcher's cost model (ZipCCL technical
summary 2.D; the time model is reading R17): a worked example computed by
hand, the break-even bandwidth where both paths take the same time, and the
limiting cases the model must respect."""
import math

import pytest

from oracle.switcher import rs_plan

EXAMPLE = dict(ranks=4, nbytes=4_000_000_000, ratio=0.5, link_gbs=100.0, link_latency_us=10.0,
               compress_gbs=1000.0, compress_fixed_us=5.0, reduce_gbs=2000.0, reduce_fixed_us=7.0)


def test_worked_example():
    # shard 1e9 B; one shard over the link 10,000 us (compressed: 5,000 us);
    # compress 3e9 B at 1000 GB/s = 3,000 us; reduce 4e9 B at 2000 GB/s = 2,000 us
    p = rs_plan(**EXAMPLE)
    assert p["native_us"] == pytest.approx(3 * (10 + 10_000), rel=1e-15)
    assert p["zipped_us"] == pytest.approx((5 + 3000) + (7 + 2000) + 3 * (10 + 5000), rel=1e-15)
    assert p["zipped"]
    assert p["breakeven_link_gbs"] == pytest.approx(3e9 * 0.5 / 5012e-6 / 1e9, rel=1e-12)


def test_breakeven_is_where_the_times_meet():
    p = rs_plan(**EXAMPLE)
    at = rs_plan(**dict(EXAMPLE, link_gbs=p["breakeven_link_gbs"]))
    assert at["native_us"] == pytest.approx(at["zipped_us"], rel=1e-12)
    for f in (0.5, 0.99):
        assert rs_plan(**dict(EXAMPLE, link_gbs=f * p["breakeven_link_gbs"]))["zipped"]
    for f in (1.01, 2.0):
        assert not rs_plan(**dict(EXAMPLE, link_gbs=f * p["breakeven_link_gbs"]))["zipped"]


def test_incompressible_payload_never_zips():
    for gbs in (0.1, 10.0, 1e4):
        p = rs_plan(**dict(EXAMPLE, ratio=1.0, link_gbs=gbs))
        assert not p["zipped"] and p["breakeven_link_gbs"] == 0.0


def test_single_rank_has_nothing_to_exchange():
    p = rs_plan(**dict(EXAMPLE, ranks=1))
    assert p == {"zipped": False, "native_us": 0.0, "zipped_us": 0.0, "breakeven_link_gbs": 0.0}


def test_latency_does_not_move_the_breakeven():
    a = rs_plan(**EXAMPLE)["breakeven_link_gbs"]
    b = rs_plan(**dict(EXAMPLE, link_latency_us=1e4))["breakeven_link_gbs"]
    assert a == pytest.approx(b, rel=1e-15)


def test_free_codec_zips_whenever_it_saves_bytes():
    p = rs_plan(**dict(EXAMPLE, compress_gbs=math.inf, reduce_gbs=math.inf, compress_fixed_us=0.0,
                       reduce_fixed_us=0.0, link_gbs=1e6))
    assert p["zipped"] and p["breakeven_link_gbs"] == math.inf


def test_library_matches_oracle_on_random_models():
    """The library's zccl_rs_plan (host C) against the oracle."""
    import numpy as np
    from lossless_bf16_exponent_split_gb300 import build
    build.build()
    import lossless_bf16_exponent_split_gb300 as z
    rng = np.random.default_rng(0)
    for _ in range(2000):
        kw = dict(ranks=int(rng.integers(1, 1025)), nbytes=int(rng.integers(0, 1 << 36)),
                  ratio=float(rng.uniform(0.05, 1.3)), link_gbs=float(10 ** rng.uniform(-1, 4)),
                  link_latency_us=float(rng.uniform(0, 100)), compress_gbs=float(10 ** rng.uniform(1, 4)),
                  compress_fixed_us=float(rng.uniform(0, 20)), reduce_gbs=float(10 ** rng.uniform(1, 4)),
                  reduce_fixed_us=float(rng.uniform(0, 20)))
        want, got = rs_plan(**kw), z.zccl_rs_plan(**kw)
        for k in ("native_us", "zipped_us", "breakeven_link_gbs"):
            assert got[k] == pytest.approx(want[k], rel=1e-12, abs=1e-12), (k, kw)
        if abs(want["native_us"] - want["zipped_us"]) > 1e-9 * max(want["native_us"], 1.0):
            assert got["zipped"] == want["zipped"], kw


def test_library_rejects_bad_models():
    from lossless_bf16_exponent_split_gb300 import build
    build.build()
    import lossless_bf16_exponent_split_gb300 as z
    for bad in (dict(ranks=0), dict(ratio=0.0), dict(ratio=math.nan), dict(link_gbs=0.0),
                dict(link_latency_us=-1.0), dict(compress_gbs=math.inf), dict(reduce_gbs=-2.0),
                dict(compress_fixed_us=math.nan), dict(reduce_fixed_us=-0.5)):
        with pytest.raises(z.ZcclError):
            z.zccl_rs_plan(**dict(EXAMPLE, **bad))
    assert z.lib().zccl_rs_plan(None, None) == z.INVALID_ARG
