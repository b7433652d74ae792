"""The reduce-scatter switcher on the GPU: the codec profile it measures is
sane, and its plans follow the cost model (ZipCCL technical summary 2.D)."""
import math

import pytest
import torch

import oracle
from oracle.switcher import rs_plan
from gpu_util import dev_u16, load_lib, require_gpu
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def switcher_cls():
    require_gpu()
    load_lib()
    from lossless_bf16_exponent_split_gb300.switcher import RsSwitcher
    return RsSwitcher


def test_profile_and_plans(switcher_cls):
    x = workloads.gaussian(1 << 22, 0.02, seed=3)
    lut = oracle.lut_from_sigma(0.02)
    slow = switcher_cls(8, link_gbs=50.0, link_latency_us=5.0, sample=dev_u16(x), lut=lut)
    p = slow.profile
    # the ratio measured on the device is the oracle's stream size
    assert p.ratio == pytest.approx(len(oracle.compress(x, lut)) / (2 * x.size), rel=1e-12)
    for v in (p.compress_gbs, p.reduce_gbs):
        assert math.isfinite(v) and 10.0 < v < 1e5
    assert p.compress_fixed_us >= 0 and p.reduce_fixed_us >= 0
    nbytes = 8 * 2 * x.size
    plan = slow.plan(nbytes)
    want = rs_plan(8, nbytes, p.ratio, 50.0, 5.0, p.compress_gbs, p.compress_fixed_us, p.reduce_gbs,
                   p.reduce_fixed_us)
    assert plan["zipped"] == want["zipped"]
    assert plan["zipped_us"] == pytest.approx(want["zipped_us"], rel=1e-12)
    # a 50 GB/s link is far below a codec running at HBM-class rates: zip
    assert plan["zipped"] and plan["breakeven_link_gbs"] > 50.0
    # an incompressible payload never zips
    assert not slow.plan(nbytes, ratio=1.0)["zipped"]
