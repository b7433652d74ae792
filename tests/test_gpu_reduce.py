"""GPU parity of the fused decompress + reduce (ZipCCL technical summary
2.D, zipped all-to-all + local reduction): bit-exact against the oracle's
in-order fp32 sum rounded to nearest-even BF16."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_bytes, host_u16, load_lib, require_gpu
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def codec():
    require_gpu()
    load_lib()
    from lossless_bf16_exponent_split_gb300 import Codec
    return Codec()


def gpu_reduce(codec, streams, n, in_bytes=None):
    devs = [dev_bytes(s) for s in streams]
    codec.reset_status()
    out = codec.decompress_reduce(devs, [len(s) for s in streams] if in_bytes is None else in_bytes, n)
    torch.cuda.synchronize()
    return codec.read_status(), host_u16(out)


@pytest.mark.parametrize("S,n", [(1, 5000), (2, 4096), (3, 3 * 4096 + 77), (8, 100_003),
                                 (5, 1), (4, 1023), (40, 9000)])
def test_reduce_matches_oracle(codec, S, n):
    shards = [workloads.special_values(n, seed=10 * S + s, frac=0.05) for s in range(S)]
    luts = [oracle.lut_from_sigma(1.0), oracle.lut_from_sigma(0.5), bytes([0, 255, 1, 2, 3, 254, 127])]
    streams = [oracle.compress(x, luts[s % 3]) for s, x in enumerate(shards)]
    want = oracle.decompress_reduce(streams, n)
    st, got = gpu_reduce(codec, streams, n)
    assert st == 0
    assert np.array_equal(got, want)


def test_reduce_order_and_specials(codec):
    lut = oracle.lut_from_sigma(1.0)
    n = 4096 + 3
    cases = [
        [np.full(n, 0x4D00, np.uint16), np.full(n, 0xCD00, np.uint16), np.full(n, 0x3F80, np.uint16)],
        [np.full(n, 0x8000, np.uint16), np.full(n, 0x8000, np.uint16)],            # -0 + -0
        [np.full(n, 0x7F7F, np.uint16), np.full(n, 0x7F7F, np.uint16)],            # overflow
        [np.full(n, 0x7F80, np.uint16), np.full(n, 0xFF80, np.uint16)],            # inf - inf
        [np.full(n, 0x0001, np.uint16), np.full(n, 0x0001, np.uint16)],            # subnormals
    ]
    for shards in cases:
        streams = [oracle.compress(x, lut) for x in shards]
        want = oracle.decompress_reduce(streams, n)
        st, got = gpu_reduce(codec, streams, n)
        assert st == 0 and np.array_equal(got, want)


def test_reduce_rejects_wrong_n(codec):
    lut = oracle.lut_from_sigma(1.0)
    s1 = oracle.compress(np.zeros(5000, np.uint16), lut)
    s2 = oracle.compress(np.zeros(5001, np.uint16), lut)
    st, _ = gpu_reduce(codec, [s1, s2], 5000)
    assert st == 3


def test_rs_local_full(codec):
    cfg = workloads.CONFIGS["rs_local"]
    shards = workloads.reduce_shards(cfg["S"], cfg["n"], cfg["sigma"], seed=0)
    lut = oracle.lut_from_sigma(cfg["sigma"])
    streams = [oracle.compress(x, lut) for x in shards]
    want = oracle.decompress_reduce(streams, cfg["n"])
    st, got = gpu_reduce(codec, streams, cfg["n"])
    assert st == 0
    assert np.array_equal(got, want)
