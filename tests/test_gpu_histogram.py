"""GPU parity: the exponent histogram kernel and the measured LUT against
the oracle, bit for bit (ZipCCL technical summary 2.A: the LUT holds the
seven most frequent exponents; the library measures them instead of
deriving them from sigma)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_u16, load_lib, require_gpu
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu

# around one lane-vector, one CTA round (1024 lanes x 2 vectors x 8 values)
# and one full grid round
EDGE_N = [0, 1, 7, 8, 9, 255, 256, 257, 16383, 16384, 16385, 16384 * 304 - 1, 16384 * 304 + 9, 1_000_003]


@pytest.fixture(scope="module")
def codec():
    require_gpu()
    load_lib()
    from lossless_bf16_exponent_split_gb300 import Codec
    return Codec()


def gpu_hist(codec, x):
    h = codec.exponent_histogram(dev_u16(x))
    torch.cuda.synchronize()
    return h.cpu().numpy().view(np.uint64)


@pytest.mark.parametrize("n", EDGE_N)
def test_histogram_edge_sizes(codec, n):
    x = workloads.random_bits(n, seed=n)
    assert np.array_equal(gpu_hist(codec, x), oracle.exponent_histogram(x))


@pytest.mark.parametrize("make", ["gaussian", "activation_mix", "special", "bits"])
def test_histogram_and_lut_match_oracle(codec, make):
    x = {"gaussian": lambda: workloads.gaussian(3_000_017, 0.02, seed=5),
         "activation_mix": lambda: workloads.activation_mix(1024, 4096, seed=6),
         "special": lambda: workloads.special_values(500_001, seed=7),
         "bits": lambda: workloads.random_bits(777_777, seed=8)}[make]()
    want = oracle.exponent_histogram(x)
    got = gpu_hist(codec, x)
    assert np.array_equal(got, want)
    assert int(got.sum()) == x.size
    assert codec.lut_from_data(dev_u16(x)) == oracle.lut_from_histogram(want)


def test_histogram_of_unaligned_tail_views(codec):
    """A 16-byte aligned view whose length is not a multiple of 8."""
    x = workloads.gaussian(100_000, 1e-3, seed=9)
    d = dev_u16(x)
    for lo, hi in [(8, 99_999), (16, 16 + 13), (1024, 1024 + 7)]:
        h = codec.exponent_histogram(d[lo:hi])
        torch.cuda.synchronize()
        assert np.array_equal(h.cpu().numpy().view(np.uint64), oracle.exponent_histogram(x[lo:hi]))


def test_histogram_single_exponent(codec):
    """Every value has one exponent: all 32 lanes of every reduction hit the
    same counter row, and each 16-bit counter takes the largest increments."""
    x = np.full(1 << 22, 0x3F80, np.uint16)  # 1.0
    h = gpu_hist(codec, x)
    assert h[127] == x.size and h.sum() == x.size


def test_histogram_folds_before_16_bit_overflow(codec):
    """1.4 G values, two exponents: each CTA folds its 16-bit counters at
    least once before the end; the exact counts are known in closed form."""
    n, k = 1_400_000_003, 700_000_001
    d = torch.empty(n, dtype=torch.int16, device="cuda")
    d[:k] = 0x3F80   # 1.0, exponent 127
    d[k:] = 0x4000   # 2.0, exponent 128
    h = codec.exponent_histogram(d).cpu().numpy().view(np.uint64)
    want = np.zeros(256, np.uint64)
    want[127], want[128] = k, n - k
    assert np.array_equal(h, want)
    del d


def test_histogram_accumulates_over_tensors(codec):
    """accumulate adds to the counts already there: the histogram of three
    tensors is the oracle's histogram of their concatenation."""
    xs = [workloads.gaussian(100_003, 0.02, seed=1), workloads.special_values(77_777, seed=2),
          workloads.random_bits(4096 * 3 + 1, seed=3)]
    h = codec.exponent_histogram(dev_u16(xs[0]))
    for x in xs[1:]:
        codec.exponent_histogram(dev_u16(x), hist=h, accumulate=True)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy().view(np.uint64), oracle.exponent_histogram(np.concatenate(xs)))
    # overwrite mode forgets the earlier counts
    codec.exponent_histogram(dev_u16(xs[1]), hist=h)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy().view(np.uint64), oracle.exponent_histogram(xs[1]))


def test_measured_lut_round_trips_through_the_codec(codec):
    """A stream coded with the measured LUT is lossless and no larger than
    with the sigma LUT, on activations that fit the Gaussian model badly."""
    x = workloads.activation_mix(2048, 4096, seed=11)
    d = dev_u16(x)
    lut = codec.lut_from_data(d)
    codec.reset_status()
    out, nb = codec.compress(d, lut)
    s_meas = int(nb.item())
    y = codec.decompress(out, s_meas, x.size)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    assert torch.equal(y, d)
    assert s_meas <= len(oracle.compress(x, oracle.lut_from_sigma(1.0)))


def test_lut_from_data_one_call(codec):
    """zccl_lut_from_data = histogram + copy back + selection, through the C ABI."""
    import lossless_bf16_exponent_split_gb300 as z
    x = workloads.activation_mix(512, 4096, seed=12)
    d = dev_u16(x)
    hist = torch.empty(256, dtype=torch.int64, device="cuda")
    lut = z.zccl_lut_from_data(d.data_ptr(), x.size, hist.data_ptr(), torch.cuda.current_stream().cuda_stream)
    want = oracle.exponent_histogram(x)
    assert lut == oracle.lut_from_histogram(want)
    assert np.array_equal(hist.cpu().numpy().view(np.uint64), want)
