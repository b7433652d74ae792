"""Oracle pins for the measured-histogram LUT (the data-driven alternative
to the sigma rule of ZipCCL technical summary 2.A): the histogram against
numpy's bincount, the LUT against a lexicographic sort, and the property
that makes it worth having -- on any data it covers at least as many values
as the sigma LUT."""
import numpy as np
import pytest

import oracle
from lossless_bf16_exponent_split_gb300 import workloads


def _numpy_lut(hist):
    order = np.lexsort((np.arange(256), -np.asarray(hist, np.int64)))  # count desc, exponent asc
    return bytes(order[:7].astype(np.uint8))


@pytest.mark.parametrize("make", [lambda: workloads.gaussian(100_003, 0.02, seed=1),
                                  lambda: workloads.activation_mix(64, 1000, seed=2),
                                  lambda: workloads.random_bits(70_000, seed=3),
                                  lambda: workloads.special_values(50_000, seed=4, frac=0.3)])
def test_histogram_and_lut_match_numpy(make):
    x = make()
    hist = oracle.exponent_histogram(x)
    assert np.array_equal(hist, np.bincount((x >> 7) & 0xFF, minlength=256).astype(np.uint64))
    assert oracle.lut_from_histogram(hist) == _numpy_lut(hist)


def test_lut_ties_go_to_the_smaller_exponent():
    hist = np.zeros(256, np.uint64)
    hist[[200, 10, 77, 5]] = [9, 9, 3, 3]  # two pairs of ties, then all zeros
    assert oracle.lut_from_histogram(hist) == bytes([10, 200, 5, 77, 0, 1, 2])
    assert oracle.lut_from_histogram(np.zeros(256, np.uint64)) == bytes(range(7))


def test_empty_input_histogram_is_zero():
    assert not oracle.exponent_histogram(np.zeros(0, np.uint16)).any()


@pytest.mark.parametrize("make,sigma", [(lambda: workloads.activation_mix(128, 2048, seed=5), 1.0),
                                        (lambda: workloads.gaussian(200_000, 0.02, seed=6), 0.02),
                                        (lambda: workloads.gaussian(200_000, 3.0, seed=7), 0.02)])
def test_data_lut_covers_at_least_the_sigma_lut(make, sigma):
    x = make()
    hist = oracle.exponent_histogram(x).astype(np.int64)
    data_cov = sum(hist[e] for e in oracle.lut_from_histogram(hist))
    sigma_cov = sum(hist[e] for e in oracle.lut_from_sigma(sigma))
    assert data_cov >= sigma_cov
    # and the stream is never larger: 11 bits per slot + 8 per escape
    assert len(oracle.compress(x, oracle.lut_from_histogram(hist))) <= len(oracle.compress(x, oracle.lut_from_sigma(sigma)))


def test_data_lut_recovers_what_the_sigma_lut_misses():
    """Two payloads the Gaussian rule fits badly.  ReLU output (half exact
    zeros): the measured LUT takes exponent 0 first and codes almost every
    value, where the sigma LUT escapes every zero.  A bucket of two layers
    with different scales: no single sigma fits both."""
    x = workloads.gaussian(1 << 20, 1.0, seed=3).copy()
    x[(x & 0x8000) != 0] = 0
    h = oracle.exponent_histogram(x).astype(np.int64)
    lut = oracle.lut_from_histogram(h)
    assert lut[0] == 0 and h[0] == (x == 0).sum()
    assert sum(h[e] for e in lut) >= 0.97 * x.size
    assert sum(h[e] for e in oracle.lut_from_sigma(1.0)) < 0.5 * x.size
    mix = np.concatenate([workloads.gaussian(1 << 19, 0.02, seed=4), workloads.gaussian(1 << 19, 1e-3, seed=5)])
    hm = oracle.exponent_histogram(mix).astype(np.int64)
    rms = float(np.sqrt((0.02 ** 2 + 1e-3 ** 2) / 2))
    assert sum(hm[e] for e in oracle.lut_from_histogram(hm)) > sum(hm[e] for e in oracle.lut_from_sigma(rms))
