"""CPU checks of the C ABI: libzccl builds for sm_103a, loads, exports every
function include/zccl.h declares, and its host-only functions agree with the
oracle; argument errors are returned before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def z():
    from lossless_bf16_exponent_split_gb300 import build
    build.build()
    import lossless_bf16_exponent_split_gb300 as z
    z.lib()
    return z


def declared_functions():
    text = open(os.path.join(ROOT, "include", "zccl.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zccl_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(z):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(z.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_function(z):
    for name in declared_functions():
        assert callable(getattr(z, name, None)), name


@pytest.mark.parametrize("sigma", [2.0 ** (f / 8) for f in range(-200, 81, 3)] + [0.02, 1e-3, 1.0])
def test_library_lut_matches_oracle(z, sigma):
    assert z.zccl_lut_from_sigma(sigma) == oracle.lut_from_sigma(sigma)


@pytest.mark.parametrize("bad", [0.0, -2.0, float("nan"), float("inf")])
def test_library_lut_rejects_bad_sigma(z, bad):
    with pytest.raises(z.ZcclError):
        z.zccl_lut_from_sigma(bad)


@pytest.mark.parametrize("n", [0, 1, 1023, 1024, 1025, 4095, 4096, 4097, 58_720_256, 10**9 + 7])
def test_sizes_match_oracle(z, n):
    if n <= 10**7:
        assert z.zccl_max_compressed_bytes(n) == oracle.max_bytes(n)
        assert z.zccl_zero_point_offset(n) == oracle.zero_point_offset(n)
    full, tail = divmod(n, 4096)
    assert z.zccl_zero_point_offset(n) == 128 + full * 5632 + (-(-tail // 1024) * 1024) * 11 // 8


def test_workspace_bytes(z):
    assert z.zccl_workspace_bytes(z.OP_COMPRESS, 0) >= 128
    assert z.zccl_workspace_bytes(z.OP_COMPRESS, 58_720_256) >= 128 + 8 * 14336
    assert z.zccl_workspace_bytes(z.OP_DECOMPRESS_REDUCE, 16 << 20, 8) >= 128 + 8 * 8 * 4096
    assert z.zccl_workspace_bytes(z.OP_COMPRESS_BATCHED, 1 << 28, 128) >= 128 + 8 * (65536 + 128)
    for op, k in [(z.OP_COMPRESS_BATCHED, 0), (z.OP_DECOMPRESS_REDUCE, 0), (9, 1),
                  (z.OP_DECOMPRESS_REDUCE, z.MAX_SHARDS + 1)]:
        with pytest.raises(z.ZcclError):
            z.zccl_workspace_bytes(op, 100, k)


def test_argument_errors_need_no_gpu(z):
    lut = oracle.lut_from_sigma(1.0)
    A = 1 << 20  # a fake, 16-byte aligned "device" address: never dereferenced
    ok = dict(d_in=A, n=4096, lut=lut, d_out=A, out_capacity=z.zccl_max_compressed_bytes(4096),
              d_out_bytes=A, d_ws=A, ws_bytes=1 << 16, d_status=A, stream=None)
    bad = [dict(d_in=A + 2), dict(d_out=A + 8), dict(d_ws=0), dict(d_out_bytes=0),
           dict(lut=bytes([3, 3, 4, 5, 6, 7, 8])), dict(n=1 << 40), dict(d_status=A + 1)]
    for b in bad:
        assert z.zccl_compress(**dict(ok, **b)) == z.INVALID_ARG, b
    assert z.zccl_compress(**dict(ok, out_capacity=100)) == z.BUFFER_TOO_SMALL
    assert z.zccl_compress(**dict(ok, ws_bytes=64)) == z.BUFFER_TOO_SMALL
    assert z.zccl_decompress(A, 64, A, 4096, A, 1 << 16, 0, None) == z.INVALID_ARG  # in_bytes too small
    assert z.zccl_decompress_split(A + 8, A, 128, A, 4096, A, 1 << 16, 0, None) == z.INVALID_ARG  # frame
    assert z.zccl_decompress_split(A, A + 4, 128, A, 4096, A, 1 << 16, 0, None) == z.INVALID_ARG  # tail
    assert z.zccl_decompress_split(A, 0, 128, A, 4096, A, 1 << 16, 0, None) == z.INVALID_ARG  # no tail
    assert z.zccl_decompress_split(A, A, 128, A, 4096, A, 64, 0, None) == z.BUFFER_TOO_SMALL
    assert z.zccl_decompress_reduce(A, A, 0, A, 100, A, 1 << 16, 0, None) == z.INVALID_ARG
    wsr = z.zccl_workspace_bytes(z.OP_DECOMPRESS_REDUCE, 100, 4)
    assert z.zccl_decompress_reduce_local(A, A, 4, A, 4, 0, A, 100, A, wsr, 0, None) == z.INVALID_ARG  # local_pos >= S
    assert z.zccl_decompress_reduce_local(A, A, 4, A + 8, 1, 0, A, 100, A, wsr, 0, None) == z.INVALID_ARG  # unaligned
    assert z.zccl_decompress_reduce_local(A, A, 0, A, 0, 1, A, 100, A, wsr, 0, None) == z.INVALID_ARG  # S == 0
    assert z.zccl_decompress_reduce_local(A, A, 4, A, 1, 1, A, 100, A, 64, 0, None) == z.BUFFER_TOO_SMALL
    assert z.zccl_compress_batched(A, 0, 100, lut, A, A, 1 << 16, 0, None) == z.INVALID_ARG
    assert z.zccl_exponent_histogram(A + 2, 100, A, 0, None) == z.INVALID_ARG  # unaligned input
    assert z.zccl_exponent_histogram(A, 100, A + 4, 0, None) == z.INVALID_ARG  # unaligned histogram
    assert z.zccl_exponent_histogram(A, 100, 0, 1, None) == z.INVALID_ARG
    assert z.zccl_exponent_histogram(A, 1 << 40, A, 0, None) == z.INVALID_ARG
    assert z.lib().zccl_lut_from_data(A, 100, A, 0, None) == z.INVALID_ARG  # no LUT out
    with pytest.raises(z.ZcclError):
        z.zccl_lut_from_data(A + 2, 100, A, None)
    assert z.zccl_status_string(0) == "ok"
    assert z.status_string(z.CORRUPT_STREAM) == "corrupt stream"


@pytest.mark.parametrize("seed", range(6))
def test_library_lut_from_histogram_matches_oracle(z, seed):
    """The host selection in the library against the oracle's, on histograms
    with many ties (small counts) and with empty bins among the top 7."""
    rng = np.random.default_rng(seed)
    hist = rng.integers(0, 4 if seed % 2 else 1 << 40, 256, dtype=np.uint64)
    if seed >= 4:
        hist[:] = 0
        hist[rng.choice(256, 3, replace=False)] = rng.integers(1, 5, 3, dtype=np.uint64)
    assert z.zccl_lut_from_histogram(hist) == oracle.lut_from_histogram(hist)


def test_library_lut_from_histogram_rejects_bad_size(z):
    with pytest.raises(ValueError):
        z.zccl_lut_from_histogram(np.zeros(255, np.uint64))


def test_noalloc_limit_is_the_exact_bound(z):
    """ZCCL_NOALLOC_MAX_ELEMS (copied into the binding) is the largest n whose
    decompress workspace fits the 1 MiB static scratch, to the chunk: the
    workspace of that n fits, one more chunk does not."""
    assert z.zccl_workspace_bytes(z.OP_DECOMPRESS, z.NOALLOC_MAX_ELEMS) <= z.NOALLOC_SCRATCH_BYTES
    assert z.zccl_workspace_bytes(z.OP_DECOMPRESS, z.NOALLOC_MAX_ELEMS + 4096) > z.NOALLOC_SCRATCH_BYTES
    assert z.NOALLOC_MAX_ELEMS % 4096 == 0
