"""zccl_decompress_noalloc: decompression for callers that cannot allocate.

Callers such as a communication library's progress thread, or a framework
hook that must stay inside the framework's memory pool, cannot call
cudaMalloc for a workspace; this entry point takes its workspace from a
static device array in the library instead.  The test calls it through the
C ABI twice in a row (different sizes) and checks each result against
zccl_decompress, bit for bit -- the codec is lossless, so the tolerance is
exact equality.  Before them, a call on a corrupt stream stops early and
leaves the shared scratch dirty; the entry point clears the part a call uses
before each call, and the valid calls that follow show it.  It lives in a
file of its own, collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_bytes, dev_u16, load_lib, require_gpu
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def z():
    require_gpu()
    load_lib()
    import lossless_bf16_exponent_split_gb300 as z
    return z


def reference_decompress(z, stream_dev, in_bytes, n):
    """The existing entry point, with a caller-allocated workspace."""
    codec = z.Codec()
    codec.reset_status()
    y = codec.decompress(stream_dev, in_bytes, n)
    torch.cuda.synchronize()
    assert codec.read_status() == z.OK
    return y


def test_noalloc_matches_decompress_twice(z):
    s = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # a stream whose header promises one escape more than its planes hold:
    # the call reports CORRUPT_STREAM after counting, with the scratch's
    # control words and flags left written
    xb = workloads.gaussian(5 * 4096 + 9, 0.02, seed=69)
    bad = bytearray(oracle.compress(xb, oracle.lut_from_sigma(0.02)))
    bad[16] += 1
    bd = dev_bytes(bytes(bad), pad=256)
    junk = torch.empty(xb.size, dtype=torch.int16, device="cuda")
    assert z.zccl_decompress_noalloc(bd.data_ptr(), len(bad) + 128, junk.data_ptr(), xb.size, status.data_ptr(),
                                     s) == z.OK
    torch.cuda.synchronize()
    assert int(status.item()) == z.CORRUPT_STREAM
    for i, n in enumerate([3 * 4096 * 257 + 11, 40_000]):  # the second call is the smaller
        x = workloads.gaussian(n, 0.02, seed=70 + i)
        stream = oracle.compress(x, oracle.lut_from_sigma(0.02))
        sd = dev_bytes(stream)
        want = reference_decompress(z, sd, len(stream), n)
        out = torch.empty(n, dtype=torch.int16, device="cuda")
        status.zero_()
        assert z.zccl_decompress_noalloc(sd.data_ptr(), len(stream), out.data_ptr(), n, status.data_ptr(), s) == z.OK
        torch.cuda.synchronize()
        assert int(status.item()) == z.OK
        assert torch.equal(out, want)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), x)


def test_noalloc_rejects_sizes_beyond_its_scratch(z):
    s = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dummy = torch.zeros(256, dtype=torch.uint8, device="cuda")
    too_big = z.NOALLOC_MAX_ELEMS + 1
    assert z.zccl_decompress_noalloc(dummy.data_ptr(), 1 << 62, dummy.data_ptr(), too_big,
                                     status.data_ptr(), s) == z.INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == 0
