"""Static-part framing (ZipCCL technical summary 2.C framing, used for the
static part of the two-phase all-to-all of 2.D): a stream splits into a frame
whose size depends on n alone (header + chunk blocks) and a zero-point tail
whose size the receiver reads from the frame's header.

The sizes are derived here from the layout (128-byte header, 11 bits per
slot, tail slots rounded up to 1024, one byte per escape padded to 128) and
checked against the oracle's streams and the library's size formula."""
import numpy as np
import pytest

import oracle
from lossless_bf16_exponent_split_gb300 import workloads

NS = [0, 1, 1000, 1024, 1025, 4096, 4097, 3 * 4096 + 5, 50_001]
PAYLOADS = {
    "gauss": lambda n: workloads.gaussian(n, 0.02, seed=n),
    "all_escape": lambda n: workloads.random_bits(n, seed=n) | 0x7F80,  # exponent 255 only
    "no_escape": lambda n: np.full(n, 0x3C00, np.uint16),                # exponent 120, in the LUT
}
LUT = oracle.lut_from_sigma(0.02)


def frame_bytes(n):
    full, tail = divmod(n, 4096)
    return 128 + (full * 4096 + -(-tail // 1024) * 1024) * 11 // 8


@pytest.mark.parametrize("n", NS)
def test_frame_size_depends_on_n_only(n):
    sizes = set()
    for make in PAYLOADS.values():
        s = oracle.compress(make(n), LUT)
        n_esc = int.from_bytes(s[16:24], "little")
        zp = int.from_bytes(s[32:40], "little")
        assert zp == frame_bytes(n) == oracle.zero_point_offset(n)
        # the receiver learns the tail's size from the header alone
        assert len(s) - zp == -(-n_esc // 128) * 128
        sizes.add(zp)
    assert len(sizes) == 1


def test_frame_and_tail_rejoin_to_the_stream():
    n = 3 * 4096 + 77
    x = workloads.special_values(n, seed=5)
    s = oracle.compress(x, LUT)
    zp = frame_bytes(n)
    frame, tail = s[:zp], s[zp:]
    assert len(tail) > 0
    assert np.array_equal(oracle.decompress(frame + tail, n), x)
    # a tail of the wrong size is a corrupt stream (the header's count is authoritative)
    st, _ = oracle.decompress_status(frame + tail[:-128], n)
    assert st != oracle.OK


def test_library_frame_size_matches():
    from lossless_bf16_exponent_split_gb300 import build
    build.build()
    import lossless_bf16_exponent_split_gb300 as z
    for n in NS + [1 << 30, (1 << 40) - 1]:
        assert z.zccl_zero_point_offset(n) == frame_bytes(n)
