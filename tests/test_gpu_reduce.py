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
                                 (5, 1), (4, 1023), (40, 9000), (2, 4 * 4096 + 3500)])
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


@pytest.mark.parametrize("off,val", [(25, None), (31, 1), (40, 1), (16, "up")])
def test_reduce_rejects_corrupt_header(codec, off, val):
    """A shard whose header breaks the format (a repeated LUT exponent, a
    nonzero reserved byte, an escape total the planes disagree with) makes
    the reduction report CORRUPT_STREAM, as the oracle rejects it."""
    lut = oracle.lut_from_sigma(1.0)
    n = 2 * 4096 + 300
    good = [oracle.compress(workloads.gaussian(n, 1.0, seed=s), lut) for s in range(3)]
    b = bytearray(good[1])
    b[off] = b[24] if val is None else (b[off] + 1 if val == "up" else val)
    streams = [good[0], bytes(b), good[2]]
    assert oracle.decompress_status(streams[1], n)[0] == oracle.CORRUPT
    st, _ = gpu_reduce(codec, streams, n)
    assert st == 3
    # the same codec, on the same workspace, then reduces good shards exactly
    st, got = gpu_reduce(codec, good, n)
    assert st == 0 and np.array_equal(got, oracle.decompress_reduce(good, n))


def test_reduce_empty_streams(codec):
    """n = 0: every stream is a bare header, the output is empty and the
    status stays 0.  A header that claims one escape is rejected as the
    oracle rejects it -- whether the zero-point array it promises is missing
    (the size check) or present (128 zero bytes: the recount of 0 escapes
    disagrees with the header)."""
    lut = oracle.lut_from_sigma(1.0)
    empty = [oracle.compress(np.zeros(0, np.uint16), lut) for _ in range(3)]
    st, got = gpu_reduce(codec, empty, 0)
    assert st == 0 and got.size == 0
    claim = bytearray(empty[1])
    claim[16] = 1  # n_esc = 1
    for bad in (bytes(claim), bytes(claim) + bytes(128)):
        assert oracle.decompress_status(bad, 0)[0] == oracle.CORRUPT
        st, got = gpu_reduce(codec, [empty[0], bad, empty[2]], 0)
        assert st == 3 and got.size == 0
    st, _ = gpu_reduce(codec, empty, 0)  # the workspace is ready again
    assert st == 0


def test_reduce_more_ranges_than_scan_ctas(codec):
    """1,024 shards (the most a call takes) of 131,073 elements: two ranges
    of 32 chunks per stream, 2,048 ranges -- more than one per CTA of the
    escape scan's grid (8 CTAs per SM), so its CTAs take several range
    tickets each and the look-back spans ranges taken in different rounds."""
    S, n = 1024, 32 * 4096 + 1
    lut = oracle.lut_from_sigma(1.0)
    shards = [workloads.special_values(n, seed=7000 + s, frac=0.01) for s in range(S)]
    streams = [oracle.compress(x, lut) for x in shards]
    want = oracle.decompress_reduce(streams, n)
    st, got = gpu_reduce(codec, streams, n)
    assert st == 0
    assert np.array_equal(got, want)


def test_rs_local_full(codec):
    cfg = workloads.CONFIGS["rs_local"]
    shards = workloads.reduce_shards(cfg["S"], cfg["n"], cfg["sigma"], seed=0)
    lut = oracle.lut_from_sigma(cfg["sigma"])
    streams = [oracle.compress(x, lut) for x in shards]
    want = oracle.decompress_reduce(streams, cfg["n"])
    st, got = gpu_reduce(codec, streams, cfg["n"])
    assert st == 0
    assert np.array_equal(got, want)


def gpu_reduce_local(codec, streams, n, local, local_pos, initial=None):
    devs = [None if s is None else dev_bytes(s) for s in streams]
    sizes = [0 if s is None else len(s) for s in streams]
    dlocal = None if local is None else torch.from_numpy(np.ascontiguousarray(local, np.uint16).view(np.int16)).cuda()
    out = None
    if initial is not None:
        out = torch.from_numpy(np.ascontiguousarray(initial, np.uint16).view(np.int16)).cuda()
    codec.reset_status()
    out = codec.decompress_reduce_local(devs, sizes, n, local=dlocal, local_pos=local_pos, out=out,
                                        accumulate=initial is not None)
    torch.cuda.synchronize()
    return codec.read_status(), host_u16(out)


@pytest.mark.parametrize("S,n,local_pos,acc", [(1, 5000, 0, False), (1, 4099, 0, True), (2, 4096, 1, False),
                                               (3, 3 * 4096 + 77, 0, True), (5, 100_003, 2, False),
                                               (8, 65_541, 7, True), (4, 7, 3, True), (6, 20_000, 5, False)])
def test_reduce_local_shard_matches_oracle(codec, S, n, local_pos, acc):
    """ZipCCL 2.D as one rank runs it: the rank's own shard enters the fold
    uncompressed at its rank position; optionally the fold starts from the
    output's current values.  Ragged n exercises the plain-BF16 tail."""
    shards = [workloads.special_values(n, seed=100 * S + s, frac=0.05) for s in range(S)]
    lut = oracle.lut_from_sigma(1.0)
    streams = [None if s == local_pos else oracle.compress(x, lut) for s, x in enumerate(shards)]
    initial = workloads.special_values(n, seed=7 + S, frac=0.05) if acc else None
    want = oracle.decompress_reduce_local(streams, n, local=shards[local_pos], local_pos=local_pos, initial=initial)
    st, got = gpu_reduce_local(codec, streams, n, shards[local_pos], local_pos, initial)
    assert st == 0
    assert np.array_equal(got, want)


def test_reduce_accumulate_without_local(codec):
    n, S = 2 * 4096 + 5, 3
    shards = [workloads.gaussian(n, 1e-3, seed=40 + s) for s in range(S)]
    lut = oracle.lut_from_sigma(1e-3)
    streams = [oracle.compress(x, lut) for x in shards]
    initial = workloads.gaussian(n, 1e-3, seed=99)
    want = oracle.decompress_reduce_local(streams, n, initial=initial)
    st, got = gpu_reduce_local(codec, streams, n, None, 0, initial)
    assert st == 0
    assert np.array_equal(got, want)


def test_reduce_local_equals_all_compressed(codec):
    """Holding one's own shard uncompressed gives the same bits as receiving
    it compressed (the codec is lossless)."""
    n, S = 50_000, 4
    shards = [workloads.gaussian(n, 1e-3, seed=60 + s) for s in range(S)]
    lut = oracle.lut_from_sigma(1e-3)
    streams = [oracle.compress(x, lut) for x in shards]
    st0, all_c = gpu_reduce(codec, streams, n)
    st1, with_local = gpu_reduce_local(codec, [streams[0], None, streams[2], streams[3]], n, shards[1], 1)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(all_c, with_local)
