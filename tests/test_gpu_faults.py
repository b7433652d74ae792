"""GPU error paths: host-side argument errors (nothing launched), corrupt
streams reported through the device status word, the bounded device waits
running out (an mbarrier phase, a counter and a flag word that nothing ever
completes), and the workspace's state after each kind of error."""
import ctypes

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


def test_host_argument_errors(z):
    lut = oracle.lut_from_sigma(1.0)
    n = 4096
    x = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    cap = z.zccl_max_compressed_bytes(n)
    out = torch.zeros(cap + 16, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    wsb = z.zccl_workspace_bytes(z.OP_COMPRESS, n)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = lambda **kw: dict(dict(d_in=x.data_ptr(), n=n, lut=lut, d_out=out.data_ptr(),
                                  out_capacity=cap, d_out_bytes=nb.data_ptr(), d_ws=ws.data_ptr(),
                                  ws_bytes=wsb, d_status=st.data_ptr(), stream=s), **kw)
    assert z.zccl_compress(**args()) == z.OK
    assert z.zccl_compress(**args(d_in=x.data_ptr() + 2)) == z.INVALID_ARG
    assert z.zccl_compress(**args(d_out=out.data_ptr() + 8)) == z.INVALID_ARG
    assert z.zccl_compress(**args(out_capacity=cap - 1)) == z.BUFFER_TOO_SMALL
    assert z.zccl_compress(**args(ws_bytes=128)) == z.BUFFER_TOO_SMALL
    assert z.zccl_compress(**args(lut=bytes([1, 1, 2, 3, 4, 5, 6]))) == z.INVALID_ARG
    assert z.zccl_compress(**args(n=1 << 40)) == z.INVALID_ARG
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def _decode_status(z, stream: bytes, n: int, in_bytes=None):
    codec = z.Codec()
    codec.reset_status()
    codec.decompress(dev_bytes(stream, pad=256), len(stream) if in_bytes is None else in_bytes, n)
    torch.cuda.synchronize()
    return codec.read_status()


def _corrupt(stream, off, val):
    b = bytearray(stream)
    b[off] = val
    return bytes(b)


def _unescape_one(stream):
    """Sets plane-0 bit of the first escaped slot of chunk 0, so the planes
    hold one escape fewer than the header says."""
    b = bytearray(stream)
    planes = [np.unpackbits(np.frombuffer(bytes(b[128 + 4096 + p * 512: 128 + 4096 + (p + 1) * 512]),
                                          np.uint8), bitorder="little") for p in range(3)]
    slot = int(np.flatnonzero((planes[0] | planes[1] | planes[2]) == 0)[0])
    b[128 + 4096 + slot // 8] |= 1 << (slot % 8)
    return bytes(b)


def test_corrupt_streams_reported(z):
    x = workloads.gaussian(3 * 4096 + 500, 1.0, seed=1)
    s = oracle.compress(x, oracle.lut_from_sigma(1.0))
    n = x.size
    assert _decode_status(z, s, n) == z.OK
    for name, b in {
        "magic": _corrupt(s, 0, 0),
        "version": _corrupt(s, 4, 2),
        "log2chunk": _corrupt(s, 6, 11),
        "n": _corrupt(s, 8, s[8] ^ 1),
        "n_esc_up": _corrupt(s, 16, s[16] + 1),
        "n_esc_down": _corrupt(s, 16, s[16] - 1),
        "zp_offset": _corrupt(s, 32, s[32] ^ 0x80),
        "dup_lut": _corrupt(s, 25, s[24]),
        "byte31": _corrupt(s, 31, 1),
        "reserved40": _corrupt(s, 40, 1),
        "reserved127": _corrupt(s, 127, 0x80),
        "escape_made_coded": _unescape_one(s),
    }.items():
        assert oracle.decompress_status(b, n)[0] == oracle.CORRUPT, name
        assert _decode_status(z, b, n) == z.CORRUPT_STREAM, name
    # zero-point array cut off (in_bytes below the header's size)
    assert _decode_status(z, s, n, in_bytes=len(s) - 128) == z.CORRUPT_STREAM


def test_bounded_wait_reports_timeout(z):
    """The mbarrier waits on the kernels' own TMA copies are bounded.
    zccl_check_bounded_wait runs that same wait on a barrier nothing
    completes: it must end (here after 2 ms) with ZCCL_ERR_TIMEOUT in the
    status word, and the context must stay usable."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert z.zccl_check_bounded_wait(2000, st.data_ptr(), s) == z.OK
    torch.cuda.synchronize()
    assert int(st.item()) == z.TIMEOUT
    assert z.zccl_check_bounded_wait(0, st.data_ptr(), s) == z.INVALID_ARG
    # the context still works: a normal round trip
    lut = oracle.lut_from_sigma(1.0)
    x = workloads.gaussian(3 * 4096 + 17, 1.0, seed=3)
    codec = z.Codec()
    out, nb = codec.compress(dev_u16(x), lut)
    torch.cuda.synchronize()
    assert codec.read_status() == z.OK
    assert out[: int(nb.item())].cpu().numpy().tobytes() == oracle.compress(x, lut)


def test_workspace_reused_across_many_calls(z):
    """The per-call arrival counter and range totals must return to their
    initial state after every call, including after a rejected batch."""
    lut = oracle.lut_from_sigma(1.0)
    codec = z.Codec()
    for i in range(30):
        n = 1 + (i * 104729) % 300_000
        x = workloads.gaussian(n, 1.0, seed=i)
        codec.reset_status()
        out, nb = codec.compress(dev_u16(x), lut)
        y = codec.decompress(out, int(nb.item()), n)
        torch.cuda.synchronize()
        assert codec.read_status() == z.OK
        assert out[: int(nb.item())].cpu().numpy().tobytes() == oracle.compress(x, lut)
        assert np.array_equal(y.cpu().numpy().view(np.uint16), x)


@pytest.mark.parametrize("kind", ["counter", "flag"])
def test_bounded_polls_report_timeout(z, kind):
    """The kernels also wait on words other CTAs write: the call's done
    counter (compress and decompress), the run-total and chunk-entry flag
    words (decompress) and the look-back words of earlier ranges (the escape
    scan of decompress-reduce).  zccl_check_bounded_poll runs those same waits
    on a zeroed word that nothing ever sets: each must end (after 3 ms) with
    ZCCL_ERR_TIMEOUT, and the context must stay usable."""
    k = z.POLL_COUNTER if kind == "counter" else z.POLL_FLAG
    word = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert z.zccl_check_bounded_poll(k, 3000, word.data_ptr(), st.data_ptr(), s) == z.OK
    torch.cuda.synchronize()
    assert int(st.item()) == z.TIMEOUT
    assert int(word.item()) == 0
    assert z.zccl_check_bounded_poll(3, 3000, word.data_ptr(), st.data_ptr(), s) == z.INVALID_ARG
    assert z.zccl_check_bounded_poll(k, 0, word.data_ptr(), st.data_ptr(), s) == z.INVALID_ARG
    assert z.zccl_check_bounded_poll(k, 3000, word.data_ptr() + 4, st.data_ptr(), s) == z.INVALID_ARG
    # a word that is already complete returns at once, with no error
    word.fill_(-(1 << 63) if kind == "flag" else 1)
    st.zero_()
    assert z.zccl_check_bounded_poll(k, 3000, word.data_ptr(), st.data_ptr(), s) == z.OK
    torch.cuda.synchronize()
    assert int(st.item()) == z.OK
    lut = oracle.lut_from_sigma(1.0)
    x = workloads.gaussian(2 * 4096 + 5, 1.0, seed=4)
    codec = z.Codec()
    out, nb = codec.compress(dev_u16(x), lut)
    y = codec.decompress(out, int(nb.item()), x.size)
    torch.cuda.synchronize()
    assert codec.read_status() == z.OK
    assert np.array_equal(y.cpu().numpy().view(np.uint16), x)


# every workspace starts with a 2 KB control block and two parity sets of
# 4096 64-bit flag words; everything past them is scratch that calls leave zero
WS_PREFIX = 2048 + 2 * 8 * 4096


def _ws_clear_past_prefix(codec, z):
    return int((codec._ws[WS_PREFIX:] != 0).sum().item()) == 0


def test_workspace_ready_after_corrupt_stream(z):
    """A call that reports CORRUPT_STREAM leaves its workspace ready: on the
    same workspace, with no re-initialisation, the next decompress and the
    next decompress-reduce are bit-exact, and the scratch past the control
    block and flag area is all zero again after each call."""
    lut = oracle.lut_from_sigma(1.0)
    n = 3 * 4096 + 500
    x = workloads.gaussian(n, 1.0, seed=5)
    good = oracle.compress(x, lut)
    bad = {"magic": _corrupt(good, 0, 0), "dup_lut": _corrupt(good, 25, good[24]),
           "reserved": _corrupt(good, 64, 1), "escape_made_coded": _unescape_one(good)}
    codec = z.Codec()
    for name, b in bad.items():
        codec.reset_status()
        codec.decompress(dev_bytes(b, pad=256), len(b), n)
        torch.cuda.synchronize()
        assert codec.read_status() == z.CORRUPT_STREAM, name
        assert _ws_clear_past_prefix(codec, z), name
        codec.reset_status()
        y = codec.decompress(dev_bytes(good, pad=256), len(good), n)
        torch.cuda.synchronize()
        assert codec.read_status() == z.OK, name
        assert np.array_equal(y.cpu().numpy().view(np.uint16), x), name
        # a reduction with the bad stream as one shard, then a good one
        shards = [good, b, good]
        devs = [dev_bytes(t) for t in shards]
        codec.reset_status()
        codec.decompress_reduce(devs, [len(t) for t in shards], n)
        torch.cuda.synchronize()
        assert codec.read_status() == z.CORRUPT_STREAM, name
        assert _ws_clear_past_prefix(codec, z), name
        codec.reset_status()
        r = codec.decompress_reduce([dev_bytes(good)] * 3, [len(good)] * 3, n)
        torch.cuda.synchronize()
        assert codec.read_status() == z.OK, name
        assert np.array_equal(r.cpu().numpy().view(np.uint16), oracle.decompress_reduce([good] * 3, n)), name


def test_workspace_init_recovers_a_call_left_midway(z):
    """After ZCCL_ERR_TIMEOUT some CTAs may have stopped mid-call, leaving the
    workspace's control words (call count, tickets, done counters, arrival
    counters) and flag words anywhere.  Such a workspace is made here by
    filling it with arbitrary bytes on the host; zccl_workspace_init then
    makes it ready, and compress, decompress and a reduction are bit-exact."""
    lut = oracle.lut_from_sigma(1.0)
    n = 5 * 4096 + 77
    x = workloads.gaussian(n, 1.0, seed=6)
    codec = z.Codec()
    wsb = max(z.zccl_workspace_bytes(z.OP_COMPRESS, n), z.zccl_workspace_bytes(z.OP_DECOMPRESS_REDUCE, n, 3))
    ptr, size = codec.workspace(wsb)
    rng = np.random.default_rng(7)
    codec._ws.copy_(torch.from_numpy(rng.integers(0, 256, size=size, dtype=np.uint8)).cuda())
    s = torch.cuda.current_stream().cuda_stream
    assert z.zccl_workspace_init(ptr, size, s) == z.OK
    codec.reset_status()
    out, nb = codec.compress(dev_u16(x), lut)
    y = codec.decompress(out, int(nb.item()), n)
    r = codec.decompress_reduce([out] * 3, [int(nb.item())] * 3, n)
    torch.cuda.synchronize()
    assert codec.read_status() == z.OK
    stream = oracle.compress(x, lut)
    assert out[: int(nb.item())].cpu().numpy().tobytes() == stream
    assert np.array_equal(y.cpu().numpy().view(np.uint16), x)
    assert np.array_equal(r.cpu().numpy().view(np.uint16), oracle.decompress_reduce([stream] * 3, n))
