"""GPU parity: libzccl compress/decompress against the oracle, byte for byte.

The oracle (plain C, CPU) defines the stream; the CUDA kernels must produce
identical stream bytes and identical decoded bits (ZipCCL technical summary
2.B, 2.C: lossless, bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
from golden_io import read_stream_fixture
from gpu_util import dev_bytes, dev_u16, host_u16, load_lib, require_gpu, stream_of
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu

LUTS = {
    "sigma0.02": oracle.lut_from_sigma(0.02),
    "sigma1": oracle.lut_from_sigma(1.0),
    "zero_inf": bytes([0, 255, 1, 2, 3, 254, 127]),
    "absent": bytes([200, 201, 202, 203, 204, 205, 206]),
}
EDGE_N = [0, 1, 7, 8, 9, 31, 32, 33, 1023, 1024, 1025, 4095, 4096, 4097, 8191, 8192,
          3 * 4096 + 5, 10 * 4096 + 1000, 100_003]


@pytest.fixture(scope="module")
def codec():
    require_gpu()
    load_lib()
    from lossless_bf16_exponent_split_gb300 import Codec
    return Codec()


def gpu_compress(codec, x, lut):
    codec.reset_status()
    out, nb = codec.compress(dev_u16(x), lut)
    s = stream_of(out, nb)
    assert codec.read_status() == 0
    return s


def gpu_decompress(codec, stream, n):
    codec.reset_status()
    y = codec.decompress(dev_bytes(stream), len(stream), n)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    return host_u16(y)


@pytest.mark.parametrize("n", EDGE_N)
@pytest.mark.parametrize("lut_name", ["sigma0.02", "zero_inf"])
def test_compress_edge_sizes(codec, n, lut_name):
    x = workloads.special_values(n, seed=n) if lut_name == "zero_inf" else workloads.gaussian(n, 0.02, seed=n)
    lut = LUTS[lut_name]
    want = oracle.compress(x, lut)
    assert gpu_compress(codec, x, lut) == want
    assert np.array_equal(gpu_decompress(codec, want, n), x)


@pytest.mark.parametrize("lut_name", list(LUTS))
def test_all_bf16_patterns(codec, lut_name):
    x = np.arange(65536, dtype=np.uint16)
    lut = LUTS[lut_name]
    want = oracle.compress(x, lut)
    assert gpu_compress(codec, x, lut) == want
    assert np.array_equal(gpu_decompress(codec, want, x.size), x)
    # shuffled, so every chunk mixes every exponent
    rng = np.random.default_rng(1)
    xs = x[rng.permutation(x.size)]
    want = oracle.compress(xs, lut)
    assert gpu_compress(codec, xs, lut) == want
    assert np.array_equal(gpu_decompress(codec, want, xs.size), xs)


def test_hand_built_fixture(codec):
    x, lut, stream = read_stream_fixture()
    assert gpu_compress(codec, x, lut) == stream
    assert np.array_equal(gpu_decompress(codec, stream, x.size), x)


def test_escape_extremes(codec):
    x = workloads.random_bits(50_000, seed=4)
    for lut in (LUTS["absent"], bytes([1, 2, 3, 4, 5, 6, 7])):
        want = oracle.compress(x, lut)
        assert gpu_compress(codec, x, lut) == want
    lut = LUTS["sigma1"]
    e = np.frombuffer(lut, np.uint8).astype(np.uint16)
    y = (e[np.arange(50_000) % 7] << 7) | (np.arange(50_000, dtype=np.uint16) & 0x807F)
    want = oracle.compress(y, lut)
    assert int.from_bytes(want[16:24], "little") == 0
    assert gpu_compress(codec, y, lut) == want
    assert np.array_equal(gpu_decompress(codec, want, y.size), y)


def test_gauss1m(codec):
    cfg = workloads.CONFIGS["gauss1m"]
    x = workloads.gaussian(cfg["n"], cfg["sigma"], seed=0)
    lut = oracle.lut_from_sigma(cfg["sigma"])
    want = oracle.compress(x, lut)
    assert gpu_compress(codec, x, lut) == want
    assert np.array_equal(gpu_decompress(codec, want, x.size), x)


def _full_size(codec, x, lut):
    """Byte-identical stream and bit-identical decode at a full config size;
    compared on the device to keep host traffic small."""
    want = oracle.compress(x, lut)
    codec.reset_status()
    xd = dev_u16(x)
    out, nb = codec.compress(xd, lut)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    assert int(nb.item()) == len(want)
    wd = dev_bytes(want)
    assert torch.equal(out[: len(want)], wd)
    codec.reset_status()
    y = codec.decompress(wd, len(want), x.size)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    assert torch.equal(y, xd)


def test_llama3_8b_allgather_full(codec):
    cfg = workloads.CONFIGS["llama3_8b_allgather"]
    _full_size(codec, workloads.gaussian(cfg["n"], cfg["sigma"], seed=0),
               oracle.lut_from_sigma(cfg["sigma"]))


def test_activation_mix_full(codec):
    _full_size(codec, workloads.activation_mix(), oracle.lut_from_sigma(1.0))


def test_shared_workspace_across_ops(codec):
    """One workspace serves compress, decompress and reduce calls in any
    order and size; each call must leave it ready for the next."""
    lut = LUTS["sigma1"]
    for i, n in enumerate([300_000, 5_000, 1_000_000, 77, 600_001]):
        x = workloads.gaussian(n, 1.0, seed=50 + i)
        want = oracle.compress(x, lut)
        assert gpu_compress(codec, x, lut) == want
        assert np.array_equal(gpu_decompress(codec, want, n), x)
        codec.reset_status()
        r = codec.decompress_reduce([dev_bytes(want), dev_bytes(want)], [len(want)] * 2, n)
        torch.cuda.synchronize()
        assert codec.read_status() == 0
        assert np.array_equal(host_u16(r), oracle.decompress_reduce([want, want], n))


def test_output_canary_untouched(codec):
    x = workloads.gaussian(20_000, 0.02, seed=9)
    lut = LUTS["sigma0.02"]
    want = oracle.compress(x, lut)
    cap = oracle.max_bytes(x.size)
    out = torch.full((cap + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    codec.reset_status()
    _, nb = codec.compress(dev_u16(x), lut, out=out)
    torch.cuda.synchronize()
    assert int(nb.item()) == len(want)
    host = out.cpu().numpy()
    assert host[: len(want)].tobytes() == want
    assert (host[len(want):] == 0xA5).all()


def test_repeated_calls_same_workspace(codec):
    lut = LUTS["sigma1"]
    for i in range(40):
        n = 1 + (i * 7919) % 60000
        x = workloads.gaussian(n, 1.0, seed=100 + i)
        want = oracle.compress(x, lut)
        assert gpu_compress(codec, x, lut) == want
        assert np.array_equal(gpu_decompress(codec, want, n), x)


def test_in_place_graph_of_calls_no_sync(codec):
    """Several calls queued back to back on one stream, one sync at the end."""
    lut = LUTS["sigma0.02"]
    xs = [workloads.gaussian(n, 0.02, seed=n) for n in (5000, 123_457, 4096 * 7, 77)]
    outs = []
    codec.reset_status()
    for x in xs:
        xd = dev_u16(x)
        outs.append((x, *codec.compress(xd, lut)))
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    for x, out, nb in outs:
        assert stream_of(out, nb) == oracle.compress(x, lut)


# Workspace bytes ahead of the per-call scratch: the control block (2048
# bytes) and two call-parity sets of 4096 run flag words.
WS_PREFIX = 2048 + 2 * 8 * 4096


def _scratch_is_zero(codec) -> bool:
    torch.cuda.synchronize()
    ws = codec._ws
    return bool((ws[WS_PREFIX:] == 0).all().item())


def test_workspace_scratch_left_zero(codec):
    """Every op leaves the workspace all zero past its control block and flag
    sets (the decoder's per-chunk entry words rely on it when ops share a
    workspace)."""
    from lossless_bf16_exponent_split_gb300 import (OP_COMPRESS, OP_COMPRESS_BATCHED, OP_DECOMPRESS,
                                                     OP_DECOMPRESS_REDUCE, zccl_workspace_bytes)
    lut = LUTS["sigma1"]
    x = workloads.activation_mix(rows=300, cols=4097, seed=3)  # ~4.5 % escapes, ragged tail
    n = x.size
    segs = [(0, 70_000), (70_000, 0), (70_000, 500_000), (570_000, n - 570_000)]
    codec.workspace(max(zccl_workspace_bytes(OP_COMPRESS, n), zccl_workspace_bytes(OP_DECOMPRESS, n),
                        zccl_workspace_bytes(OP_DECOMPRESS_REDUCE, n, 3),
                        zccl_workspace_bytes(OP_COMPRESS_BATCHED, n, len(segs))))
    want = oracle.compress(x, lut)
    assert gpu_compress(codec, x, lut) == want
    assert _scratch_is_zero(codec)
    assert np.array_equal(gpu_decompress(codec, want, n), x)
    assert _scratch_is_zero(codec)
    codec.reset_status()
    r = codec.decompress_reduce([dev_bytes(want)] * 3, [len(want)] * 3, n)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    assert np.array_equal(host_u16(r), oracle.decompress_reduce([want] * 3, n))
    assert _scratch_is_zero(codec)
    xd = dev_u16(x)
    pairs = []
    for lo, cnt in segs:
        pairs.append((xd[lo:lo + cnt], torch.empty(oracle.max_bytes(cnt), dtype=torch.uint8, device="cuda")))
    codec.reset_status()
    nb = codec.compress_batched(pairs, lut, total_n=n)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    for (lo, cnt), (_, o), m in zip(segs, pairs, nb.cpu().tolist()):
        assert o[:m].cpu().numpy().tobytes() == oracle.compress(x[lo:lo + cnt], lut)
    assert _scratch_is_zero(codec)


def test_long_runs_full_parity(codec):
    """700M elements: each CTA's run of chunks spans more than one 128-chunk
    batch in both kernels (grid <= 1216 CTAs), with a ragged tail, and both
    kernels hand out chunks in tickets of 4, then 2, then 1 consecutive
    chunks as the call nears its end; stream and round trip bit-exact
    against the oracle."""
    n = 700_000_000
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    xd = (torch.randn(n, device="cuda", generator=g) * 0.02).to(torch.bfloat16).view(torch.int16)
    lut = LUTS["sigma0.02"]
    codec.reset_status()
    out, nb = codec.compress(xd, lut)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    m = int(nb.item())
    x = xd.cpu().numpy().view(np.uint16)
    want = oracle.compress(x, lut)
    assert m == len(want)
    assert out[:m].cpu().numpy().tobytes() == want
    codec.reset_status()
    y = codec.decompress(out, m, n)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    assert torch.equal(y, xd)


@pytest.mark.parametrize("n", [0, 1, 1025, 4096, 3 * 4096 + 5, 100_003])
@pytest.mark.parametrize("kind", ["gauss", "special", "no_escape"])
def test_decompress_split_frame_and_tail(codec, n, kind):
    """The stream received as two separate buffers: its frame (header and
    blocks, a size fixed by n) and its zero-point tail."""
    x = {"gauss": lambda: workloads.gaussian(n, 0.02, seed=n + 1),
         "special": lambda: workloads.special_values(n, seed=n + 2),
         "no_escape": lambda: np.full(n, 0x3C00, np.uint16)}[kind]()
    lut = LUTS["sigma0.02"]
    stream = oracle.compress(x, lut)
    zp = oracle.zero_point_offset(n)
    frame = dev_bytes(stream[:zp])
    tail_b = stream[zp:]
    tail = dev_bytes(tail_b) if tail_b else None
    if kind == "no_escape":
        assert not tail_b
    codec.reset_status()
    y = codec.decompress_split(frame, tail, len(tail_b), n)
    torch.cuda.synchronize()
    assert codec.read_status() == 0
    assert np.array_equal(host_u16(y), x)


def test_decompress_split_short_tail_is_corrupt(codec):
    n = 2 * 4096 + 3
    x = workloads.special_values(n, seed=9)
    stream = oracle.compress(x, LUTS["sigma0.02"])
    zp = oracle.zero_point_offset(n)
    assert len(stream) - zp >= 256
    codec.reset_status()
    codec.decompress_split(dev_bytes(stream[:zp]), dev_bytes(stream[zp:-128]), len(stream) - zp - 128, n)
    torch.cuda.synchronize()
    assert codec.read_status() == 3  # CORRUPT_STREAM
