"""GPU: each call reads what the work queued right before it in the stream
wrote, with no host synchronisation in between.

Some of the library's kernels are launched as programmatic dependents of the
preceding work, so they start during its tail and must wait for it before
reading anything. These tests queue producer and consumer back to back, with
inputs that change from one round to the next, and compare every result with
the oracle at the end. (Technical summary 2.A for the histogram, 2.B/2.D for
the codec and the local reduction of zipped all-to-all.)"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_u16, host_u16, load_lib, require_gpu
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def z():
    require_gpu()
    load_lib()
    import lossless_bf16_exponent_split_gb300 as z
    return z


def _handle():
    return torch.cuda.current_stream().cuda_stream


def test_histogram_behind_writer_kernel(z):
    """A torch kernel rewrites the input, then the histogram runs; overwrite
    and accumulate alternate, and back-to-back histogram calls follow each
    other directly."""
    n = 2_000_003
    datas = [workloads.gaussian(n, 0.02, seed=1), workloads.special_values(n, seed=2, frac=0.3),
             workloads.random_bits(n, seed=3)]
    srcs = [dev_u16(d) for d in datas]
    buf = torch.empty(n, dtype=torch.int16, device="cuda")
    hists = [torch.zeros(256, dtype=torch.int64, device="cuda") for _ in range(4)]
    torch.cuda.synchronize()
    h = _handle()
    # round r: hist[r] = histogram(datas[r % 3]) then += histogram(datas[(r + 1) % 3])
    for r in range(4):
        torch.bitwise_xor(srcs[r % 3], 0, out=buf)  # the writer kernel
        z.check(z.zccl_exponent_histogram(buf.data_ptr(), n, hists[r].data_ptr(), 0, h), "histogram")
        torch.bitwise_xor(srcs[(r + 1) % 3], 0, out=buf)
        z.check(z.zccl_exponent_histogram(buf.data_ptr(), n, hists[r].data_ptr(), 1, h), "histogram")
    torch.cuda.synchronize()
    want = [oracle.exponent_histogram(d) for d in datas]
    for r in range(4):
        got = hists[r].cpu().numpy().view(np.uint64)
        assert np.array_equal(got, want[r % 3] + want[(r + 1) % 3]), f"round {r}"


def test_reduce_behind_compress(z):
    """S shards are compressed into the same stream buffers every round, and
    the fused decompress-reduce is queued right behind the last compress;
    each round's output must be that round's reduction."""
    S, n, rounds = 4, 300_007, 3
    lut = z.zccl_lut_from_sigma(1.0)
    data = [[workloads.special_values(n, seed=100 * r + s, frac=0.05) for s in range(S)] for r in range(rounds)]
    xs = [[dev_u16(x) for x in row] for row in data]
    cap = z.zccl_max_compressed_bytes(n)
    outs = [torch.zeros(cap, dtype=torch.uint8, device="cuda") for _ in range(S)]
    inb = torch.zeros(S, dtype=torch.int64, device="cuda")  # compress writes each size here
    ptrs = torch.tensor([o.data_ptr() for o in outs], dtype=torch.int64, device="cuda")
    ys = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(rounds)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsc_b = z.zccl_workspace_bytes(z.OP_COMPRESS, n)
    wsc = torch.zeros(wsc_b, dtype=torch.uint8, device="cuda")
    wsr_b = z.zccl_workspace_bytes(z.OP_DECOMPRESS_REDUCE, n, S)
    wsr = torch.zeros(wsr_b, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    h = _handle()
    for r in range(rounds):
        for s in range(S):
            z.check(z.zccl_compress(xs[r][s].data_ptr(), n, lut, outs[s].data_ptr(), cap, inb.data_ptr() + 8 * s,
                                    wsc.data_ptr(), wsc_b, status.data_ptr(), h), "compress")
        z.check(z.zccl_decompress_reduce(ptrs.data_ptr(), inb.data_ptr(), S, ys[r].data_ptr(), n, wsr.data_ptr(),
                                         wsr_b, status.data_ptr(), h), "decompress_reduce")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for r in range(rounds):
        want = oracle.decompress_reduce([oracle.compress(x, lut) for x in data[r]], n)
        assert np.array_equal(host_u16(ys[r]), want), f"round {r}"


def test_reduces_back_to_back(z):
    """Two reductions over different shard sets follow each other directly,
    the second one's scan kernel starting under the first one's tail."""
    S, n = 3, 150_001
    lut = z.zccl_lut_from_sigma(0.5)
    sets = [[workloads.special_values(n, seed=7 * k + s, frac=0.05) for s in range(S)] for k in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs, sizes = [], []
    for row in sets:
        streams = [oracle.compress(x, lut) for x in row]
        bufs.append([torch.frombuffer(bytearray(b), dtype=torch.uint8).cuda() for b in streams])
        sizes.append(torch.tensor([len(b) for b in streams], dtype=torch.int64, device="cuda"))
    ptrs = [torch.tensor([t.data_ptr() for t in row], dtype=torch.int64, device="cuda") for row in bufs]
    ys = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(4)]
    wsb = z.zccl_workspace_bytes(z.OP_DECOMPRESS_REDUCE, n, S)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    h = _handle()
    for i in range(4):
        k = i % 2
        z.check(z.zccl_decompress_reduce(ptrs[k].data_ptr(), sizes[k].data_ptr(), S, ys[i].data_ptr(), n,
                                         ws.data_ptr(), wsb, status.data_ptr(), h), "decompress_reduce")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = [oracle.decompress_reduce([oracle.compress(x, lut) for x in row], n) for row in sets]
    for i in range(4):
        assert np.array_equal(host_u16(ys[i]), want[i % 2]), f"call {i}"


def test_decompress_behind_compress(z):
    """compress then decompress of the same buffers, round after round with
    new data, with nothing in between."""
    n, rounds = 1_000_003, 3
    lut = z.zccl_lut_from_sigma(0.02)
    data = [workloads.gaussian(n, 0.02, seed=20 + r) for r in range(rounds)]
    xs = [dev_u16(d) for d in data]
    cap = z.zccl_max_compressed_bytes(n)
    out = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    nb = torch.zeros(1, dtype=torch.int64, device="cuda")
    ys = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(rounds)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = z.zccl_workspace_bytes(z.OP_COMPRESS, n)
    wsc = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    wsd = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    h = _handle()
    for r in range(rounds):
        z.check(z.zccl_compress(xs[r].data_ptr(), n, lut, out.data_ptr(), cap, nb.data_ptr(), wsc.data_ptr(), wsb,
                                status.data_ptr(), h), "compress")
        z.check(z.zccl_decompress(out.data_ptr(), cap, ys[r].data_ptr(), n, wsd.data_ptr(), wsb, status.data_ptr(),
                                  h), "decompress")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for r in range(rounds):
        assert np.array_equal(host_u16(ys[r]), data[r]), f"round {r}"
