"""GPU parity of the batched compression of ragged MoE segments (ZipCCL
technical summary 2.D: per-expert static part + dynamic remainder), one
launch for all segments; every segment's stream must equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_u16, load_lib, require_gpu
from lossless_bf16_exponent_split_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def z():
    require_gpu()
    load_lib()
    import lossless_bf16_exponent_split_gb300 as z
    return z


def run_batched(z, payload_dev, hidden, segments, lut, total_n=None, caps=None):
    codec = z.Codec()
    pairs = []
    for i, (r0, rows) in enumerate(segments):
        n = rows * hidden
        x = payload_dev[r0 * hidden: r0 * hidden + n]
        cap = z.zccl_max_compressed_bytes(n) if caps is None else caps[i]
        pairs.append((x, torch.zeros(cap + 256, dtype=torch.uint8, device="cuda")[:cap]))
    codec.reset_status()
    nb = codec.compress_batched(pairs, lut, total_n=total_n)
    torch.cuda.synchronize()
    return codec.read_status(), nb.cpu().numpy(), [o for _, o in pairs]


def check_segments(payload, hidden, segments, lut, nb, outs, skip=()):
    for i, (r0, rows) in enumerate(segments):
        if i in skip:
            assert nb[i] == 0
            continue
        x = payload[r0 * hidden:(r0 + rows) * hidden]
        want = oracle.compress(x, lut)
        assert nb[i] == len(want), i
        assert outs[i][: len(want)].cpu().numpy().tobytes() == want, i


def test_small_moe(z):
    m = workloads.moe_payload(tokens=512, top_k=4, experts=16, hidden=192, seed=5)
    lut = oracle.lut_from_sigma(1.0)
    st, nb, outs = run_batched(z, dev_u16(m.payload), m.hidden, m.segments, lut)
    assert st == 0
    check_segments(m.payload, m.hidden, m.segments, lut, nb, outs)


def test_ragged_sizes_and_empty_segments(z):
    rng = np.random.default_rng(7)
    hidden = 1
    sizes = [0, 1, 7, 4096, 4097, 0, 12_345, 33, 8192, 0, 70_001, 5]
    rows = []
    r0 = 0
    # segment starts padded to 8 elements so every input is 16-byte aligned
    for n in sizes:
        rows.append((r0, n))
        r0 += -(-n // 8) * 8
    payload = workloads.special_values(r0, seed=8)
    lut = oracle.lut_from_sigma(0.5)
    st, nb, outs = run_batched(z, dev_u16(payload), hidden, rows, lut)
    assert st == 0
    check_segments(payload, hidden, rows, lut, nb, outs)


def test_invalid_segments_skipped(z):
    hidden = 1
    rows = [(0, 5000), (5000, 3000), (8000, 9000), (17000, 100)]
    payload = workloads.gaussian(17100, 1.0, seed=2)
    lut = oracle.lut_from_sigma(1.0)
    caps = [oracle.max_bytes(n) for _, n in rows]
    caps[1] -= 1  # too small -> BUFFER_TOO_SMALL, segment skipped
    st, nb, outs = run_batched(z, dev_u16(payload), hidden, rows, lut, caps=caps)
    assert st == z.BUFFER_TOO_SMALL
    check_segments(payload, hidden, rows, lut, nb, outs, skip=(1,))


def test_total_n_undercount_rejected(z):
    hidden = 1
    rows = [(0, 50_000), (50_000, 50_000)]
    payload = workloads.gaussian(100_000, 1.0, seed=2)
    st, nb, _ = run_batched(z, dev_u16(payload), hidden, rows, oracle.lut_from_sigma(1.0),
                            total_n=10_000)
    assert st == z.INVALID_ARG


def test_moe_a2a_full(z):
    cfg = workloads.CONFIGS["moe_a2a"]
    m = workloads.moe_payload(tokens=cfg["tokens"], top_k=cfg["top_k"], experts=cfg["experts"],
                              hidden=cfg["hidden"], seed=0)
    lut = oracle.lut_from_sigma(cfg["sigma"])
    st, nb, outs = run_batched(z, dev_u16(m.payload), m.hidden, m.segments, lut)
    assert st == 0
    check_segments(m.payload, m.hidden, m.segments, lut, nb, outs)
