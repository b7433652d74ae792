"""Host logic of bench.py that decides what is measured (no GPU)."""
import bench


def test_decompress_offset_avoids_l2_resident_stream():
    for R in (3, 4, 5):
        for warmup in range(3, 12):
            for steps in range(1, 64):
                off = bench.decompress_offset(warmup, steps, R)
                assert off in (-1, 1)
                # the first timed decompress reads a buffer other than the one
                # the last timed compress wrote
                last_written = (warmup + steps) % R
                assert (warmup + 1 + off) % R != last_written
                # interleaved single launches: compress k, then decompress
                # (k + off), never the buffer just written
                assert off % R != 0


def test_decompress_offset_prefers_previous_stream():
    # K not a multiple of 3 with R = 3: the previous step's stream
    assert bench.decompress_offset(5, 30, 3) == 1      # 35 % 3 == 5 % 3: the conflict case
    assert bench.decompress_offset(5, 31, 3) == -1
    assert bench.decompress_offset(3, 2, 3) == -1


def test_group_bounds_cover_every_launch_once():
    for steps in range(1, 200):
        b = bench.group_bounds(steps)
        assert b[0] == 0 and b[-1] == steps
        assert len(b) - 1 == min(steps, 6)
        sizes = [b[i + 1] - b[i] for i in range(len(b) - 1)]
        assert all(x >= 1 for x in sizes)
        assert max(sizes) - min(sizes) <= 1


def test_every_workload_is_a_bench_choice_with_a_kind(monkeypatch):
    """Each entry of the workload table is accepted by --workload and maps to
    one of the measurement kinds (the generators are stubbed, so no payload
    is built)."""
    import sys
    from lossless_bf16_exponent_split_gb300 import workloads as w
    tiny = w.gaussian(16, 0.02, seed=0)
    monkeypatch.setattr(w, "gaussian", lambda n, sigma, seed=0: tiny)
    monkeypatch.setattr(w, "activation_mix", lambda *a, **k: tiny)
    monkeypatch.setattr(w, "moe_payload", lambda **k: type("M", (), {"payload": tiny})())
    monkeypatch.setattr(w, "reduce_shards", lambda S, n, sigma, seed=0: [tiny] * S)
    for name in w.CONFIGS:
        monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", name])
        assert bench.parse_args().workload == name
        assert bench.make_inputs(name, 0)[0] in ("roundtrip", "histogram", "batched", "reduce")
    assert bench.make_inputs("gauss268m", 0)[0] == "roundtrip"
    assert w.CONFIGS["gauss268m"]["n"] == 1 << 28
    assert "gauss268m" not in bench.CONFIG_WORKLOADS  # opt-in: not part of the default run
