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
