"""Pins of the oracle's encoder/decoder (ZipCCL technical summary 2.B, 2.C).

Independent pins: the hand-built stream fixture (byte layout), exhaustive
round trips over every BF16 bit pattern, escape counts and stream sizes
derived here with numpy from the page's "11 bits per element + full 8-bit
exponent for each zero-point" statement, and the corrupt-stream rules.
"""
import numpy as np
import pytest

import oracle
from golden_io import read_stream_fixture
from lossless_bf16_exponent_split_gb300 import workloads

ALL_PATTERNS = np.arange(65536, dtype=np.uint16)
LUTS = {
    "sigma1": oracle.lut_from_sigma(1.0),
    "sigma0.02": oracle.lut_from_sigma(0.02),
    "zero_inf": bytes([0, 255, 1, 2, 3, 254, 127]),     # holds exponents 0 and 255
    "absent": bytes([200, 201, 202, 203, 204, 205, 206]),
}


def expected_size(n, n_esc):
    """Header 128 B, then per chunk of 4096 slots (tail slots rounded up to
    1024) one sign-mantissa byte + 3 code bits per slot, then one byte per
    escape padded to 128 B."""
    full, tail = divmod(n, 4096)
    slots = full * 4096 + (-(-tail // 1024) * 1024)
    return 128 + slots * 11 // 8 + (-(-n_esc // 128) * 128)


def independent_escape_count(x, lut):
    return int((~np.isin((x >> 7) & 0xFF, np.frombuffer(lut, np.uint8))).sum())


def test_hand_built_fixture_encodes_and_decodes():
    x, lut, stream = read_stream_fixture()
    assert oracle.compress(x, lut) == stream
    assert np.array_equal(oracle.decompress(stream, x.size), x)


@pytest.mark.parametrize("name", list(LUTS))
def test_all_bf16_patterns_round_trip(name):
    lut = LUTS[name]
    s = oracle.compress(ALL_PATTERNS, lut)
    assert np.array_equal(oracle.decompress(s, ALL_PATTERNS.size), ALL_PATTERNS)
    n_esc = independent_escape_count(ALL_PATTERNS, lut)
    assert n_esc == 65536 - 7 * 256          # each LUT exponent covers 256 patterns
    assert int.from_bytes(s[16:24], "little") == n_esc
    assert len(s) == expected_size(65536, n_esc)


@pytest.mark.parametrize("name", list(LUTS))
def test_every_pattern_alone(name):
    """Each of the 65,536 patterns as a 1-element stream (a tail chunk)."""
    lut = LUTS[name]
    lutset = set(lut)
    for v in range(0, 65536, 1):
        if v % 97 and v not in (0, 0x7F80, 0xFF80, 0x7FC0, 0x8000):
            continue
        x = np.array([v], np.uint16)
        s = oracle.compress(x, lut)
        esc = 0 if ((v >> 7) & 0xFF) in lutset else 1
        assert len(s) == expected_size(1, esc)
        assert oracle.decompress(s, 1)[0] == v


@pytest.mark.parametrize("n", [0, 1, 7, 8, 31, 32, 33, 1023, 1024, 1025, 4095, 4096, 4097,
                               8191, 8192, 12289, 65536 + 17])
def test_sizes_and_round_trip(n):
    x = workloads.gaussian(n, 0.02, seed=n)
    lut = LUTS["sigma0.02"]
    s = oracle.compress(x, lut)
    n_esc = independent_escape_count(x, lut)
    assert len(s) == expected_size(n, n_esc)
    assert len(s) == oracle.stream_bytes(n, n_esc)
    assert oracle.max_bytes(n) == expected_size(n, n)
    assert np.array_equal(oracle.decompress(s, n), x)


def test_empty_stream_is_header_only():
    s = oracle.compress(np.zeros(0, np.uint16), LUTS["sigma1"])
    assert len(s) == 128
    assert s[:4] == b"ZCCL"[::1] and int.from_bytes(s[32:40], "little") == 128


def test_escape_extremes():
    x = workloads.gaussian(10000, 1.0, seed=3)
    # LUT without any exponent present in the data: everything escapes
    s = oracle.compress(x, LUTS["absent"])
    assert len(s) == oracle.max_bytes(x.size)
    # data made only of LUT exponents: nothing escapes
    lut = LUTS["sigma1"]
    e = np.frombuffer(lut, np.uint8).astype(np.uint16)
    y = (e[np.arange(10000) % 7] << 7) | (np.arange(10000, dtype=np.uint16) & 0x807F)
    s = oracle.compress(y, lut)
    assert int.from_bytes(s[16:24], "little") == 0
    assert len(s) == expected_size(10000, 0)
    assert np.array_equal(oracle.decompress(s, 10000), y)


def test_compression_ratio_near_page_figure():
    """16 -> 11 bits (about 31 % saved) plus one byte per escape: at
    sigma = 0.02 (2.13 % escapes) the ratio is about 11/16 + 0.0213/2."""
    x = workloads.gaussian(1 << 20, 0.02, seed=0)
    s = oracle.compress(x, LUTS["sigma0.02"])
    r = len(s) / (2 * x.size)
    assert abs(r - (11 / 16 + 0.02126 / 2)) < 1e-3
    assert 0.30 < 1 - 11 / 16 < 0.32


def test_plane_bits_match_codes():
    """Reads the planes back with numpy's bit unpacking and compares them with
    codes computed from exponents (rank in the LUT + 1, else 0)."""
    n = 4096 * 2 + 1500
    x = workloads.special_values(n, seed=5)
    lut = LUTS["sigma1"]
    s = np.frombuffer(oracle.compress(x, lut), np.uint8)
    lut_a = np.frombuffer(lut, np.uint8)
    e = (x >> 7) & 0xFF
    codes = np.zeros(n, np.uint8)
    for r in range(7):
        codes[e == lut_a[r]] = r + 1
    pos = 128
    for c0 in range(0, n, 4096):
        cnt = min(4096, n - c0)
        L = 4096 if cnt == 4096 else -(-cnt // 1024) * 1024
        sm = s[pos:pos + L]
        assert np.array_equal(sm[:cnt], (((x[c0:c0 + cnt] >> 8) & 0x80) | (x[c0:c0 + cnt] & 0x7F)).astype(np.uint8))
        assert not sm[cnt:].any()
        got = np.zeros(L, np.uint8)
        for p in range(3):
            bits = np.unpackbits(s[pos + L + p * L // 8: pos + L + (p + 1) * L // 8], bitorder="little")
            got |= (bits << p).astype(np.uint8)
        assert np.array_equal(got[:cnt], codes[c0:c0 + cnt])
        assert not got[cnt:].any()
        pos += L * 11 // 8
    esc = e[codes == 0].astype(np.uint8)
    assert np.array_equal(s[pos:pos + esc.size], esc)


def _corrupt(stream, off, val):
    b = bytearray(stream)
    b[off] = val
    return bytes(b)


def test_corrupt_streams_rejected():
    x = workloads.gaussian(5000, 1.0, seed=1)
    s = oracle.compress(x, LUTS["sigma1"])
    n = x.size
    assert oracle.decompress_status(s, n)[0] == oracle.OK
    assert int.from_bytes(s[16:24], "little") % 128 != 0   # last byte is padding
    bad = {
        "magic": _corrupt(s, 0, 0x00),
        "version": _corrupt(s, 4, 2),
        "log2chunk": _corrupt(s, 6, 11),
        "n": _corrupt(s, 8, s[8] ^ 1),
        "n_esc_up": _corrupt(s, 16, s[16] + 1),
        "n_esc_down": _corrupt(s, 16, s[16] - 1),
        "zp_offset": _corrupt(s, 32, s[32] ^ 0x80),
        "dup_lut": _corrupt(s, 25, s[24]),
        "reserved": _corrupt(s, 100, 1),
        "padding_slot": _corrupt(s, 128 + 4096 * 11 // 8 + 950, 1),
        "padding_plane": _corrupt(s, 128 + 4096 * 11 // 8 + 1024 + 127, 0x80),
        "zp_padding": _corrupt(s, len(s) - 1, 7),
        "truncated": s[:-128],
        "short_header": s[:64],
    }
    for name, b in bad.items():
        assert oracle.decompress_status(b, n)[0] == oracle.CORRUPT, name
    # wrong n requested by the caller
    assert oracle.decompress_status(s, n + 1)[0] == oracle.CORRUPT


def test_invalid_lut_rejected():
    with pytest.raises(oracle.OracleError) as e:
        oracle.compress(np.zeros(4, np.uint16), bytes([1, 1, 2, 3, 4, 5, 6]))
    assert e.value.status == oracle.INVALID_ARG
