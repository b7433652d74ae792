"""Oracle for the lossless BF16 exponent codec -- TEST INFRASTRUCTURE ONLY.

The oracle is the plain C file ``zccl_oracle.c`` beside this module, compiled
with gcc into ``oracle/_build/libzccl_oracle.so`` and called through ctypes,
plus ``switcher.py``, the reduce-scatter switcher's time model in plain
Python (fp64).
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it and shares no code with it.

Each wrapper below names the section of the ZipCCL page ("ZipCCL: Efficient
Lossless Data Compression of Communication Collectives for Accelerating LLM
Training", technical summary) whose step the C function follows.

Parity pins live in ``tests/test_oracle_*.py``; every oracle function has at
least one pin that does not go through its own code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zccl_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libzccl_oracle.so")

OK, INVALID_ARG, TOO_SMALL, CORRUPT = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        sig = {
            "zo_lut_from_sigma": ([ctypes.c_double, u8p], ctypes.c_int),
            "zo_binade_mass": ([ctypes.c_double, ctypes.c_int], ctypes.c_double),
            "zo_zero_point_offset": ([ctypes.c_uint64], ctypes.c_uint64),
            "zo_stream_bytes": ([ctypes.c_uint64, ctypes.c_uint64], ctypes.c_uint64),
            "zo_max_bytes": ([ctypes.c_uint64], ctypes.c_uint64),
            "zo_compress": ([u16p, ctypes.c_uint64, u8p, u8p, ctypes.c_uint64, u64p],
                            ctypes.c_int),
            "zo_decompress": ([u8p, ctypes.c_uint64, u16p, ctypes.c_uint64], ctypes.c_int),
            "zo_decompress_reduce": ([ctypes.POINTER(u8p), u64p, ctypes.c_uint32, u16p,
                                      ctypes.c_uint64], ctypes.c_int),
            "zo_decompress_reduce_local": ([ctypes.POINTER(u8p), u64p, ctypes.c_uint32, u16p, ctypes.c_uint32,
                                            ctypes.c_int, u16p, ctypes.c_uint64], ctypes.c_int),
            "zo_exponent_histogram": ([u16p, ctypes.c_uint64, u64p], None),
            "zo_lut_from_histogram": ([u64p, u8p], ctypes.c_int),
            "zo_round_bf16": ([ctypes.c_float], ctypes.c_uint16),
            "zo_round_bf16_n": ([ctypes.POINTER(ctypes.c_float), u16p, ctypes.c_uint64], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} failed with status {status}")
        self.status = status


def lut_from_sigma(sigma: float) -> bytes:
    """ZipCCL 2.A: the 7 most probable BF16 exponents under N(0, sigma^2)."""
    lut = np.zeros(7, np.uint8)
    st = _load().zo_lut_from_sigma(float(sigma), _ptr(lut, ctypes.c_uint8))
    if st != OK:
        raise OracleError(st, "lut_from_sigma")
    return lut.tobytes()


def binade_mass(sigma: float, E: int) -> float:
    """ZipCCL 2.A: Gaussian mass of the binade with biased exponent E."""
    return _load().zo_binade_mass(float(sigma), int(E))


def zero_point_offset(n: int) -> int:
    return int(_load().zo_zero_point_offset(n))


def stream_bytes(n: int, n_esc: int) -> int:
    return int(_load().zo_stream_bytes(n, n_esc))


def max_bytes(n: int) -> int:
    return int(_load().zo_max_bytes(n))


def compress(x: np.ndarray, lut: bytes) -> bytes:
    """ZipCCL 2.B + 2.C: BF16 bit patterns (uint16) -> stream bytes."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    n = x.size
    cap = max_bytes(n)
    out = np.zeros(cap, np.uint8)
    lut_a = np.frombuffer(bytes(lut), np.uint8).copy()
    nbytes = ctypes.c_uint64(0)
    st = _load().zo_compress(_ptr(x, ctypes.c_uint16), n, _ptr(lut_a, ctypes.c_uint8),
                             _ptr(out, ctypes.c_uint8), cap, ctypes.byref(nbytes))
    if st != OK:
        raise OracleError(st, "compress")
    return out[: nbytes.value].tobytes()


def compress_batched(segments, lut: bytes):
    """ZipCCL 2.D static/dynamic parts: one independent stream per segment,
    compressed one after another."""
    return [compress(seg, lut) for seg in segments]


def decompress_status(stream, n: int):
    """(status, decoded uint16 array) of decoding ``stream``; never raises."""
    buf = np.frombuffer(bytes(stream), np.uint8).copy()
    x = np.zeros(max(n, 1), np.uint16)
    st = _load().zo_decompress(_ptr(buf, ctypes.c_uint8), buf.size, _ptr(x, ctypes.c_uint16), n)
    return int(st), x[:n]


def decompress(stream, n: int) -> np.ndarray:
    """Inverse of ZipCCL 2.B: stream bytes -> BF16 bit patterns (uint16)."""
    st, x = decompress_status(stream, n)
    if st != OK:
        raise OracleError(st, "decompress")
    return x


def decompress_reduce(streams, n: int) -> np.ndarray:
    """ZipCCL 2.D local reduction: decode S streams, add in fp32 in shard
    order, round to nearest-even BF16."""
    bufs = [np.frombuffer(bytes(s), np.uint8).copy() for s in streams]
    S = len(bufs)
    ptrs = (ctypes.POINTER(ctypes.c_uint8) * S)(*[_ptr(b, ctypes.c_uint8) for b in bufs])
    sizes = np.array([b.size for b in bufs], np.uint64)
    out = np.zeros(max(n, 1), np.uint16)
    st = _load().zo_decompress_reduce(ptrs, _ptr(sizes, ctypes.c_uint64), S,
                                      _ptr(out, ctypes.c_uint16), n)
    if st != OK:
        raise OracleError(st, "decompress_reduce")
    return out[:n]


def decompress_reduce_local(streams, n: int, local=None, local_pos: int = 0, initial=None) -> np.ndarray:
    """ZipCCL 2.D local reduction as one rank sees it: `streams` in rank
    order, where position local_pos is the rank's own uncompressed BF16
    shard `local` (its entry in `streams` is ignored); with `initial` (BF16
    bits) the fold starts from those values (accumulate into an existing
    output)."""
    S = len(streams)
    bufs = [np.frombuffer(bytes(s if s is not None else b"\0"), np.uint8).copy() for s in streams]
    ptrs = (ctypes.POINTER(ctypes.c_uint8) * S)(*[_ptr(b, ctypes.c_uint8) for b in bufs])
    sizes = np.array([b.size for b in bufs], np.uint64)
    out = np.zeros(max(n, 1), np.uint16)
    if initial is not None:
        out[:n] = np.asarray(initial, np.uint16)[:n]
    loc = None
    if local is not None:
        loc = np.ascontiguousarray(np.asarray(local, np.uint16)[:n])
        if loc.size == 0:
            loc = np.zeros(1, np.uint16)
    st = _load().zo_decompress_reduce_local(ptrs, _ptr(sizes, ctypes.c_uint64), S,
                                            _ptr(loc, ctypes.c_uint16) if loc is not None else None,
                                            local_pos, 1 if initial is not None else 0,
                                            _ptr(out, ctypes.c_uint16), n)
    if st != OK:
        raise OracleError(st, "decompress_reduce_local")
    return out[:n]


def round_bf16(f: float) -> int:
    """fp32 -> BF16 by distance, ties to even; NaN -> 0x7FC0."""
    return int(_load().zo_round_bf16(ctypes.c_float(f)))


def round_bf16_array(f: np.ndarray) -> np.ndarray:
    """Vector form of :func:`round_bf16`."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.zeros(max(f.size, 1), np.uint16)
    _load().zo_round_bf16_n(_ptr(f, ctypes.c_float), _ptr(out, ctypes.c_uint16), f.size)
    return out[: f.size]


def exponent_histogram(x) -> np.ndarray:
    """hist[e] = number of BF16 values with biased exponent e (0..255)."""
    x = np.ascontiguousarray(np.asarray(x, np.uint16))
    hist = np.zeros(256, np.uint64)
    buf = x if x.size else np.zeros(1, np.uint16)
    _load().zo_exponent_histogram(_ptr(buf, ctypes.c_uint16), x.size, _ptr(hist, ctypes.c_uint64))
    return hist


def lut_from_histogram(hist) -> bytes:
    """The 7 most frequent exponents, rank order, ties to the smaller one."""
    h = np.ascontiguousarray(np.asarray(hist, np.uint64))
    lut = np.zeros(7, np.uint8)
    st = _load().zo_lut_from_histogram(_ptr(h, ctypes.c_uint64), _ptr(lut, ctypes.c_uint8))
    if st != OK:
        raise OracleError(st, "lut_from_histogram")
    return lut.tobytes()
