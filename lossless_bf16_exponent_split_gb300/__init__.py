"""lossless_bf16_exponent_split_gb300 -- Python binding of libzccl, the GB300
lossless BF16 exponent codec ("ZipCCL: Efficient Lossless Data Compression of
Communication Collectives for Accelerating LLM Training", technical summary
2.A-2.D).

The functions named ``zccl_*`` mirror the C ABI in ``include/zccl.h`` one to
one: they only marshal arguments (integers are device addresses, streams are
``cudaStream_t`` handles as integers) and return the C status code.  Every step
of the codec runs in the library's CUDA kernels; there is no Python or CPU
fallback -- if ``libzccl.so`` is missing, every call raises.

``Codec`` is a convenience layer over the same calls that allocates buffers
with PyTorch (device memory and streams only).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

OK, INVALID_ARG, BUFFER_TOO_SMALL, CORRUPT_STREAM, CUDA_ERROR, TIMEOUT = range(6)
OP_COMPRESS, OP_DECOMPRESS, OP_COMPRESS_BATCHED, OP_DECOMPRESS_REDUCE = range(4)
POLL_COUNTER, POLL_FLAG = 1, 2
MAX_SEGMENTS = 4096
MAX_SHARDS = 1024
CHUNK = 4096
NOALLOC_SCRATCH_BYTES = 1 << 20
NOALLOC_MAX_ELEMS = 502267904

LIB_PATH = _build.LIB
_lib = None
_lock = threading.Lock()

# C function signatures: name -> (argtypes, restype)
_u8p = ctypes.c_void_p
_SIGS = {
    "zccl_lut_from_sigma": ([ctypes.c_double, ctypes.c_void_p], ctypes.c_int),
    "zccl_max_compressed_bytes": ([ctypes.c_uint64], ctypes.c_uint64),
    "zccl_zero_point_offset": ([ctypes.c_uint64], ctypes.c_uint64),
    "zccl_workspace_bytes": ([ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32,
                              ctypes.POINTER(ctypes.c_uint64)], ctypes.c_int),
    "zccl_workspace_init": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p], ctypes.c_int),
    "zccl_compress": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64,
                       ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "zccl_decompress": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_uint64,
                         ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p],
                        ctypes.c_int),
    "zccl_decompress_split": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                               ctypes.c_uint64, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                               ctypes.c_void_p], ctypes.c_int),
    "zccl_compress_batched": ([ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                               ctypes.c_void_p], ctypes.c_int),
    "zccl_decompress_reduce": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p,
                                ctypes.c_uint64, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                ctypes.c_void_p], ctypes.c_int),
    "zccl_decompress_reduce_local": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p,
                                      ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64,
                                      ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p],
                                     ctypes.c_int),
    "zccl_decompress_noalloc": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_uint64,
                                 ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "zccl_check_bounded_wait": ([ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "zccl_check_bounded_poll": ([ctypes.c_int, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                                ctypes.c_int),
    "zccl_exponent_histogram": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int,
                                 ctypes.c_void_p], ctypes.c_int),
    "zccl_lut_from_histogram": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "zccl_lut_from_data": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                           ctypes.c_int),
    "zccl_rs_plan": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "zccl_status_string": ([ctypes.c_int], ctypes.c_char_p),
}


class RsModel(ctypes.Structure):
    """zccl_rs_model_t"""
    _fields_ = [("ranks", ctypes.c_uint32), ("bytes", ctypes.c_uint64), ("ratio", ctypes.c_double),
                ("link_gbs", ctypes.c_double), ("link_latency_us", ctypes.c_double),
                ("compress_gbs", ctypes.c_double), ("compress_fixed_us", ctypes.c_double),
                ("reduce_gbs", ctypes.c_double), ("reduce_fixed_us", ctypes.c_double)]


class RsPlan(ctypes.Structure):
    """zccl_rs_plan_t"""
    _fields_ = [("zipped", ctypes.c_int), ("native_us", ctypes.c_double), ("zipped_us", ctypes.c_double),
                ("breakeven_link_gbs", ctypes.c_double)]


class ZcclError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libzccl (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libzccl not built ({LIB_PATH} missing): run "
                                   "lossless_bf16_exponent_split_gb300.build.build()")
            cdll = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(cdll, name)
                fn.argtypes = args
                fn.restype = res
            _lib = cdll
        return _lib


def _lut_buf(lut) -> ctypes.Array:
    b = bytes(lut)
    if len(b) != 7:
        raise ValueError("a LUT is 7 exponent bytes")
    return (ctypes.c_uint8 * 7)(*b)


# ---- the C ABI, one to one ---------------------------------------------------
def zccl_lut_from_sigma(sigma: float) -> bytes:
    buf = (ctypes.c_uint8 * 7)()
    st = lib().zccl_lut_from_sigma(float(sigma), ctypes.byref(buf))
    if st != OK:
        raise ZcclError(st, "zccl_lut_from_sigma")
    return bytes(buf)


def zccl_max_compressed_bytes(n: int) -> int:
    return int(lib().zccl_max_compressed_bytes(n))


def zccl_zero_point_offset(n: int) -> int:
    return int(lib().zccl_zero_point_offset(n))


def zccl_workspace_bytes(op: int, n: int, k: int = 0) -> int:
    out = ctypes.c_uint64(0)
    st = lib().zccl_workspace_bytes(op, n, k, ctypes.byref(out))
    if st != OK:
        raise ZcclError(st, "zccl_workspace_bytes")
    return int(out.value)


def zccl_workspace_init(d_ws: int, ws_bytes: int, stream: int) -> int:
    return lib().zccl_workspace_init(d_ws, ws_bytes, stream)


def zccl_compress(d_in, n, lut, d_out, out_capacity, d_out_bytes, d_ws, ws_bytes, d_status,
                  stream) -> int:
    return lib().zccl_compress(d_in, n, ctypes.byref(_lut_buf(lut)), d_out, out_capacity,
                               d_out_bytes, d_ws, ws_bytes, d_status, stream)


def zccl_decompress(d_in, in_bytes, d_out, n, d_ws, ws_bytes, d_status, stream) -> int:
    return lib().zccl_decompress(d_in, in_bytes, d_out, n, d_ws, ws_bytes, d_status, stream)


def zccl_decompress_split(d_frame, d_tail, tail_bytes, d_out, n, d_ws, ws_bytes, d_status, stream) -> int:
    """zccl_decompress of a stream held as its fixed-size frame (the first
    zccl_zero_point_offset(n) bytes) and its zero-point tail, apart."""
    return lib().zccl_decompress_split(d_frame, d_tail, tail_bytes, d_out, n, d_ws, ws_bytes, d_status, stream)


def zccl_compress_batched(d_segs, n_segs, total_n, lut, d_out_bytes, d_ws, ws_bytes, d_status,
                          stream) -> int:
    return lib().zccl_compress_batched(d_segs, n_segs, total_n, ctypes.byref(_lut_buf(lut)),
                                       d_out_bytes, d_ws, ws_bytes, d_status, stream)


def zccl_decompress_reduce(d_streams, d_in_bytes, S, d_out, n, d_ws, ws_bytes, d_status,
                           stream) -> int:
    return lib().zccl_decompress_reduce(d_streams, d_in_bytes, S, d_out, n, d_ws, ws_bytes,
                                        d_status, stream)


def zccl_decompress_reduce_local(d_streams, d_in_bytes, S, d_local, local_pos, accumulate, d_out, n, d_ws,
                                 ws_bytes, d_status, stream) -> int:
    """zccl_decompress_reduce with the rank's own shard as plain BF16 at
    local_pos (d_local may be 0 for none) and, with accumulate, the fold
    starting from the values already in d_out."""
    return lib().zccl_decompress_reduce_local(d_streams, d_in_bytes, S, d_local, local_pos, accumulate, d_out,
                                              n, d_ws, ws_bytes, d_status, stream)


def zccl_exponent_histogram(d_in, n, d_hist, accumulate, stream) -> int:
    """256 uint64 exponent counts of n BF16 values into device d_hist
    (added to the counts there when accumulate is true)."""
    return lib().zccl_exponent_histogram(d_in, n, d_hist, 1 if accumulate else 0, stream)


def zccl_lut_from_histogram(hist) -> bytes:
    """The 7 most frequent exponents of a host histogram (256 counts)."""
    import numpy as _np
    h = _np.ascontiguousarray(_np.asarray(hist, _np.uint64))
    if h.size != 256:
        raise ValueError("a histogram has 256 counts")
    lut = (ctypes.c_uint8 * 7)()
    check(lib().zccl_lut_from_histogram(h.ctypes.data, ctypes.addressof(lut)), "zccl_lut_from_histogram")
    return bytes(lut)


def zccl_lut_from_data(d_in, n, d_hist, stream) -> bytes:
    """The measured LUT of n BF16 values (d_hist: 2 KB device scratch);
    synchronises the stream."""
    lut = (ctypes.c_uint8 * 7)()
    check(lib().zccl_lut_from_data(d_in, n, d_hist, ctypes.addressof(lut), stream), "zccl_lut_from_data")
    return bytes(lut)


def zccl_decompress_noalloc(d_in, in_bytes, d_out, n, d_status, stream) -> int:
    """zccl_decompress without a caller workspace (static 1 MiB device
    scratch inside the library; for callers that cannot allocate)."""
    return lib().zccl_decompress_noalloc(d_in, in_bytes, d_out, n, d_status, stream)


def zccl_check_bounded_wait(limit_us, d_status, stream) -> int:
    return lib().zccl_check_bounded_wait(limit_us, d_status, stream)


def zccl_check_bounded_poll(kind, limit_us, d_word, d_status, stream) -> int:
    return lib().zccl_check_bounded_poll(kind, limit_us, d_word, d_status, stream)


def zccl_rs_plan(ranks, nbytes, ratio, link_gbs, link_latency_us, compress_gbs, compress_fixed_us,
                 reduce_gbs, reduce_fixed_us) -> dict:
    """The switcher's choice and both paths' modelled times (host only)."""
    m = RsModel(ranks, nbytes, ratio, link_gbs, link_latency_us, compress_gbs, compress_fixed_us, reduce_gbs,
                reduce_fixed_us)
    p = RsPlan()
    check(lib().zccl_rs_plan(ctypes.addressof(m), ctypes.addressof(p)), "zccl_rs_plan")
    return {"zipped": bool(p.zipped), "native_us": p.native_us, "zipped_us": p.zipped_us,
            "breakeven_link_gbs": p.breakeven_link_gbs}


def zccl_status_string(status: int) -> str:
    return lib().zccl_status_string(status).decode()


def status_string(status: int) -> str:
    try:
        return zccl_status_string(status)
    except Exception:  # library missing: still give a readable message
        return "unknown"


def check(status: int, what: str) -> None:
    if status != OK:
        raise ZcclError(status, what)


from .codec import Codec  # noqa: E402  (torch-based convenience layer)

__all__ = [n for n in list(globals()) if n.startswith("zccl_")] + [
    "Codec", "ZcclError", "check", "lib", "status_string"]
