"""Codec: a thin convenience layer over the zccl_* C calls.

It allocates outputs and the workspace with PyTorch (device memory and
streams only) and passes raw device addresses to libzccl; all codec work runs
in the library's kernels.  Inputs are BF16 tensors (or 16-bit integer views
of BF16 bit patterns) on the current CUDA device.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (OP_COMPRESS, OP_COMPRESS_BATCHED, OP_DECOMPRESS, OP_DECOMPRESS_REDUCE, OK,
               ZcclError, check, zccl_compress, zccl_compress_batched, zccl_decompress,
               zccl_decompress_reduce, zccl_decompress_reduce_local, zccl_decompress_split,
               zccl_exponent_histogram,
               zccl_lut_from_histogram, zccl_max_compressed_bytes, zccl_workspace_bytes)

SEGMENT_DTYPE = np.dtype([("in", "<u8"), ("n", "<u8"), ("out", "<u8"), ("cap", "<u8")])


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _as_u16_ptr(x: torch.Tensor) -> int:
    if x.element_size() != 2 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("expected a contiguous 16-bit CUDA tensor (BF16 bit patterns)")
    return x.data_ptr()


class Codec:
    """Owns a workspace and a device status word; one instance per stream."""

    def __init__(self, device=None, stream=None):
        self.device = torch.device(device if device is not None else "cuda")
        self.stream = stream
        self._ws = None
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    # -- workspace ------------------------------------------------------------
    def workspace(self, nbytes: int):
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self._ws.data_ptr(), self._ws.numel()

    def reset_status(self):
        self.status.zero_()

    def read_status(self) -> int:
        return int(self.status.item())

    def check_status(self, what="device"):
        st = self.read_status()
        if st != OK:
            raise ZcclError(st, what)

    # -- calls ----------------------------------------------------------------
    def compress(self, x: torch.Tensor, lut: bytes, out: torch.Tensor | None = None,
                 out_bytes: torch.Tensor | None = None):
        """Returns (stream buffer uint8 of max size, device int64 size tensor)."""
        n = x.numel()
        cap = zccl_max_compressed_bytes(n)
        if out is None:
            out = torch.empty(cap, dtype=torch.uint8, device=self.device)
        if out_bytes is None:
            out_bytes = torch.zeros(1, dtype=torch.int64, device=self.device)
        ws, wsb = self.workspace(zccl_workspace_bytes(OP_COMPRESS, n))
        check(zccl_compress(_as_u16_ptr(x) if n else 0, n, lut, out.data_ptr(), out.numel(),
                            out_bytes.data_ptr(), ws, wsb, self.status.data_ptr(),
                            _stream_handle(self.stream)), "zccl_compress")
        return out, out_bytes

    def decompress(self, stream_buf: torch.Tensor, in_bytes: int, n: int,
                   out: torch.Tensor | None = None) -> torch.Tensor:
        if out is None:
            out = torch.empty(max(n, 1), dtype=torch.int16, device=self.device)[:n]
        ws, wsb = self.workspace(zccl_workspace_bytes(OP_DECOMPRESS, n))
        check(zccl_decompress(stream_buf.data_ptr(), in_bytes, out.data_ptr() if n else 0, n, ws,
                              wsb, self.status.data_ptr(), _stream_handle(self.stream)),
              "zccl_decompress")
        return out

    def decompress_split(self, frame: torch.Tensor, tail: torch.Tensor | None, tail_bytes: int, n: int,
                         out: torch.Tensor | None = None):
        """Decompress a stream held as its frame (header + blocks, exactly
        zccl_zero_point_offset(n) bytes) and its zero-point tail, apart."""
        if out is None:
            out = torch.empty(max(n, 1), dtype=torch.int16, device=self.device)[:n]
        ws, wsb = self.workspace(zccl_workspace_bytes(OP_DECOMPRESS, n))
        check(zccl_decompress_split(frame.data_ptr(), tail.data_ptr() if tail is not None and tail_bytes else 0,
                                    tail_bytes, out.data_ptr() if n else 0, n, ws, wsb, self.status.data_ptr(),
                                    _stream_handle(self.stream)), "zccl_decompress_split")
        return out

    def segment_table(self, segments) -> torch.Tensor:
        """Device array of zccl_segment_t from [(in_tensor, out_tensor), ...]."""
        tab = np.zeros(len(segments), SEGMENT_DTYPE)
        for i, (x, o) in enumerate(segments):
            tab[i] = (x.data_ptr() if x.numel() else 0, x.numel(), o.data_ptr(), o.numel())
        host = torch.from_numpy(tab.view(np.uint8).copy())
        return host.to(self.device, non_blocking=False)

    def compress_batched(self, segments, lut: bytes, total_n: int | None = None,
                         table: torch.Tensor | None = None, out_bytes: torch.Tensor | None = None):
        """segments: [(in_tensor, out_tensor)]; returns the device size array."""
        k = len(segments)
        if total_n is None:
            total_n = sum(x.numel() for x, _ in segments)
        if table is None:
            table = self.segment_table(segments)
        if out_bytes is None:
            out_bytes = torch.zeros(k, dtype=torch.int64, device=self.device)
        ws, wsb = self.workspace(zccl_workspace_bytes(OP_COMPRESS_BATCHED, total_n, k))
        check(zccl_compress_batched(table.data_ptr(), k, total_n, lut, out_bytes.data_ptr(), ws,
                                    wsb, self.status.data_ptr(), _stream_handle(self.stream)),
              "zccl_compress_batched")
        return out_bytes

    def decompress_reduce(self, streams, in_bytes, n: int, out: torch.Tensor | None = None):
        """streams: list of uint8 stream tensors; in_bytes: list of sizes or a
        device int64 tensor."""
        S = len(streams)
        ptrs = torch.tensor([s.data_ptr() for s in streams], dtype=torch.int64).to(self.device)
        if not torch.is_tensor(in_bytes):
            in_bytes = torch.tensor(list(in_bytes), dtype=torch.int64).to(self.device)
        if out is None:
            out = torch.empty(max(n, 1), dtype=torch.int16, device=self.device)[:n]
        ws, wsb = self.workspace(zccl_workspace_bytes(OP_DECOMPRESS_REDUCE, n, S))
        check(zccl_decompress_reduce(ptrs.data_ptr(), in_bytes.data_ptr(), S,
                                     out.data_ptr() if n else 0, n, ws, wsb,
                                     self.status.data_ptr(), _stream_handle(self.stream)),
              "zccl_decompress_reduce")
        self._keep = (ptrs, in_bytes)  # alive until the next call
        return out

    def decompress_reduce_local(self, streams, in_bytes, n: int, local: torch.Tensor | None = None,
                                local_pos: int = 0, out: torch.Tensor | None = None, accumulate: bool = False):
        """Like decompress_reduce, with the rank's own shard `local` (plain
        BF16, 16-bit tensor) at position local_pos (its entry in `streams`
        is ignored and may be None) and, with accumulate, the fold starting
        from the values already in `out`."""
        S = len(streams)
        ptrs = torch.tensor([0 if st is None else st.data_ptr() for st in streams], dtype=torch.int64)
        ptrs = ptrs.to(self.device)
        if not torch.is_tensor(in_bytes):
            in_bytes = torch.tensor([int(v) for v in in_bytes], dtype=torch.int64).to(self.device)
        if out is None:
            if accumulate:
                raise ValueError("accumulate needs an existing out")
            out = torch.empty(max(n, 1), dtype=torch.int16, device=self.device)[:n]
        ws, wsb = self.workspace(zccl_workspace_bytes(OP_DECOMPRESS_REDUCE, n, S))
        check(zccl_decompress_reduce_local(ptrs.data_ptr(), in_bytes.data_ptr(), S,
                                           _as_u16_ptr(local) if local is not None and n else 0, local_pos,
                                           1 if accumulate else 0, out.data_ptr() if n else 0, n, ws, wsb,
                                           self.status.data_ptr(), _stream_handle(self.stream)),
              "zccl_decompress_reduce_local")
        self._keep = (ptrs, in_bytes)
        return out

    def exponent_histogram(self, x: torch.Tensor, hist: torch.Tensor | None = None,
                           accumulate: bool = False) -> torch.Tensor:
        """256 exponent counts of the BF16 tensor x, as an int64 device tensor
        (the library writes unsigned 64-bit counts); with accumulate, added
        to the counts already in `hist`."""
        if hist is None:
            if accumulate:
                raise ValueError("accumulate needs an existing hist")
            hist = torch.empty(256, dtype=torch.int64, device=self.device)
        n = x.numel()
        check(zccl_exponent_histogram(_as_u16_ptr(x) if n else 0, n, hist.data_ptr(), accumulate,
                                      _stream_handle(self.stream)), "zccl_exponent_histogram")
        return hist

    def lut_from_data(self, x: torch.Tensor) -> bytes:
        """The LUT of x's 7 most frequent exponents (one histogram pass on the
        device, the selection on the host)."""
        return zccl_lut_from_histogram(self.exponent_histogram(x).cpu().numpy().view(np.uint64))
