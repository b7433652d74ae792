"""Helpers for the GPU tests: device buffers from oracle inputs and back."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def load_lib():
    """Builds (if needed) and loads libzccl; the GPU tests must use it."""
    from lossless_bf16_exponent_split_gb300 import build, lib
    build.build()
    return lib()


def dev_u16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.uint16).view(np.int16)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def dev_bytes(b: bytes, pad: int = 0) -> torch.Tensor:
    t = torch.zeros(len(b) + pad, dtype=torch.uint8)
    if b:
        t[: len(b)] = torch.frombuffer(bytearray(b), dtype=torch.uint8)
    return t.cuda()


def stream_of(out: torch.Tensor, out_bytes: torch.Tensor) -> bytes:
    nb = int(out_bytes.item())
    return out[:nb].cpu().numpy().tobytes()
