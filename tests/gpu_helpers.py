"""Helpers for the GPU tests: move seeded host arrays through the C ABI and back."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from lossless_bf16_compression_gb300 import binding as zc  # noqa: E402


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zc.lib()


def to_device(x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def gpu_round_trip(x: np.ndarray, base: int = -1):
    """Compress and decompress on the GPU; return (status, stream bytes, decoded values)."""
    xd = to_device(x)
    zc.status(reset=True)
    out, out_bytes = zc.compress(xd, base)
    back = zc.decompress(out, x.size)
    st = zc.status(reset=True)
    total = int(out_bytes.item())
    return st, out[:total].cpu().numpy(), back.cpu().numpy().view(np.uint16)


def gpu_compress(x: np.ndarray, base: int = -1):
    xd = to_device(x)
    zc.status(reset=True)
    out, out_bytes = zc.compress(xd, base)
    st = zc.status(reset=True)
    return st, out, int(out_bytes.item())


def gpu_decompress_bytes(stream: np.ndarray, n: int, capacity: int):
    """Decompress host stream bytes placed at the start of a zeroed device buffer of
    `capacity` bytes (so every read the kernel may make stays inside the buffer)."""
    buf = torch.zeros(max(capacity, stream.size, 48), dtype=torch.uint8, device="cuda")
    buf[:stream.size] = torch.from_numpy(stream)
    zc.status(reset=True)
    out = zc.decompress(buf, n)
    st = zc.status(reset=True)
    return st, out.cpu().numpy().view(np.uint16)
