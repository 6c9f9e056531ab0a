"""ctypes binding of ``libzc.so`` (the sm_103a codec library).

The functions below carry the C ABI's names and only marshal arguments; every step of the
codec runs in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzc.so")

ZC_OK = 0
ZC_ERR_INVALID_ARG = 1
ZC_ERR_MISALIGNED = 2
ZC_ERR_CUDA = 3
ZC_ERR_CORRUPT = 4
ZC_ERR_SIZE_MISMATCH = 5
ZC_ERR_TIMEOUT = 6
ZC_BASE_AUTO = -1
ZC_STATIC_SCRATCH_MAX_N = 1065222144
ZC_CHUNK_VALUES = 4096
ZC_KERNEL_STATS = 1
ZC_KERNEL_ENCODE = 2
ZC_KERNEL_DECODE = 3
ZC_KERNEL_RAW = 4
ZC_KERNEL_SMALL = 5
ZC_KERNEL_MEDIUM = 6
ZC_KERNEL_FUSED = 7
ZC_KERNEL_REFIT_STATS = 8
ZC_KERNEL_REFIT_ENCODE = 9

ERROR_NAMES = {
    ZC_OK: "ZC_OK",
    ZC_ERR_INVALID_ARG: "ZC_ERR_INVALID_ARG",
    ZC_ERR_MISALIGNED: "ZC_ERR_MISALIGNED",
    ZC_ERR_CUDA: "ZC_ERR_CUDA",
    ZC_ERR_CORRUPT: "ZC_ERR_CORRUPT",
    ZC_ERR_SIZE_MISMATCH: "ZC_ERR_SIZE_MISMATCH",
    ZC_ERR_TIMEOUT: "ZC_ERR_TIMEOUT",
}

# (name, restype, argtypes) of every exported entry point.
_SIG = {
    "zc_max_compressed_bytes": (ctypes.c_size_t, [ctypes.c_size_t]),
    "zc_max_stream_bytes": (ctypes.c_size_t, [ctypes.c_size_t]),
    "zc_compress": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p]),
    "zc_decompress": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "zc_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "zc_timing_enable": (ctypes.c_int, [ctypes.c_int]),
    "zc_timing_collect": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]),
    "zc_compress_static_scratch": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p]),
    "zc_compress_stall_test": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_uint]),
    "zc_loopback_bytes": (ctypes.c_size_t, [ctypes.c_size_t]),
    "zc_loopback": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "zc_loopback_stall_test": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_uint]),
}

_lock = threading.Lock()
_lib = None


class ZcError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ERROR_NAMES.get(code, code)}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libzc.so (built in-tree by ``build.build()``); raise if it is not there."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIG.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIG)


# ------------------------------------------------------------------ C ABI, same names


def zc_max_compressed_bytes(n: int) -> int:
    return int(lib().zc_max_compressed_bytes(n))


def zc_max_stream_bytes(n: int) -> int:
    return int(lib().zc_max_stream_bytes(n))


def zc_compress(in_ptr: int, n: int, base_or_auto: int, out_ptr: int, out_bytes_ptr: int, stream: int) -> int:
    return int(lib().zc_compress(in_ptr, n, base_or_auto, out_ptr, out_bytes_ptr, stream))


def zc_decompress(in_ptr: int, out_ptr: int, n: int, stream: int) -> int:
    return int(lib().zc_decompress(in_ptr, out_ptr, n, stream))


def zc_status(stream: int, reset: int = 0) -> int:
    return int(lib().zc_status(stream, reset))


def zc_timing_enable(enable: int) -> int:
    return int(lib().zc_timing_enable(enable))


def zc_timing_collect(max_records: int = 4096) -> list[tuple[int, float]]:
    ids = (ctypes.c_int * max_records)()
    ms = (ctypes.c_float * max_records)()
    k = int(lib().zc_timing_collect(ids, ms, max_records))
    if k < 0:
        raise ZcError(-k, "zc_timing_collect")
    return [(ids[i], ms[i]) for i in range(k)]


def zc_compress_static_scratch(in_ptr: int, n: int, base_or_auto: int, out_ptr: int, out_bytes_ptr: int,
                               stream: int) -> int:
    return int(lib().zc_compress_static_scratch(in_ptr, n, base_or_auto, out_ptr, out_bytes_ptr, stream))


def zc_compress_stall_test(in_ptr: int, n: int, base_or_auto: int, out_ptr: int, out_bytes_ptr: int,
                           stream: int, stalled_chunk: int, spin_limit: int) -> int:
    return int(lib().zc_compress_stall_test(in_ptr, n, base_or_auto, out_ptr, out_bytes_ptr, stream,
                                            stalled_chunk, spin_limit))


def zc_loopback_bytes(n: int) -> int:
    return int(lib().zc_loopback_bytes(n))


def zc_loopback(in_ptr: int, n: int, base_or_auto: int, out_ptr: int, out_bytes_ptr: int, values_ptr: int,
                stream: int) -> int:
    return int(lib().zc_loopback(in_ptr, n, base_or_auto, out_ptr, out_bytes_ptr, values_ptr, stream))


def zc_loopback_stall_test(in_ptr: int, n: int, base_or_auto: int, out_ptr: int, out_bytes_ptr: int,
                           values_ptr: int, stream: int, stalled_chunk: int, spin_limit: int) -> int:
    return int(lib().zc_loopback_stall_test(in_ptr, n, base_or_auto, out_ptr, out_bytes_ptr, values_ptr, stream,
                                            stalled_chunk, spin_limit))


# ------------------------------------------------------------------ torch conveniences


def _stream_handle(stream) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check(code: int, what: str) -> None:
    if code != ZC_OK:
        raise ZcError(code, what)


def compress(x, base: int = ZC_BASE_AUTO, stream=None, out=None, out_bytes=None):
    """Compress a CUDA tensor of BF16 values (dtype bfloat16, int16 or uint16).

    Returns (out, out_bytes): ``out`` is a uint8 CUDA tensor of capacity
    zc_max_compressed_bytes(n) holding the stream at its start, ``out_bytes`` a 1-element
    int64 CUDA tensor with the stream length (valid once the stream's work has run)."""
    import torch

    if not x.is_cuda or x.element_size() != 2:
        raise TypeError("compress expects a CUDA tensor of 16-bit values")
    x = x.contiguous()
    n = x.numel()
    cap = zc_max_compressed_bytes(n)
    if out is None:
        out = torch.empty(cap, dtype=torch.uint8, device=x.device)
    if out_bytes is None:
        out_bytes = torch.zeros(1, dtype=torch.int64, device=x.device)
    _check(zc_compress(x.data_ptr(), n, base, out.data_ptr(), out_bytes.data_ptr(), _stream_handle(stream)),
           "zc_compress")
    return out, out_bytes


def decompress(stream_bytes, n: int, stream=None, out=None):
    """Decompress a uint8 CUDA tensor holding a stream into n BF16 bit patterns (int16 tensor)."""
    import torch

    if out is None:
        out = torch.empty(n, dtype=torch.int16, device=stream_bytes.device)
    _check(zc_decompress(stream_bytes.data_ptr(), out.data_ptr(), n, _stream_handle(stream)), "zc_decompress")
    return out


def loopback(x, base: int = ZC_BASE_AUTO, stream=None):
    """Compress a CUDA tensor of BF16 values and decode the stream in the same launch.

    Returns (out, out_bytes, values): the stream at the start of ``out`` (uint8, capacity
    zc_loopback_bytes(n)), its length (1-element int64 CUDA tensor) and the decoded values
    (int16 CUDA tensor)."""
    import torch

    if not x.is_cuda or x.element_size() != 2:
        raise TypeError("loopback expects a CUDA tensor of 16-bit values")
    x = x.contiguous()
    n = x.numel()
    out = torch.empty(zc_loopback_bytes(n), dtype=torch.uint8, device=x.device)
    out_bytes = torch.zeros(1, dtype=torch.int64, device=x.device)
    values = torch.empty(max(n, 1), dtype=torch.int16, device=x.device)[:n]
    _check(zc_loopback(x.data_ptr(), n, base, out.data_ptr(), out_bytes.data_ptr(), values.data_ptr(),
                       _stream_handle(stream)), "zc_loopback")
    return out, out_bytes, values


def status(stream=None, reset: bool = False) -> int:
    return zc_status(_stream_handle(stream), 1 if reset else 0)
