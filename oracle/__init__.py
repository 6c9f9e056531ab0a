"""Plain single-threaded reference of the lossless BF16 exponent codec (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its binding) never
imports this package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` do.  The C source (``zc_oracle.c``) shares nothing with the CUDA library.

Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution", first technique --
exponent coding with a window taken from the tensor's standard deviation -- and the third
technique's switch to the native form where coding does not pay.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libzc_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_INVALID_ARG = 1
ERR_CORRUPT = 4
ERR_SIZE_MISMATCH = 5
ERR_CAPACITY = 7


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no fused multiply-add contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "zc_oracle.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, c_int, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            for name in ("zco_num_chunks", "zco_records_base", "zco_max_stream_bytes", "zco_raw_stream_bytes"):
                getattr(lib, name).argtypes = [u64]
                getattr(lib, name).restype = u64
            lib.zco_record_bytes.argtypes = [u64, u64]
            lib.zco_record_bytes.restype = u64
            lib.zco_window_constant.argtypes = []
            lib.zco_window_constant.restype = ctypes.c_double
            lib.zco_sum_squares.argtypes = [p, u64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(u64)]
            lib.zco_sum_squares.restype = c_int
            lib.zco_select_e0.argtypes = [ctypes.c_double, u64]
            lib.zco_select_e0.restype = c_int
            lib.zco_choose_e0.argtypes = [p, u64]
            lib.zco_choose_e0.restype = c_int
            lib.zco_compress.argtypes = [p, u64, c_int, p, u64]
            lib.zco_compress.restype = i64
            lib.zco_decompress.argtypes = [p, u64, p, u64]
            lib.zco_decompress.restype = c_int
            _lib = lib
    return _lib


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 BF16 bit patterns, got {a.dtype}")
    return a.reshape(-1)


def num_chunks(n: int) -> int:
    return int(_load().zco_num_chunks(n))


def records_base(n: int) -> int:
    return int(_load().zco_records_base(n))


def record_bytes(m: int, k: int) -> int:
    return int(_load().zco_record_bytes(m, k))


def max_stream_bytes(n: int) -> int:
    return int(_load().zco_max_stream_bytes(n))


def raw_stream_bytes(n: int) -> int:
    return int(_load().zco_raw_stream_bytes(n))


def window_constant() -> float:
    return float(_load().zco_window_constant())


def sum_squares(x) -> tuple[float, int]:
    a = _u16(x)
    s = ctypes.c_double()
    nf = ctypes.c_uint64()
    _load().zco_sum_squares(a.ctypes.data, a.size, ctypes.byref(s), ctypes.byref(nf))
    return s.value, nf.value


def select_e0(S_d: float, n_f: int) -> int:
    return int(_load().zco_select_e0(S_d, n_f))


def choose_e0(x) -> int:
    a = _u16(x)
    return int(_load().zco_choose_e0(a.ctypes.data, a.size))


def compress(x, base: int = -1) -> np.ndarray:
    """Return the stream (uint8 array) for BF16 bit patterns x with window base ``base``
    (-1 = from the data)."""
    a = _u16(x)
    cap = max_stream_bytes(a.size)
    out = np.empty(cap, dtype=np.uint8)
    r = _load().zco_compress(a.ctypes.data, a.size, base, out.ctypes.data, cap)
    if r < 0:
        raise ValueError(f"oracle compress failed with status {-r}")
    return out[:r].copy()


def decompress(stream, n: int) -> tuple[int, np.ndarray]:
    """Return (status, values).  values is meaningful only when status == OK."""
    s = np.ascontiguousarray(stream, dtype=np.uint8).reshape(-1)
    out = np.zeros(max(n, 1), dtype=np.uint16)
    st = _load().zco_decompress(s.ctypes.data, s.size, out.ctypes.data, n)
    return int(st), out[:n]
