"""The C ABI library without a GPU: it builds for sm_103a, loads, exports every entry point
include/zc.h declares, and its pure host functions and host-side argument checks behave."""
import ctypes
import os
import re

import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import build as zbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return zc.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "zc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:size_t|int|void)\s+(zc_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(zc.exported_symbols()) == names


def test_binding_constants_match_the_header():
    """Every numeric #define of include/zc.h that the binding names has the header's value."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "zc.h")).read(), flags=re.S)
    defines = {k: int(v, 0) for k, v in re.findall(r"^#define\s+(ZC_\w+)\s+\(?(-?\w+)\)?\s*$", text, flags=re.M)
               if re.fullmatch(r"-?(0x[0-9a-fA-F]+|\d+)[uUlL]*", v) and not v.endswith(("u", "U", "l", "L"))}
    assert {"ZC_OK", "ZC_ERR_TIMEOUT", "ZC_KERNEL_SMALL", "ZC_BASE_AUTO"} <= set(defines)
    for name, value in defines.items():
        if hasattr(zc, name):
            assert getattr(zc, name) == value, name
    for name in ("ZC_KERNEL_STATS", "ZC_KERNEL_ENCODE", "ZC_KERNEL_DECODE", "ZC_KERNEL_RAW", "ZC_KERNEL_SMALL",
                 "ZC_KERNEL_MEDIUM", "ZC_KERNEL_FUSED", "ZC_KERNEL_REFIT_STATS", "ZC_KERNEL_REFIT_ENCODE"):
        assert getattr(zc, name) == defines[name]


def _pad16(v):
    return (v + 15) // 16 * 16


def _fixed_region_end(n):
    """End of the coded form's fixed parts: header, table, then 5632 B per full chunk."""
    N = (n + 4095) // 4096
    rem = n % 4096
    return _pad16(32 + 8 * (N + 1)) + (n // 4096) * 5632 + (_pad16((3 * rem + 7) // 8) + _pad16(rem) if rem else 0)


def test_max_stream_bytes_matches_oracle(lib):
    """Room for the stream: the longest stream (the raw form, the oracle's bound) or the coded
    fixed parts, whichever ends later."""
    for n in [0, 1, 7, 8, 50, 100, 4095, 4096, 4097, 10 ** 6, 58_720_256, 117_440_512, 268_435_456, 1 << 29]:
        assert oracle.max_stream_bytes(n) == oracle.raw_stream_bytes(n) == 32 + _pad16(2 * n)
        assert zc.zc_max_stream_bytes(n) == max(oracle.max_stream_bytes(n), _fixed_region_end(n))
        N = (n + 4095) // 4096
        assert zc.zc_max_compressed_bytes(n) >= zc.zc_max_stream_bytes(n) + 8 * N
    assert zc.zc_max_stream_bytes(1) == 80 > oracle.max_stream_bytes(1) == 48  # tiny n: the fixed parts
    assert zc.zc_max_stream_bytes(1000) == oracle.max_stream_bytes(1000)


def test_max_stream_bytes_closed_form_large(lib):
    n = (1 << 40) - 3
    assert zc.zc_max_stream_bytes(n) == 32 + _pad16(2 * n)


def test_sizes_beyond_limit(lib):
    assert zc.zc_max_stream_bytes((1 << 40) + 1) == 0
    assert zc.zc_max_compressed_bytes((1 << 40) + 1) == 0


def test_host_argument_checks(lib):
    A = 1 << 20  # an aligned fake address; never dereferenced by these calls
    out_len = ctypes.c_uint64()
    p_len = ctypes.addressof(out_len)
    assert zc.zc_compress(0, 10, -1, A, p_len, 0) == zc.ZC_ERR_INVALID_ARG       # null input
    assert zc.zc_compress(A, 10, -1, 0, p_len, 0) == zc.ZC_ERR_INVALID_ARG       # null output
    assert zc.zc_compress(A, 10, -1, A * 4, 0, 0) == zc.ZC_ERR_INVALID_ARG       # null length
    assert zc.zc_compress(A, 10, 250, A * 4, p_len, 0) == zc.ZC_ERR_INVALID_ARG  # base too big
    assert zc.zc_compress(A, 10, -2, A * 4, p_len, 0) == zc.ZC_ERR_INVALID_ARG
    assert zc.zc_compress(A, (1 << 40) + 1, -1, A * 4, p_len, 0) == zc.ZC_ERR_INVALID_ARG
    assert zc.zc_compress(A + 2, 10, -1, A * 4, p_len, 0) == zc.ZC_ERR_MISALIGNED
    assert zc.zc_compress(A, 10, -1, A * 4 + 8, p_len, 0) == zc.ZC_ERR_MISALIGNED
    assert zc.zc_compress(A, 10, -1, A * 4, p_len + 4, 0) == zc.ZC_ERR_MISALIGNED
    assert zc.zc_compress(A, 100, -1, A + 64, p_len, 0) == zc.ZC_ERR_INVALID_ARG  # overlap
    assert zc.zc_decompress(0, A, 10, 0) == zc.ZC_ERR_INVALID_ARG
    assert zc.zc_decompress(A, 0, 10, 0) == zc.ZC_ERR_INVALID_ARG
    assert zc.zc_decompress(A + 8, A * 4, 10, 0) == zc.ZC_ERR_MISALIGNED
    assert zc.zc_decompress(A, A + 16, 100, 0) == zc.ZC_ERR_INVALID_ARG          # overlap


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-GPU failure path")
def test_no_gpu_fails_loudly(lib):
    A = 1 << 20
    out_len = ctypes.c_uint64()
    # valid arguments reach the CUDA runtime, which reports that there is no device
    assert zc.zc_compress(A, 10, -1, A * 4, ctypes.addressof(out_len), 0) == zc.ZC_ERR_CUDA
    assert zc.zc_decompress(A, A * 4, 10, 0) == zc.ZC_ERR_CUDA
