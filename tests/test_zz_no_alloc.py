"""zc_compress_static_scratch: compression for callers that cannot allocate device memory.

A caller such as a communication layer whose send buffers are registered once, at exactly the
worst-case stream size, and that must not call cudaMalloc on its progress path (it can
synchronize the device, and it is not allowed during stream capture) cannot give zc_compress the
extra workspace it keeps in the tail of `out`.  The static-scratch entry point takes its
workspace from a fixed array inside the library instead.  These checks run it through the C ABI
and require its streams to equal zc_compress's streams byte for byte, on calls made one after
the other (the shared array must not carry anything over), and its size limit to be enforced.
"""
import ctypes

import numpy as np
import pytest

from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import require_gpu, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs():
    rng = np.random.default_rng(2024)
    a = workloads.fp32_to_bf16_bits((rng.standard_normal(3 * 4096 + 77) * 0.02).astype(np.float32))
    a[rng.choice(a.size, 500, replace=False)] = workloads.random_patterns(500, 1)
    b = workloads.sweep(20)  # larger, and a different window base
    return a, b


def _reference_stream(x):
    """The stream zc_compress writes for x (its `out` includes the workspace tail)."""
    out, ob = zc.compress(to_device(x))
    torch.cuda.synchronize()
    return out[:int(ob.item())].cpu().numpy()


def test_static_scratch_matches_compress_on_consecutive_calls():
    s = torch.cuda.current_stream().cuda_stream
    zc.status(reset=True)
    for x in _inputs():  # two calls in a row through the shared array
        want = _reference_stream(x)
        xd = to_device(x)
        out = torch.full((zc.zc_max_stream_bytes(x.size),), 0xEE, dtype=torch.uint8, device="cuda")
        ob = torch.zeros(1, dtype=torch.int64, device="cuda")
        assert zc.zc_compress_static_scratch(xd.data_ptr(), x.size, zc.ZC_BASE_AUTO, out.data_ptr(),
                                             ob.data_ptr(), s) == zc.ZC_OK
        assert zc.zc_status(s, 1) == zc.ZC_OK
        total = int(ob.item())
        assert total == want.size
        assert out[:total].cpu().numpy().tobytes() == want.tobytes()
        back = zc.decompress(out, x.size)
        assert zc.status(reset=True) == zc.ZC_OK
        assert np.array_equal(back.cpu().numpy().view(np.uint16), x)


def test_static_scratch_supplied_base_and_host_length():
    x = _inputs()[0]
    s = torch.cuda.current_stream().cuda_stream
    xd = to_device(x)
    out = torch.empty(zc.zc_max_stream_bytes(x.size), dtype=torch.uint8, device="cuda")
    length = ctypes.c_uint64(0)  # pageable host memory: the call copies the length back
    e0 = int(_reference_stream(x)[7])
    zc.status(reset=True)
    assert zc.zc_compress_static_scratch(xd.data_ptr(), x.size, e0, out.data_ptr(), ctypes.addressof(length),
                                         s) == zc.ZC_OK
    assert zc.zc_status(s, 1) == zc.ZC_OK
    want = _reference_stream(x)
    assert length.value == want.size
    assert out[:want.size].cpu().numpy().tobytes() == want.tobytes()


def test_static_scratch_rejects_sizes_beyond_its_limit():
    s = torch.cuda.current_stream().cuda_stream
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    big = zc.ZC_STATIC_SCRATCH_MAX_N + 1
    # rejected before any device memory is touched, so the (unused) addresses may be small
    assert zc.zc_compress_static_scratch(1 << 20, big, zc.ZC_BASE_AUTO, 1 << 24, ob.data_ptr(), s) == \
        zc.ZC_ERR_INVALID_ARG
