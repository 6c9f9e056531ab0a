"""zc_compress_static_scratch: compression for callers that cannot allocate device memory.

A caller such as a communication layer whose send buffers are registered once, at exactly the
worst-case stream size, and that must not call cudaMalloc on its progress path (it can
synchronize the device, and it is not allowed during stream capture) cannot give zc_compress the
extra workspace it keeps in the tail of `out`.  The static-scratch entry point takes its
workspace from a fixed array inside the library instead.  These checks run it through the C ABI
and require its streams to equal the oracle's byte for byte on calls made one after the other
(the shared array must not carry anything over), the device's free memory to stay the same
across those calls, its writes to stay inside zc_max_stream_bytes(n) bytes of `out`, and its
size limit to be enforced.
"""
import ctypes

import numpy as np
import pytest

import oracle
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


def _static_call(xd, n, base, out, ob_ptr):
    s = torch.cuda.current_stream().cuda_stream
    rc = zc.zc_compress_static_scratch(xd.data_ptr(), n, base, out.data_ptr(), ob_ptr, s)
    torch.cuda.synchronize()
    return rc, zc.zc_status(s, 1)


def test_static_scratch_matches_oracle_on_consecutive_calls():
    inputs = _inputs()
    wants = [oracle.compress(x) for x in inputs]
    devs = [to_device(x) for x in inputs]
    outs = [torch.full((zc.zc_max_stream_bytes(x.size),), 0xEE, dtype=torch.uint8, device="cuda") for x in inputs]
    obs = [torch.zeros(1, dtype=torch.int64, device="cuda") for _ in inputs]
    backs = [torch.empty(x.size, dtype=torch.int16, device="cuda") for x in inputs]
    zc.status(reset=True)
    # a first call loads the library's kernels (and with them its device arrays) on this device
    assert _static_call(devs[1], inputs[1].size, zc.ZC_BASE_AUTO, outs[1], obs[1].data_ptr()) == (zc.ZC_OK, zc.ZC_OK)
    for x, xd, out, ob, want in zip(inputs, devs, outs, obs, wants):  # two calls in a row
        free_before = torch.cuda.mem_get_info()[0]
        assert _static_call(xd, x.size, zc.ZC_BASE_AUTO, out, ob.data_ptr()) == (zc.ZC_OK, zc.ZC_OK)
        assert torch.cuda.mem_get_info()[0] == free_before, "the call changed the device's free memory"
        total = int(ob.item())
        assert total == want.size
        assert out[:total].cpu().numpy().tobytes() == want.tobytes()
    for x, out, back in zip(inputs, outs, backs):
        zc.decompress(out, x.size, out=back)
        assert zc.status(reset=True) == zc.ZC_OK
        assert np.array_equal(back.cpu().numpy().view(np.uint16), x)


def test_static_scratch_supplied_base_and_host_length():
    x = _inputs()[0]
    want = oracle.compress(x, 116)
    xd = to_device(x)
    out = torch.empty(zc.zc_max_stream_bytes(x.size), dtype=torch.uint8, device="cuda")
    length = ctypes.c_uint64(0)  # pageable host memory: the call copies the length back
    zc.status(reset=True)
    assert _static_call(xd, x.size, 116, out, ctypes.addressof(length)) == (zc.ZC_OK, zc.ZC_OK)
    assert length.value == want.size
    assert out[:want.size].cpu().numpy().tobytes() == want.tobytes()


@pytest.mark.parametrize("n", [2 * 4096 + 50, 3 * 4096, 40 * 4096 + 50, 70 * 4096 + 50])
def test_static_scratch_stays_inside_its_stream_bound(n):
    """Random bit patterns give the longest stream n values can give (the raw form: written after
    the coded form was found longer by the single-launch path for small tensors, and by the raw
    pass beyond); 4 KiB of 0xA5 right before `out` and right after zc_max_stream_bytes(n) bytes
    of it must survive."""
    G = 4096
    x = workloads.random_patterns(n, 600 + n)
    want = oracle.compress(x)
    cap = zc.zc_max_stream_bytes(n)
    buf = torch.full((G + cap + G,), 0xA5, dtype=torch.uint8, device="cuda")
    out = buf[G:G + cap]
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    zc.status(reset=True)
    assert _static_call(to_device(x), n, zc.ZC_BASE_AUTO, out, ob.data_ptr()) == (zc.ZC_OK, zc.ZC_OK)
    h = buf.cpu().numpy()
    assert np.all(h[:G] == 0xA5) and np.all(h[G + cap:] == 0xA5), "a guard band was written"
    total = int(ob.item())
    assert total == want.size == cap
    assert h[G:G + total].tobytes() == want.tobytes()


def test_static_scratch_rejects_sizes_beyond_its_limit():
    s = torch.cuda.current_stream().cuda_stream
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    big = zc.ZC_STATIC_SCRATCH_MAX_N + 1
    # rejected before any device memory is touched, so the (unused) addresses may be small
    assert zc.zc_compress_static_scratch(1 << 20, big, zc.ZC_BASE_AUTO, 1 << 24, ob.data_ptr(), s) == \
        zc.ZC_ERR_INVALID_ARG
