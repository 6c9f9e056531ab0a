"""The codec's calls captured once in a CUDA graph and replayed on new input contents.

A caller that runs the same message sizes every step (a training job's gradient buckets) can
capture its compress and decompress calls once and replay them, which drops the host's per-call
cost.  That works only if a call decides on the host nothing that depends on the values (the
route follows from n alone; e0, the escape sections and the stream's form are found on the
device), makes no allocation or synchronization while capturing, and resets its own device
state on every run.  Each test captures the calls for one size, then replays the graph on two
inputs of that size with different windows (and one that comes out raw), and requires every
replayed stream to equal the oracle's byte for byte and every decoded tensor to equal its input.
The sizes reach each route of a compress call: one cluster, the cooperative grid, the fused
L2-resident kernel and the speculative persistent encoder.
"""
import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SIZES = [3 * 4096 + 77, (1 << 20) + 333, (1 << 24) + 77, (1 << 25) + 3 * 4096 + 5]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(n):
    """Three inputs of n values: N(0, 1), N(0, 1e-3) (another e0), random bit patterns (raw)."""
    rng = np.random.default_rng(n % 100003)
    a = workloads.fp32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32))
    b = workloads.fp32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32) * np.float32(1e-3))
    c = workloads.random_patterns(n, 7 + n % 1000)
    return a, b, c


def _replay_each(g, xd, inputs, check):
    for x in inputs:
        xd.copy_(torch.from_numpy(x.view(np.int16)))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check(x)


def _capture(calls):
    """Capture `calls(stream_handle)` on a side stream into a new graph."""
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            calls(side.cuda_stream)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("n", SIZES)
def test_compress_and_decompress_replayed(n):
    inputs = _inputs(n)
    xd = torch.empty(n, dtype=torch.int16, device="cuda")
    out = torch.empty(zc.zc_max_compressed_bytes(n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    back = torch.empty(n, dtype=torch.int16, device="cuda")

    def calls(s):
        assert zc.zc_compress(xd.data_ptr(), n, zc.ZC_BASE_AUTO, out.data_ptr(), ob.data_ptr(), s) == zc.ZC_OK
        assert zc.zc_decompress(out.data_ptr(), back.data_ptr(), n, s) == zc.ZC_OK

    xd.copy_(torch.from_numpy(inputs[0].view(np.int16)))
    zc.status(reset=True)
    calls(torch.cuda.current_stream().cuda_stream)  # loads the kernels before the capture
    assert zc.status(reset=True) == zc.ZC_OK
    g = _capture(calls)

    def check(x):
        assert zc.status(reset=True) == zc.ZC_OK
        want = oracle.compress(x)
        total = int(ob.item())
        assert total == want.size
        assert out[:total].cpu().numpy().tobytes() == want.tobytes()
        assert np.array_equal(back.cpu().numpy().view(np.uint16), x)

    _replay_each(g, xd, inputs, check)
    del g


@pytest.mark.parametrize("n", [SIZES[0], SIZES[3]])
def test_static_scratch_replayed(n):
    """The entry point that allocates nothing: captured, it must also reset its shared array on
    every replay (the replays follow one another on one stream)."""
    inputs = _inputs(n)
    xd = torch.empty(n, dtype=torch.int16, device="cuda")
    out = torch.empty(zc.zc_max_stream_bytes(n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")

    def calls(s):
        assert zc.zc_compress_static_scratch(xd.data_ptr(), n, zc.ZC_BASE_AUTO, out.data_ptr(), ob.data_ptr(),
                                             s) == zc.ZC_OK

    xd.copy_(torch.from_numpy(inputs[1].view(np.int16)))
    zc.status(reset=True)
    calls(torch.cuda.current_stream().cuda_stream)  # the first call looks up the array's address
    assert zc.status(reset=True) == zc.ZC_OK
    g = _capture(calls)

    def check(x):
        assert zc.status(reset=True) == zc.ZC_OK
        want = oracle.compress(x)
        total = int(ob.item())
        assert total == want.size
        assert out[:total].cpu().numpy().tobytes() == want.tobytes()

    _replay_each(g, xd, inputs, check)
    del g


@pytest.mark.parametrize("n", [SIZES[1], SIZES[3]])
def test_loopback_replayed(n):
    inputs = _inputs(n)
    xd = torch.empty(n, dtype=torch.int16, device="cuda")
    out = torch.empty(zc.zc_loopback_bytes(n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    values = torch.empty(n, dtype=torch.int16, device="cuda")

    def calls(s):
        assert zc.zc_loopback(xd.data_ptr(), n, zc.ZC_BASE_AUTO, out.data_ptr(), ob.data_ptr(), values.data_ptr(),
                              s) == zc.ZC_OK

    xd.copy_(torch.from_numpy(inputs[0].view(np.int16)))
    zc.status(reset=True)
    calls(torch.cuda.current_stream().cuda_stream)
    assert zc.status(reset=True) == zc.ZC_OK
    g = _capture(calls)

    def check(x):
        assert zc.status(reset=True) == zc.ZC_OK
        want = oracle.compress(x)
        total = int(ob.item())
        assert total == want.size
        assert out[:total].cpu().numpy().tobytes() == want.tobytes()
        assert np.array_equal(values.cpu().numpy().view(np.uint16), x)

    _replay_each(g, xd, inputs, check)
    del g
