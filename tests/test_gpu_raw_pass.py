"""The raw pass, against the oracle, through the C ABI.

In auto mode the statistics pass also counts the exponents of a sample (two values in every 256)
and predicts the coded stream's length from the sample's share of escapes.  When the prediction
is clearly past the raw form's length, the encode kernel first counts every chunk's escapes exactly
while it copies the values to their place in the raw form, and keeps the form that the rule
gives: the raw form when the coded one is longer, else (ties included) the coded form, which the
encode kernel then writes over the copy.  A prediction only picks the route, so every stream
must equal the oracle's byte for byte whichever route was taken; the control block at the start
of the workspace (the tail of `out`) tells which one was (`raw_predicted` at byte 80,
`raw_done` at byte 84).
"""
import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import gpu_compress, require_gpu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def raw_bytes(n):
    return 32 + (2 * n + 15) // 16 * 16


def compress_and_route(x, base=-1):
    """GPU stream (checked against the oracle and decoded back) and (raw_predicted, raw_done)."""
    st, out, total = gpu_compress(x, base)
    assert st == zc.ZC_OK, zc.ERROR_NAMES.get(st, st)
    stream = out[:total].cpu().numpy()
    want = oracle.compress(x, base)
    assert stream.size == want.size, f"length {stream.size} vs oracle {want.size}"
    if stream.tobytes() != want.tobytes():
        diff = np.flatnonzero(stream != want)
        pytest.fail(f"stream differs from the oracle at {diff.size} bytes, first at {diff[0]}")
    back = zc.decompress(out, x.size)
    assert zc.status(reset=True) == zc.ZC_OK
    assert np.array_equal(back.cpu().numpy().view(np.uint16), x)
    ws = (zc.zc_max_stream_bytes(x.size) + 255) // 256 * 256
    flags = out[ws + 80:ws + 88].cpu().numpy().view(np.uint32)
    return stream, (int(flags[0]), int(flags[1]))


def in_window(rng, k):
    """k values of exponent 127 (magnitudes in [1, 2)): inside the window [122, 128] that the
    tensors below get."""
    return ((rng.integers(0, 2, k) << 15) | (127 << 7) | rng.integers(0, 128, k)).astype(np.uint16)


def tiny(rng, k):
    """k values of exponent 20: escapes that add almost nothing to the sum of squares."""
    return ((rng.integers(0, 2, k) << 15) | (20 << 7) | rng.integers(0, 128, k)).astype(np.uint16)


def planes_and_list(planes, list_k, extra=0, chunks=16400, tail=0, seed=7):
    """`planes` chunks of escapes only (each keeps a 4096-byte plane), then one chunk with
    list_k escapes, one with `extra`, the rest (and a ragged tail of `tail` values) with none."""
    rng = np.random.default_rng(seed)
    parts = []
    for c in range(chunks):
        x = in_window(rng, 4096)
        k = 4096 if c < planes else (list_k if c == planes else (extra if c == planes + 1 else 0))
        if k:
            pos = rng.choice(4096, k, replace=False)
            x[pos] = tiny(rng, k)
        parts.append(x)
    parts.append(in_window(rng, tail))
    return np.concatenate(parts)


# (tensors beyond the single-launch paths -- 2^26 values on a GB300 -- which decide the form from
# exact sizes before writing)
@pytest.mark.parametrize("n", [(1 << 26) + 1, (1 << 26) + 77, 16500 * 4096, 16500 * 4096 + 8, 70_000_001])
def test_random_patterns_take_the_raw_pass(n):
    x = workloads.random_patterns(n, 900 + n % 1000)
    s, route = compress_and_route(x)
    assert route == (1, 1), "the raw pass did not write the stream"
    assert s[6] == 0 and s.size == raw_bytes(n)
    assert s[32:32 + 2 * n].tobytes() == x.tobytes()


def test_gaussian_tensor_is_not_predicted_raw():
    x = workloads.sweep(20)
    s, route = compress_and_route(x)
    assert route == (0, 0)
    assert s[6] == 12


def test_prediction_raw_but_coded_is_shorter():
    """5200 of 16400 chunks escape everywhere and keep planes (one byte per value): the sample
    sees ~32% escapes, which at three bytes each would make the coded stream longer, but the
    planes make it shorter.  The exact count keeps the coded form."""
    x = planes_and_list(5200, 100, tail=1000)
    s, route = compress_and_route(x)
    assert route == (1, 0), "the sample did not predict a raw stream, or the raw form was kept"
    assert s[6] == 12 and s.size < raw_bytes(x.size)


def test_tie_after_the_raw_pass_keeps_the_coded_form():
    """10217 plane chunks and one list of 1317 escapes (3951 bytes, padded to 3952) make the coded
    stream exactly as long as the raw form (134,348,832 bytes): the coded form is kept.  One
    escape more, in another chunk, makes it 16 bytes longer: the raw form."""
    x = planes_and_list(10217, 1317)
    s, route = compress_and_route(x)
    assert route == (1, 0)
    assert s[6] == 12 and s.size == raw_bytes(x.size)
    x = planes_and_list(10217, 1317, extra=1)
    s, route = compress_and_route(x)
    assert route == (1, 1)
    assert s[6] == 0 and s.size == raw_bytes(x.size)


def test_supplied_base_takes_no_prediction():
    """With e0 supplied there is no statistics pass: a raw stream comes from the raw-form step
    after coding, and it is the same stream."""
    x = workloads.random_patterns(67_200_003, 31)
    s, route = compress_and_route(x, base=int(oracle.choose_e0(x)))
    assert route == (0, 0)
    assert s[6] == 0
    s_auto, route = compress_and_route(x)
    assert route == (1, 1) and s_auto.tobytes() == s.tobytes()


def test_raw_pass_length_on_the_host():
    """The length reaches pageable host memory through the control block as well."""
    import ctypes

    x = workloads.random_patterns(67_200_000, 77)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    out = torch.empty(zc.zc_max_compressed_bytes(x.size), dtype=torch.uint8, device="cuda")
    length = ctypes.c_uint64(0)
    zc.status(reset=True)
    s = torch.cuda.current_stream().cuda_stream
    assert zc.zc_compress(xd.data_ptr(), x.size, zc.ZC_BASE_AUTO, out.data_ptr(), ctypes.addressof(length), s) == 0
    assert zc.status(reset=True) == zc.ZC_OK
    assert length.value == raw_bytes(x.size)
    assert out[:length.value].cpu().numpy().tobytes() == oracle.compress(x).tobytes()
