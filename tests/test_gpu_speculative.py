"""The speculative path (auto mode, tensors above the single-launch sizes), against the oracle,
through the C ABI.

Every CTA of the encode kernel reads the same sample -- 512 chunks spread evenly over the tensor,
chunk c giving its 16-byte vector (37 c + 11) mod 512 -- and guesses e0 from it; when it trusts
the guess it codes with it while summing the squares of every value exactly as the statistics
kernel does, and the CTA whose chunks complete the count applies the rule to the whole tensor's
sum.  When the rule settles the guessed e0 the stream is final; otherwise, or when the sample was
not trusted, the fallback word is set and the statistics kernel and the encode kernel run again
after it, as without the speculation.  Every stream must equal the oracle's byte for byte
whichever way it went; the fallback word (bytes 240..243 of the control block at the start of the
workspace, in the tail of `out`) tells which way that was.
"""
import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import require_gpu, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SINGLE_MAX = 1 << 25  # the largest tensor that compresses in one launch on a GB300


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def ctrl_word(out, n, offset):
    ws = (zc.zc_max_stream_bytes(n) + 255) // 256 * 256
    return int(out[ws + offset:ws + offset + 4].cpu().numpy().view(np.uint32)[0])


def compress_checked(x, base=-1):
    """(stream, kernels run, fallback word): the stream equal to the oracle's, decoded back."""
    xd = to_device(x)
    zc.zc_timing_enable(1)
    zc.zc_timing_collect()
    try:
        zc.status(reset=True)
        out, ob = zc.compress(xd, base)
        st = zc.status(reset=True)
        kernels = [k for k, _ in zc.zc_timing_collect()]
    finally:
        zc.zc_timing_enable(0)
    assert st == zc.ZC_OK, zc.ERROR_NAMES.get(st, st)
    total = int(ob.item())
    stream = out[:total].cpu().numpy()
    want = oracle.compress(x, base)
    assert stream[7] == want[7], f"e0 {stream[7]} vs oracle {want[7]}"
    assert stream.size == want.size, f"length {stream.size} vs oracle {want.size}"
    if stream.tobytes() != want.tobytes():
        diff = np.flatnonzero(stream != want)
        pytest.fail(f"stream differs from the oracle at {diff.size} bytes, first at {diff[0]}")
    back = zc.decompress(out, x.size)
    assert zc.status(reset=True) == zc.ZC_OK
    assert bool(torch.equal(back, xd))
    return stream, kernels, ctrl_word(out, x.size, 240)


def sampled_positions(n):
    """Start of every sampled vector."""
    full = n // 4096
    c = np.arange(512, dtype=np.int64) * full // 512
    return 4096 * c + 8 * ((37 * c + 11) % 512)


def gaussian(n, seed, sigma=1.0):
    rng = np.random.default_rng(seed)
    return workloads.fp32_to_bf16_bits((rng.standard_normal(n) * sigma).astype(np.float32))


SPEC_KERNELS = [zc.ZC_KERNEL_ENCODE, zc.ZC_KERNEL_REFIT_STATS, zc.ZC_KERNEL_REFIT_ENCODE, zc.ZC_KERNEL_RAW]


@pytest.mark.parametrize("n", [SINGLE_MAX + 1, SINGLE_MAX + 3 * 4096 + 5, 40_000_001, 3 * SINGLE_MAX])
def test_guess_holds(n):
    s, kernels, route = compress_checked(gaussian(n, n % 1000))
    assert kernels == SPEC_KERNELS
    assert route == 0 and s[6] == 12 and s[7] == 122


@pytest.mark.parametrize("log2_sigma,e0", [(-46, 76), (-34.5, 87), (58.5, 180), (62, 184)])
def test_guess_holds_at_every_scale(log2_sigma, e0):
    """The speculative sums take the plain fp32 squares only for e0 in [87, 180], where the
    window's squares are normal fp32 numbers; outside that range every block goes through the
    careful (scaled) block sum.  Both ends of the plain range and a scale beyond each: the guess
    holds and the stream is the oracle's."""
    x = gaussian(SINGLE_MAX + 4096 * 5 + 11, 12, 2.0 ** log2_sigma)
    s, kernels, route = compress_checked(x)
    assert kernels == SPEC_KERNELS
    assert route == 0 and s[6] == 12 and s[7] == e0


def test_gradient_bucket_is_not_speculated():
    """0.1% of the values are 100x the rest and make most of the sum of squares: a sample of 4096
    values estimates it far too loosely (relative standard error over 30%), so the encode kernel
    does not speculate."""
    x = workloads.make("grad_bucket_4096x14336")
    s, _, route = compress_checked(x)
    assert route == 1 and s[6] == 12 and s[7] == 114


def misleading_sample(n, seed):
    """N(0, 1) values whose sampled vectors are scaled by 1/4: the sample's e0 is 120, the
    tensor's 122."""
    x = gaussian(n, seed).view(np.uint16).copy()
    pos = sampled_positions(n)
    idx = (pos[:, None] + np.arange(8)[None, :]).ravel()
    v = (x[idx].astype(np.uint32) << 16).view(np.float32) * np.float32(0.25)
    x[idx] = workloads.fp32_to_bf16_bits(v)
    assert oracle.choose_e0(x) == 122
    return x


def test_guess_wrong_falls_back_to_the_coded_form():
    """The coding pass codes with the sample's 120, its own sums settle 122, and the statistics
    and encode kernels redo it."""
    x = misleading_sample(SINGLE_MAX + 4096 * 11 + 3, 7)
    s, _, route = compress_checked(x)
    assert route == 1 and s[6] == 12 and s[7] == 122


def test_guess_wrong_falls_back_to_the_raw_form():
    """One huge value outside the sample: the tensor's e0 is far above the sample's, almost every
    value escapes, and the stream is raw."""
    n = SINGLE_MAX + 77
    x = gaussian(n, 8)
    x[1] = workloads.fp32_to_bf16_bits(np.array([1e20], np.float32))[0]
    s, _, route = compress_checked(x)
    assert route == 1 and s[6] == 0


def test_guess_holds_and_the_stream_is_raw():
    """Outside the sampled vectors, 60% of the value pairs (a, b) become (sqrt(a^2 + b^2), 0): the
    sum of squares and the finite count barely move, so the sample's e0 (122) holds (and 70% of
    every CTA's values stay inside the window, so its fast sums are trusted), but 30% of the
    values are now zeros -- escapes below the window -- so every chunk's list makes the coded form
    longer than the raw one.  The raw-form step must write the raw form, the oracle's."""
    n = SINGLE_MAX + 4096 * 7 + 5
    f = (gaussian(n, 61).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    sampled = np.zeros(n, bool)
    sampled[(sampled_positions(n)[:, None] + np.arange(8)[None, :]).ravel()] = True
    a, b = f[0:n - 1:2].copy(), f[1:n:2].copy()
    pair = ~sampled[0:n - 1:2] & ~sampled[1:n:2] & (np.random.default_rng(62).random(n // 2) < 0.6)
    a[pair] = np.sign(a[pair]) * np.sqrt(a[pair] ** 2 + b[pair] ** 2)
    b[pair] = 0.0
    f[0:n - 1:2], f[1:n:2] = a, b
    x = workloads.fp32_to_bf16_bits(f.astype(np.float32))
    assert oracle.choose_e0(x) == 122
    s, kernels, route = compress_checked(x)
    assert kernels == SPEC_KERNELS
    assert route == 0 and s[6] == 0 and s[7] == 122


def test_sample_not_confident_on_random_patterns():
    """A sample that predicts a raw stream keeps the encode kernel from speculating at all."""
    n = SINGLE_MAX + 4096
    s, _, route = compress_checked(workloads.random_patterns(n, 3))
    assert route == 1 and s[6] == 0


def test_nonfinite_values_in_the_speculative_sums():
    n = SINGLE_MAX + 999
    x = gaussian(n, 9)
    x[::97] = 0x7FC0   # NaN
    x[5::4096] = 0xFF80  # -Inf
    s, _, route = compress_checked(x)
    assert route == 0 and s[6] == 12


def test_supplied_base_takes_no_speculation():
    x = gaussian(SINGLE_MAX + 5, 10)
    s, kernels, _ = compress_checked(x, base=122)
    assert kernels == [zc.ZC_KERNEL_ENCODE, zc.ZC_KERNEL_RAW]


def test_static_scratch_entry_takes_the_speculative_path():
    x = gaussian(SINGLE_MAX + 4096 + 1, 11)
    xd = to_device(x)
    out = torch.zeros(zc.zc_max_stream_bytes(x.size), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    zc.zc_timing_enable(1)
    zc.zc_timing_collect()
    try:
        zc.status(reset=True)
        s = torch.cuda.current_stream().cuda_stream
        assert zc.zc_compress_static_scratch(xd.data_ptr(), x.size, zc.ZC_BASE_AUTO, out.data_ptr(),
                                             ob.data_ptr(), s) == 0
        assert zc.status(reset=True) == zc.ZC_OK
        kernels = [k for k, _ in zc.zc_timing_collect()]
    finally:
        zc.zc_timing_enable(0)
    assert kernels == SPEC_KERNELS
    total = int(ob.item())
    assert out[:total].cpu().numpy().tobytes() == oracle.compress(x).tobytes()


@pytest.mark.parametrize("n", [3 * 4096 + 17, 40 * 4096 + 5, (1 << 21) + 4096 * 3 + 1, (1 << 23) + 9, (1 << 24) + 77])
def test_single_launch_own_e0_differs(n):
    """The cooperative grid codes each CTA's chunks at once with that CTA's own e0 (the rule at its
    own partial) and settles the tensor's e0 at the barrier that also publishes the sections'
    sizes.  Here the first half is N(0, 1) and the second N(0, 16^2): the halves' own e0 (122 and
    126) both differ from the tensor's (125), so the chunks are coded again with 125.  (The
    cluster and the L2-resident kernel settle e0 before coding: the same tensor as a check.)"""
    x = np.concatenate([gaussian(n // 2, 51), gaussian(n - n // 2, 52, 16.0)])
    assert oracle.choose_e0(x) == 125
    s, _, _ = compress_checked(x)
    assert s[6] == 12 and s[7] == 125


@pytest.mark.parametrize("n", [1, 7, 8, 4096 * 2 + 3, 40 * 4096 + 5, (1 << 20) + 3, (1 << 23) + 9, (1 << 25) - 5])
def test_single_launch_guess_holds(n):
    """Tiny to 2^25 - 5 values (every single-launch kernel): the stream, e0 included, is the
    oracle's."""
    compress_checked(gaussian(n, 41 + n % 89))


def test_concurrent_calls_on_two_streams():
    """Two large tensors compressed at once on two streams, each with its own buffers: the
    persistent encode kernels share the GPU, their CTAs wait only on work that running CTAs of
    their own launch have taken, and each stream must be the oracle's (one speculates, the
    other's sample is not trusted and takes the statistics route)."""
    xs = [gaussian(SINGLE_MAX + 4096 * 3 + 5, 71), workloads.make("grad_bucket_4096x14336")]
    devs = [to_device(x) for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    zc.status(reset=True)
    outs = []
    for xd, st in zip(devs, streams):
        with torch.cuda.stream(st):
            outs.append(zc.compress(xd, stream=st))
    torch.cuda.synchronize()
    assert zc.status(reset=True) == zc.ZC_OK
    for x, xd, (out, ob) in zip(xs, devs, outs):
        total = int(ob.item())
        want = oracle.compress(x)
        assert total == want.size and out[:total].cpu().numpy().tobytes() == want.tobytes()
        back = zc.decompress(out, x.size)
        assert zc.status(reset=True) == zc.ZC_OK
        assert bool(torch.equal(back, xd))
