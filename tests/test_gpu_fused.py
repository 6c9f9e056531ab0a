"""The L2-resident single launch (tensors above the medium size, up to 2^25 values), against the
oracle, through the C ABI.

That kernel reads the input three times in one cooperative grid -- the sum of squares, an exact
escape count per chunk, then the coding -- and writes every part of the stream straight to its
place, having known the stream's form and every offset before the first byte.  Each case checks
the stream byte for byte against the oracle, decodes it back, and checks from the library's own
timing records that this kernel, alone, compressed the tensor (the one above 2^25 must not).
"""
import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import require_gpu, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FUSED_MAX = 1 << 25          # the largest tensor the L2-resident launch takes on a GB300
MEDIUM_MAX = 2432 * 4096     # the largest one of the medium launch (608 resident CTAs)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def raw_bytes(n):
    return 32 + (2 * n + 15) // 16 * 16


def compress_checked(x, base=-1):
    """The GPU stream, equal to the oracle's and decoded back; the library kernels it ran."""
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
    assert stream.size == want.size, f"length {stream.size} vs oracle {want.size}"
    if stream.tobytes() != want.tobytes():
        diff = np.flatnonzero(stream != want)
        pytest.fail(f"stream differs from the oracle at {diff.size} bytes, first at {diff[0]}")
    back = zc.decompress(out, x.size)
    assert zc.status(reset=True) == zc.ZC_OK
    assert bool(torch.equal(back, xd))
    return stream, kernels, out


def mixed(n, seed, frac=0.02):
    """N(0, 1) values (window [122, 128]); a fraction `frac` scaled by 2^-40 .. 2^3 (escapes
    below the window, a few above); every 37th chunk scaled by 2^-30 (escapes only: a plane)."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n).astype(np.float32)
    k = int(n * frac)
    pos = rng.choice(n, k, replace=False)
    v[pos] *= np.float32(2.0) ** rng.integers(-40, 4, k).astype(np.float32)
    for c in range(5, (n + 4095) // 4096, 37):
        v[4096 * c:4096 * (c + 1)] *= np.float32(2.0 ** -30)
    return workloads.fp32_to_bf16_bits(v)


@pytest.mark.parametrize("n", [MEDIUM_MAX + 1, MEDIUM_MAX + 4096 * 7 + 3, 1 << 24, (1 << 24) + 77,
                               FUSED_MAX - 3, FUSED_MAX])
@pytest.mark.parametrize("base", [-1, 122])
def test_fused_launch(n, base):
    _, kernels, _ = compress_checked(mixed(n, 300 + n % 997), base)
    assert kernels == [zc.ZC_KERNEL_FUSED]


def test_beyond_the_fused_launch():
    _, kernels, _ = compress_checked(np.concatenate([workloads.sweep(25), workloads.sweep(12)[:5]]))
    assert zc.ZC_KERNEL_FUSED not in kernels and zc.ZC_KERNEL_ENCODE in kernels


@pytest.mark.parametrize("base", [0, 249])
def test_extreme_bases(base):
    """Window bases at both ends: nearly every value escapes (planes) or all do."""
    compress_checked(mixed(MEDIUM_MAX + 12345, 17, frac=0.001), base)


@pytest.mark.parametrize("n", [MEDIUM_MAX + 1, 16_800_001, FUSED_MAX])
def test_random_patterns_raw_form(n):
    s, kernels, _ = compress_checked(workloads.random_patterns(n, 700 + n % 1000))
    assert kernels == [zc.ZC_KERNEL_FUSED]
    assert s[6] == 0 and s.size == raw_bytes(n)


def in_window(rng, k):
    return ((rng.integers(0, 2, k) << 15) | (127 << 7) | rng.integers(0, 128, k)).astype(np.uint16)


def tiny(rng, k):
    return ((rng.integers(0, 2, k) << 15) | (20 << 7) | rng.integers(0, 128, k)).astype(np.uint16)


def planes_and_list(planes, list_k, extra=0, chunks=4100, tail=0, seed=7):
    """`planes` chunks of escapes only, one chunk with list_k escapes, one with `extra`, the rest
    (and a ragged tail of `tail` values) with none; every value inside [122, 128] but the escapes,
    which are tiny (exponent 20), so e0 stays 122."""
    rng = np.random.default_rng(seed)
    parts = []
    for c in range(chunks):
        x = in_window(rng, 4096)
        k = 4096 if c < planes else (list_k if c == planes else (extra if c == planes + 1 else 0))
        if k:
            x[rng.choice(4096, k, replace=False)] = tiny(rng, k)
        parts.append(x)
    parts.append(in_window(rng, tail))
    return np.concatenate(parts)


def test_tie_keeps_the_coded_form():
    """2554 plane chunks and one list of 662 escapes make the coded stream exactly as long as the
    raw form: the coded form is kept.  One escape more makes it 16 bytes longer: the raw form."""
    x = planes_and_list(2554, 662)
    s, kernels, _ = compress_checked(x)
    assert kernels == [zc.ZC_KERNEL_FUSED]
    assert s[6] == 12 and s.size == raw_bytes(x.size)
    s, _, _ = compress_checked(planes_and_list(2554, 662, extra=1))
    assert s[6] == 0 and s.size == raw_bytes(x.size)


def test_planes_lists_and_a_ragged_tail():
    """Planes, a list at the list/plane boundary (1365 escapes: 4095 bytes), empty sections and a
    ragged last chunk, side by side."""
    x = planes_and_list(1300, 1365, extra=1366, tail=1000)
    s, _, _ = compress_checked(x)
    assert s[6] == 12 and s.size < raw_bytes(x.size)


def test_nonfinite_values():
    x = np.tile(workloads.sweep(20), 12)[:12_000_017].copy()
    x[::97] = 0x7FC0
    x[5::4096] = 0xFF80
    s, kernels, _ = compress_checked(x)
    assert kernels == [zc.ZC_KERNEL_FUSED] and s[6] == 12


def test_exact_path_flag():
    """A tensor on a switching point of the window rule: every CTA must reach the same exact e0
    (the oracle's), and the control block records that the exact sums decided it."""
    from test_gpu_parity import _near_boundary_tensor

    x = _near_boundary_tensor(-3, 12_000_000, 19, 0.0)
    _, kernels, out = compress_checked(x)
    assert kernels == [zc.ZC_KERNEL_FUSED]
    ws = (zc.zc_max_stream_bytes(x.size) + 255) // 256 * 256
    assert int(out[ws + 12:ws + 16].cpu().numpy().view(np.uint32)[0]) == 1


def test_static_scratch_entry_takes_the_same_launch():
    x = mixed(MEDIUM_MAX + 99, 5)
    xd = to_device(x)
    out = torch.zeros(zc.zc_max_stream_bytes(x.size), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    zc.status(reset=True)
    s = torch.cuda.current_stream().cuda_stream
    assert zc.zc_compress_static_scratch(xd.data_ptr(), x.size, zc.ZC_BASE_AUTO, out.data_ptr(),
                                         ob.data_ptr(), s) == 0
    assert zc.status(reset=True) == zc.ZC_OK
    total = int(ob.item())
    assert out[:total].cpu().numpy().tobytes() == oracle.compress(x).tobytes()
