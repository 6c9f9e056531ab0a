"""GPU path against the oracle, element by element, through the C ABI.

Bar (all integer/byte work, so everything is bit-exact): the decoded tensor equals the
input; the stream equals the oracle's stream for the same input and base; in auto mode the
chosen e0 equals the oracle's (the GPU decides e0 exactly, falling back to an exact integer
sum when its fp32-block estimate cannot settle the binade, so no boundary exception is
taken).  Sizes span several chunks and ragged tails; the full-size workloads run in the same
launch configuration as the benchmark.
"""
import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import gpu_compress, gpu_round_trip, require_gpu, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def check_parity(x, base=-1, compare_stream=True):
    st, stream, back = gpu_round_trip(x, base)
    assert st == zc.ZC_OK, zc.ERROR_NAMES.get(st, st)
    assert np.array_equal(back, x), "round trip is not exact"
    if compare_stream:
        want = oracle.compress(x, base)
        assert stream[7] == want[7], f"e0 {stream[7]} vs oracle {want[7]}"
        assert stream.size == want.size, f"length {stream.size} vs oracle {want.size}"
        if stream.tobytes() != want.tobytes():
            diff = np.flatnonzero(stream != want)
            pytest.fail(f"stream differs from the oracle at {diff.size} bytes, first at {diff[0]}")
    return stream


def mixed(n, seed, sigma=0.02, frac=0.1):
    rng = np.random.default_rng(seed)
    x = workloads.fp32_to_bf16_bits((rng.standard_normal(n) * sigma).astype(np.float32))
    mask = rng.random(n) < frac
    x[mask] = workloads.random_patterns(int(mask.sum()), seed + 1)
    return x


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 15, 16, 17, 43, 171, 4095, 4096, 4097, 4139, 8191,
                               3 * 4096 + 5, 100_003])
@pytest.mark.parametrize("base", [-1, 0, 122, 249])
def test_sizes_and_bases(n, base):
    check_parity(mixed(n, n), base)


def test_all_patterns_every_base():
    x = workloads.all_patterns()
    xd = to_device(x)
    for base in [-1] + list(range(250)):
        zc.status(reset=True)
        out, ob = zc.compress(xd, base)
        back = zc.decompress(out, x.size)
        assert zc.status(reset=True) == zc.ZC_OK
        total = int(ob.item())
        want = oracle.compress(x, base)
        assert out[:total].cpu().numpy().tobytes() == want.tobytes(), base
        assert np.array_equal(back.cpu().numpy().view(np.uint16), x), base


def test_weight_1m():
    check_parity(workloads.weight_1m())


def test_escape_free_and_all_escape():
    rng = np.random.default_rng(3)
    n = 5 * 4096 + 77
    e = rng.integers(120, 127, n)
    x = ((rng.integers(0, 2, n) << 15) | (e << 7) | rng.integers(0, 128, n)).astype(np.uint16)
    s = check_parity(x, 120)
    assert s.size == oracle.records_base(n) + 5 * 5632 + oracle.record_bytes(77, 0)
    check_parity(np.zeros(n, np.uint16), 5)  # every value escapes
    check_parity(np.zeros(n, np.uint16))      # all zeros: e0 = 0, exponent 0 is in the window


@pytest.mark.parametrize("k", [1361, 1365, 1366, 2048])
def test_full_chunks_at_the_list_plane_boundary(k):
    """Full chunks with k escapes.  Up to 1365 escapes (3k <= 4096) they keep a list.  From
    1361 on, that list pads to 4096 bytes, the size of a plane, so the decoder builds from it
    as a plane first and must rebuild the values from the codes.  From 1366 on they keep a
    plane.  Seven escape-free chunks after them keep the stream in the coded form."""
    rng = np.random.default_rng(k)
    chunks = []
    for j in range(10):
        x = np.full(4096, 0x3F80, np.uint16)  # 1.0: exponent 127, in the window for e0 = 127
        x |= rng.integers(0, 128, 4096).astype(np.uint16)  # random mantissas
        if j < 3:
            pos = rng.choice(4096, k, replace=False)
            x[pos] = rng.integers(0, 0x0100, k).astype(np.uint16)  # exponents 0 and 1: escapes
        chunks.append(x)
    x = np.concatenate(chunks)
    s = check_parity(x, 127)
    section = (4096 if 3 * k > 4096 else (3 * k + 15) // 16 * 16)
    assert s[6] == 12 and s.size == oracle.records_base(x.size) + 3 * (5632 + section) + 7 * 5632


@pytest.mark.parametrize("n", [0, 1, 5, 37, 38, 4095, 4097, 3 * 4096 + 3, 100_000])
def test_raw_form(n):
    """Tensors whose coded form would be longer come out in the raw form: the header, then the
    values as they are.  Random bit patterns escape almost everywhere; tiny tensors pay more
    for the coded header and table than they save."""
    x = workloads.random_patterns(n, 500 + n)
    s = check_parity(x)
    assert s[6] == 0 and s.size == 32 + (2 * n + 15) // 16 * 16
    assert s[32:32 + 2 * n].tobytes() == x.tobytes()


def test_raw_and_coded_at_the_tie():
    """37 values of 1.0 under e0 = 127 cost 112 bytes either way: the coded form is kept; one
    escape more tips the stream into the raw form."""
    x = np.full(37, 0x3F80, np.uint16)
    s = check_parity(x, 127)
    assert s.size == 112 and s[6] == 12
    x[5] = 0
    s = check_parity(x, 127)
    assert s.size == 112 and s[6] == 0


@pytest.mark.parametrize("n", [64 * 4096 + 1, 100_003 * 3, 1 << 20, 4 * (1 << 20) + 77, 2432 * 4096, 2432 * 4096 + 1])
@pytest.mark.parametrize("base", [-1, 122])
def test_single_cooperative_launch(n, base):
    """Sizes past the cluster launch: up to four chunks per CTA of one cooperative grid (2432
    chunks on a GB300: 608 resident CTAs), then, one value more, the multi-launch path."""
    check_parity(mixed(n, 500 + n % 1000, sigma=1.0, frac=0.02), base)


@pytest.mark.parametrize("n", [300_001, 5_000_000])
def test_single_cooperative_launch_raw_and_special(n):
    """The raw form and non-finite blocks on the cooperative-grid path."""
    s = check_parity(workloads.random_patterns(n, 61))
    assert s[6] == 0
    x = workloads.sweep(20)[: n % (1 << 20)].copy() if n < (1 << 20) else np.tile(workloads.sweep(20), 5)[:n].copy()
    x[::97] = 0x7FC0
    check_parity(x)


def test_special_tensors():
    check_parity(np.full(9000, 0x7FC0, np.uint16))           # only NaN: no finite value
    check_parity(np.full(9000, 0x3F80, np.uint16))           # constant 1.0
    check_parity(np.array([0x7F7F] * 5000 + [0x0001] * 5000, np.uint16))  # extremes
    check_parity(workloads.random_patterns(70_000, 5))


@pytest.mark.parametrize("case", ["mixed_1pct", "nan_every_64th", "all_patterns_x4"])
def test_nonfinite_blocks_beyond_the_small_path(case):
    """Blocks of 64 values holding Inf or NaN clear and count them inside the vectorized sum (the
    statistics kernel of the multi-launch path): e0 and the stream must still equal the oracle's."""
    if case == "mixed_1pct":
        x = mixed(2_000_003, 41, sigma=1.0, frac=0.01)
    elif case == "nan_every_64th":
        x = workloads.sweep(21).copy()
        x[::64] = 0x7FC1
        x[5::4096] = 0xFF80  # -Inf
    else:
        x = np.concatenate([np.tile(workloads.all_patterns(), 4), workloads.all_patterns()[:1234]])
    check_parity(x)


def _near_boundary_tensor(k4, n, seed, rel, zero_frac=0.0):
    """A tensor whose sum of squares is within ~1e-15 of (1 + rel) 4**k4 n / c^2, i.e. whose
    mean square times c^2 sits `rel` away from a switching point of the window rule (with about
    `zero_frac` of its values zero)."""
    rng = np.random.default_rng(seed)
    T = (4.0 ** k4) * n / oracle.window_constant() * (1.0 + rel)
    bulk = n - 48
    v = rng.standard_normal(bulk)
    if zero_frac:
        v[rng.random(bulk) < zero_frac] = 0.0
    v *= np.sqrt(T * (1 - 1e-3) / np.sum(v * v))
    x = workloads.fp32_to_bf16_bits(v.astype(np.float32))
    as_float = lambda b: float(np.array([int(b) << 16], np.uint32).view(np.float32)[0])  # noqa: E731
    f = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    R = T - float(np.sum(f * f))
    tail = []
    for _ in range(48):  # greedy: the largest BF16 whose square still fits in what is left
        r = min(np.sqrt(max(R, 0.0)), float(np.finfo(np.float32).max))  # (no overflow to Inf in the cast)
        t = int(workloads.fp32_to_bf16_bits(np.array([r], np.float32))[0])
        while t > 0 and as_float(t) ** 2 > R:
            t -= 1
        tail.append(t)
        R -= as_float(t) ** 2
    return np.concatenate([x, np.array(tail, np.uint16)])


@pytest.mark.parametrize("k4,rel", [(-8, -1e-9), (-8, 1e-9), (-3, 0.0), (-11, 1e-9), (2, -1e-9), (-5, 3e-6)])
def test_auto_base_at_binade_boundaries(k4, rel):
    """Tensors built to sit on a switching point of the window rule: the fast fp32 estimate
    cannot decide, the exact integer fallback must, and it must agree with the oracle."""
    x = _near_boundary_tensor(k4, 20_000, 100 + k4, rel)
    st, out, total = gpu_compress(x)
    assert st == zc.ZC_OK
    stream = out[:total].cpu().numpy()
    assert stream[7] == oracle.choose_e0(x)
    ws = (zc.zc_max_stream_bytes(x.size) + 255) // 256 * 256
    exact_path = int(out[ws + 12:ws + 16].cpu().numpy().view(np.uint32)[0])
    assert exact_path == 1, "the exact fallback did not run"
    check_parity(x)


@pytest.mark.parametrize("n,k4,zeros", [((1 << 20) + 3, -8, 0.0), (1 << 26, -3, 0.0),
                                        ((1 << 25) + 3 * 4096 + 5, -114, 0.0),
                                        ((1 << 25) + 3 * 4096 + 5, 118, 0.0),
                                        ((1 << 25) + 4096 + 3, -8, 0.3)])
def test_auto_base_at_binade_boundaries_large(n, k4, zeros):
    """Boundary tensors beyond the cluster launch: the exact sum runs over the whole grid (in the
    cooperative-grid launch at 2^20 + 3 values, in the encode kernel's first phase beyond 2^25)
    and must agree with the oracle.  In the first phase, e0 = 13 puts the exact sums' 24-binade
    window at its lowest anchor (exponent 1: subnormals inside it), e0 = 245 at its highest
    (exponent 230), and a tensor with 30% zeros sends many values down the out-of-window path
    that skips them."""
    x = _near_boundary_tensor(k4, n, 200 + k4, 1e-9, zeros)
    st, out, total = gpu_compress(x)
    assert st == zc.ZC_OK
    stream = out[:total].cpu().numpy()
    assert stream[7] == oracle.choose_e0(x)
    ws = (zc.zc_max_stream_bytes(x.size) + 255) // 256 * 256
    assert int(out[ws + 12:ws + 16].cpu().numpy().view(np.uint32)[0]) == 1, "the exact fallback did not run"
    check_parity(x)


@pytest.mark.parametrize("n,k4,rel", [(20_000, -8, 1e-4), (20_000, -3, -5e-5), ((1 << 20) + 3, -8, -1e-4),
                                      ((1 << 24) + 5, -5, 5e-5), ((1 << 25) + 4096 * 2 + 7, -8, 1e-4)])
def test_auto_base_near_binade_boundaries(n, k4, rel):
    """Mean squares 5e-5 to 1e-4 from a switching point: closer than the margin of the quick fp32
    check of the window rule (2^-12, about 2.4e-4), farther than the fp64 rule's interval (2^-16
    plus the estimate's 2^-17): e0 is settled by the rule's two fp64 ends, with no exact sums, and
    must be the oracle's -- in the cluster, the cooperative grid, the L2-resident kernel and the
    statistics kernel."""
    x = _near_boundary_tensor(k4, n, 300 + k4, rel)
    st, out, total = gpu_compress(x)
    assert st == zc.ZC_OK
    assert out[7].item() == oracle.choose_e0(x)
    ws = (zc.zc_max_stream_bytes(x.size) + 255) // 256 * 256
    assert int(out[ws + 12:ws + 16].cpu().numpy().view(np.uint32)[0]) == 0, "the exact fallback ran"
    check_parity(x)


def test_supplied_base_matches_auto_stream():
    x = mixed(50_000, 4)
    s_auto = check_parity(x, -1)
    s_given = check_parity(x, int(s_auto[7]))
    assert s_auto.tobytes() == s_given.tobytes()


def test_deterministic_and_concurrent_streams():
    """Four compressions on four streams at once: two on the single-launch path for small
    tensors, two on the multi-launch path."""
    xs = [mixed((200_000 if i % 2 else 600_000) + 17 * i, 20 + i) for i in range(4)]
    devs = [to_device(x) for x in xs]
    streams = [torch.cuda.Stream() for _ in xs]
    outs = []
    zc.status(reset=True)
    for xd, s in zip(devs, streams):
        with torch.cuda.stream(s):
            outs.append(zc.compress(xd, stream=s))
    torch.cuda.synchronize()
    assert zc.status(reset=True) == zc.ZC_OK
    for x, (out, ob) in zip(xs, outs):
        total = int(ob.item())
        assert out[:total].cpu().numpy().tobytes() == oracle.compress(x).tobytes()


@pytest.mark.parametrize("n", [4095, 3 * 4096, 3 * 4096 + 5])
def test_buffers_at_16_byte_offsets(n):
    """Input, stream and output buffers that start 16 bytes past an allocation's start (the
    alignment the C ABI asks for, below what the caching allocator hands out)."""
    x = mixed(n, 70 + n)
    pad = np.zeros(8, dtype=np.uint16)
    xd = to_device(np.concatenate([pad, x]))[8:]
    assert xd.data_ptr() % 256 == 16
    cap = zc.zc_max_compressed_bytes(n)
    out_all = torch.zeros(cap + 16, dtype=torch.uint8, device="cuda")
    out = out_all[16:]
    zc.status(reset=True)
    _, ob = zc.compress(xd, out=out)
    total = int(ob.item())
    assert zc.status(reset=True) == zc.ZC_OK
    assert out[:total].cpu().numpy().tobytes() == oracle.compress(x).tobytes()
    back_all = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    zc.decompress(out, n, out=back_all[8:])
    assert zc.status(reset=True) == zc.ZC_OK
    assert np.array_equal(back_all[8:].cpu().numpy().view(np.uint16), x)
    assert not back_all[:8].any()


def test_out_bytes_in_host_memory():
    import ctypes

    x = mixed(30_000, 9)
    xd = to_device(x)
    cap = zc.zc_max_compressed_bytes(x.size)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    want = oracle.compress(x)
    # pageable: the call copies the length back and synchronizes
    n_host = ctypes.c_uint64(0)
    st = zc.zc_compress(xd.data_ptr(), x.size, -1, out.data_ptr(), ctypes.addressof(n_host),
                        torch.cuda.current_stream().cuda_stream)
    assert st == zc.ZC_OK and n_host.value == want.size
    # pinned: written by the kernel
    pinned = torch.zeros(1, dtype=torch.int64).pin_memory()
    st = zc.zc_compress(xd.data_ptr(), x.size, -1, out.data_ptr(), pinned.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == zc.ZC_OK and int(pinned[0]) == want.size
    assert out[:want.size].cpu().numpy().tobytes() == want.tobytes()


# ---------------------------------------------------------------- full-size workloads


@pytest.mark.parametrize("name", ["grad_bucket_4096x14336", "moe_a2a_16384x7168", "adversarial_256m"])
def test_full_size_workload(name):
    check_parity(workloads.make(name))


@pytest.mark.parametrize("k", [15, 16, 17, 20, 23, 26, 29])
def test_sweep_sizes(k):
    check_parity(workloads.sweep(k))
