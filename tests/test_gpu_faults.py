"""Device-side error detection, without faulting the GPU.

Corrupt streams are made on the host; the decoder must report them through zc_status (and
agree with the oracle on which streams are invalid) while reading only inside the buffer.
The scan's wait is made to run out by a chunk that never publishes; the call must report
ZC_ERR_TIMEOUT and leave the context usable.  Canary bytes around every buffer must survive.
"""
import ctypes

import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import gpu_decompress_bytes, require_gpu, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_VALUES = 3 * 4096 + 100


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def sample():
    """N(0, 0.02^2) with 300 random bit patterns, coded with the window of the Gaussian part
    (e0 = 116), so that every chunk keeps its escapes as a list.  (In auto mode the random
    patterns' huge values pull e0 up to 243 and every chunk keeps a plane instead.)"""
    rng = np.random.default_rng(42)
    x = workloads.fp32_to_bf16_bits((rng.standard_normal(N_VALUES) * 0.02).astype(np.float32))
    x[rng.choice(N_VALUES, 300, replace=False)] = workloads.random_patterns(300, 43)
    s = oracle.compress(x, 116)
    N = (N_VALUES + 4095) // 4096
    assert all(escape_offset(s, c + 1) - escape_offset(s, c) < 1024 for c in range(N)), "lists expected"
    return x, s


def u64_at(s, off, v):
    t = s.copy()
    t[off:off + 8] = np.frombuffer(np.uint64(v).tobytes(), np.uint8)
    return t


def oracle_status(stream, n, capacity):
    buf = np.zeros(capacity, np.uint8)
    buf[:stream.size] = stream
    return oracle.decompress(buf, n)


def escape_offset(s, c):
    return int(s[32 + 8 * c:40 + 8 * c].view(np.uint64)[0])


def targeted_mutations(s, x):
    pad16 = lambda v: (v + 15) // 16 * 16  # noqa: E731
    N = (N_VALUES + 4095) // 4096
    R0 = pad16(32 + 8 * (N + 1))
    e0 = int(s[7])
    E = (x[:4096].astype(np.int64) >> 7) & 0xFF
    k0 = int(((E < e0) | (E > e0 + 6)).sum())
    esc0 = escape_offset(s, 0)
    last = R0 + (N - 1) * 5632  # fixed part of the last chunk (100 values)
    muts = {
        "magic": (0, 0x00),
        "version": (4, 1),
        "log2_chunk": (6, 11),
        "base_250": (7, 250),
        "N": (16, 5),
        "total_bytes": (24, s[24] ^ 0x10),
        "offset_0": (32, s[32] ^ 0x10),
        "offset_1_misaligned": (40, s[40] ^ 0x01),
        "escape_position": (esc0, s[esc0] ^ 0x01),
        "escape_exponent_in_window": (esc0 + 2 * k0, e0),
        "last_codes_padding": (last + (3 * 100 + 7) // 8 + 1, 0x80),
        "last_byte_plane_padding": (last + 48 + 100 + 1, 0x01),
    }
    if (3 * k0) % 16:
        muts["escape_padding"] = (esc0 + 3 * k0 + 1, 0x55)
    if not (E[0] < e0 or E[0] > e0 + 6):  # value 0's code is in bits 0..2 of the first code byte
        muts["code_to_escape"] = (R0, s[R0] | 0x07)
    out = {}
    for name, (pos, val) in muts.items():
        t = s.copy()
        t[pos] = np.uint8(val)
        out[name] = t
    out["n_mismatch"] = u64_at(s, 8, N_VALUES + 1)
    out["table_end"] = u64_at(s, 32 + 8 * N, int(s[24:32].view(np.uint64)[0]) + 16)
    return out


def test_targeted_corruptions_are_reported(sample):
    x, s = sample
    cap = zc.zc_max_compressed_bytes(N_VALUES)
    for name, t in targeted_mutations(s, x).items():
        ost, _ = oracle_status(t, N_VALUES, cap)
        assert ost != oracle.OK, f"{name}: the oracle accepts it, the mutation is not a corruption"
        st, _ = gpu_decompress_bytes(t, N_VALUES, cap)
        want = zc.ZC_ERR_SIZE_MISMATCH if ost == oracle.ERR_SIZE_MISMATCH else zc.ZC_ERR_CORRUPT
        assert st == want, f"{name}: status {zc.ERROR_NAMES.get(st, st)}"


def test_random_bit_flips_match_oracle_verdict(sample):
    x, s = sample
    cap = zc.zc_max_compressed_bytes(N_VALUES)
    rng = np.random.default_rng(5)
    accepted = rejected = 0
    for _ in range(400):
        t = s.copy()
        pos = int(rng.integers(0, s.size))
        t[pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, ovals = oracle_status(t, N_VALUES, cap)
        st, gvals = gpu_decompress_bytes(t, N_VALUES, cap)
        if ost == oracle.OK:
            assert st == zc.ZC_OK, f"flip at {pos}: GPU rejects a valid stream"
            assert np.array_equal(gvals, ovals), f"flip at {pos}: different values"
            accepted += 1
        else:
            assert st != zc.ZC_OK, f"flip at {pos}: GPU accepts an invalid stream"
            rejected += 1
    assert accepted > 50 and rejected > 50


PLANE_CHUNKS = (6, 7)  # chunks of random bit patterns among escape-free ones


@pytest.fixture(scope="module")
def dense_sample():
    """Six escape-free chunks (exponents 127..133, in the window of e0 = 127), two chunks and 50
    values of random bit patterns: nearly every value of the last three escapes, so they keep
    their escapes as exponent planes (one byte per value) rather than lists, and the clean
    chunks keep the stream in the coded form."""
    rng = np.random.default_rng(91)
    clean = 6 * 4096
    e = rng.integers(127, 134, clean)
    head = ((rng.integers(0, 2, clean) << 15) | (e << 7) | rng.integers(0, 128, clean)).astype(np.uint16)
    x = np.concatenate([head, workloads.random_patterns(2 * 4096 + 50, 91)])
    s = oracle.compress(x, 127)
    assert s[6] == 12
    return x, s


def test_plane_corruptions_are_reported(dense_sample):
    x, s = dense_sample
    n = x.size
    N = (n + 4095) // 4096
    cap = zc.zc_max_compressed_bytes(n)
    c0 = PLANE_CHUNKS[0]
    off0, off1 = escape_offset(s, c0), escape_offset(s, c0 + 1)
    assert off1 - off0 == 4096, "the first random chunk keeps a plane"
    e0 = int(s[7])
    E = (x[4096 * c0:4096 * (c0 + 1)].astype(np.int64) >> 7) & 0xFF
    inside = np.flatnonzero((E >= e0) & (E <= e0 + 6))
    outside = np.flatnonzero((E < e0) | (E > e0 + 6))
    assert inside.size > 0 and outside.size > 0
    st, vals = gpu_decompress_bytes(s, n, cap)
    assert st == zc.ZC_OK and np.array_equal(vals, x)
    R0 = (32 + 8 * (N + 1) + 15) // 16 * 16
    codes0 = R0 + 5632 * c0
    i_in, i_out = int(inside[0]), int(outside[-1])
    last_off = escape_offset(s, N - 1)  # the last chunk's 50 values: a plane of pad16(50) = 64 bytes
    muts = {
        "escaped_exponent_into_window": (off0 + i_out, e0 + 2),
        "in_window_exponent_changed": (off0 + i_in, (int(E[i_in]) + 1) & 0xFF if E[i_in] < e0 + 6 else e0),
        "last_plane_padding": (last_off + 50 + 3, 0x01),
    }
    for name, (pos, val) in muts.items():
        t = s.copy()
        t[pos] = np.uint8(val)
        ost, _ = oracle_status(t, n, cap)
        assert ost != oracle.OK, f"{name}: the oracle accepts it, the mutation is not a corruption"
        st, _ = gpu_decompress_bytes(t, n, cap)
        assert st == zc.ZC_ERR_CORRUPT, f"{name}: status {zc.ERROR_NAMES.get(st, st)}"
    # an escaped value's exponent moved to another out-of-window exponent is a valid stream of
    # another tensor: both sides must accept it and agree on the values
    t = s.copy()
    t[off0 + i_out] = np.uint8(0 if E[i_out] != 0 else 1)
    ost, ovals = oracle_status(t, n, cap)
    st, gvals = gpu_decompress_bytes(t, n, cap)
    assert ost == oracle.OK and st == zc.ZC_OK and np.array_equal(gvals, ovals)
    rng = np.random.default_rng(8)
    for _ in range(60):  # flips in the plane chunk's codes and plane: the GPU's verdict is the oracle's
        t = s.copy()
        pos = int(rng.choice([rng.integers(codes0, codes0 + 1536), rng.integers(off0, off1)]))
        t[pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, ovals = oracle_status(t, n, cap)
        st, gvals = gpu_decompress_bytes(t, n, cap)
        if ost == oracle.OK:
            assert st == zc.ZC_OK and np.array_equal(gvals, ovals), f"flip at {pos}"
        else:
            assert st != zc.ZC_OK, f"flip at {pos}: GPU accepts an invalid stream"


@pytest.fixture(scope="module")
def raw_sample():
    """Random bit patterns: the coded form would be longer, so the stream is in the raw form."""
    x = workloads.random_patterns(3 * 4096 + 77, 92)
    s = oracle.compress(x)
    assert s[6] == 0 and s.size == 32 + (2 * x.size + 15) // 16 * 16
    return x, s


def test_raw_corruptions_are_reported(raw_sample):
    x, s = raw_sample
    n = x.size
    cap = zc.zc_max_compressed_bytes(n)
    st, vals = gpu_decompress_bytes(s, n, cap)
    assert st == zc.ZC_OK and np.array_equal(vals, x)
    muts = {"form_12": (6, 12), "form_1": (6, 1), "version": (4, 3), "base_250": (7, 250), "N_1": (16, 1),
            "total": (24, s[24] ^ 0x10), "padding": (32 + 2 * n + 1, 0x01), "magic": (1, 0)}
    for name, (pos, val) in muts.items():
        t = s.copy()
        t[pos] = np.uint8(val)
        ost, _ = oracle_status(t, n, cap)
        assert ost == oracle.ERR_CORRUPT, f"{name}: the oracle accepts it"
        st, _ = gpu_decompress_bytes(t, n, cap)
        assert st == zc.ZC_ERR_CORRUPT, f"{name}: status {zc.ERROR_NAMES.get(st, st)}"
    st, _ = gpu_decompress_bytes(s, n + 1, zc.zc_max_compressed_bytes(n + 1))
    assert st == zc.ZC_ERR_SIZE_MISMATCH
    rng = np.random.default_rng(9)
    for _ in range(100):  # flips anywhere in a raw stream: the GPU's verdict and values are the oracle's
        t = s.copy()
        pos = int(rng.integers(0, s.size))
        t[pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, ovals = oracle_status(t, n, cap)
        st, gvals = gpu_decompress_bytes(t, n, cap)
        assert (st == zc.ZC_OK) == (ost == oracle.OK), f"flip at {pos}"
        if st == zc.ZC_OK:
            assert np.array_equal(gvals, ovals), f"flip at {pos}"


def test_valid_stream_and_wrong_n(sample):
    x, s = sample
    cap = zc.zc_max_compressed_bytes(N_VALUES)
    st, vals = gpu_decompress_bytes(s, N_VALUES, cap)
    assert st == zc.ZC_OK and np.array_equal(vals, x)
    st, _ = gpu_decompress_bytes(s, N_VALUES - 1, cap)
    assert st == zc.ZC_ERR_SIZE_MISMATCH


def test_valid_small_stream_with_much_larger_n(sample):
    """A caller's n far above the stream's: the header check reports it before any read that
    depends on n.  The stream sits at the start of a zeroed buffer large enough for every read
    a decoder could make for the larger n, so this test cannot fault whatever the kernel does."""
    x, s = sample
    big = 64 * 4096 + 5
    st, _ = gpu_decompress_bytes(s, big, zc.zc_max_compressed_bytes(big))
    assert st == zc.ZC_ERR_SIZE_MISMATCH
    st, _ = gpu_decompress_bytes(s, 0, zc.zc_max_compressed_bytes(big))
    assert st == zc.ZC_ERR_SIZE_MISMATCH


@pytest.mark.parametrize("total", [0, 16, 48, 64])
def test_total_below_the_fixed_region(sample, total):
    """A header whose total_bytes ends before the fixed parts (below records_base(n), or below the
    start of the escape region) is corrupt.  The stream is cut to total_bytes bytes and followed
    by a 4 KiB guard band inside the same allocation; the decoder reports ZC_ERR_CORRUPT and
    writes nothing."""
    x, s = sample
    G = 4096
    t = u64_at(s, 24, total)[:max(total, 32)]
    ost, _ = oracle_status(t, N_VALUES, t.size)
    assert ost == oracle.ERR_CORRUPT
    buf = torch.full((t.size + G,), 0xA5, dtype=torch.uint8, device="cuda")
    buf[:t.size] = torch.from_numpy(t.copy())
    out = torch.full((N_VALUES + 16,), 0x5A5A, dtype=torch.int16, device="cuda")
    s_ = torch.cuda.current_stream().cuda_stream
    zc.status(reset=True)
    assert zc.zc_decompress(buf.data_ptr(), out.data_ptr(), N_VALUES, s_) == zc.ZC_OK
    assert zc.zc_status(s_, 1) == zc.ZC_ERR_CORRUPT
    assert bool((out == 0x5A5A).all()), "the decoder wrote values from a corrupt stream"
    assert bool((buf[t.size:] == 0xA5).all())


def test_empty_stream():
    s = oracle.compress(np.zeros(0, np.uint16))
    st, _ = gpu_decompress_bytes(s, 0, 64)
    assert st == zc.ZC_OK
    st, _ = gpu_decompress_bytes(u64_at(s, 24, 64), 0, 128)
    assert st == zc.ZC_ERR_CORRUPT


@pytest.mark.parametrize("stalled", [0, 1, 17])
def test_scan_wait_is_bounded(stalled):
    x = workloads.sweep(18)  # 64 chunks
    xd = to_device(x)
    cap = zc.zc_max_compressed_bytes(x.size)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    zc.status(reset=True)
    assert zc.zc_compress_stall_test(xd.data_ptr(), x.size, -1, out.data_ptr(), ob.data_ptr(), s,
                                     stalled, 2000) == zc.ZC_OK
    assert zc.zc_status(s, 1) == zc.ZC_ERR_TIMEOUT
    # the context is still usable: a normal call afterwards is exact
    out2, ob2 = zc.compress(xd)
    back = zc.decompress(out2, x.size)
    assert zc.status(reset=True) == zc.ZC_OK
    assert np.array_equal(back.cpu().numpy().view(np.uint16), x)
    assert out2[:int(ob2.item())].cpu().numpy().tobytes() == oracle.compress(x).tobytes()


def test_guard_bands():
    """4 KiB of 0xA5 before and after the input, the output and the decoded buffer."""
    G = 4096
    rng = np.random.default_rng(77)
    for n in (1, 4097, 3 * 4096 + 5, 70_001):
        x = workloads.random_patterns(n, int(rng.integers(1 << 30)))
        cap = zc.zc_max_compressed_bytes(n)
        inb = torch.full((G + 2 * n + G,), 0xA5, dtype=torch.uint8, device="cuda")
        inb[G:G + 2 * n] = torch.from_numpy(x.view(np.uint8).copy())
        outb = torch.full((G + cap + G,), 0xA5, dtype=torch.uint8, device="cuda")
        decb = torch.full((G + 2 * n + 16 + G,), 0xA5, dtype=torch.uint8, device="cuda")
        ob = torch.zeros(1, dtype=torch.int64, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        zc.status(reset=True)
        assert zc.zc_compress(inb.data_ptr() + G, n, -1, outb.data_ptr() + G, ob.data_ptr(), s) == zc.ZC_OK
        assert zc.zc_decompress(outb.data_ptr() + G, decb.data_ptr() + G, n, s) == zc.ZC_OK
        assert zc.zc_status(s, 1) == zc.ZC_OK
        for buf, lo, hi in ((inb, G, G + 2 * n), (outb, G, G + cap), (decb, G, G + 2 * n)):
            h = buf.cpu().numpy()
            assert np.all(h[:lo] == 0xA5) and np.all(h[hi:] == 0xA5), "a guard band was written"
        got = decb[G:G + 2 * n].cpu().numpy().view(np.uint16)
        assert np.array_equal(got, x)
        total = int(ob.item())
        assert outb[G:G + total].cpu().numpy().tobytes() == oracle.compress(x).tobytes()
