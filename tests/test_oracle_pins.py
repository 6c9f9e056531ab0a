"""Pins for the oracle against facts that do not come from the oracle itself.

Each test checks the plain C reference against something fixed by the pages or by
mathematics: a hand-derived stream, the correctly rounded sum (math.fsum), the Gaussian
escape-rate argmin the window rule stands for, the constant re-derived with mpmath, the
closed-form size and "about 11 bits per value" (ZipCCL, "Key idea and contribution"), and
exhaustive round trips.  A plausible mistake in the oracle -- a wrong shift, a dropped
rounding, an off-by-one window, a transposed section -- fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import workloads

CHUNK = 4096


def pad16(v):
    return (v + 15) // 16 * 16


def bf16_to_float(bits):
    """Exact Python floats of BF16 bit patterns (through fp32, which holds them exactly)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def escape_section(m, k):
    """Bytes of a chunk's escape section: a list of k (u16, u8) pairs, or a plane of all m
    exponents when 3k > m; zero-padded to 16."""
    return pad16(m) if 3 * k > m else pad16(3 * k)


def coded_size(x, e0):
    """Length of the coded form from the size formula, escapes counted per chunk."""
    n = x.size
    N = (n + CHUNK - 1) // CHUNK
    E = (x.astype(np.int64) >> 7) & 0xFF
    escape = (E < e0) | (E > e0 + 6)
    total = pad16(32 + 8 * (N + 1))
    for c in range(N):
        m = min(CHUNK, n - c * CHUNK)
        k = int(escape[c * CHUNK:c * CHUNK + m].sum())
        total += pad16((3 * m + 7) // 8) + pad16(m) + escape_section(m, k)
    return total


def raw_size(n):
    """The raw form: 32-byte header, then the n values, zero-padded to 16 bytes."""
    return 32 + pad16(2 * n)


def closed_form_size(x, e0):
    """Stream length: the coded form, or the raw form when the coded one is longer."""
    return min(coded_size(x, e0), raw_size(x.size))


# ----------------------------------------------------------------------------- golden


@pytest.mark.parametrize("fixture", ["golden_raw", "golden_plane", "golden_list"])
def test_golden_streams_match_hand_derivation(fixture, request):
    e0, values, stream = request.getfixturevalue(fixture)
    got = oracle.compress(values, e0)
    assert got.tobytes() == stream.tobytes()
    st, back = oracle.decompress(stream, values.size)
    assert st == oracle.OK and np.array_equal(back, values)


def test_list_or_plane_at_the_boundary():
    """3k <= m keeps a list, 3k > m a plane, whichever is smaller; the codes are the same.  A
    first chunk of 4096 in-window values keeps the stream in the coded form."""
    e0 = 127
    inside, outside = 0x3F80, 0x0000  # exponents 127 (code 0) and 0 (an escape)
    head = [inside] * CHUNK
    for m in range(1, 40):
        for k in range(0, m + 1):
            x = np.array(head + [outside] * k + [inside] * (m - k), np.uint16)
            s = oracle.compress(x, e0)
            fixed_end = pad16(32 + 8 * 3) + 5632 + pad16((3 * m + 7) // 8) + pad16(m)
            section = len(s) - fixed_end
            assert section == (pad16(m) if 3 * k > m else pad16(3 * k)), (m, k)
            assert section == min(pad16(m), pad16(3 * k))
            if 3 * k > m:  # a plane: one exponent byte per value, in value order
                assert s[-section:][:m].tolist() == [0] * k + [127] * (m - k)
            st, back = oracle.decompress(s, CHUNK + m)
            assert st == oracle.OK and np.array_equal(back, x)


def test_raw_form_exactly_when_the_coded_form_is_longer():
    """The native form is chosen exactly when the coded form would be longer than the 32-byte
    header plus the values; ties keep the coded form."""
    rng = np.random.default_rng(21)
    seen = {True: 0, False: 0}
    for n in [1, 2, 7, 37, 38, 100, 171, 600, 4095, 4096, 4097, 9000]:
        for frac in (0.0, 0.01, 0.05, 0.2, 0.3, 0.5, 1.0):
            e = rng.integers(120, 127, n)  # in the window of e0 = 120
            x = ((rng.integers(0, 2, n) << 15) | (e << 7) | rng.integers(0, 128, n)).astype(np.uint16)
            esc = rng.random(n) < frac
            x[esc] = rng.integers(0, 0x0100, int(esc.sum())).astype(np.uint16)  # exponents 0, 1
            s = oracle.compress(x, 120)
            raw = coded_size(x, 120) > raw_size(n)
            seen[raw] += 1
            assert len(s) == (raw_size(n) if raw else coded_size(x, 120)), (n, frac)
            assert (s[6] == 0) == raw  # byte 6: 0 for the raw form, 12 for the coded one
            if raw:
                assert s[32:32 + 2 * n].tobytes() == x.tobytes()  # the values as they are
            st, back = oracle.decompress(s, n)
            assert st == oracle.OK and np.array_equal(back, x)
    assert seen[True] > 10 and seen[False] > 10
    # a tie: 37 in-window values cost 48 + 16 + 48 = 112 bytes either way -> coded
    x = np.full(37, 0x3F80, np.uint16)
    assert coded_size(x, 127) == raw_size(37) == 112
    assert oracle.compress(x, 127)[6] == 12


# ----------------------------------------------------------------------------- window rule


def _derive_c2_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    f = lambda t: mp.erf(t / mp.sqrt(2)) + mp.erfc(128 * t / mp.sqrt(2))  # noqa: E731
    u = mp.findroot(lambda u: f(u) - f(2 * u), 0.019)
    return mp, (2 * u) ** 2


def test_window_constant_rederived():
    """c = 2u with f(u) = f(2u): the switching point between adjacent 7-binade windows."""
    mp, c2 = _derive_c2_mpmath()
    assert oracle.window_constant() == float(c2)


def _gaussian_escape_rate(mp, e0, sigma):
    lo = mp.mpf(2) ** (e0 - 127)
    hi = mp.mpf(2) ** (e0 - 120)
    s = mp.mpf(sigma) * mp.sqrt(2)
    return mp.erf(lo / s) + mp.erfc(hi / s)


def test_window_is_gaussian_escape_argmin():
    """For a tensor whose RMS is sigma (a constant tensor), e0 must be the integer base whose
    7-binade window has the fewest expected escapes under N(0, sigma^2)."""
    mp, _ = _derive_c2_mpmath()
    mp.mp.dps = 30
    checked = 0
    for bits in range(0x3000, 0x5000, 7):  # sigma from about 5e-10 to 3e9
        sigma = float(bf16_to_float([bits])[0])
        rates = {e: _gaussian_escape_rate(mp, e, sigma) for e in range(0, 250)
                 if abs(e - (math.log2(sigma) + 122.3)) < 4}
        best = min(rates, key=lambda e: rates[e])
        second = sorted(rates.values())[1]
        if abs(second - rates[best]) < 1e-9 * rates[best]:
            continue  # a tie: both windows are optimal
        x = np.full(3, bits, dtype=np.uint16)
        assert oracle.choose_e0(x) == best, hex(bits)
        checked += 1
    assert checked > 1000


def test_constant_tensors_follow_log2_rule():
    """Every positive finite BF16 constant: e0 = clamp(floor(log2(|v| c)) + 127, 0, 249)."""
    mp, c2 = _derive_c2_mpmath()
    c = mp.sqrt(c2)
    for bits in range(1, 0x7F80):
        v = mp.mpf(float(bf16_to_float([bits])[0]))
        t = mp.log(v * c, 2)
        if abs(t - mp.nint(t)) < 1e-12:
            continue
        want = min(249, max(0, int(mp.floor(t)) + 127))
        x = np.array([bits, bits | 0x8000], dtype=np.uint16)  # sign does not matter
        assert oracle.choose_e0(x) == want, hex(bits)


def test_special_cases():
    assert oracle.choose_e0(np.zeros(0, np.uint16)) == 0
    assert oracle.choose_e0(np.zeros(1000, np.uint16)) == 0
    assert oracle.choose_e0(np.full(10, 0x8000, np.uint16)) == 0  # -0.0
    assert oracle.choose_e0(np.array([0x7F80, 0xFF80, 0x7FC0], np.uint16)) == 0  # no finite value
    assert oracle.choose_e0(np.full(10, 0x3F80, np.uint16)) == 122  # 1.0: window 122..128
    # a non-finite value changes neither the sum nor the count
    x = np.full(10, 0x3F80, np.uint16)
    assert oracle.choose_e0(np.concatenate([x, [0x7FC0, 0xFF80]]).astype(np.uint16)) == 122


# ----------------------------------------------------------------------------- exact sum


def _fsum_reference(bits):
    v = bf16_to_float(bits)
    fin = np.isfinite(v)
    return math.fsum((v[fin] * v[fin]).tolist()), int(fin.sum())


@pytest.mark.parametrize("case", ["gauss", "patterns", "tiny", "huge", "mixed", "weight_1m"])
def test_sum_of_squares_is_correctly_rounded(case):
    rng = np.random.default_rng(11)
    if case == "gauss":
        x = workloads.fp32_to_bf16_bits(rng.standard_normal(300_000).astype(np.float32))
    elif case == "patterns":
        x = workloads.random_patterns(300_000, 12)
    elif case == "tiny":  # subnormals and the smallest normals only
        x = rng.integers(0, 0x0200, 50_000).astype(np.uint16)
    elif case == "huge":  # the largest finite values
        x = rng.integers(0x7E00, 0x7F80, 50_000).astype(np.uint16)
    elif case == "mixed":  # one huge value among many tiny ones: the sum must not lose either
        x = rng.integers(0x0001, 0x0080, 200_000).astype(np.uint16)
        x[::50_000] = 0x7F7F
    else:
        x = workloads.weight_1m()
    S_d, n_f = oracle.sum_squares(x)
    want_S, want_nf = _fsum_reference(x)
    assert n_f == want_nf
    assert S_d == want_S


def test_sum_tie_rounds_to_even():
    # 128 squares of 2^23 sum to 2^53, where the fp64 spacing is 2; adding squares of 1.0
    # lands exactly halfway between two neighbours, so the rounding must pick the even one.
    one = 0x3F80  # 1.0 -> square 1
    big = 0x4B00  # 2^23 -> square 2^46
    x = np.array([big] * 128 + [one], dtype=np.uint16)  # 2^53 + 1: a tie between 2^53 and 2^53+2
    S_d, _ = oracle.sum_squares(x)
    assert S_d == 2.0 ** 53  # ties to even
    x = np.array([big] * 128 + [one, one, one], dtype=np.uint16)  # 2^53 + 3: tie -> 2^53 + 4
    S_d, _ = oracle.sum_squares(x)
    assert S_d == 2.0 ** 53 + 4
    assert S_d == math.fsum([2.0 ** 46] * 128 + [1.0] * 3)


# ----------------------------------------------------------------------------- size


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 15, 16, 17, 43, 171, 4095, 4096, 4097, 4139, 8191, 12288, 12345])
def test_size_closed_form_around_chunk_edges(n):
    rng = np.random.default_rng(n)
    x = workloads.fp32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    mask = rng.random(n) < 0.1
    x[mask] = rng.integers(0, 1 << 16, int(mask.sum())).astype(np.uint16)
    for e0 in (-1, 0, 100, 122, 249):
        s = oracle.compress(x, e0)
        used = s[7] if e0 == -1 else e0
        assert len(s) == closed_form_size(x, int(used))
        st, back = oracle.decompress(s, n)
        assert st == oracle.OK and np.array_equal(back, x)


def test_about_eleven_bits_per_value():
    """No escapes: 16 -> about 11 bits per value, about 31% less volume (the page's ideal):
    3 code bits + 8 sign|mantissa bits per value, plus the header and offset table."""
    rng = np.random.default_rng(5)
    n = 1 << 20
    e0 = 122
    exps = rng.integers(e0, e0 + 7, n)
    x = ((rng.integers(0, 2, n) << 15) | (exps << 7) | rng.integers(0, 128, n)).astype(np.uint16)
    s = oracle.compress(x, e0)
    bits_per_value = 8 * len(s) / n
    assert 11.0 <= bits_per_value < 11.02  # 3 + 8 bits, plus 8 table bytes per 4096 values
    assert abs((1 - len(s) / (2 * n)) - 0.31) < 0.005
    assert len(s) == closed_form_size(x, e0)


def test_worst_case_matches_max_stream_bytes():
    for n in (1, 4096, 4097, 10000):
        x = np.zeros(n, np.uint16)  # exponent 0 is outside every window with e0 >= 1
        s = oracle.compress(x, 5)
        assert len(s) == oracle.max_stream_bytes(n)


# ----------------------------------------------------------------------------- round trips


def test_all_patterns_round_trip_every_base():
    x = workloads.all_patterns()
    for e0 in [-1] + list(range(250)):
        s = oracle.compress(x, e0)
        used = int(s[7])
        if e0 >= 0:
            assert used == e0
        assert len(s) == closed_form_size(x, used)
        st, back = oracle.decompress(s, x.size)
        assert st == oracle.OK
        assert np.array_equal(back, x)


def test_every_pattern_as_single_value():
    """One value: the coded form takes at least 48 + 16 + 16 bytes, the raw form 48."""
    x = workloads.all_patterns()
    for b in x:
        one = np.array([b], np.uint16)
        s = oracle.compress(one)
        assert len(s) == 48 and s[6] == 0 and s[32:34].tobytes() == one.tobytes()
        st, back = oracle.decompress(s, 1)
        assert st == oracle.OK and back[0] == b


_ALPHABET = np.array(
    [0x0000, 0x8000, 0x0001, 0x807F, 0x0080, 0x00FF, 0x3C00, 0x3D00, 0x3D80, 0x3E00, 0x3E80,
     0x3F00, 0x3F80, 0xBF80, 0x4000, 0x4080, 0x4100, 0x4180, 0x4200, 0x4280, 0x4300, 0x4380,
     0x7F00, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81, 0x3FFF, 0xBFFF, 0x0100,
     0x1000, 0x2000, 0x3000, 0x3800, 0x3A00, 0x3B00, 0x3B80, 0x3C80, 0x3E7F, 0x3EFF, 0x3F7F,
     0x407F, 0x40FF, 0x417F, 0x41FF, 0x427F, 0x42FF, 0x437F, 0x4400, 0x4500, 0x5000, 0x6000,
     0x7000, 0x7E00, 0xC000, 0xC100, 0xC300, 0xC400, 0xBE00, 0xBD00, 0x3D40],
    dtype=np.uint16)


def test_brute_force_pairs():
    """Every 2-value tensor over a 64-pattern alphabet, under several bases."""
    assert len(set(_ALPHABET.tolist())) == 64
    bases = [-1, 0, 1, 60, 120, 121, 122, 123, 124, 125, 126, 127, 248, 249]
    for a in _ALPHABET:
        for b in _ALPHABET:
            x = np.array([a, b], np.uint16)
            for e0 in bases:
                s = oracle.compress(x, e0)
                assert len(s) == closed_form_size(x, int(s[7]))
                st, back = oracle.decompress(s, 2)
                assert st == oracle.OK and np.array_equal(back, x)


def test_brute_force_triples():
    alpha = _ALPHABET[::4]
    assert alpha.size == 16
    for a in alpha:
        for b in alpha:
            for c in alpha:
                x = np.array([a, b, c], np.uint16)
                for e0 in (-1, 0, 122, 249):
                    s = oracle.compress(x, e0)
                    assert len(s) == closed_form_size(x, int(s[7]))
                    st, back = oracle.decompress(s, 3)
                    assert st == oracle.OK and np.array_equal(back, x)


# ----------------------------------------------------------------------------- canonical form


def _bijection_under_flips(stream, n, positions=None):
    """Every single-bit flip is rejected, or decodes to values whose stream is the flipped one.
    The one exception the format allows: a raw stream is accepted for values whose coded form
    is shorter (the decoder does not recompute the form choice)."""
    accepted = 0
    for pos in (range(len(stream)) if positions is None else positions):
        for bit in range(8):
            t = stream.copy()
            t[pos] ^= 1 << bit
            st, back = oracle.decompress(t, n)
            if st == oracle.OK:
                again = oracle.compress(back, int(t[7]))
                if t[6] == 0 and again[6] != 0:
                    assert len(again) <= len(t), (pos, bit)
                else:
                    assert again.tobytes() == t.tobytes(), (pos, bit)
                accepted += 1
    return accepted


def _interesting_positions(stream):
    """Header, table, chunk 1's fixed part, the escape region, and every 61st byte of chunk 0."""
    return sorted(set(range(64)) | set(range(0, 5696, 61)) | {1599} | set(range(5696, len(stream))))


def test_decoder_accepts_only_canonical_streams(golden_raw, golden_plane, golden_list):
    for e0, values, stream in (golden_raw, golden_plane, golden_list):
        pos = None if stream.size < 100 else _interesting_positions(stream)
        assert _bijection_under_flips(stream, values.size, pos) > 0
    rng = np.random.default_rng(3)
    x = workloads.fp32_to_bf16_bits(rng.standard_normal(300).astype(np.float32))
    s = oracle.compress(x)
    assert s[6] == 12
    _bijection_under_flips(s, x.size)


def test_decoder_rejections_plane(golden_plane):
    """The plane form (chunk 1: five values, two escapes; its section at 5744)."""
    e0, values, stream = golden_plane
    n = values.size
    assert oracle.decompress(stream, n + 1)[0] == oracle.ERR_SIZE_MISMATCH
    assert oracle.decompress(stream[:-16], n)[0] == oracle.ERR_CORRUPT  # truncated
    for pos, val in [(0, 0),          # magic
                     (4, 3),          # version 3
                     (6, 11),         # another chunk size
                     (7, 250),        # base out of range
                     (5744 + 6, 1),   # nonzero plane padding (after 5 bytes)
                     (5744 + 4, 130),  # an escaped value's exponent inside the window
                     (5744 + 1, 129),  # an in-window value's exponent other than e0 + code
                     (5696, 0xCF)]:   # code 0 -> 7: the plane holds 127, inside the window
        t = stream.copy()
        t[pos] = val
        assert oracle.decompress(t, n)[0] == oracle.ERR_CORRUPT, (pos, val)


def test_decoder_rejections_list(golden_list):
    """The list form (chunk 0: one escape, its section at 5728; chunk 1: two, at 5744)."""
    e0, values, stream = golden_list
    n = values.size
    for pos, val in [(5744, 3),       # first position names an in-window value
                     (5746, 2),       # positions not increasing
                     (5744 + 4, 130),  # escape exponent inside the window
                     (5744 + 6, 1),   # nonzero list padding (after 2 + 2 + 1 + 1 bytes)
                     (5696, 0xCF),    # code 0 -> 7: three escapes, the section must be a plane
                     (5728, 0xFE),    # chunk 0's escape names value 4094 (code 0)
                     (1599, 0x60),    # chunk 0's escape loses its code 7
                     (40, 0x71)]:     # chunk 1's escape offset moved
        t = stream.copy()
        t[pos] = val
        assert oracle.decompress(t, n)[0] == oracle.ERR_CORRUPT, (pos, val)


def test_decoder_rejections_raw(golden_raw):
    """The raw form: byte 6 = 0, N = 0, total = 32 + pad16(2n), zero padding."""
    e0, values, stream = golden_raw
    assert oracle.decompress(stream, 6)[0] == oracle.ERR_SIZE_MISMATCH
    assert oracle.decompress(stream[:-16], 5)[0] == oracle.ERR_CORRUPT  # truncated
    for pos, val in [(6, 12),   # read as a coded stream: N = 0 is not ceil(5/4096)
                     (16, 1),   # N = 1 in a raw stream
                     (24, 64),  # total is not 48
                     (42, 1),   # nonzero padding after the 10 value bytes
                     (4, 3),    # version 3
                     (7, 250)]:  # base out of range
        t = stream.copy()
        t[pos] = val
        assert oracle.decompress(t, 5)[0] == oracle.ERR_CORRUPT, (pos, val)


def test_raw_stream_of_a_compressible_tensor_is_accepted(golden_plane):
    """The decoder checks a raw stream's bytes but does not recompute the form choice: the raw
    form of a tensor whose coded form is shorter still decodes to its values."""
    e0, values, stream = golden_plane
    n = values.size
    raw = np.zeros(raw_size(n), np.uint8)
    raw[:4] = np.frombuffer(b"ZCB1", np.uint8)
    raw[4], raw[7] = 4, e0
    raw[8:16] = np.frombuffer(np.uint64(n).tobytes(), np.uint8)
    raw[24:32] = np.frombuffer(np.uint64(raw.size).tobytes(), np.uint8)
    raw[32:32 + 2 * n] = np.frombuffer(values.tobytes(), np.uint8)
    st, back = oracle.decompress(raw, n)
    assert st == oracle.OK and np.array_equal(back, values)


# ----------------------------------------------------------------------------- statistics


def stream_escape_count(s, n):
    """Escapes in a stream, counted from the 3-bit codes of its fixed parts."""
    N = (n + CHUNK - 1) // CHUNK
    base = pad16(32 + 8 * (N + 1))
    k = 0
    for c in range(N):
        m = min(CHUNK, n - c * CHUNK)
        codes = s[base + 5632 * c: base + 5632 * c + (3 * m + 7) // 8]
        bits = np.unpackbits(codes, bitorder="little")[:3 * m].reshape(m, 3)
        k += int(np.all(bits == 1, axis=1).sum())
    return k


def test_gaussian_escape_rate_matches_model():
    """N(0,1): window 122..128, so escapes are |x| < 2^-5 or |x| >= 4."""
    x = workloads.sweep(20)
    s = oracle.compress(x)
    assert s[7] == 122
    k = stream_escape_count(s, x.size)
    p = math.erf(2.0 ** -5 / math.sqrt(2)) + math.erfc(4.0 / math.sqrt(2))
    n = x.size
    assert abs(k - p * n) < 5 * math.sqrt(n * p * (1 - p))
