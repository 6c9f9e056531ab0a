"""Planted mistakes: every plausible slip in the oracle must fail an independent check.

Each mutant is one small edit of oracle/zc_oracle.c (a wrong shift or index, an off-by-one
window, a dropped case, a transposed field, the wrong side of the list/plane rule ...),
compiled on the CPU into a private library.  The checks below do not use the oracle: they are
the hand-derived streams in tests/golden, math.fsum for the sum of squares, the window rule
evaluated in Python for constant tensors, the size formula written out in Python, and round
trips.  The unmutated source must pass all of them and every mutant must fail at least one.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

from conftest import ROOT, golden_stream

SRC = os.path.join(ROOT, "oracle", "zc_oracle.c")
C2 = float.fromhex("0x1.79a1e790e0f01p-10")

MUTANTS = {
    "plane_rule_ge": ("static int exponent_plane(uint64_t m, uint64_t k) { return 3u * k > m; }",
                      "static int exponent_plane(uint64_t m, uint64_t k) { return 3u * k >= m; }"),
    "plane_escapes_only": ("        esc[i] = (uint8_t)E; /* every exponent, in value order */",
                           "        if (code == 7u) esc[i] = (uint8_t)E;"),
    "plane_unchecked": ("        if (exponent_code(E, e0) != code) return ZCO_ERR_CORRUPT; /* the plane must agree with the codes */",
                        "        (void)code;"),
    "window_one_narrower": ("  return (d >= 0 && d < WINDOW) ? (unsigned)d : 7u;",
                            "  return (d >= 0 && d < WINDOW - 1) ? (unsigned)d : 7u;"),
    "code_bits_reversed": ("        if ((code >> b) & 1u) set_bit(codes, 3u * i + b); /* code i at bits [3i, 3i+3) */",
                           "        if ((code >> b) & 1u) set_bit(codes, 3u * i + (2u - b));"),
    "sign_bit_shift": ("      sm[i] = (uint8_t)((bf16_sign(xc[i]) << 7) | bf16_mantissa(xc[i]));",
                       "      sm[i] = (uint8_t)((bf16_sign(xc[i]) << 6) | bf16_mantissa(xc[i]));"),
    "position_off_by_one": ("        put_u16(esc + 2u * r, (uint16_t)i); /* positions, ascending */",
                            "        put_u16(esc + 2u * r, (uint16_t)(i + 1u));"),
    "exponents_before_positions": ("        esc[2u * k + r] = (uint8_t)E;       /* full exponents, same order */",
                                   "        esc[r] = (uint8_t)E;"),
    "offset_table_shifted": ("    put_u64(out + HEADER_BYTES + 8u * c, esc_pos);",
                             "    put_u64(out + HEADER_BYTES + 8u * c, esc_pos + 16u);"),
    "version_3": ("#define FORMAT_VERSION 4u", "#define FORMAT_VERSION 3u"),
    "raw_rule_ge": ("  const int raw_form = coded > raw; /* R7: ties keep the coded form */",
                    "  const int raw_form = coded >= raw;"),
    "raw_never": ("  const int raw_form = coded > raw; /* R7: ties keep the coded form */",
                  "  const int raw_form = 0; (void)raw;"),
    "raw_values_byte_swapped": ("    for (uint64_t i = 0; i < n; ++i) put_u16(out + HEADER_BYTES + 2u * i, x[i]);",
                                "    for (uint64_t i = 0; i < n; ++i) put_u16(out + HEADER_BYTES + 2u * i, (uint16_t)((x[i] << 8) | (x[i] >> 8)));"),
    "raw_unpadded": ("uint64_t zco_raw_stream_bytes(uint64_t n) { return HEADER_BYTES + pad16(2u * n); }",
                     "uint64_t zco_raw_stream_bytes(uint64_t n) { return HEADER_BYTES + 2u * n; }"),
    "raw_form_marker": ("#define RAW_FORM 0u /* header byte 6 of a raw stream (R7) */", "#define RAW_FORM 1u"),
    "coded_length_unbounded": ("  if (total > in_bytes || total > zco_raw_stream_bytes(n) || total < escape_base(n)) return ZCO_ERR_CORRUPT;",
                               "  if (total > in_bytes || total < escape_base(n)) return ZCO_ERR_CORRUPT;"),
    "floor_half_truncates": ("static int floor_half(int v) { return v >= 0 ? v / 2 : -((-v + 1) / 2); }",
                             "static int floor_half(int v) { return v / 2; }"),
    "constant_typo": ("static const double WINDOW_C2 = 0x1.79a1e790e0f01p-10;",
                      "static const double WINDOW_C2 = 0x1.79a1e790e0f01p-9;"),
}


def _build(tmp_path, name, edit):
    src = open(SRC).read()
    if edit is not None:
        old, new = edit
        assert src.count(old) == 1, f"{name}: the edit target must occur once in the oracle"
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    c = d / "zc_oracle.c"
    c.write_text(src)
    so = d / "lib.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                    f"-I{os.path.join(ROOT, 'oracle')}", "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    u64, i64, c_int, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.zco_max_stream_bytes.argtypes = [u64]
    lib.zco_max_stream_bytes.restype = u64
    lib.zco_sum_squares.argtypes = [p, u64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(u64)]
    lib.zco_sum_squares.restype = c_int
    lib.zco_compress.argtypes = [p, u64, c_int, p, u64]
    lib.zco_compress.restype = i64
    lib.zco_decompress.argtypes = [p, u64, p, u64]
    lib.zco_decompress.restype = c_int
    return lib


class Oracle:
    def __init__(self, lib):
        self.lib = lib

    def compress(self, x, base=-1):
        cap = int(self.lib.zco_max_stream_bytes(x.size)) + 4096  # room for a mutant that overruns
        out = np.zeros(cap, np.uint8)
        r = self.lib.zco_compress(x.ctypes.data, x.size, base, out.ctypes.data, cap)
        return None if r < 0 else out[:r].copy()

    def decompress(self, s, n):
        out = np.zeros(max(n, 1), np.uint16)
        st = self.lib.zco_decompress(s.ctypes.data, s.size, out.ctypes.data, n)
        return st, out[:n]

    def sum_squares(self, x):
        S, nf = ctypes.c_double(), ctypes.c_uint64()
        self.lib.zco_sum_squares(x.ctypes.data, x.size, ctypes.byref(S), ctypes.byref(nf))
        return S.value, nf.value


# ----------------------------------------------------------------------------- independent checks


def pad16(v):
    return (v + 15) // 16 * 16


def bf16_value(b):
    E, mant, sign = (b >> 7) & 0xFF, b & 0x7F, -1.0 if b >> 15 else 1.0
    return sign * (mant * 2.0 ** -133 if E == 0 else (128 + mant) * 2.0 ** (E - 134))


def size_formula(x, e0):
    """The coded form's length from the size formula, or the raw form's when that is shorter."""
    n = x.size
    N = (n + 4095) // 4096
    E = (x.astype(np.int64) >> 7) & 0xFF
    esc = (E < e0) | (E > e0 + 6)
    total = pad16(32 + 8 * (N + 1))
    for c in range(N):
        m = min(4096, n - 4096 * c)
        k = int(esc[4096 * c:4096 * c + m].sum())
        total += pad16((3 * m + 7) // 8) + pad16(m) + (pad16(m) if 3 * k > m else pad16(3 * k))
    return min(total, 32 + pad16(2 * n))


# The coded form of the five values of tiny_raw_stream.txt under e0 = 127, worked out by hand
# there (96 bytes: header, table, codes, sign|mantissa plane, an exponent plane).  It is longer
# than the raw form (48 bytes), so no encoder writes it and the decoder must reject it.
NONCANONICAL_CODED = bytes.fromhex(
    "5a43423104000c7f0500000000000000" "01000000000000006000000000000000"
    "50000000000000006000000000000000" "c87d0000000000000000000000000000"
    "00a00048410000000000000000000000" "7f800085ff0000000000000000000000")


def window_rule_for_constant(v, n):
    """e0 for n copies of the finite nonzero value v: q = v^2 exactly, y = q * c^2 rounded."""
    y = (v * v) * C2
    e = math.frexp(y)[1] - 1  # floor(log2(y)) for a positive normal y
    return min(max(math.floor(e / 2) + 127, 0), 249)


def checks(o):
    """Names of the independent checks that fail for this oracle build."""
    failed = []
    for fixture in ("tiny_raw_stream.txt", "two_chunk_plane_stream.txt", "two_chunk_list_stream.txt"):
        e0, vals, want = golden_stream(fixture)
        got = o.compress(vals, e0)
        if got is None or got.tobytes() != want.tobytes():
            failed.append(f"golden {fixture}")
        st, back = o.decompress(want, vals.size)
        if st != 0 or not np.array_equal(back, vals):
            failed.append(f"golden decode {fixture}")
    e0, vals, bad = golden_stream("two_chunk_plane_stream.txt")  # a plane byte moved into the window
    bad[5744 + 1] = 129
    if o.decompress(bad, vals.size)[0] == 0:
        failed.append("plane corruption accepted")
    if o.decompress(np.frombuffer(NONCANONICAL_CODED, np.uint8).copy(), 5)[0] == 0:
        failed.append("coded stream longer than the raw form accepted")
    tie = np.full(37, 0x3F80, np.uint16)  # coded: 48 + 16 + 48 = 112 bytes; raw: 32 + 80 = 112
    s = o.compress(tie, 127)
    if s is None or len(s) != 112 or s[6] != 12:
        failed.append("a tie keeps the coded form")
    rng = np.random.default_rng(11)
    samples = [rng.integers(0, 1 << 16, 5000).astype(np.uint16),
               rng.integers(0, 0x0100, 3000).astype(np.uint16),  # subnormals and zeros
               (rng.integers(0x3E00, 0x4100, 4097)).astype(np.uint16)]
    for x in samples:
        fin = [bf16_value(int(b)) for b in x if (int(b) >> 7) & 0xFF != 0xFF]
        S, nf = o.sum_squares(x)
        if nf != len(fin) or S != math.fsum(v * v for v in fin):
            failed.append("sum of squares")
            break
    for b in (0x3F80, 0x3FC0, 0x0D00, 0x2A10, 0x5F00, 0x0180):  # constants, small and large
        x = np.full(3, b, np.uint16)
        s = o.compress(x)
        if s is None or int(s[7]) != window_rule_for_constant(bf16_value(b), 3):
            failed.append(f"e0 of constant {b:#06x}")
            break
    for n, e0 in ((1, 127), (100, 122), (4097, 5), (9000, 122)):
        x = rng.integers(0, 1 << 16, n).astype(np.uint16)
        s = o.compress(x, e0)
        if s is None or len(s) != size_formula(x, e0):
            failed.append("size formula")
            break
        st, back = o.decompress(s, n)
        if st != 0 or not np.array_equal(back, x):
            failed.append("round trip")
            break
    for n in (1, 5000, 12345):
        if o.lib.zco_max_stream_bytes(n) != 32 + pad16(2 * n):
            failed.append("worst-case size")
            break
    for m in range(1, 24):  # the list-or-plane boundary, both sides of 3k = m
        for k in (m // 3, m // 3 + 1):
            if k > m:
                continue
            # a chunk of 1.0s keeps the coded form; then k zeros (exponent 0, escapes for
            # e0 = 127) and 1.0s (exponent 127, code 0)
            x = np.array([0x3F80] * 4096 + [0x0000] * k + [0x3F80] * (m - k), np.uint16)
            if 3 * k > m:  # a plane: every exponent in value order
                section = bytes([0] * k + [127] * (m - k))
            else:  # a list: u16 positions 0..k-1, then k exponent bytes 0
                section = b"".join(i.to_bytes(2, "little") for i in range(k)) + bytes(k)
            section += bytes(pad16(len(section)) - len(section))
            s = o.compress(x, 127)
            ok = s is not None and len(s) == size_formula(x, 127) and o.decompress(s, x.size)[0] == 0
            if not ok or (section and s[len(s) - len(section):].tobytes() != section):
                failed.append("list/plane boundary")
                break
        else:
            continue
        break
    return failed


def test_unmutated_oracle_passes_every_check(tmp_path):
    assert checks(Oracle(_build(tmp_path, "original", None))) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    failed = checks(Oracle(_build(tmp_path, name, MUTANTS[name])))
    assert failed, f"mutant {name} passes every independent check"
