"""The encoder's ring placement (lossless_bf16_compression_gb300/csrc/zc_ring.h), replayed on the
CPU.  The same header the kernel includes is compiled here with g++ into a small shim, and random
traces of sections placed and retired in order check what the kernel relies on: every section
lies inside the ring, never overlaps a section still waiting, and a drained ring takes any
section (so no coding thread can wait for room that never comes)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "lossless_bf16_compression_gb300", "csrc")
MAX_SECTION = 4096  # an exponent plane of a full chunk, the largest escape section

SHIM = r"""
#include "zc_ring.h"
extern "C" void place(unsigned head, unsigned need, unsigned ring, unsigned* where, unsigned* gap) {
  zc::ring_place(head, need, ring, where, gap);
}
extern "C" int fits(unsigned waiting, unsigned gap, unsigned need, unsigned ring) {
  return zc::ring_fits(waiting, gap, need, ring) ? 1 : 0;
}
"""


@pytest.fixture(scope="module")
def ring(tmp_path_factory):
    d = tmp_path_factory.mktemp("ring")
    src = d / "shim.cpp"
    src.write_text(SHIM)
    so = d / "shim.so"
    subprocess.run(["g++", "-std=c++17", "-O2", "-fPIC", "-shared", f"-I{CSRC}", "-o", str(so), str(src)], check=True)
    lib = ctypes.CDLL(str(so))
    u = ctypes.c_uint
    lib.place.argtypes = [u, u, u, ctypes.POINTER(u), ctypes.POINTER(u)]
    lib.place.restype = None
    lib.fits.argtypes = [u, u, u, u]
    lib.fits.restype = ctypes.c_int

    def place(head, need, R):
        w, g = u(), u()
        lib.place(head, need, R, ctypes.byref(w), ctypes.byref(g))
        return w.value, g.value

    return place, lambda waiting, gap, need, R: bool(lib.fits(waiting, gap, need, R))


def encoder_ring_bytes():
    """The ring size the encoder is built with by default (ZC_ENCODE_RING_KB KiB)."""
    text = open(os.path.join(CSRC, "zc_encode.cu")).read()
    assert re.search(r"constexpr unsigned kRingBytes = ZC_ENCODE_RING_KB \* 1024;", text)
    return 1024 * int(re.search(r"#define ZC_ENCODE_RING_KB (\d+)", text).group(1))


def test_edge_cases(ring):
    place, fits = ring
    R = encoder_ring_bytes()
    assert R >= 2 * MAX_SECTION
    assert place(R, 1024, R) == (0, 0)          # a section that ended exactly at the end
    assert place(R - 256, 1024, R) == (0, 256)  # does not fit before the end: skip the rest
    assert place(R - 256, 256, R) == (R - 256, 0)
    assert place(100, 0, R) == (100, 0)         # an empty section takes no room
    assert not fits(R - 64, 0, 128, R) and fits(R - 128, 0, 128, R)
    for head in range(0, R + 1, 16):            # a drained ring takes any section
        for need in range(0, MAX_SECTION + 1, 16):
            w, g = place(head, need, R)
            assert fits(0, g, need, R) and w + need <= R


@pytest.mark.parametrize("seed", range(8))
def test_random_traces(ring, seed):
    place, fits = ring
    R = encoder_ring_bytes()
    rng = np.random.default_rng(seed)
    head = made = freed = 0
    fifo = []  # (where, size, gap) of the sections waiting, oldest first
    placed = 0
    for _ in range(6000):
        kind = rng.random()
        need = 16 * int(rng.integers(0, 257)) if kind < 0.3 else (MAX_SECTION if kind < 0.4 else 16 * int(rng.integers(0, 90)))
        w, g = place(head, need, R)
        while not fits(made - freed, g, need, R):  # the coding threads wait; the retiring warp frees in order
            assert fifo, "a drained ring refused a section"
            _, s, gg = fifo.pop(0)
            freed += s + gg
        assert 0 <= w and w + need <= R, (head, need, w)
        if need:
            for (w2, s2, _) in fifo:
                assert w + need <= w2 or w2 + s2 <= w or s2 == 0, "overlaps a waiting section"
        if g:
            assert w == 0 and head + need > R
        fifo.append((w, need, g))
        made += g + need
        head = w + need
        placed += 1
        while fifo and rng.random() < 0.4:
            _, s, gg = fifo.pop(0)
            freed += s + gg
        assert made - freed == sum(s + gg for (_, s, gg) in fifo)
    assert placed == 6000
