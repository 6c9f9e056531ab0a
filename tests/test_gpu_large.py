"""The largest tensor the tests move through the GPU: 2^32 + 4097 values (8.6 GB), whose stream
(about 6.2 GB) puts offsets past 2^32 bytes, chunk indices past 2^20 and value indices past
2^32 (the ragged last chunk, which the encoder reads without a tiled copy, starts at 2^32 + 4096).

The input repeats one 2^20-value N(0, 1) block, so every chunk's bytes can be checked against
the oracle's stream of that block under the same e0: the fixed part and the escape section of
sampled chunks, their offsets (from the block's section sizes), the header and the length.  e0
is the oracle's window rule on the exact sum of squares of the whole tensor, summed per
exponent in integers and rounded once to fp64.  The round trip is compared on the device.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

BLOCK = 1 << 20            # values of the repeated block (256 chunks)
COPIES = 4 * 1024          # whole copies of the block
TAIL = 4097                # then the block's first 4097 values: one full chunk and one value
N_VALUES = COPIES * BLOCK + TAIL


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    if torch.cuda.mem_get_info()[0] < 32 << 30:
        pytest.skip("needs about 26 GB of free device memory")


def exact_sum_of_squares(x):
    """(S * 2^268 as an integer, finite count): x = sig * 2^(E' - 134), E' = max(E, 1), so
    x^2 = sig^2 * 2^(2E' - 268); per-exponent sums of sig^2 are exact in float64 (< 2^53)."""
    E = ((x >> 7) & 0xFF).astype(np.int64)
    m = (x & 0x7F).astype(np.int64)
    finite = E != 255
    sig = np.where(E > 0, 128 + m, m)
    Ep = np.maximum(E, 1)
    T = np.bincount(Ep[finite], weights=(sig[finite] ** 2).astype(np.float64), minlength=256)
    assert T.max() < 2.0 ** 53
    return sum(int(T[e]) << (2 * e) for e in range(1, 255)), int(finite.sum())


def sections(stream, n):
    """Offsets table and per-chunk (fixed part, escape section) bytes of a coded oracle stream."""
    N = oracle.num_chunks(n)
    table = stream[32:32 + 8 * (N + 1)].view(np.uint64).astype(np.int64)
    R0 = oracle.records_base(n)
    fixed = [stream[R0 + 5632 * c: R0 + 5632 * (c + 1)] for c in range(N)]
    secs = [stream[table[c]:table[c + 1]] for c in range(N)]
    return table, fixed, secs


def test_stream_past_four_gigabytes():
    block = workloads.sweep(20)
    S_block, nf_block = exact_sum_of_squares(block)
    S_tail, nf_tail = exact_sum_of_squares(block[:TAIL])
    S = COPIES * S_block + S_tail
    e0 = oracle.select_e0(float(Fraction(S, 1 << 268)), COPIES * nf_block + nf_tail)
    assert e0 == oracle.choose_e0(block) == 122

    want = oracle.compress(block, e0)
    assert want[6] == 12  # the coded form
    b_table, b_fixed, b_secs = sections(want, BLOCK)
    b_sizes = np.diff(b_table)
    b_prefix = np.concatenate([[0], np.cumsum(b_sizes)])
    # the final one-value chunk holds block[4096]: the oracle's stream of the block followed by it
    last = oracle.compress(np.concatenate([block, block[TAIL - 1:TAIL]]), e0)
    assert last[6] == 12
    _, l_fixed, l_secs = sections(last, BLOCK + 1)
    l_fixed, l_sec = l_fixed[-1][:32], l_secs[-1]

    n = N_VALUES
    N = oracle.num_chunks(n)
    R0 = oracle.records_base(n)
    E0 = R0 + 5632 * (N - 1) + (16 + 16)  # fixed parts; the last chunk's is 32 bytes
    total = E0 + COPIES * int(b_prefix[-1]) + int(b_prefix[TAIL // 4096]) + len(l_sec)
    assert total > 1 << 32

    x = np.concatenate([np.tile(block, COPIES), block[:TAIL]])
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    del x
    zc.status(reset=True)
    out, ob = zc.compress(xd)
    assert zc.status(reset=True) == zc.ZC_OK
    assert int(ob.item()) == total

    def dev(lo, hi):
        return out[lo:hi].cpu().numpy()

    hdr = dev(0, 32)
    assert hdr[6] == 12 and hdr[7] == e0
    assert hdr[8:16].view(np.uint64)[0] == n and hdr[16:24].view(np.uint64)[0] == N
    assert hdr[24:32].view(np.uint64)[0] == total

    def offset(c):  # start of chunk c's escape section
        return E0 + (c // 256) * int(b_prefix[-1]) + int(b_prefix[c % 256])

    rng = np.random.default_rng(5)
    sample = sorted(set([0, 1, 255, 256, 257, 12345, N // 2, N - 3, N - 2, N - 1] +
                        [int(c) for c in rng.integers(0, N - 1, 24)]))
    for c in sample:
        assert dev(32 + 8 * c, 40 + 8 * c).view(np.uint64)[0] == offset(c), c
        if c < N - 1:
            assert dev(R0 + 5632 * c, R0 + 5632 * (c + 1)).tobytes() == b_fixed[c % 256].tobytes(), c
            assert dev(offset(c), offset(c) + int(b_sizes[c % 256])).tobytes() == b_secs[c % 256].tobytes(), c
        else:
            assert dev(R0 + 5632 * c, R0 + 5632 * c + 32).tobytes() == l_fixed.tobytes()
            assert dev(offset(c), total).tobytes() == l_sec.tobytes()
    assert dev(32 + 8 * N, 40 + 8 * N).view(np.uint64)[0] == total

    back = zc.decompress(out, n)
    assert zc.status(reset=True) == zc.ZC_OK
    assert bool(torch.equal(back, xd))
