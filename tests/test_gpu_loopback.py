"""zc_loopback: compress and decompress in one launch, chunks decoded as their bytes reach the
stream (the split-send pipeline with the transfer taken out).  Against the oracle: the final
stream equals oracle.compress byte for byte (coded or raw), and the decoded values equal the
input bit for bit; the decoding's bounded wait reports ZC_ERR_TIMEOUT on a planted stall."""
import numpy as np
import pytest

import oracle
from lossless_bf16_compression_gb300 import binding as zc
from lossless_bf16_compression_gb300 import workloads

from gpu_helpers import require_gpu, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def mixed(n, seed, sigma=0.02, frac=0.1):
    rng = np.random.default_rng(seed)
    x = workloads.fp32_to_bf16_bits((rng.standard_normal(n) * sigma).astype(np.float32))
    mask = rng.random(n) < frac
    x[mask] = workloads.random_patterns(int(mask.sum()), seed + 1)
    return x


def check_loopback(x, base=-1):
    xd = to_device(x)
    zc.status(reset=True)
    out, ob, values = zc.loopback(xd, base)
    st = zc.status(reset=True)
    assert st == zc.ZC_OK, zc.ERROR_NAMES.get(st, st)
    assert np.array_equal(values.cpu().numpy().view(np.uint16), x), "decoded values differ from the input"
    total = int(ob.item())
    want = oracle.compress(x, base)
    got = out[:total].cpu().numpy()
    assert total == want.size and got.tobytes() == want.tobytes(), "stream differs from the oracle"
    return got


@pytest.mark.parametrize("n", [1, 7, 4095, 4096, 4097, 3 * 4096 + 5, 100_003])
@pytest.mark.parametrize("base", [-1, 116])
def test_sizes(n, base):
    check_loopback(mixed(n, 300 + n), base)


def test_all_patterns_and_planes():
    check_loopback(workloads.all_patterns())
    x = np.concatenate([np.full(6 * 4096, 0x3F80, np.uint16), workloads.random_patterns(2 * 4096 + 50, 3)])
    s = check_loopback(x, 127)  # escape-free chunks, then chunks with planes: the coded form
    assert s[6] == 12


@pytest.mark.parametrize("name", ["weight_1m", "grad_bucket_4096x14336", "moe_a2a_16384x7168", "adversarial_256m"])
def test_workloads(name):
    check_loopback(workloads.make(name))


@pytest.mark.parametrize("k", [20, 26, 29])
def test_sweep(k):
    check_loopback(workloads.sweep(k))


def test_exact_e0_in_the_loopback():
    """A tensor on a switching point of the window rule: the encode kernel's first phase settles
    e0 exactly before any CTA codes or decodes (the decoding-only CTAs take part too)."""
    from test_gpu_parity import _near_boundary_tensor

    x = _near_boundary_tensor(-8, (1 << 20) + 3, 192, 1e-9)
    s = check_loopback(x)
    assert s[7] == oracle.choose_e0(x)


def loopback_fallback_word(out, n):
    """The fallback word of the loopback's control block (bytes 240..243; the workspace is the
    last workspace-size bytes of the loopback's buffer)."""
    ws_bytes = zc.zc_max_compressed_bytes(n) - (zc.zc_max_stream_bytes(n) + 255) // 256 * 256
    at = zc.zc_loopback_bytes(n) - ws_bytes
    return int(out[at + 240:at + 244].cpu().numpy().view(np.uint32)[0])


def test_speculative_loopback_guess_holds():
    """From 512 full chunks on, the loopback takes the speculative route: it codes and decodes
    with the sample's e0, which the whole tensor's sums then confirm."""
    x = workloads.sweep(23)
    xd = to_device(x)
    zc.status(reset=True)
    out, ob, values = zc.loopback(xd)
    assert zc.status(reset=True) == zc.ZC_OK
    assert loopback_fallback_word(out, x.size) == 0
    assert np.array_equal(values.cpu().numpy().view(np.uint16), x)
    want = oracle.compress(x)
    assert out[:int(ob.item())].cpu().numpy().tobytes() == want.tobytes()


def test_speculative_loopback_falls_back():
    """A sample that names the wrong e0 (120 for a tensor of 122): the chunks coded and decoded
    with 120 are coded and decoded again after the statistics pass, and the final stream and
    values are the oracle's and the input."""
    from test_gpu_speculative import misleading_sample

    x = misleading_sample((1 << 25) + 4096 * 3 + 9, 21)
    xd = to_device(x)
    zc.status(reset=True)
    out, ob, values = zc.loopback(xd)
    assert zc.status(reset=True) == zc.ZC_OK
    assert loopback_fallback_word(out, x.size) == 1
    assert np.array_equal(values.cpu().numpy().view(np.uint16), x)
    want = oracle.compress(x)
    assert out[:int(ob.item())].cpu().numpy().tobytes() == want.tobytes()


@pytest.mark.parametrize("stalled", [0, 37])
def test_decode_wait_is_bounded(stalled):
    x = workloads.sweep(18)  # 64 chunks
    xd = to_device(x)
    out = torch.empty(zc.zc_loopback_bytes(x.size), dtype=torch.uint8, device="cuda")
    values = torch.empty(x.size, dtype=torch.int16, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    zc.status(reset=True)
    assert zc.zc_loopback_stall_test(xd.data_ptr(), x.size, -1, out.data_ptr(), ob.data_ptr(), values.data_ptr(), s,
                                     stalled, 2000) == zc.ZC_OK
    assert zc.zc_status(s, 1) == zc.ZC_ERR_TIMEOUT
    check_loopback(x)  # the context is still usable
