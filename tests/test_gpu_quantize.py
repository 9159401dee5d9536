"""GPU quantiser (fsops_quantize_mxfp8) against the oracle: bit-exact codes
and scales, both scale layouts, random workloads and an edge-case corpus."""
import numpy as np
import pytest

import oracle
from workloads import inputs
from tests._util import to_dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fs():
    import mxfp8_swiglu_mlp_gb300 as fs

    return fs


def _run(fs, bits, layout):
    import torch

    rows, K = bits.shape
    x = to_dev_u16(bits)
    codes = torch.full((rows, K), 0xAB, dtype=torch.uint8, device="cuda")
    nsc = fs.fsops_scale_bytes(rows, K, layout)
    scales = torch.full((nsc + 64,), 0xCD, dtype=torch.uint8, device="cuda")  # 64-byte guard band
    fs.fsops_quantize_mxfp8(x, rows, K, K, codes, scales, layout)
    torch.cuda.synchronize()
    sc = scales.cpu().numpy()
    assert np.all(sc[nsc:] == 0xCD), "write past the scale buffer"
    return codes.cpu().numpy(), sc[:nsc]


def _check(fs, bits):
    rows, K = bits.shape
    oc, os_ = oracle.quantize_bf16(bits)
    c, s = _run(fs, bits, fs.SCALES_ROWMAJOR)
    assert np.array_equal(c, oc)
    assert np.array_equal(s.reshape(rows, K // 32), os_)
    if K % 128 == 0:
        c2, s2 = _run(fs, bits, fs.SCALES_TCGEN05)
        assert np.array_equal(c2, oc)
        assert np.array_equal(s2, oracle.scales_rowmajor_to_tiled(os_))   # padding bytes are zero too


@pytest.mark.parametrize("rows,K", [(1, 128), (17, 256), (128, 1024), (300, 384), (2816, 1024), (1, 32)])
def test_random_weights_bit_exact(fs, rows, K):
    wl = inputs.make_workload_small("q", 1, K, rows, seed=rows + K)
    rng = np.random.Generator(np.random.PCG64(rows * 7 + K))
    w = rng.standard_normal((rows, K), dtype=np.float32) / np.sqrt(K)
    w.reshape(-1)[rng.choice(rows * K, max(1, rows * K // 1000), replace=False)] *= 20
    _check(fs, inputs.bf16_bits_from_f32(w))


def _edge_corpus() -> np.ndarray:
    """Blocks of 32 bf16 values hitting every special case of the rule."""
    f = lambda v: inputs.bf16_bits_from_f32(np.asarray(v, np.float32))
    blocks = []
    blocks.append(np.zeros(32, np.uint16))                                 # all zero -> byte 0
    b = np.zeros(32, np.uint16); b[::2] = 0x8000; blocks.append(b)         # negative zeros
    sub = np.arange(1, 33, dtype=np.uint16); blocks.append(sub)            # bf16 subnormals
    blocks.append(sub | 0x8000)                                            # negative subnormals
    amax = 1.0
    ties = [amax, 76 / 256, 68 / 256, 1.5 * 2 ** -17, 2 ** -18, -2 ** -18, 15 * 2 ** -18, 0.3]
    blocks.append(f(np.pad(ties, (0, 32 - len(ties)))))                    # E4M3 ties (amax 1)
    blocks.append(f(np.pad([1.9, 1.0, 1.78125, -1.99], (0, 28))))          # saturation
    blocks.append(f(np.full(32, 2.0 ** 100)))                              # large
    blocks.append(f(np.pad([2.0 ** -126, 2.0 ** -130], (0, 30))))          # tiny, clamped scale
    blocks.append(f(np.linspace(-448, 448, 32)))                           # amax 448 exactly
    blocks.append(f(np.float32(3.3895314e38) * np.linspace(-1, 1, 32)))    # near bf16 max
    rng = np.random.default_rng(0)
    for e in (-140, -100, -20, 0, 20, 100, 126):                           # random magnitudes
        blocks.append(f(rng.standard_normal(32) * 2.0 ** e))
    corpus = np.concatenate(blocks)
    n = (len(corpus) + 127) // 128 * 128
    corpus = np.pad(corpus, (0, n - len(corpus)))
    return corpus.reshape(-1, 128)


def test_edge_corpus_bit_exact(fs):
    _check(fs, _edge_corpus())


def test_all_bf16_patterns(fs):
    """All 65536 bf16 bit patterns except Inf/NaN, in blocks of mixed magnitude."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]
    n = len(bits) // 128 * 128
    _check(fs, bits[:n].reshape(-1, 128))


def test_strided_input(fs):
    import torch

    rng = np.random.default_rng(3)
    full = inputs.bf16_bits_from_f32(rng.standard_normal((40, 384), dtype=np.float32))
    x = to_dev_u16(full)
    codes = torch.empty((40, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty(fs.fsops_scale_bytes(40, 256, fs.SCALES_ROWMAJOR), dtype=torch.uint8, device="cuda")
    fs.fsops_quantize_mxfp8(x, 40, 256, 384, codes, scales, fs.SCALES_ROWMAJOR)
    oc, os_ = oracle.quantize_bf16(full[:, :256])
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().reshape(40, 8), os_)
