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


# ------------------------------------------------------------------ SwiGLU + requantisation
# The kernel forms h = SiLU(g) * u in fp32 (fast exponential and divide) and
# the oracle in fp64.  Their h differ by a relative error below 2^-19, so an
# E4M3 code may differ only where the fp64 value, scaled by its block's
# exponent, lies within that distance of a rounding boundary (a midpoint
# between neighbouring E4M3 values); a block's scale byte may differ only
# where its fp64 amax lies that close to a power of two.
_H_REL = 2.0 ** -19


def _flip_allowed(t: np.ndarray) -> np.ndarray:
    table = oracle.e4m3_table()
    mids = (table[1:] + table[:-1]) / 2
    lo = np.searchsorted(mids, t * (1 - _H_REL), side="left")
    hi = np.searchsorted(mids, t * (1 + _H_REL), side="right")
    return hi > lo


def _paired(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """[M, 2I] with the columns in W_gateup's paired order: block j of 128
    columns = gate features 64j..64j+63, then up features 64j..64j+63."""
    M, I = g.shape
    return np.stack([g.reshape(M, I // 64, 64), u.reshape(M, I // 64, 64)], axis=2).reshape(M, 2 * I)


@pytest.mark.parametrize("M,I,seed", [(1, 128, 1), (37, 512, 2), (128, 1280, 3), (200, 256, 4)])
def test_swiglu_quantize_against_oracle(fs, M, I, seed):
    import torch

    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((M, I)) * np.power(10.0, rng.uniform(-2, 1.5, size=(M, 1)))).astype(np.float32)
    u = rng.standard_normal((M, I)).astype(np.float32)
    g[0, :32] = 0.0                                   # a zero block: scale byte 0, codes +-0
    g[-1, 32:64] = -np.abs(g[-1, 32:64]) - 20.0       # SiLU deep in its negative tail
    gu = torch.from_numpy(_paired(g, u)).cuda()
    codes = torch.full((M, I), 0xAB, dtype=torch.uint8, device="cuda")
    nsc = fs.fsops_scale_bytes(M, I, fs.SCALES_TCGEN05)
    scales = torch.zeros((nsc + 64,), dtype=torch.uint8, device="cuda")
    scales[nsc:] = 0xCD
    fs.fsops_swiglu_quantize_mxfp8(gu, M, I, codes, scales)
    torch.cuda.synchronize()
    sc = scales.cpu().numpy()
    assert np.all(sc[nsc:] == 0xCD), "write past the scale buffer"
    got_c = codes.cpu().numpy()
    got_s = oracle.scales_tiled_to_rowmajor(sc[:nsc], M, I)
    want_c, want_s = oracle.swiglu_quantize(np.concatenate([g, u], axis=1).astype(np.float64))
    h = oracle.silu(g.astype(np.float64)) * u.astype(np.float64)
    amax = np.abs(h.reshape(M, I // 32, 32)).max(axis=2)
    lg = np.log2(np.where(amax > 0, amax, 1.0))
    near_pow2 = (amax > 0) & (np.abs(lg - np.round(lg)) < 2 * _H_REL)
    # scales: bit-exact except where amax sits on a power of two
    s_diff = got_s != want_s
    assert not np.any(s_diff & ~near_pow2), np.argwhere(s_diff & ~near_pow2)[:5]
    # codes of blocks whose scale agrees: equal except near a rounding boundary
    same_block = np.repeat(got_s == want_s, 32, axis=1)
    e = want_s.astype(np.int64) - 127
    t = np.abs(h) * np.power(2.0, -np.repeat(e, 32, axis=1))
    allowed = _flip_allowed(t)
    flips = (got_c != want_c) & same_block
    assert not np.any(flips & ~allowed), np.argwhere(flips & ~allowed)[:5]
    # such boundary cases are rare: nearly every code is identical
    assert np.mean(got_c == want_c) > 0.999, np.mean(got_c == want_c)


@pytest.mark.parametrize("I,H,seed", [(64, 128, 5), (2816, 1024, 6), (320, 384, 7)])
def test_gateup_quantize_pairs_rows(fs, I, H, seed):
    """fsops_quantize_mxfp8_gateup writes W_gate and W_up quantised in the
    paired row order, bit for bit the oracle's quantisation of that matrix."""
    import torch

    rng = np.random.default_rng(seed)
    wg = inputs.bf16_bits_from_f32(rng.standard_normal((I, H), dtype=np.float32) / np.sqrt(H))
    wu = inputs.bf16_bits_from_f32(rng.standard_normal((I, H), dtype=np.float32) / np.sqrt(H))
    paired = np.stack([wg.reshape(I // 64, 64, H), wu.reshape(I // 64, 64, H)], axis=1).reshape(2 * I, H)
    oc, os_ = oracle.quantize_bf16(paired)
    codes = torch.full((2 * I, H), 0xAB, dtype=torch.uint8, device="cuda")
    nsc = fs.fsops_scale_bytes(2 * I, H, fs.SCALES_TCGEN05)
    scales = torch.full((nsc + 64,), 0xCD, dtype=torch.uint8, device="cuda")
    fs.fsops_quantize_mxfp8_gateup(to_dev_u16(wg), to_dev_u16(wu), I, H, H, codes, scales)
    torch.cuda.synchronize()
    sc = scales.cpu().numpy()
    assert np.all(sc[nsc:] == 0xCD)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sc[:nsc], oracle.scales_rowmajor_to_tiled(os_))
