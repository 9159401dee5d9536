"""FP8 with 128 x 128 block scales (the "bsgemm" format): the GPU quantiser
bit for bit against the oracle's quantize_blockscale, and the GEMM against the
oracle's gemm_blockscale, end to end from bf16 A and W."""
import numpy as np
import pytest

import oracle
from workloads import inputs
from tests._util import to_dev_u16, from_dev_bf16, bf16_bits_to_f64, rel_l2, max_abs_norm, REL_L2_TOL, MAX_ABS_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fs():
    import mxfp8_swiglu_mlp_gb300 as fs

    return fs


def _bits(rng, rows, K, scale=1.0, spread=None, zero_rows=()):
    v = rng.standard_normal((rows, K)).astype(np.float32) * np.float32(scale)
    if spread is not None:
        v *= np.power(10.0, rng.uniform(*spread, size=(rows, 1))).astype(np.float32)
    for r in zero_rows:
        v[r] = 0.0
    return inputs.bf16_bits_from_f32(v)


def _gpu_quantize(fs, bits, block_rows):
    import torch

    rows, K = bits.shape
    codes, scales = fs.quantize_blockscale(to_dev_u16(bits), block_rows)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("rows,K,block_rows,seed", [(1, 128, 1, 1), (37, 384, 1, 2), (128, 256, 128, 3),
                                                    (300, 384, 128, 4), (200, 1280, 1, 5)])
def test_blockscale_quantize_bit_exact(fs, rows, K, block_rows, seed):
    rng = np.random.default_rng(seed)
    bits = _bits(rng, rows, K, spread=(-3, 3), zero_rows=(0,) if rows > 1 else ())
    c, s = _gpu_quantize(fs, bits, block_rows)
    oc, os_ = oracle.quantize_blockscale(bits, block_rows)
    assert np.array_equal(s.view(np.uint32), os_.astype(np.float32).view(np.uint32))
    assert np.array_equal(c, oc)


def test_blockscale_quantize_edge_values(fs):
    """Subnormal bf16 inputs, values at the saturation edge, negative zeros,
    a block of one outlier, huge magnitudes."""
    f = lambda v: inputs.bf16_bits_from_f32(np.asarray(v, np.float32))
    rows = []
    rows.append(np.arange(1, 129, dtype=np.uint16))                        # bf16 subnormals
    rows.append(np.arange(1, 129, dtype=np.uint16) | 0x8000)
    rows.append(f(np.linspace(-448.0, 448.0, 128)))
    r = np.zeros(128, np.float32); r[7] = 3.0e5; rows.append(f(r))          # one outlier, rest zero
    r = np.zeros(128, np.uint16); r[::3] = 0x8000; rows.append(r)           # negative zeros only
    rows.append(f(np.full(128, 2.0 ** 120)))
    rows.append(f(np.random.default_rng(9).standard_normal(128) * 2.0 ** -130))
    bits = np.stack(rows)
    for block_rows in (1, 128):
        c, s = _gpu_quantize(fs, bits, block_rows)
        oc, os_ = oracle.quantize_blockscale(bits, block_rows)
        assert np.array_equal(s.view(np.uint32), os_.astype(np.float32).view(np.uint32))
        assert np.array_equal(c, oc), block_rows


def _run_gemm(fs, a_bits, w_bits, c_f32):
    import torch

    M, K = a_bits.shape
    N = w_bits.shape[0]
    ac, asc = fs.quantize_blockscale(to_dev_u16(a_bits), 1)
    wc, wsc = fs.quantize_blockscale(to_dev_u16(w_bits), 128)
    n = fs.fsops_blockscale_gemm_workspace_bytes(M, N, K)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    ws_ptr = ws.data_ptr() + (-ws.data_ptr()) % 256
    c = torch.empty((M, N), dtype=torch.float32 if c_f32 else torch.bfloat16, device="cuda")
    outs = []
    for _ in range(2):  # the second call runs on what the first left in the workspace
        c.fill_(7.0)
        fs.fsops_fp8_blockscale_gemm(ac, asc, wc, wsc, c, fs.DTYPE_F32 if c_f32 else fs.DTYPE_BF16, M, N, K,
                                     ws_ptr, n)
        torch.cuda.synchronize()
        assert fs.fsops_read_kernel_status(ws_ptr) == 0
        outs.append(c.cpu().numpy().astype(np.float64) if c_f32 else bf16_bits_to_f64(from_dev_bf16(c)))
    assert int(ws[(ws_ptr - ws.data_ptr()):][:n].count_nonzero()) == 0, "workspace not left zero"
    return outs


# (M, N, K): whole row tiles per block (few units), and tiles split over many
# blocks (N = 1024, K = 5120: 320 units), ragged token counts up to 128
GEMMS = [(1, 128, 128), (5, 384, 512), (16, 1024, 1280), (33, 256, 640), (64, 512, 384), (100, 640, 256),
         (128, 384, 1024), (16, 1024, 5120), (3, 8192, 128)]


@pytest.mark.parametrize("M,N,K", GEMMS)
def test_blockscale_gemm_fp32_out(fs, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    a = _bits(rng, M, K, spread=(-1, 1))
    w = _bits(rng, N, K, scale=1.0 / np.sqrt(K))
    want = oracle.gemm_blockscale(a, w)["c"]
    for got in _run_gemm(fs, a, w, True):
        assert rel_l2(got, want) < 1e-5, rel_l2(got, want)
        for m in range(M):
            assert rel_l2(got[m], want[m]) < 1e-5


@pytest.mark.parametrize("M,N,K", GEMMS[:5])
def test_blockscale_gemm_bf16_out(fs, M, N, K):
    rng = np.random.default_rng(M * 11 + N + K)
    a = _bits(rng, M, K)
    w = _bits(rng, N, K, scale=1.0 / np.sqrt(K))
    want = bf16_bits_to_f64(oracle.gemm_blockscale(a, w)["c_bf16"])
    for got in _run_gemm(fs, a, w, False):
        assert rel_l2(got, want) <= REL_L2_TOL
        assert max_abs_norm(got, want) <= MAX_ABS_TOL
        assert np.mean(got == want) > 0.99


def test_blockscale_gemm_decode_shape_sampled(fs):
    """The H = 5120, I = 17408 gate/up shape (N = 34816, K = 5120) at 16
    tokens: the whole output is finite, and 256 outputs of 2 sampled 128-row
    blocks of W match the oracle, which quantises those blocks itself."""
    import torch

    M, N, K = 16, 34816, 5120
    g = torch.Generator(device="cuda").manual_seed(21)
    w = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    rng = np.random.default_rng(22)
    a = _bits(rng, M, K)
    ac, asc = fs.quantize_blockscale(to_dev_u16(a), 1)
    wc, wsc = fs.quantize_blockscale(w, 128)
    n = fs.fsops_blockscale_gemm_workspace_bytes(M, N, K)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    ws_ptr = ws.data_ptr() + (-ws.data_ptr()) % 256
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fs.fsops_fp8_blockscale_gemm(ac, asc, wc, wsc, c, fs.DTYPE_F32, M, N, K, ws_ptr, n)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(c).all())
    for blk in (3, 201):
        rows = slice(blk * 128, blk * 128 + 128)
        w_bits = w[rows].view(torch.int16).cpu().numpy().view(np.uint16)
        want = oracle.gemm_blockscale(a, w_bits)["c"]
        got = c[:, rows].cpu().numpy().astype(np.float64)
        assert rel_l2(got, want) < 1e-5, rel_l2(got, want)
    del w, wc, wsc, ws, c
    torch.cuda.empty_cache()
