"""Block-scaled MXFP8 GEMM (fsops_mxfp8_gemm / _ex) against the oracle's fp64
GEMM of the dequantised operands."""
import numpy as np
import pytest

import oracle
from workloads import inputs
from tests._util import to_dev_u16, from_dev_bf16, bf16_bits_to_f64, rel_l2, max_abs_norm, control_words_clear

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fs():
    import mxfp8_swiglu_mlp_gb300 as fs

    return fs


def _operands(M, N, K, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    a = inputs.bf16_bits_from_f32(rng.standard_normal((M, K), dtype=np.float32))
    w = rng.standard_normal((N, K), dtype=np.float32) / np.sqrt(K)
    w.reshape(-1)[rng.choice(N * K, max(1, N * K // 1000), replace=False)] *= 20
    return a, inputs.bf16_bits_from_f32(w)


def _gpu_gemm(fs, a_bits, b_bits, c_f32=False, prequant=False):
    import torch

    M, K = a_bits.shape
    N = b_bits.shape[0]
    bc, bs = fs.quantize_weight(to_dev_u16(b_bits))
    ws_n = fs.fsops_gemm_workspace_bytes(M, N, K)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32 if c_f32 else torch.bfloat16, device="cuda")
    outs = []
    for _ in range(2):  # the second call reuses the workspace the first one left behind
        if prequant:
            ac, asc = fs.quantize_weight(to_dev_u16(a_bits))
            fs.fsops_mxfp8_gemm_ex(ac, asc, fs.DTYPE_MXFP8, bc, bs, c, fs.DTYPE_F32 if c_f32 else fs.DTYPE_BF16,
                                   M, N, K, ws, ws_n)
        elif c_f32:
            fs.fsops_mxfp8_gemm_ex(to_dev_u16(a_bits), None, fs.DTYPE_BF16, bc, bs, c, fs.DTYPE_F32, M, N, K, ws,
                                   ws_n)
        else:
            fs.fsops_mxfp8_gemm(to_dev_u16(a_bits), bc, bs, c, M, N, K, ws, ws_n)
        torch.cuda.synchronize()
        assert fs.fsops_read_kernel_status(ws) == 0
        assert control_words_clear(ws[:16384]), "control words not reset"
        outs.append(c.cpu().numpy().astype(np.float64) if c_f32 else bf16_bits_to_f64(from_dev_bf16(c)))
    # split-K sums are added in arrival order: repeated calls agree to fp32
    # rounding (a bf16 output can then differ by one bf16 step in a few places)
    assert rel_l2(outs[1], outs[0]) < (1e-6 if c_f32 else 1e-3)
    if not c_f32:
        assert np.mean(outs[1] == outs[0]) > 0.99
    return outs[1]


SHAPES = [(1, 256, 128), (3, 384, 256), (16, 512, 1024), (17, 256, 384), (64, 1024, 512), (127, 128, 256),
          (128, 768, 2048), (2, 2560, 9728)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_fp32_out_matches_oracle(fs, M, N, K):
    a, b = _operands(M, N, K, seed=M * 1000 + N + K)
    bc, bs = oracle.quantize_bf16(b)
    ref = oracle.gemm(a, bc, bs)["c"]
    got = _gpu_gemm(fs, a, b, c_f32=True)
    assert rel_l2(got, ref) < 1e-5, rel_l2(got, ref)


@pytest.mark.parametrize("M,N,K", SHAPES[:6])
def test_gemm_bf16_out_matches_oracle(fs, M, N, K):
    a, b = _operands(M, N, K, seed=M + N + K)
    bc, bs = oracle.quantize_bf16(b)
    res = oracle.gemm(a, bc, bs)
    got = _gpu_gemm(fs, a, b)
    ref = bf16_bits_to_f64(res["c_bf16"])
    assert rel_l2(got, ref) < 2e-3
    assert max_abs_norm(got, ref) < 1e-2
    # fp32 accumulation differs from fp64 only in the last bits: most outputs are the same bf16
    assert np.mean(got == ref) > 0.9


@pytest.mark.parametrize("M,N,K", [(5, 384, 256), (128, 512, 640)])
def test_gemm_prequantised_a(fs, M, N, K):
    a, b = _operands(M, N, K, seed=7 * M + K)
    bc, bs = oracle.quantize_bf16(b)
    ref = oracle.gemm(a, bc, bs)["c"]
    got = _gpu_gemm(fs, a, b, c_f32=True, prequant=True)
    assert rel_l2(got, ref) < 1e-5


def test_gemm_zero_blocks_and_scale_spread(fs):
    M, N, K = 8, 256, 512
    rng = np.random.default_rng(11)
    a = rng.standard_normal((M, K)).astype(np.float32) * (10.0 ** rng.uniform(-3, 3, (M, 1)))
    a[:, 64:96] = 0.0
    b = rng.standard_normal((N, K)).astype(np.float32) * 0.05
    b.reshape(-1, 32)[rng.choice(N * K // 32, N * K // 320, replace=False)] = 0.0
    a, b = inputs.bf16_bits_from_f32(a), inputs.bf16_bits_from_f32(b)
    bc, bs = oracle.quantize_bf16(b)
    ref = oracle.gemm(a, bc, bs)["c"]
    got = _gpu_gemm(fs, a, b, c_f32=True)
    assert rel_l2(got, ref) < 1e-5
    for m in range(M):
        assert rel_l2(got[m], ref[m]) < 1e-5


# M > 128 (prefill): whole 128 x 256 output tiles per block, A quantised by
# its own launch; ragged last row tile and half-width last column tile.
PREFILL = [(129, 256, 128), (300, 384, 256), (1000, 640, 640), (4096, 256, 256)]


@pytest.mark.parametrize("M,N,K", PREFILL)
@pytest.mark.parametrize("form", [0, 1])
def test_gemm_prefill_fp32_out_matches_oracle(fs, M, N, K, form, knob):
    """Both launch forms: one block per tile (0) and the 256-row pair MMA (1;
    shapes with an odd number of 128-column halves fall back to form 0)."""
    knob("GEMM_FORM", form)
    a, b = _operands(M, N, K, seed=3 * M + N + K)
    bc, bs = oracle.quantize_bf16(b)
    ref = oracle.gemm(a, bc, bs)["c"]
    got = _gpu_gemm(fs, a, b, c_f32=True)
    assert rel_l2(got, ref) < 1e-5, rel_l2(got, ref)


@pytest.mark.parametrize("M,N,K", PREFILL[:3])
@pytest.mark.parametrize("form", [0, 1])
def test_gemm_prefill_bf16_out_matches_oracle(fs, M, N, K, form, knob):
    knob("GEMM_FORM", form)
    a, b = _operands(M, N, K, seed=5 * M + N + K)
    bc, bs = oracle.quantize_bf16(b)
    res = oracle.gemm(a, bc, bs)
    got = _gpu_gemm(fs, a, b)
    ref = bf16_bits_to_f64(res["c_bf16"])
    assert rel_l2(got, ref) < 2e-3
    assert max_abs_norm(got, ref) < 1e-2
    assert np.mean(got == ref) > 0.9


@pytest.mark.parametrize("form", [0, 1])
def test_gemm_prefill_pair_shapes(fs, form, knob):
    """N a multiple of 256 (the pair MMA's shapes): an odd number of row
    tiles leaves the last pair's second tile wholly past M."""
    knob("GEMM_FORM", form)
    for M, N, K, seed in ((384, 512, 640, 41), (1000, 768, 256, 42), (256, 256, 1152, 43)):
        a, b = _operands(M, N, K, seed=seed)
        bc, bs = oracle.quantize_bf16(b)
        ref = oracle.gemm(a, bc, bs)["c"]
        got = _gpu_gemm(fs, a, b, c_f32=True)
        assert rel_l2(got, ref) < 1e-5, (M, N, K, rel_l2(got, ref))


def test_gemm_prefill_prequantised_a(fs):
    M, N, K = 515, 384, 384
    a, b = _operands(M, N, K, seed=99)
    bc, bs = oracle.quantize_bf16(b)
    ref = oracle.gemm(a, bc, bs)["c"]
    got = _gpu_gemm(fs, a, b, c_f32=True, prequant=True)
    assert rel_l2(got, ref) < 1e-5


def test_two_library_copies_in_one_process(fs, tmp_path):
    """A second copy of the library loaded in the same process launches its
    own kernels (each copy raises its own kernels' shared-memory limits)."""
    import ctypes
    import shutil

    import torch

    from mxfp8_swiglu_mlp_gb300 import build

    path = str(tmp_path / "libfsops_copy.so")
    shutil.copy(build.LIB, path)
    other = ctypes.CDLL(path)
    for name, (args, res) in fs._SIGS.items():
        f = getattr(other, name)
        f.argtypes = args
        f.restype = res
    for M, N, K in ((16, 512, 256), (256, 512, 256)):  # the persistent and the tiled kernel
        a_bits, b_bits = _operands(M, N, K, 90 + M)
        bc, bs = fs.quantize_weight(to_dev_u16(b_bits))
        a = to_dev_u16(a_bits)
        outs = []
        for lib in (fs.lib, other):
            ws_n = lib.fsops_gemm_workspace_bytes(M, N, K)
            ws = torch.zeros(ws_n, dtype=torch.uint8, device="cuda")
            c = torch.empty((M, N), dtype=torch.float32, device="cuda")
            st = lib.fsops_mxfp8_gemm_ex(a.data_ptr(), None, fs.DTYPE_BF16, bc.data_ptr(), bs.data_ptr(),
                                         c.data_ptr(), fs.DTYPE_F32, M, N, K, ws.data_ptr(), ws_n,
                                         torch.cuda.current_stream().cuda_stream)
            assert st == fs.OK, (M, lib.fsops_last_cuda_error())
            torch.cuda.synchronize()
            outs.append(c.cpu().numpy().astype(np.float64))
        assert rel_l2(outs[1], outs[0]) < 1e-6


@pytest.mark.parametrize("form", [0, 1])
def test_gemm_square_16384_sampled(fs, form, knob):
    """The largest square GEMM (16384^3, bf16 A quantised on the device): the
    whole output is finite, and 16 sampled rows x 128 sampled columns match
    the oracle, which quantises the sampled rows of A and B itself."""
    import torch

    knob("GEMM_FORM", form)
    M = N = K = 16384
    g = torch.Generator(device="cuda").manual_seed(11)
    a = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    bc, bs = fs.quantize_weight(w)
    ws_n = fs.fsops_gemm_workspace_bytes(M, N, K)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device="cuda")
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    fs.fsops_mxfp8_gemm(a, bc, bs, c, M, N, K, ws, ws_n)
    torch.cuda.synchronize()
    assert fs.fsops_read_kernel_status(ws) == 0
    assert bool(torch.isfinite(c).all())
    rng = np.random.default_rng(int(form) + 1)
    rows = np.sort(rng.choice(M, 16, replace=False))
    cols = np.sort(rng.choice(N, 128, replace=False))
    a_bits = a[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    b_bits = w[torch.from_numpy(cols).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    bc_o, bs_o = oracle.quantize_bf16(b_bits)
    ref = oracle.gemm(a_bits, bc_o, bs_o)["c_bf16"]
    got = c[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].view(torch.int16).cpu().numpy()
    got = bf16_bits_to_f64(got.view(np.uint16))
    want = bf16_bits_to_f64(ref)
    assert rel_l2(got, want) < 2e-3, rel_l2(got, want)
    assert max_abs_norm(got, want) < 1e-2
    del a, w, bc, bs, ws, c
    torch.cuda.empty_cache()
