"""The MLP above 128 token rows (prefill shapes): x quantised, the gate/up
GEMM whose epilogue writes h = SiLU(g) * u requantised to MXFP8, the down GEMM
on h; against the oracle, element by element on small shapes and on sampled
tokens and output features at the m16 layer's size with 4096 tokens."""
import numpy as np
import pytest

import oracle
from workloads import inputs
from tests._util import to_dev_u16, from_dev_bf16, bf16_bits_to_f64, rel_l2
from tests.test_gpu_mlp import Layer, _assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fs():
    import mxfp8_swiglu_mlp_gb300 as fs

    return fs


# ragged row tiles (129, 200, 300, 513), one and several feature tiles, H and
# I from one to several 128-blocks
PREFILL = [(129, 256, 384, 20), (200, 384, 256, 21), (256, 512, 640, 22), (300, 256, 1024, 23),
           (513, 640, 384, 24), (384, 128, 128, 25)]


@pytest.mark.parametrize("M,H,I,seed", PREFILL)
@pytest.mark.parametrize("fused", [True, False])
def test_prefill_small_shapes(fs, M, H, I, seed, fused):
    wl = inputs.make_workload_small("s", M, H, I, seed)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs, fused), L.oracle())


@pytest.mark.parametrize("form", [0, 1])
def test_prefill_cluster_forms(fs, form, knob):
    """Both launch forms of the tiled GEMMs: single blocks and 256-row pair
    MMAs of 2-block clusters."""
    knob("GEMM_FORM", form)
    wl = inputs.make_workload_small("s", 640, 512, 768, 26)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs), L.oracle())


def test_prefill_token_scale_spread_and_zero_blocks(fs):
    wl = inputs.make_workload_small("s", 260, 384, 512, 27, token_scale_log10=(-2.0, 2.0), zero_block_frac=0.05)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs), L.oracle())


def test_prefill_full_size_sampled(fs):
    """The m16 layer (H=2560, I=9728) with 4096 tokens: 48 sampled tokens x 256
    sampled output features.  Token rows are independent through the whole
    MLP, so the oracle runs on the sampled tokens alone."""
    wl = inputs.WORKLOADS["m16"]
    L = Layer(fs, wl, M=4096)
    y = L.run(fs)
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(L.M, 48, replace=False))
    feats = np.sort(rng.choice(L.H, 256, replace=False))
    qw = oracle.quantize_weights(L.wg, L.wu, L.wd)
    ref = oracle.swiglu_mlp(L.x[toks], qw, rows_down=feats)
    _assert_parity(y[toks][:, feats], ref)


def test_prefill_deterministic_and_graph_safe(fs):
    """No split-K above 128 rows: every call and every graph replay gives the
    same bits."""
    import torch

    wl = inputs.make_workload_small("s", 320, 512, 512, 28)
    L = Layer(fs, wl)
    ref = L.run(fs)
    assert np.array_equal(L.run(fs), ref)
    y = torch.empty((L.M, L.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fs.fsops_mxfp8_swiglu_mlp(L.x_dev, L.w.gateup_codes, L.w.down_codes, L.w.scales, y, L.M, L.H, L.I,
                                      stream=s)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(from_dev_bf16(y), ref)


def test_prefill_matches_three_launch_path(fs):
    """The SwiGLU epilogue and the standalone SwiGLU-quantise launch compute
    the same h, so the two paths agree far inside the oracle tolerance."""
    wl = inputs.make_workload_small("s", 384, 768, 1024, 29)
    L = Layer(fs, wl)
    a = bf16_bits_to_f64(L.run(fs, True))
    b = bf16_bits_to_f64(L.run(fs, False))
    assert rel_l2(a, b) < 1e-3


def test_noalloc_rejects_prefill(fs):
    import torch

    wl = inputs.make_workload_small("s", 200, 256, 256, 30)
    L = Layer(fs, wl)
    y = torch.empty((L.M, L.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fs.FsopsError) as e:
        fs.fsops_mxfp8_swiglu_mlp_noalloc(L.x_dev, L.w.gateup_codes, L.w.down_codes, L.w.scales, y, L.M, L.H, L.I)
    assert e.value.status == fs.ERR_UNSUPPORTED_SHAPE
