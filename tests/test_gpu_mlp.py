"""Fused single-launch MXFP8 SwiGLU MLP (and the three-launch path) against
the oracle, on the workloads' shapes and distributions."""
import numpy as np
import pytest

import oracle
from workloads import inputs
from tests._util import (to_dev_u16, from_dev_bf16, bf16_bits_to_f64, rel_l2, max_abs_norm, per_row_rel_l2,
                         REL_L2_TOL, MAX_ABS_TOL, PER_ROW_TOL, assert_repeat_close, control_words_clear)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fs():
    import mxfp8_swiglu_mlp_gb300 as fs

    return fs


class Layer:
    def __init__(self, fs, wl, layer=0, M=None):
        import torch

        self.M = wl.M if M is None else M
        self.H, self.I = wl.H, wl.I
        self.x = inputs.make_activations(wl, self.M)
        self.wg, self.wu, self.wd = inputs.make_layer(wl, layer)
        self.w = fs.prepare_mlp_weights(to_dev_u16(self.wg), to_dev_u16(self.wu), to_dev_u16(self.wd))
        self.x_dev = to_dev_u16(self.x)
        self.ws = fs.Workspace(self.M, self.H, self.I)
        torch.cuda.synchronize()

    def run(self, fs, fused=True, scales=None):
        import torch

        y = torch.empty((self.M, self.H), dtype=torch.bfloat16, device="cuda")
        f = fs.fsops_mxfp8_swiglu_mlp if fused else fs.fsops_mxfp8_swiglu_mlp_unfused
        f(self.x_dev, self.w.gateup_codes, self.w.down_codes, scales or self.w.scales, y, self.M, self.H, self.I)
        torch.cuda.synchronize()
        assert fs.fsops_read_kernel_status() == 0
        return from_dev_bf16(y)

    def oracle(self, rows=None):
        qw = oracle.quantize_weights(self.wg, self.wu, self.wd)
        return oracle.swiglu_mlp(self.x, qw, rows_down=rows)


def _assert_parity(got_bits, ref, per_row=True):
    got = bf16_bits_to_f64(got_bits)
    want = bf16_bits_to_f64(ref["y_bf16"])
    assert rel_l2(got, want) <= REL_L2_TOL, rel_l2(got, want)
    assert max_abs_norm(got, want) <= MAX_ABS_TOL, max_abs_norm(got, want)
    if per_row:
        pr = per_row_rel_l2(got, want)
        assert np.max(pr) <= PER_ROW_TOL, pr


SMALL = [(1, 256, 384, 0), (5, 512, 640, 1), (16, 1024, 1280, 2), (33, 384, 512, 3), (128, 256, 256, 4),
         (64, 1152, 896, 5), (100, 640, 2048, 6),
         # small H, large I: many gate/up tiles, short K loops
         (8, 256, 4864, 7), (32, 384, 5120, 8),
         # more 128-feature chunks than 2-block clusters: 2, 3 and 4 chunks per cluster
         (17, 256, 9856, 17), (4, 256, 25600, 18), (3, 512, 38912, 19),
         # H of one row tile of 128 (the grid-wide kernel) and an odd number of row tiles
         (6, 128, 512, 20), (20, 640, 768, 21)]


@pytest.mark.parametrize("M,H,I,seed", SMALL)
@pytest.mark.parametrize("fused", [True, False])
def test_small_shapes(fs, M, H, I, seed, fused):
    wl = inputs.make_workload_small("s", M, H, I, seed)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs, fused), L.oracle())


@pytest.mark.parametrize("M,H,I,seed", [s for s in SMALL if s[0] <= 32 and s[1] >= 256])
def test_small_shapes_sliced(fs, M, H, I, seed, knob):
    """The cluster-sliced kernel forced on every small shape it serves
    (1-4 chunks per cluster, one row tile, odd row tiles, M up to 32)."""
    knob("DECODE_PATH", 1)
    wl = inputs.make_workload_small("s", M, H, I, seed)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs), L.oracle())


@pytest.mark.parametrize("M,kn", [
    (16, {"TR0": 128, "WHOLE_TILES": 0, "DECODE_PATH": 0}),   # 128-row gate/up tiles, split-K
    (16, {"TR0": 256, "WHOLE_TILES": 1, "DECODE_PATH": 0}),   # 256-row whole tiles, staged epilogue
    (16, {"TR1": 128, "DECODE_PATH": 0}),                     # 128-row down tiles, staged epilogue
    (64, {"TR1": 128, "WHOLE_TILES": 0}),                     # 128-row down tiles, split gate/up from TMEM
    (100, {"TR1": 128}),                                      # 128-row down tiles, per-owner finishing
    (64, {"TR0": 128}),                                       # 128-row whole gate/up tiles from TMEM
    (16, {"I": 5120, "DECODE_PATH": 0}),                      # gate/up tiles split by 2-block clusters
    (16, {"I": 5120, "PAIRS": 0, "DECODE_PATH": 0}),          # the same shape split over all blocks
    (16, {"LOCAL_XQ": 0, "DECODE_PATH": 0}),                  # x quantised grid-wide at M <= 16
    (16, {"PRIME": 3, "MAX_INFLIGHT": 2, "DECODE_PATH": 0}),  # other weight-load depths
    (16, {"COOPERATIVE": 1, "DECODE_PATH": 0}),               # cooperative launch of the grid-wide kernel
    (64, {"COOPERATIVE": 1}),
    # tile-aligned splits (each block on one tile) and stream-K forced, where
    # both phases allow either (KS >= blocks per tile)
    (16, {"H": 2560, "ALIGNED": 1, "PAIRS": 0, "DECODE_PATH": 0}),
    (16, {"H": 2560, "ALIGNED": 0, "PAIRS": 0, "DECODE_PATH": 0}),
    (5, {"H": 1280, "I": 4096, "ALIGNED": 1, "DECODE_PATH": 0}),
    (64, {"H": 2560, "ALIGNED": 1}),
    (64, {"H": 2560, "ALIGNED": 0}),
])
def test_tile_plans(fs, M, kn, knob):
    """Every tile height / split combination the grid-wide kernel supports,
    forced through the plan knobs, against the oracle."""
    kn = dict(kn)
    I = int(kn.pop("I", 2560))
    H = int(kn.pop("H", 512))
    for k, v in kn.items():
        knob(k, v)
    wl = inputs.make_workload_small("s", M, H, I, 9)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs, True), L.oracle())


@pytest.mark.parametrize("M,H,I,seed", [(1, 512, 1024, 30), (16, 768, 2560, 31), (32, 512, 896, 32),
                                        (8, 1024, 2816, 33), (2, 2048, 1024, 34)])
def test_decode_paths_agree(fs, M, H, I, seed, knob):
    """The cluster-sliced kernel, the grid-wide kernel and (M <= 8) the
    small-M kernel on the same inputs: each within the oracle's tolerance,
    and close to one another."""
    wl = inputs.make_workload_small("s", M, H, I, seed)
    L = Layer(fs, wl)
    ref = L.oracle()
    outs = []
    for path in ([0, 1, 2] if M <= 8 else [0, 1]):
        knob("DECODE_PATH", path)
        outs.append(L.run(fs))
        _assert_parity(outs[-1], ref)
    for o in outs[1:]:
        assert rel_l2(bf16_bits_to_f64(o), bf16_bits_to_f64(outs[0])) < 1e-3


@pytest.mark.parametrize("M,H,I,seed", [s for s in SMALL if s[0] <= 8])
def test_small_shapes_grid_wide(fs, M, H, I, seed, knob):
    """The shapes of up to 8 tokens (which the small-M kernel takes by
    default where it applies) on the grid-wide kernel."""
    knob("DECODE_PATH", 0)
    wl = inputs.make_workload_small("s", M, H, I, seed)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs), L.oracle())


def test_token_scale_spread(fs):
    """Rows scaled by 10^U(-2, 2) (the m128 workload's activations)."""
    wl = inputs.make_workload_small("s", 48, 512, 768, 9, token_scale_log10=(-2.0, 2.0))
    L = Layer(fs, wl)
    _assert_parity(L.run(fs), L.oracle())


def test_zero_blocks(fs):
    wl = inputs.make_workload_small("s", 8, 640, 1024, 10, zero_block_frac=0.05)
    L = Layer(fs, wl)
    _assert_parity(L.run(fs), L.oracle())


@pytest.mark.parametrize("name", ["m1", "m16"])
def test_full_size_workloads(fs, name):
    wl = inputs.WORKLOADS[name]
    L = Layer(fs, wl)
    ref = L.oracle()
    _assert_parity(L.run(fs, True), ref)
    _assert_parity(L.run(fs, False), ref)


@pytest.mark.parametrize("name", ["m64", "m128"])
def test_full_size_sampled_rows(fs, name):
    """Full-size layer (one of the 32), checked on 256 sampled output features."""
    wl = inputs.WORKLOADS[name]
    L = Layer(fs, wl, layer=3)
    rows = np.sort(np.random.default_rng(1).choice(wl.H, 256, replace=False))
    ref = L.oracle(rows)
    y = L.run(fs)
    _assert_parity(y[:, rows], ref)


def test_sweep_shape_sampled(fs):
    wl = inputs.WORKLOADS["sweep"]
    for M in (1, 32):
        L = Layer(fs, wl, layer=0, M=M)
        rows = np.sort(np.random.default_rng(M).choice(wl.H, 128, replace=False))
        _assert_parity(L.run(fs)[:, rows], L.oracle(rows))


@pytest.mark.parametrize("M,path", [(16, 0), (16, 1), (64, 0), (1, 1)])
def test_repeat_calls_agree(fs, M, path, knob):
    """Split-K partial sums are added into L2 in arrival order, so repeated
    calls agree to fp32 rounding (one bf16 step at most, element by element:
    the stand-in race detector), and every call leaves the workspace ready
    for the next one."""
    if M <= 32:
        knob("DECODE_PATH", path)
    wl = inputs.make_workload_small("s", M, 1024, 1536, 12)
    L = Layer(fs, wl)
    ref = L.oracle()
    runs = [L.run(fs) for _ in range(4)]
    for r in runs:
        _assert_parity(r, ref)
    for r in runs[1:]:
        assert_repeat_close(runs[0], r)


def test_repeat_calls_full_size(fs):
    """The m1, m16, m64 and m128 layers, four calls each: every element within
    one bf16 step of the first call's."""
    for name in ("m1", "m16", "m64", "m128"):
        wl = inputs.WORKLOADS[name]
        L = Layer(fs, wl, layer=wl.layers - 1)
        runs = [L.run(fs) for _ in range(4)]
        for r in runs[1:]:
            assert_repeat_close(runs[0], r)


def test_wrong_scale_layout_is_caught(fs):
    """The pages' bug: scales in another layout give large errors at full speed."""
    import torch

    wl = inputs.make_workload_small("s", 16, 512, 512, 13)
    L = Layer(fs, wl)
    qw = oracle.quantize_weights(L.wg, L.wu, L.wd)
    rm_gu = torch.from_numpy(np.ascontiguousarray(qw["gateup_scales"]).reshape(-1)).cuda()
    rm_d = torch.from_numpy(np.ascontiguousarray(qw["down_scales"]).reshape(-1)).cuda()
    y = L.run(fs, scales=(rm_gu, rm_d))
    got = bf16_bits_to_f64(y)
    want = bf16_bits_to_f64(L.oracle()["y_bf16"])
    assert rel_l2(got, want) > 0.1


def test_cuda_graph_replay(fs):
    import torch

    wl = inputs.make_workload_small("s", 16, 768, 1024, 14)
    L = Layer(fs, wl)
    ref = L.run(fs)
    y = torch.empty((L.M, L.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fs.fsops_mxfp8_swiglu_mlp(L.x_dev, L.w.gateup_codes, L.w.down_codes, L.w.scales, y, L.M, L.H, L.I,
                                      stream=s)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_repeat_close(from_dev_bf16(y), ref)


def test_output_guard_band(fs):
    import torch

    wl = inputs.make_workload_small("s", 7, 384, 512, 15)
    L = Layer(fs, wl)
    buf = torch.full((L.M * L.H + 4096,), -7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[2048:2048 + L.M * L.H].view(L.M, L.H)
    fs.fsops_mxfp8_swiglu_mlp(L.x_dev, L.w.gateup_codes, L.w.down_codes, L.w.scales, y, L.M, L.H, L.I)
    torch.cuda.synchronize()
    b = buf.float().cpu().numpy()
    assert np.all(b[:2048] == -7.0) and np.all(b[2048 + L.M * L.H:] == -7.0)
    _assert_parity(from_dev_bf16(y), L.oracle())


# (M, H, I, knobs): the cluster-sliced kernel; the grid-wide kernel with
# stream-K gate/up; with 2-block cluster pairs exchanging gate/up halves through
# distributed shared memory (I / 128 = 40 tiles for 76 pairs); with whole
# gate/up tiles and per-owner finishing (M = 64); cooperative.
TIMEOUT_CASES = [(4, 256, 384, {"DECODE_PATH": 1}), (4, 256, 384, {"DECODE_PATH": 0}), (16, 256, 5120, {"DECODE_PATH": 0}),
                 (64, 256, 1024, {}), (16, 256, 5120, {"DECODE_PATH": 0, "COOPERATIVE": 1}),
                 (4, 256, 384, {"DECODE_PATH": 2}), (8, 256, 4864, {"DECODE_PATH": 2})]


@pytest.mark.parametrize("M,H,I,knobs", TIMEOUT_CASES)
def test_wait_timeout_reports_and_recovers(fs, knob, M, H, I, knobs):
    """A wait that can never be satisfied (one arrival more than any block
    makes) runs out, the kernel reports FSOPS_ERR_TIMEOUT and returns; every
    block of a cluster pair leaves together; the next launch is correct."""
    import torch

    for k, v in knobs.items():
        knob(k, v)
    wl = inputs.make_workload_small("s", M, H, I, 16)
    L = Layer(fs, wl)
    y = torch.empty((L.M, L.H), dtype=torch.bfloat16, device="cuda")
    fs.fsops_set_wait_timeout_ns(20_000_000)
    fs.fsops_debug_set_extra_arrivals(1)
    try:
        fs.fsops_mxfp8_swiglu_mlp(L.x_dev, L.w.gateup_codes, L.w.down_codes, L.w.scales, y, L.M, L.H, L.I)
        torch.cuda.synchronize()
        word = fs.fsops_read_kernel_status()
    finally:
        fs.fsops_debug_set_extra_arrivals(0)
        fs.fsops_set_wait_timeout_ns(1_000_000_000)
    assert (word >> 24) == fs.ERR_TIMEOUT, hex(word)
    assert control_words_clear(L.ws.buf[(L.ws.ptr - L.ws.buf.data_ptr()):][:16384])
    _assert_parity(L.run(fs), L.oracle())
