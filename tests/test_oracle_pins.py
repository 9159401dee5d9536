"""Pins for the CPU oracle: it is checked against things other than itself.

* the OCP E4M3 encoding landmarks (tests/golden/ocp_e4m3_landmarks.txt);
* torch's float8_e4m3fn conversion (a library routine, round-to-nearest-even)
  for every in-range value, exhaustively over bf16 bit patterns;
* hand-worked block quantisations (tests/golden/mx_worked_examples.txt);
* closed forms: power-of-two blocks round-trip exactly, all-zero blocks,
  single-outlier saturation;
* exact rational arithmetic (fractions.Fraction) for the block-scaled GEMM;
* torch.nn.functional.silu for SiLU;
* the whole MLP rebuilt from torch pieces (float8 conversion, fp64 matmul);
* the quantisation-error band against the unquantised fp64 SwiGLU MLP;
* the decoder block: RMSNorm against torch.nn.functional.rms_norm and its
  closed forms (unit mean square, scale invariance, per-feature gain), and the
  block y = x + MLP(RMSNorm(x) * gamma) rebuilt from torch pieces.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from workloads import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ E4M3 table
def _torch_e4m3_decode(code: int) -> float:
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64))


def test_e4m3_table_matches_ocp_landmarks():
    table = oracle.e4m3_table()
    with open(os.path.join(GOLDEN, "ocp_e4m3_landmarks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code_s, val_s = line.split()[:2]
            assert table[int(code_s, 16)] == float.fromhex(val_s), line


def test_e4m3_table_matches_torch_decode():
    table = oracle.e4m3_table()
    assert len(table) == 127
    for c in range(127):
        assert table[c] == _torch_e4m3_decode(c), c
    assert np.all(np.diff(table) > 0)


def _torch_e4m3_code(t: np.ndarray) -> np.ndarray:
    """Magnitude code of torch's float8_e4m3fn conversion (valid for 0 <= t <= 448).

    torch converts float64 through float32, which could round twice, so the
    inputs must be float32 values (or so small that they round to zero)."""
    t = np.ascontiguousarray(t, np.float64)
    t32 = t.astype(np.float32)
    assert np.all((t32.astype(np.float64) == t) | (t < 2.0 ** -12))
    x = torch.from_numpy(t32)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy() & 0x7F


def test_e4m3_rounding_matches_torch_random():
    rng = np.random.default_rng(123)
    t = np.concatenate([rng.uniform(0, 448, 4000), rng.uniform(0, 1e-2, 2000),
                        np.exp(rng.uniform(-12, math.log(448), 4000))]).astype(np.float32)
    ours = np.array([oracle.e4m3_round_code(v) for v in t])
    assert np.array_equal(ours, _torch_e4m3_code(t))


def test_e4m3_rounding_all_midpoints_and_values():
    table = oracle.e4m3_table()
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)   # exact in float32
    pts = np.concatenate([table.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
                          np.nextafter(mids, np.float32(1000))])
    ours = np.array([oracle.e4m3_round_code(v) for v in pts])
    assert np.array_equal(ours, _torch_e4m3_code(pts))
    # saturation: everything above 448 maps to the largest finite code
    for v in (448.0, 448.0001, 463.99, 464.0, 480.0, 1e6):
        assert oracle.e4m3_round_code(v) == 0x7E


def test_quantize_exhaustive_bf16_against_torch():
    """Every finite bf16 pattern, placed in blocks with a known amax, quantises
    exactly as torch's float8 conversion of v * 2^-e (in range)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    bits, vals = bits[finite], vals[finite]
    for amax_exp in (-130, -60, -8, 0, 5, 40, 120):
        # each block: 31 arbitrary entries no larger than amax plus amax itself
        amax = 2.0 ** amax_exp * 1.5
        ok = np.abs(vals) <= amax
        sel = vals[ok]
        n = (len(sel) // 31) * 31
        blocks = sel[:n].reshape(-1, 31)
        blocks = np.concatenate([blocks, np.full((blocks.shape[0], 1), amax)], axis=1)
        codes, scales = oracle.quantize_f64(blocks)
        e = oracle.block_exponent(amax)
        assert np.all(scales == e + 127)
        t = np.abs(blocks) * 2.0 ** (-e)
        expect = _torch_e4m3_code(np.minimum(t, 448.0)) | np.where(np.signbit(blocks), 0x80, 0)
        assert np.array_equal(codes, expect.astype(np.uint8)), amax_exp


# ------------------------------------------------------------------ worked examples
def _parse_worked():
    out = []
    with open(os.path.join(GOLDEN, "mx_worked_examples.txt")) as f:
        for line in f:
            if line.startswith("#") or "|" not in line:
                continue
            head, body = line.split("|")
            entries = []
            for tok in body.split():
                v, c = tok.split("=")
                entries.append((float.fromhex(v), int(c, 16)))
            out.append((int(head.strip(), 16), entries))
    return out


def test_worked_examples():
    cases = _parse_worked()
    assert len(cases) >= 7
    for scale_byte, entries in cases:
        block = np.zeros((1, 32))
        for i, (v, _) in enumerate(entries):
            block[0, i] = v
        codes, scales = oracle.quantize_f64(block)
        assert scales[0, 0] == scale_byte, (scale_byte, entries)
        for i, (_, c) in enumerate(entries):
            assert codes[0, i] == c, (i, entries[i], hex(codes[0, i]))
        assert np.all(codes[0, len(entries):] == 0)


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("a", [-120, -20, -3, 0, 7, 60, 127])
def test_power_of_two_block_round_trips(a):
    """amax = 2^a gives scale byte a - 8 + 127 (clamped); every value that is
    E4M3-representable after scaling by 2^(8-a) survives quantise/dequantise."""
    e = max(-127, a - 8)
    vals = [2.0 ** a]
    for k in range(a - 14, a + 1):          # normal range after scaling: 3 mantissa bits
        for m in range(8):
            v = (1 + m / 8) * 2.0 ** k
            if v <= 2.0 ** a and k - e >= -6:
                vals.append(v)
    for k in range(a - 17, a - 14):         # subnormal range: multiples of 2^-9 after scaling
        if k - e >= -9:
            vals.append(2.0 ** k)
    vals = np.array(vals)
    n = (len(vals) + 31) // 32 * 32
    blocks = np.zeros(n)
    blocks[:len(vals)] = vals
    blocks = blocks.reshape(-1, 32)
    blocks[:, 0] = 2.0 ** a                    # every block carries the amax
    codes, scales = oracle.quantize_f64(blocks)
    assert np.all(scales == e + 127)
    assert np.array_equal(oracle.dequantize(codes, scales), blocks)


def test_zero_blocks_and_negative_zero():
    block = np.zeros((2, 32))
    block[1, ::2] = -0.0
    codes, scales = oracle.quantize_f64(block)
    assert np.all(scales == 0)
    assert np.all(codes[0] == 0)
    assert np.all(codes[1, ::2] == 0x80) and np.all(codes[1, 1::2] == 0)
    assert np.all(oracle.dequantize(codes, scales) == 0)


@pytest.mark.parametrize("a", [-50, 0, 13])
def test_single_outlier_saturates(a):
    block = np.full((1, 32), 2.0 ** (a - 6))
    block[0, 5] = 1.9 * 2.0 ** a
    codes, scales = oracle.quantize_f64(block)
    assert scales[0, 0] == a - 8 + 127
    assert codes[0, 5] == 0x7E                 # 1.9 * 2^8 = 486.4 > 448
    assert oracle.dequantize(codes, scales)[0, 5] == 448.0 * 2.0 ** (a - 8)
    # the others: 2^(a-6) * 2^(8-a) = 4 = 2^2 -> E = 9, m = 0 -> code 0x48
    assert np.all(np.delete(codes[0], 5) == 0x48)


def test_block_exponent_closed_form():
    rng = np.random.default_rng(5)
    for amax in np.exp(rng.uniform(-80, 80, 500)):
        e = oracle.block_exponent(amax)
        assert 2.0 ** (e + 8) <= amax < 2.0 ** (e + 9)
    assert oracle.block_exponent(0.0) == -127
    assert oracle.block_exponent(2.0 ** -140) == -127
    assert oracle.block_exponent(5e-324) == -127


# ------------------------------------------------------------------ GEMM, exact
def _exact_value(code: int, scale: int) -> Fraction:
    """Exact rational value of an MXFP8 element, decoded from the bits here."""
    E, m = (code >> 3) & 0xF, code & 7
    mag = Fraction(m, 8) * Fraction(2) ** -6 if E == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (E - 7)
    mag *= Fraction(2) ** (scale - 127)
    return -mag if code & 0x80 else mag


@pytest.mark.parametrize("M,N,K", [(1, 3, 32), (2, 4, 64), (4, 2, 128), (3, 5, 96)])
def test_gemm_exact_rational(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a = inputs.bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    b = inputs.bf16_bits_from_f32((rng.standard_normal((N, K)) * 0.1).astype(np.float32))
    bc, bs = oracle.quantize_bf16(b)
    res = oracle.gemm(a, bc, bs)
    ac, as_ = res["a_codes"], res["a_scales"]
    for i in range(M):
        for j in range(N):
            s = sum(_exact_value(int(ac[i, k]), int(as_[i, k // 32])) *
                    _exact_value(int(bc[j, k]), int(bs[j, k // 32])) for k in range(K))
            assert res["c"][i, j] == float(s)


# ------------------------------------------------------------------ SiLU
def test_silu_matches_torch():
    g = np.concatenate([np.linspace(-40, 40, 2001), [-800.0, 800.0, 0.0, -0.0]])
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy()
    ours = oracle.silu(g)
    np.testing.assert_allclose(ours, ref, rtol=1e-15, atol=1e-300)


# ------------------------------------------------------------------ bf16 rounding
def test_round_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(9)
    f = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16_bits(f.astype(np.float64)), ref)


def test_round_bf16_single_rounding():
    # 1 + 2^-8 + 2^-30: just above the bf16 midpoint between 1 and 1 + 2^-7.
    # Rounding directly gives 1 + 2^-7; going through float32 first would drop
    # the 2^-30, land on the midpoint and round to 1.
    y = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30, -(1.0 + 2.0 ** -8 + 2.0 ** -30)])
    got = oracle.bf16_bits_to_f64(oracle.round_bf16_bits(y))
    assert got[0] == 1.0 + 2.0 ** -7 and got[1] == -(1.0 + 2.0 ** -7)


# ------------------------------------------------------------------ scale layout
def test_tiled_layout_worked_offsets():
    rows, K = 256, 256
    sc = np.zeros((rows, K // 32), np.uint8)
    with open(os.path.join(GOLDEN, "tiled_scale_layout_examples.txt")) as f:
        pts = [tuple(int(t) for t in line.split()) for line in f
               if line.strip() and not line.startswith("#")]
    for n, (r, kb, off) in enumerate(pts):
        sc[r, kb] = n + 1
    tiled = oracle.scales_rowmajor_to_tiled(sc)
    assert tiled.size == oracle.tiled_scale_bytes(rows, K) == 2 * 2 * 512
    for n, (r, kb, off) in enumerate(pts):
        assert tiled[off] == n + 1, (r, kb, off)


def test_tiled_layout_is_a_permutation():
    rows, K = 384, 512
    sc = np.arange(rows * (K // 32), dtype=np.int64).reshape(rows, K // 32)
    tiled = oracle.mx_oracle._tiled_offsets(rows, K // 32)
    assert len(np.unique(tiled)) == tiled.size == oracle.tiled_scale_bytes(rows, K)
    # each 512-byte tile holds one 128-row x 4-block patch
    tile_of = tiled // 512
    for rt in range(3):
        for kg in range(4):
            patch = tile_of[rt * 128:(rt + 1) * 128, kg * 4:(kg + 1) * 4]
            assert np.all(patch == rt * 4 + kg)
    rm = (sc % 251).astype(np.uint8)
    back = oracle.scales_tiled_to_rowmajor(oracle.scales_rowmajor_to_tiled(rm), rows, K)
    assert np.array_equal(back, rm)


# ------------------------------------------------------------------ the MLP, rebuilt from torch
def _torch_mx_qdq(v: torch.Tensor) -> torch.Tensor:
    """MXFP8 quantise/dequantise from torch pieces: the block exponent from
    torch.frexp, the element rounding from torch's float8_e4m3fn conversion
    (saturation applied first, as the MX rule saturates)."""
    rows, K = v.shape
    blk = v.reshape(rows, K // 32, 32)
    amax = blk.abs().amax(dim=-1, keepdim=True)
    _, ex = torch.frexp(amax)
    e = torch.where(amax == 0, torch.full_like(ex, -127), (ex - 1 - 8).clamp(-127, 127))
    scale = torch.ldexp(torch.ones_like(amax), e.to(torch.float64))
    t = (blk / scale).clamp(-448.0, 448.0)
    q = t.to(torch.float8_e4m3fn).to(torch.float64)
    return (q * scale).reshape(rows, K)


def _torch_mlp(x, wg, wu, wd, quantize=True):
    qd = _torch_mx_qdq if quantize else (lambda a: a)
    xq, wgq, wuq, wdq = qd(x), qd(wg), qd(wu), qd(wd)
    g = xq @ wgq.T
    u = xq @ wuq.T
    h = torch.nn.functional.silu(g) * u
    return qd(h) @ wdq.T, h


def _small_layer(M=5, H=256, I=384, seed=11, **kw):
    wl = inputs.make_workload_small("t", M, H, I, seed, **kw)
    x = inputs.make_activations(wl)
    wg, wu, wd = inputs.make_layer(wl, 0)
    return x, wg, wu, wd


def _f64(bits):
    return torch.from_numpy(oracle.bf16_bits_to_f64(bits))


@pytest.mark.parametrize("kw", [{}, {"zero_block_frac": 0.05}, {"token_scale_log10": (-2.0, 2.0)}])
def test_mlp_matches_torch_rebuild(kw):
    x, wg, wu, wd = _small_layer(**kw)
    qw = oracle.quantize_weights(wg, wu, wd)
    res = oracle.swiglu_mlp(x, qw)
    y_t, h_t = _torch_mlp(_f64(x), _f64(wg), _f64(wu), _f64(wd))
    np.testing.assert_allclose(res["h"], h_t.numpy(), rtol=1e-12, atol=1e-300)
    assert oracle.rel_l2(res["y"], y_t.numpy()) < 1e-12
    # y_bf16 is the single rounding of y
    assert np.array_equal(res["y_bf16"], oracle.round_bf16_bits(y_t.numpy()))


def test_mlp_quantisation_error_band():
    """rel-L2 of the quantised MLP against the unquantised fp64 SwiGLU MLP lies
    within 2x of the estimate built from each tensor's own round-trip error."""
    x, wg, wu, wd = _small_layer(M=16, H=512, I=1024, seed=3)
    qw = oracle.quantize_weights(wg, wu, wd)
    res = oracle.swiglu_mlp(x, qw)
    xf, wgf, wuf, wdf = (_f64(a) for a in (x, wg, wu, wd))
    y_ref, h_ref = _torch_mlp(xf, wgf, wuf, wdf, quantize=False)
    rt = lambda a: oracle.rel_l2(oracle.quant_dequant(a.numpy()), a.numpy())
    ex, eg, eu, ed, eh = rt(xf), rt(wgf), rt(wuf), rt(wdf), rt(h_ref)
    est = math.sqrt(2 * ex ** 2 + eg ** 2 + eu ** 2 + eh ** 2 + ed ** 2)
    got = oracle.rel_l2(res["y"], y_ref.numpy())
    assert 0.5 * est < got < 2.0 * est, (got, est)
    assert 0.01 < got < 0.2


def test_oracle_is_deterministic():
    x, wg, wu, wd = _small_layer(seed=4)
    a = oracle.swiglu_mlp(x, oracle.quantize_weights(wg, wu, wd))
    b = oracle.swiglu_mlp(x, oracle.quantize_weights(wg, wu, wd))
    assert np.array_equal(a["y_bf16"], b["y_bf16"]) and np.array_equal(a["h_codes"], b["h_codes"])


def test_sampled_rows_equal_full():
    x, wg, wu, wd = _small_layer(seed=6)
    qw = oracle.quantize_weights(wg, wu, wd)
    full = oracle.swiglu_mlp(x, qw)
    rows = np.array([0, 7, 100, 255])
    part = oracle.swiglu_mlp(x, qw, rows_down=rows)
    assert np.array_equal(part["y_bf16"], full["y_bf16"][:, rows])


# ------------------------------------------------------------------ planted mistakes
def _pin_error(y_candidate, x, wg, wu, wd):
    y_t, _ = _torch_mlp(_f64(x), _f64(wg), _f64(wu), _f64(wd))
    return oracle.rel_l2(y_candidate, y_t.numpy())


@pytest.mark.parametrize("mistake", ["swap_gate_up", "skip_h_requant", "scale_rule_minus7",
                                     "transpose_down", "scale_layout"])
def test_planted_mistakes_are_caught(mistake):
    """Each plausible oracle bug, planted here on the CPU, breaks the torch
    rebuild pin by far more than its 1e-12 tolerance."""
    x, wg, wu, wd = _small_layer(M=4, H=256, I=256, seed=8)
    qw = oracle.quantize_weights(wg, wu, wd)
    I = wg.shape[0]
    xd = oracle.dequantize(*oracle.quantize_bf16(x))
    wgu = oracle.dequantize(qw["gateup_codes"], qw["gateup_scales"])
    wdd = oracle.dequantize(qw["down_codes"], qw["down_scales"])
    g, u = xd @ wgu[:I].T, xd @ wgu[I:].T
    if mistake == "swap_gate_up":
        g, u = u, g
    h = oracle.silu(g) * u
    hd = h if mistake == "skip_h_requant" else oracle.quant_dequant(h)
    if mistake == "scale_rule_minus7":
        c, s = oracle.quantize_f64(h)
        hd = oracle.dequantize(c, (s.astype(np.int64) + 1).astype(np.uint8))
    if mistake == "transpose_down":
        wdd = wdd.T
    if mistake == "scale_layout":
        # scales read in the tiled order as if they were row-major (the pages' bug)
        tiled = oracle.scales_rowmajor_to_tiled(qw["down_scales"])
        wrong = tiled[: qw["down_scales"].size].reshape(qw["down_scales"].shape)
        wdd = oracle.dequantize(qw["down_codes"], wrong)
    y = hd @ wdd.T
    assert _pin_error(y, x, wg, wu, wd) > 1e-3


# ------------------------------------------------------------------ the decoder block
def _gain(H, seed):
    rng = np.random.default_rng(seed)
    return inputs.bf16_bits_from_f32((1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32))


def _ones(H):
    return inputs.bf16_bits_from_f32(np.ones(H, np.float32))


def test_rmsnorm_matches_torch():
    x, *_ = _small_layer(M=7, H=384, seed=31, token_scale_log10=(-2.0, 2.0))
    g = _gain(384, 1)
    for eps in (0.0, 1e-6, 0.5):
        want = torch.nn.functional.rms_norm(_f64(x), (384,), weight=_f64(g), eps=eps)
        np.testing.assert_allclose(oracle.rmsnorm(x, g, eps), want.numpy(), rtol=1e-13, atol=0)


def test_rmsnorm_closed_forms():
    x, *_ = _small_layer(M=6, H=512, seed=32, token_scale_log10=(-2.0, 2.0))
    n = oracle.rmsnorm(x, _ones(512), 0.0)
    # every row has mean square 1 (a norm over the wrong axis, or a missing
    # square root, breaks this)
    np.testing.assert_allclose(np.mean(n * n, axis=1), 1.0, rtol=1e-12)
    # scaling a row by 2^k (exact in bf16) leaves it unchanged; -1 flips it
    xf = oracle.bf16_bits_to_f64(x)
    for c in (4.0, 0.125, -1.0):
        xc = inputs.bf16_bits_from_f32((xf * c).astype(np.float32))
        np.testing.assert_allclose(oracle.rmsnorm(xc, _ones(512), 0.0), np.sign(c) * n, rtol=1e-13)
    # the gain multiplies each feature (column), not each token
    g = _gain(512, 2)
    np.testing.assert_allclose(oracle.rmsnorm(x, g, 0.0), n * oracle.bf16_bits_to_f64(g)[None, :], rtol=1e-15)
    # [3, 4] has mean square 12.5
    x2 = inputs.bf16_bits_from_f32(np.array([[3.0, 4.0]], np.float32))
    np.testing.assert_allclose(oracle.rmsnorm(x2, _ones(2), 0.0), [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]],
                               rtol=1e-15)
    # eps keeps an all-zero row at zero
    z = np.zeros((1, 64), np.uint16)
    assert np.all(oracle.rmsnorm(z, _ones(64), 1e-6) == 0.0)


def _torch_block(x, g, eps, wg, wu, wd, residual=True):
    xf = _f64(x)
    n = torch.nn.functional.rms_norm(xf, (xf.shape[1],), weight=_f64(g), eps=eps)
    qd = _torch_mx_qdq
    gg = qd(n) @ qd(_f64(wg)).T
    uu = qd(n) @ qd(_f64(wu)).T
    y = qd(torch.nn.functional.silu(gg) * uu) @ qd(_f64(wd)).T
    return y + xf if residual else y


@pytest.mark.parametrize("residual", [True, False])
def test_mlp_block_matches_torch_rebuild(residual):
    x, wg, wu, wd = _small_layer(M=5, H=256, I=384, seed=33, token_scale_log10=(-1.0, 1.0))
    g = _gain(256, 3)
    qw = oracle.quantize_weights(wg, wu, wd)
    res = oracle.mlp_block(x, g, 1e-6, qw, residual=residual)
    y_t = _torch_block(x, g, 1e-6, wg, wu, wd, residual)
    assert oracle.rel_l2(res["y"], y_t.numpy()) < 1e-12
    assert np.array_equal(res["y_bf16"], oracle.round_bf16_bits(y_t.numpy()))
    rows = np.array([1, 100, 255])
    part = oracle.mlp_block(x, g, 1e-6, qw, residual=residual, rows_down=rows)
    assert np.array_equal(part["y_bf16"], res["y_bf16"][:, rows])


@pytest.mark.parametrize("mistake", ["no_gain", "no_residual", "eps_outside_sqrt", "bf16_rounded_norm",
                                     "norm_over_tokens"])
def test_mlp_block_planted_mistakes_are_caught(mistake):
    """Each plausible bug in the block, planted here on the CPU, breaks the
    torch rebuild pin by far more than its 1e-12 tolerance."""
    x, wg, wu, wd = _small_layer(M=4, H=256, I=256, seed=34, token_scale_log10=(-1.0, 1.0))
    g = _gain(256, 4)
    eps = 1e-2  # large enough for the eps placement to show
    qw = oracle.quantize_weights(wg, wu, wd)
    xf = oracle.bf16_bits_to_f64(x)
    gf = oracle.bf16_bits_to_f64(g)
    if mistake == "norm_over_tokens":
        n = xf / np.sqrt(np.mean(xf * xf, axis=0, keepdims=True) + eps) * gf
    elif mistake == "eps_outside_sqrt":
        n = xf / (np.sqrt(np.mean(xf * xf, axis=1, keepdims=True)) + eps) * gf
    else:
        n = xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + eps) * (1.0 if mistake == "no_gain" else gf)
    if mistake == "bf16_rounded_norm":
        n = oracle.bf16_bits_to_f64(oracle.round_bf16_bits(n))
    y = oracle.mx_oracle._mlp_from_quantised(*oracle.quantize_f64(n), qw, None)["y"]
    if mistake != "no_residual":
        y = y + xf
    want = _torch_block(x, g, eps, wg, wu, wd).numpy()
    assert oracle.rel_l2(y, want) > 1e-6, mistake


# ------------------------------------------------------------------ paged decode attention
def _attn_case(B=3, Hq=8, Hkv=2, D=128, P=16, lo=5, hi=70, seed=1):
    wl = inputs.AttnWorkload("t", B, Hq, Hkv, D, P, lo, hi, seed)
    d = inputs.make_attention(wl)
    npages = d["k"].shape[0]
    kc, ks = oracle.quantize_bf16(d["k"].reshape(-1, D))
    vc, vs = oracle.quantize_bf16(d["v"].reshape(-1, D))
    cache = (kc.reshape(npages, Hkv, P, D), ks.reshape(npages, Hkv, P, D // 32),
             vc.reshape(npages, Hkv, P, D), vs.reshape(npages, Hkv, P, D // 32))
    return wl, d, cache


def _torch_attention(wl, d, cache, sm_scale, gqa=True):
    """The same step from torch pieces: the pages gathered into contiguous
    [Hkv, n, D] tensors, then torch's scaled_dot_product_attention with its
    GQA broadcast, in float64."""
    kc, ks, vc, vs = cache
    npages, Hkv, P, D = kc.shape
    kd = torch.from_numpy(oracle.dequantize(kc.reshape(-1, D), ks.reshape(-1, D // 32))).reshape(npages, Hkv, P, D)
    vd = torch.from_numpy(oracle.dequantize(vc.reshape(-1, D), vs.reshape(-1, D // 32))).reshape(npages, Hkv, P, D)
    q = _f64(d["q"])
    out = []
    for b in range(wl.B):
        n = int(d["seq_lens"][b])
        pages = torch.from_numpy(d["block_table"][b, : -(-n // P)].astype(np.int64))
        kb = kd[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :n]
        vb = vd[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :n]
        o = torch.nn.functional.scaled_dot_product_attention(q[b][None, :, None, :], kb[None], vb[None], scale=sm_scale,
                                                             enable_gqa=gqa)
        out.append(o[0, :, 0, :])
    return torch.stack(out).numpy()


@pytest.mark.parametrize("kw", [{}, {"Hq": 8, "Hkv": 8}, {"Hq": 16, "Hkv": 2, "P": 32, "lo": 1, "hi": 64},
                                {"B": 2, "Hq": 4, "Hkv": 1, "lo": 32, "hi": 32}])
def test_attention_matches_torch_sdpa(kw):
    wl, d, cache = _attn_case(**kw)
    sm = 1.0 / math.sqrt(wl.D)
    res = oracle.paged_decode_attention(d["q"], *cache, d["block_table"], d["seq_lens"], sm)
    want = _torch_attention(wl, d, cache, sm)
    np.testing.assert_allclose(res["out"], want, rtol=1e-10, atol=1e-12)
    assert np.array_equal(res["out_bf16"], oracle.round_bf16_bits(want))


def test_attention_closed_forms():
    wl, d, cache = _attn_case(B=2, lo=40, hi=60, seed=3)
    kc, ks, vc, vs = cache
    npages, Hkv, P, D = kc.shape
    table, lens = d["block_table"], d["seq_lens"]
    # one token: the output is that token's V row
    one = np.array([1, 1], np.int32)
    res = oracle.paged_decode_attention(d["q"], kc, ks, vc, vs, table, one, 0.1)
    for b in range(2):
        for h in range(wl.Hq):
            np.testing.assert_array_equal(res["out"][b, h], oracle.dequantize(vc[table[b, 0], h // 4, :1],
                                                                               vs[table[b, 0], h // 4, :1])[0])
    # identical keys (or a zero scale): the uniform average of the V rows
    same_k = np.broadcast_to(kc[:1, :, :1], kc.shape).copy()  # one key per head, in every slot
    same_s = np.broadcast_to(ks[:1, :, :1], ks.shape).copy()
    r1 = oracle.paged_decode_attention(d["q"], same_k, same_s, vc, vs, table, lens, 0.1)
    r2 = oracle.paged_decode_attention(d["q"], kc, ks, vc, vs, table, lens, 0.0)
    for b in range(2):
        n = int(lens[b])
        pages = table[b, : -(-n // P)]
        for hk in range(Hkv):
            vrows = oracle.dequantize(np.concatenate([vc[p, hk] for p in pages])[:n],
                                      np.concatenate([vs[p, hk] for p in pages])[:n])
            mean = vrows.mean(axis=0)
            for g in range(4):
                np.testing.assert_allclose(r1["out"][b, hk * 4 + g], mean, rtol=1e-12, atol=1e-14)
                np.testing.assert_allclose(r2["out"][b, hk * 4 + g], mean, rtol=1e-12, atol=1e-14)
    # moving the physical pages (and the table with them) changes nothing
    perm = np.random.default_rng(5).permutation(npages)
    inv = np.argsort(perm)
    moved = tuple(a[perm] for a in cache)
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1).astype(np.int32)
    r3 = oracle.paged_decode_attention(d["q"], *moved, table2, lens, 0.1)
    r4 = oracle.paged_decode_attention(d["q"], *cache, table, lens, 0.1)
    np.testing.assert_array_equal(r3["out"], r4["out"])


@pytest.mark.parametrize("mistake", ["gqa_modulo", "padding_slots", "no_scale", "k_scales_from_v"])
def test_attention_planted_mistakes_are_caught(mistake):
    """Each plausible bug, planted here on the CPU, moves the result far from
    the torch rebuild."""
    wl, d, cache = _attn_case(B=2, Hq=8, Hkv=2, lo=20, hi=45, seed=7)
    kc, ks, vc, vs = cache
    npages, Hkv, P, D = kc.shape
    sm = 1.0 / math.sqrt(D)
    q = oracle.bf16_bits_to_f64(d["q"])
    out = np.zeros_like(q)
    for b in range(wl.B):
        n = int(d["seq_lens"][b])
        npg = -(-n // P)
        pages = d["block_table"][b, :npg]
        use = npg * P if mistake == "padding_slots" else n
        for h in range(wl.Hq):
            hk = h % Hkv if mistake == "gqa_modulo" else h // (wl.Hq // Hkv)
            kscale = vs if mistake == "k_scales_from_v" else ks
            k = oracle.dequantize(np.concatenate([kc[p, hk] for p in pages])[:use],
                                  np.concatenate([kscale[p, hk] for p in pages])[:use])
            v = oracle.dequantize(np.concatenate([vc[p, hk] for p in pages])[:use],
                                  np.concatenate([vs[p, hk] for p in pages])[:use])
            s = (1.0 if mistake == "no_scale" else sm) * (k @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ v
    want = _torch_attention(wl, d, cache, sm)
    assert oracle.rel_l2(out, want) > 1e-3, mistake


# ------------------------------------------------------------------ 128x128 block scales (bsgemm)
def _torch_blockscale(bits, block_rows, block_cols=128):
    """Codes and scales from torch pieces: block amax in float32, the scale
    amax / 448 in float32, v / scale in float32, saturated, then torch's
    float8_e4m3fn conversion (round-to-nearest-even)."""
    v = torch.from_numpy(oracle.bf16_bits_to_f64(bits)).to(torch.float32)
    rows, K = v.shape
    rb = -(-rows // block_rows)
    pad = torch.zeros(rb * block_rows, K, dtype=torch.float32)
    pad[:rows] = v
    blk = pad.reshape(rb, block_rows, K // block_cols, block_cols)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / torch.tensor(448.0, dtype=torch.float32), torch.ones_like(amax))
    t = blk / scale[:, None, :, None]
    codes = t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).reshape(rb * block_rows, K)[:rows]
    return codes.numpy(), scale.numpy()


@pytest.mark.parametrize("rows,K,block_rows,seed", [(3, 256, 1, 1), (130, 384, 128, 2), (256, 128, 128, 3),
                                                    (5, 512, 1, 4)])
def test_blockscale_codes_match_torch(rows, K, block_rows, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-6, 6, size=(rows, 1)))
    v.reshape(-1)[rng.choice(v.size, 3, replace=False)] = 0.0
    bits = inputs.bf16_bits_from_f32(v.astype(np.float32))
    c, s = oracle.quantize_blockscale(bits, block_rows)
    tc, ts = _torch_blockscale(bits, block_rows)
    assert np.array_equal(s, ts)
    assert np.array_equal(c, tc)


def test_blockscale_gemm_exact_rational():
    rng = np.random.default_rng(5)
    a = inputs.bf16_bits_from_f32(rng.standard_normal((2, 256)).astype(np.float32))
    w = inputs.bf16_bits_from_f32((rng.standard_normal((130, 256)) * 0.05).astype(np.float32))
    res = oracle.gemm_blockscale(a, w)
    table = [Fraction(float(x)) for x in oracle.e4m3_table()]
    val = lambda code: (-1 if code & 0x80 else 1) * table[code & 0x7F]
    for m in range(2):
        for n in (0, 77, 129):
            exact = Fraction(0)
            for kb in range(2):
                dot = sum(val(int(res["a_codes"][m, k])) * val(int(res["w_codes"][n, k]))
                          for k in range(128 * kb, 128 * kb + 128))
                exact += Fraction(float(res["a_scales"][m, kb])) * Fraction(float(res["w_scales"][n // 128, kb])) * dot
            assert abs(float(exact) - res["c"][m, n]) <= 1e-12 * max(abs(float(exact)), 1e-30)


def test_blockscale_closed_forms():
    # a block of exact E4M3 values whose amax is 448 * 2^-3 has scale 2^-3
    # and round-trips exactly
    rng = np.random.default_rng(6)
    table = oracle.e4m3_table()
    vals = rng.choice(table, size=(1, 128)) * rng.choice([-1.0, 1.0], size=(1, 128))
    vals[0, 17] = 448.0
    v = vals * 0.125
    bits = inputs.bf16_bits_from_f32(v.astype(np.float32))
    c, s = oracle.quantize_blockscale(bits, 1)
    assert s[0, 0] == np.float32(0.125)
    np.testing.assert_array_equal(oracle.dequantize_blockscale(c, s, 1), v)
    # an all-zero block: scale 1, codes 0
    z = np.zeros((1, 128), np.uint16)
    cz, sz = oracle.quantize_blockscale(z, 1)
    assert sz[0, 0] == 1.0 and np.all(cz == 0)
    # blocks are independent: changing one 128x128 block leaves the others' bytes
    w = inputs.bf16_bits_from_f32(rng.standard_normal((256, 256)).astype(np.float32))
    c1, s1 = oracle.quantize_blockscale(w, 128)
    w2 = w.copy()
    w2[200, 200] = inputs.bf16_bits_from_f32(np.array([[1000.0]], np.float32))[0, 0]
    c2, s2 = oracle.quantize_blockscale(w2, 128)
    assert np.array_equal(c1[:128], c2[:128]) and np.array_equal(c1[128:, :128], c2[128:, :128])
    assert s1[1, 1] != s2[1, 1] and np.array_equal(np.delete(s1.ravel(), 3), np.delete(s2.ravel(), 3))


@pytest.mark.parametrize("mistake", ["int8_scale", "groups_along_m", "per_tensor"])
def test_blockscale_planted_mistakes_are_caught(mistake):
    """Each plausible bug in the scale rule or the block shape, planted here on
    the CPU, changes the codes the torch pin fixes."""
    rng = np.random.default_rng(7)
    v = rng.standard_normal((4, 256)) * np.exp(rng.uniform(-3, 3, size=(4, 1)))
    bits = inputs.bf16_bits_from_f32(v.astype(np.float32))
    tc, _ = _torch_blockscale(bits, 1)
    f = oracle.bf16_bits_to_f64(bits).astype(np.float32)
    if mistake == "int8_scale":
        s = np.abs(f.reshape(4, 2, 128)).max(axis=2) / np.float32(127.0)
        t = f.reshape(4, 2, 128) / s[:, :, None]
    elif mistake == "groups_along_m":
        s = np.abs(f).max(axis=0, keepdims=True) / np.float32(448.0)  # one scale per column over the tokens
        t = (f / s).reshape(4, 2, 128)
    else:
        t = (f / (np.abs(f).max() / np.float32(448.0))).reshape(4, 2, 128)
    t = torch.from_numpy(t.astype(np.float32)).clamp(-448.0, 448.0)
    codes = t.to(torch.float8_e4m3fn).view(torch.uint8).reshape(4, 256).numpy()
    assert np.mean(codes != tc) > 0.05, mistake


# ------------------------------------------------------------------ SwiGLU + requantisation (the unfused middle step)
def _torch_mx_codes(v: torch.Tensor):
    """MXFP8 codes and row-major scale bytes of float64 rows, from torch
    pieces: the block exponent from torch.frexp, the element rounding from
    torch's float8_e4m3fn conversion after the saturation of the MX rule."""
    rows, K = v.shape
    blk = v.reshape(rows, K // 32, 32)
    amax = blk.abs().amax(dim=-1, keepdim=True)
    _, ex = torch.frexp(amax)
    e = torch.where(amax == 0, torch.full_like(ex, -127), (ex - 1 - 8).clamp(-127, 127))
    t = (blk / torch.ldexp(torch.ones_like(amax), e.to(torch.float64))).clamp(-448.0, 448.0)
    codes = t.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, K)
    return codes.numpy(), (e[..., 0] + 127).to(torch.uint8).numpy()


def test_swiglu_quantize_matches_torch_rebuild():
    """oracle.swiglu_quantize (h = SiLU(g) * u, requantised along I) against
    torch's silu and float8 conversion, bit for bit, on gate sums spread over
    six decades, a zero block and a block of negative gates."""
    rng = np.random.default_rng(21)
    M, I = 9, 256
    g = rng.standard_normal((M, I)) * np.power(10.0, rng.uniform(-3, 3, size=(M, 1)))
    u = rng.standard_normal((M, I))
    g[2, 32:64] = 0.0
    g[3, 64:96] = -np.abs(g[3, 64:96]) - 5.0
    codes, scales = oracle.swiglu_quantize(np.concatenate([g, u], axis=1))
    h = torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)
    tc, ts = _torch_mx_codes(h)
    assert np.array_equal(codes, tc)
    assert np.array_equal(scales, ts)


def test_swiglu_quantize_closed_forms():
    """SiLU(64) = 64 exactly in float64 (1 + e^-64 rounds to 1), so gate 64
    with up values on the E4M3 grid gives h = 64 u, which requantises
    exactly; a zero gate gives a zero block (scale byte 0) whose codes carry
    the sign of u; swapping gate and up is caught."""
    rng = np.random.default_rng(22)
    I = 64
    # block maximum 14 = 1.75 * 2^3: h's amax 896 gives e = 9 - 8 = 1 and
    # 896 / 2 = 448 exactly (a mantissa above 1.75 would saturate); every
    # other value is at most 14 and at least 2^-4, so h / 2 stays on the grid
    mags = np.array([(1 + m / 8) * 2.0 ** k for k in range(-4, 4) for m in range(8)])
    mags = mags[mags <= 14.0]
    u = rng.choice(mags, size=(1, I)) * rng.choice([-1.0, 1.0], size=(1, I))
    u[0, 0] = 14.0
    g = np.full((1, I), 64.0)
    codes, scales = oracle.swiglu_quantize(np.concatenate([g, u], axis=1))
    back = oracle.dequantize(codes, scales)
    assert np.array_equal(back, 64.0 * u)
    zc, zs = oracle.swiglu_quantize(np.concatenate([np.zeros((1, I)), u], axis=1))
    assert np.all(zs == 0)
    assert np.array_equal(zc[0] & 0x7F, np.zeros(I, np.uint8))
    assert np.array_equal(zc[0] >> 7, (u[0] < 0).astype(np.uint8))
    gr = rng.standard_normal((3, I)) * 3
    ur = rng.standard_normal((3, I))
    right = oracle.swiglu_quantize(np.concatenate([gr, ur], axis=1))[0]
    swapped = oracle.swiglu_quantize(np.concatenate([ur, gr], axis=1))[0]
    assert np.mean(right == swapped) < 0.5
