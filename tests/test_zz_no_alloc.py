"""The no-allocation MLP entry point (fsops_mxfp8_swiglu_mlp_noalloc), called
through the C ABI, against the workspace entry point (fsops_mxfp8_swiglu_mlp).

It serves callers that cannot allocate device memory, so its scratch is a
fixed buffer inside the library; this file runs last so that a failure here
leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest

import oracle
from workloads import inputs
from tests._util import (to_dev_u16, from_dev_bf16, bf16_bits_to_f64, rel_l2, REL_L2_TOL, MAX_ABS_TOL, max_abs_norm,
                         assert_repeat_close)

pytestmark = pytest.mark.gpu


def _call_noalloc(fs, xd, w, y, M, H, I):
    import torch

    sc = fs._MlpScales(w.gateup_scales.data_ptr(), w.down_scales.data_ptr())
    return fs.lib.fsops_mxfp8_swiglu_mlp_noalloc(xd.data_ptr(), w.gateup_codes.data_ptr(), w.down_codes.data_ptr(),
                                                 ctypes.byref(sc), y.data_ptr(), M, H, I,
                                                 torch.cuda.current_stream().cuda_stream)


def _read_status(fs):
    word = ctypes.c_uint32(0)
    assert fs.lib.fsops_read_noalloc_status(ctypes.byref(word)) == fs.OK
    return word.value


# (workload, M, sampled output features for the oracle check or None for all).
# m64 and m128 take the plans whose scratch layout differs most from the small
# cases: whole gate/up tiles (no gate/up split-K sums) and, at m128, 128-row
# down tiles; m128 is the case the 8 MiB limit is sized for.
CASES = [("m16", None, None), ("m1", None, None), ("m16", 3, None), ("m64", None, 256), ("m128", None, 256)]


@pytest.mark.parametrize("name,M,nrows", CASES)
def test_noalloc_matches_workspace_entry_point(name, M, nrows):
    import torch

    import mxfp8_swiglu_mlp_gb300 as fs

    wl = inputs.WORKLOADS[name]
    M = wl.M if M is None else M
    x = inputs.make_activations(wl, M)
    wg, wu, wd = inputs.make_layer(wl, 0)
    w = fs.prepare_mlp_weights(to_dev_u16(wg), to_dev_u16(wu), to_dev_u16(wd))
    xd = to_dev_u16(x)
    ws = fs.Workspace(M, wl.H, wl.I)
    y_ref = torch.empty((M, wl.H), dtype=torch.bfloat16, device="cuda")
    fs.fsops_mxfp8_swiglu_mlp(xd, w.gateup_codes, w.down_codes, w.scales, y_ref, M, wl.H, wl.I)
    torch.cuda.synchronize()
    ref_bits = from_dev_bf16(y_ref)
    rows = None if nrows is None else np.sort(np.random.default_rng(M).choice(wl.H, nrows, replace=False))
    want = bf16_bits_to_f64(oracle.swiglu_mlp(x, oracle.quantize_weights(wg, wu, wd), rows_down=rows)["y_bf16"])
    for _ in range(2):  # the second call runs on what the first one left in the buffer
        y = torch.full((M, wl.H), 7.0, dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(fs, xd, w, y, M, wl.H, wl.I) == fs.OK
        torch.cuda.synchronize()
        assert _read_status(fs) == 0
        got_bits = from_dev_bf16(y)
        # split-K sums are added in arrival order: the two entry points agree to
        # fp32 rounding, one bf16 step at most per element
        assert_repeat_close(got_bits, ref_bits)
        got = bf16_bits_to_f64(got_bits)
        sub = got if rows is None else got[:, rows]
        assert rel_l2(sub, want) <= REL_L2_TOL and max_abs_norm(sub, want) <= MAX_ABS_TOL
    del ws


def test_noalloc_timeout_is_reported_and_cleared():
    """A wait that can never be satisfied runs out inside the no-allocation
    call; the status word of its fixed buffer reports FSOPS_ERR_TIMEOUT, and
    the next call (which clears the buffer first) is correct again."""
    import torch

    import mxfp8_swiglu_mlp_gb300 as fs

    wl = inputs.make_workload_small("s", 4, 256, 384, 16)
    x = inputs.make_activations(wl)
    wg, wu, wd = inputs.make_layer(wl, 0)
    w = fs.prepare_mlp_weights(to_dev_u16(wg), to_dev_u16(wu), to_dev_u16(wd))
    xd = to_dev_u16(x)
    y = torch.empty((wl.M, wl.H), dtype=torch.bfloat16, device="cuda")
    fs.fsops_set_wait_timeout_ns(20_000_000)
    fs.fsops_debug_set_extra_arrivals(1)
    try:
        assert _call_noalloc(fs, xd, w, y, wl.M, wl.H, wl.I) == fs.OK
        torch.cuda.synchronize()
        word = _read_status(fs)
    finally:
        fs.fsops_debug_set_extra_arrivals(0)
        fs.fsops_set_wait_timeout_ns(1_000_000_000)
    assert (word >> 24) == fs.ERR_TIMEOUT, hex(word)
    assert _read_status(fs) == 0  # read and cleared
    want = bf16_bits_to_f64(oracle.swiglu_mlp(x, oracle.quantize_weights(wg, wu, wd))["y_bf16"])
    for _ in range(2):
        assert _call_noalloc(fs, xd, w, y, wl.M, wl.H, wl.I) == fs.OK
        torch.cuda.synchronize()
        assert _read_status(fs) == 0
        got = bf16_bits_to_f64(from_dev_bf16(y))
        assert rel_l2(got, want) <= REL_L2_TOL and max_abs_norm(got, want) <= MAX_ABS_TOL


def test_noalloc_rejects_shapes_beyond_its_buffer():
    import torch

    import mxfp8_swiglu_mlp_gb300 as fs

    # M = 128, H = I = 65536 needs far more than the 8 MiB buffer: rejected
    # before any pointer is touched (the pointers below are never dereferenced)
    fake = 1 << 20
    sc = fs._MlpScales(fake, fake)
    st = fs.lib.fsops_mxfp8_swiglu_mlp_noalloc(fake, fake, fake, ctypes.byref(sc), fake, 128, 65536, 65536,
                                               torch.cuda.current_stream().cuda_stream)
    assert st == fs.ERR_UNSUPPORTED_SHAPE
    st = fs.lib.fsops_mxfp8_swiglu_mlp_noalloc(fake, fake, fake, ctypes.byref(sc), fake, 129, 256, 256,
                                               torch.cuda.current_stream().cuda_stream)
    assert st == fs.ERR_UNSUPPORTED_SHAPE
