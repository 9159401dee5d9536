"""The C ABI library loads without a GPU, exports every function that
include/fsops.h declares, and rejects bad arguments on the host before any
CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "fsops.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(fsops_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def fs():
    import __graft_entry__

    __graft_entry__.build()
    import mxfp8_swiglu_mlp_gb300 as fs

    return fs


def test_every_declared_symbol_is_exported(fs):
    names = _declared_functions()
    assert len(names) >= 15, names
    for n in names:
        assert hasattr(fs.lib, n), n


def test_status_strings(fs):
    for s in range(7):
        assert fs.fsops_status_string(s) != "unknown status"
    assert fs.fsops_status_string(99) == "unknown status"
    assert fs.fsops_version() >= 100


def test_scale_bytes(fs):
    assert fs.fsops_scale_bytes(300, 384, fs.SCALES_ROWMAJOR) == 300 * 12
    assert fs.fsops_scale_bytes(300, 384, fs.SCALES_TCGEN05) == 3 * 3 * 512
    assert fs.fsops_scale_bytes(1, 128, fs.SCALES_TCGEN05) == 512
    assert fs.fsops_scale_bytes(10, 128, 7) == 0


FAKE = 0x100000  # 16-byte aligned, never dereferenced: every call below fails validation first


def test_mlp_validation(fs):
    lib = fs.lib
    sc = fs._MlpScales(FAKE, FAKE)
    call = lambda x=FAKE, w1=FAKE, w2=FAKE, s=ctypes.byref(sc), y=FAKE, M=16, H=256, I=256: \
        lib.fsops_mxfp8_swiglu_mlp(x, w1, w2, s, y, M, H, I, None)
    assert call(x=None) == fs.ERR_INVALID_ARG
    assert call(y=None) == fs.ERR_INVALID_ARG
    assert call(s=None) == fs.ERR_INVALID_ARG
    for M in (0, 16385, -1):
        assert call(M=M) == fs.ERR_UNSUPPORTED_SHAPE
    for H, I in ((200, 256), (256, 100), (0, 256), (128 * 513, 256)):
        assert call(H=H, I=I) == fs.ERR_UNSUPPORTED_SHAPE
    assert call(x=FAKE + 2) == fs.ERR_MISALIGNED
    assert call(w2=FAKE + 8) == fs.ERR_MISALIGNED
    assert call(y=FAKE + 4) == fs.ERR_MISALIGNED
    bad = fs._MlpScales(FAKE + 1, FAKE)
    assert call(s=ctypes.byref(bad)) == fs.ERR_MISALIGNED
    nul = fs._MlpScales(None, FAKE)
    assert call(s=ctypes.byref(nul)) == fs.ERR_INVALID_ARG
    assert lib.fsops_mxfp8_swiglu_mlp_unfused(FAKE, FAKE, FAKE, ctypes.byref(sc), FAKE, 0, 256, 256, None) \
        == fs.ERR_UNSUPPORTED_SHAPE


def test_gemm_validation(fs):
    lib = fs.lib
    g = lambda a=FAKE, asc=None, adt=fs.DTYPE_BF16, b=FAKE, bs=FAKE, c=FAKE, cdt=fs.DTYPE_BF16, M=4, N=256, K=256, \
        ws=FAKE, n=1 << 30: lib.fsops_mxfp8_gemm_ex(a, asc, adt, b, bs, c, cdt, M, N, K, ws, n, None)
    assert g(a=None) == fs.ERR_INVALID_ARG
    assert g(ws=None) == fs.ERR_INVALID_ARG
    assert g(adt=fs.DTYPE_F32) == fs.ERR_INVALID_ARG
    assert g(cdt=fs.DTYPE_MXFP8) == fs.ERR_INVALID_ARG
    assert g(asc=FAKE) == fs.ERR_INVALID_ARG                 # bf16 A takes no scales
    assert g(adt=fs.DTYPE_MXFP8) == fs.ERR_INVALID_ARG      # MXFP8 A needs scales
    for M, N, K in ((0, 256, 256), (16385, 256, 256), (4, 200, 256), (4, 256, 100), (4, 256, 65536 + 128)):
        assert g(M=M, N=N, K=K) == fs.ERR_UNSUPPORTED_SHAPE
    assert g(c=FAKE + 2) == fs.ERR_MISALIGNED
    assert g(b=FAKE + 8) == fs.ERR_MISALIGNED
    assert lib.fsops_mxfp8_gemm(FAKE, FAKE, FAKE, FAKE, 0, 256, 256, FAKE, 1 << 30, None) == fs.ERR_UNSUPPORTED_SHAPE


def test_quantize_validation(fs):
    lib = fs.lib
    q = lambda x=FAKE, rows=4, K=256, ld=256, c=FAKE, s=FAKE, layout=fs.SCALES_TCGEN05: \
        lib.fsops_quantize_mxfp8(x, rows, K, ld, c, s, layout, None)
    assert q(layout=5) == fs.ERR_INVALID_ARG
    assert q(K=96) == fs.ERR_UNSUPPORTED_SHAPE                # tiled layout wants K % 128
    assert q(K=100, layout=fs.SCALES_ROWMAJOR, ld=104) == fs.ERR_UNSUPPORTED_SHAPE
    assert q(ld=100) == fs.ERR_UNSUPPORTED_SHAPE              # ld < K
    assert q(ld=260) == fs.ERR_UNSUPPORTED_SHAPE              # ld % 8
    assert q(rows=-1) == fs.ERR_UNSUPPORTED_SHAPE
    assert q(rows=0, x=None) == fs.OK                         # empty input: nothing to do
    assert q(x=None) == fs.ERR_INVALID_ARG
    assert q(x=FAKE + 2) == fs.ERR_MISALIGNED
    assert lib.fsops_swiglu_quantize_mxfp8(FAKE, 0, 256, FAKE, FAKE, None) == fs.ERR_UNSUPPORTED_SHAPE
    assert lib.fsops_swiglu_quantize_mxfp8(FAKE, 4, 200, FAKE, FAKE, None) == fs.ERR_UNSUPPORTED_SHAPE
    assert lib.fsops_swiglu_quantize_mxfp8(None, 4, 256, FAKE, FAKE, None) == fs.ERR_INVALID_ARG


def test_size_queries_reject_bad_shapes(fs):
    assert fs.fsops_mlp_workspace_bytes(0, 256, 256) == 0
    assert fs.fsops_mlp_workspace_bytes(16385, 256, 256) == 0
    assert fs.fsops_gemm_workspace_bytes(4, 100, 256) == 0
    assert fs.lib.fsops_set_wait_timeout_ns(0) == fs.ERR_INVALID_ARG


def test_rmsnorm_quantize_validation(fs):
    lib = fs.lib
    q = lambda x=FAKE, g=FAKE, eps=1e-6, rows=4, K=256, ld=256, c=FAKE, s=FAKE, layout=fs.SCALES_TCGEN05: \
        lib.fsops_rmsnorm_quantize_mxfp8(x, g, eps, rows, K, ld, c, s, layout, None)
    assert q(layout=7) == fs.ERR_INVALID_ARG
    assert q(eps=-1.0) == fs.ERR_INVALID_ARG
    assert q(eps=float("nan")) == fs.ERR_INVALID_ARG
    assert q(K=96) == fs.ERR_UNSUPPORTED_SHAPE                 # tiled layout wants K % 128
    assert q(ld=100) == fs.ERR_UNSUPPORTED_SHAPE               # ld < K
    assert q(rows=-1) == fs.ERR_UNSUPPORTED_SHAPE
    assert q(rows=0) == fs.OK                                  # nothing to do, no device needed
    assert q(g=None) == fs.ERR_INVALID_ARG
    assert q(g=FAKE + 4) == fs.ERR_MISALIGNED


def test_mlp_block_validation(fs):
    lib = fs.lib
    sc = fs._MlpScales(FAKE, FAKE)
    call = lambda g=FAKE, eps=1e-6, res=1, M=16, H=256, I=256: lib.fsops_mxfp8_swiglu_mlp_block(
        FAKE, g, eps, res, FAKE, FAKE, ctypes.byref(sc), FAKE, M, H, I, None)
    assert call(g=None) == fs.ERR_INVALID_ARG
    assert call(eps=float("nan")) == fs.ERR_INVALID_ARG
    assert call(res=2) == fs.ERR_INVALID_ARG
    assert call(g=FAKE + 2) == fs.ERR_MISALIGNED
    for M in (0, 16385):
        assert call(M=M) == fs.ERR_UNSUPPORTED_SHAPE
    assert call(H=200) == fs.ERR_UNSUPPORTED_SHAPE


def test_paged_attention_validation(fs):
    """Host-side checks of fsops_mxfp8_paged_decode_attention, before any
    device work."""
    lib = fs.lib
    F4 = FAKE

    def call(q=FAKE, kc=FAKE, ks=FAKE, vc=FAKE, vs=FAKE, num_pages=10, table=F4, max_pages=4, lens=F4, out=FAKE,
             B=2, Hq=8, Hkv=2, D=128, P=16, sm=0.088, ws=FAKE, ws_n=1 << 20):
        return lib.fsops_mxfp8_paged_decode_attention(q, kc, ks, vc, vs, num_pages, table, max_pages, lens, out, B,
                                                      Hq, Hkv, D, P, sm, ws, ws_n, None)

    for kw in ({"D": 64}, {"P": 8}, {"P": 48}, {"Hq": 6, "Hkv": 4}, {"Hq": 24, "Hkv": 2}, {"B": 0},
               {"num_pages": 0}, {"max_pages": 0}, {"Hq": 1, "Hkv": 2}):
        assert call(**kw) == fs.ERR_UNSUPPORTED_SHAPE, kw
    assert call(q=None) == fs.ERR_INVALID_ARG
    assert call(table=None) == fs.ERR_INVALID_ARG
    assert call(ws=None) == fs.ERR_INVALID_ARG
    assert call(sm=float("nan")) == fs.ERR_INVALID_ARG
    assert call(kc=FAKE + 8) == fs.ERR_MISALIGNED
    assert call(ws=FAKE + 16) == fs.ERR_MISALIGNED  # the workspace wants 256-byte alignment
    assert call(lens=FAKE + 2) == fs.ERR_MISALIGNED
    assert fs.fsops_paged_attention_workspace_bytes(2, 8, 2, 64, 16, 4) == 0


def test_gateup_quantize_validation(fs):
    lib = fs.lib
    q = lambda g=FAKE, u=FAKE, I=256, H=256, ld=256, c=FAKE, s=FAKE: \
        lib.fsops_quantize_mxfp8_gateup(g, u, I, H, ld, c, s, None)
    for kw in ({"I": 96}, {"I": 0}, {"H": 200}, {"ld": 128}, {"ld": 260}, {"I": 1 << 20, "H": 1 << 14}):
        assert q(**kw) == fs.ERR_UNSUPPORTED_SHAPE, kw
    assert q(g=None) == fs.ERR_INVALID_ARG
    assert q(u=None) == fs.ERR_INVALID_ARG
    assert q(s=None) == fs.ERR_INVALID_ARG
    assert q(u=FAKE + 2) == fs.ERR_MISALIGNED
    assert q(c=FAKE + 8) == fs.ERR_MISALIGNED


def test_knobs_and_noalloc_status_validation(fs):
    lib = fs.lib
    assert lib.fsops_debug_set_knob(-1, 0) == fs.ERR_INVALID_ARG
    assert lib.fsops_debug_set_knob(len(fs.KNOBS), 0) == fs.ERR_INVALID_ARG
    for k in fs.KNOBS.values():
        assert lib.fsops_debug_set_knob(k, -1) == fs.OK
    assert lib.fsops_read_noalloc_status(None) == fs.ERR_INVALID_ARG


def test_blockscale_validation(fs):
    lib = fs.lib
    q = lambda x=FAKE, rows=4, K=256, ld=256, br=1, c=FAKE, s=FAKE: \
        lib.fsops_quantize_fp8_blockscale(x, rows, K, ld, br, c, s, None)
    assert q(br=64) == fs.ERR_INVALID_ARG
    assert q(K=96) == fs.ERR_UNSUPPORTED_SHAPE
    assert q(ld=128) == fs.ERR_UNSUPPORTED_SHAPE
    assert q(ld=260) == fs.ERR_UNSUPPORTED_SHAPE
    assert q(rows=0, x=None) == fs.OK
    assert q(x=None) == fs.ERR_INVALID_ARG
    assert q(x=FAKE + 2) == fs.ERR_MISALIGNED
    assert q(s=FAKE + 2) == fs.ERR_MISALIGNED
    assert fs.fsops_blockscale_scale_count(300, 384, 128) == 3 * 3
    assert fs.fsops_blockscale_scale_count(300, 384, 1) == 300 * 3
    assert fs.fsops_blockscale_scale_count(300, 100, 1) == 0
    g = lambda a=FAKE, sa=FAKE, w=FAKE, sw=FAKE, c=FAKE, cdt=fs.DTYPE_BF16, M=4, N=256, K=256, ws=FAKE, n=1 << 30: \
        lib.fsops_fp8_blockscale_gemm(a, sa, w, sw, c, cdt, M, N, K, ws, n, None)
    assert g(a=None) == fs.ERR_INVALID_ARG
    assert g(sw=None) == fs.ERR_INVALID_ARG
    assert g(cdt=fs.DTYPE_MXFP8) == fs.ERR_INVALID_ARG
    for M, N, K in ((0, 256, 256), (129, 256, 256), (4, 200, 256), (4, 256, 100)):
        assert g(M=M, N=N, K=K) == fs.ERR_UNSUPPORTED_SHAPE
    assert g(n=16) == fs.ERR_INVALID_ARG
    assert g(ws=FAKE + 16) == fs.ERR_MISALIGNED
    assert g(c=FAKE + 2) == fs.ERR_MISALIGNED
    assert fs.fsops_blockscale_gemm_workspace_bytes(129, 256, 256) == 0
    assert fs.fsops_blockscale_gemm_workspace_bytes(16, 256, 256) == 16384 + 16 * 256 * 4
