"""Python binding of the GB300 MXFP8 SwiGLU MLP library (libfsops.so).

Argument marshalling only: every function below takes torch tensors (device
memory from PyTorch), passes their pointers and the current CUDA stream to the
C ABI of ``include/fsops.h`` under the same name, and raises ``FsopsError`` on
a non-OK status.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and importing this package fails
if the library is missing.

Build the library with ``python mxfp8_swiglu_mlp_gb300/build.py`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

from . import build as _build

__all__ = [
    "FsopsError", "lib", "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED_SHAPE", "ERR_MISALIGNED", "ERR_CUDA",
    "ERR_TIMEOUT", "ERR_NO_DEVICE", "SCALES_ROWMAJOR", "SCALES_TCGEN05", "DTYPE_BF16", "DTYPE_F32",
    "DTYPE_MXFP8", "fsops_quantize_mxfp8", "fsops_quantize_mxfp8_gateup", "fsops_scale_bytes", "fsops_mxfp8_gemm", "fsops_mxfp8_gemm_ex",
    "fsops_gemm_workspace_bytes", "fsops_swiglu_quantize_mxfp8", "fsops_mxfp8_swiglu_mlp",
    "fsops_mxfp8_swiglu_mlp_unfused", "fsops_mxfp8_swiglu_mlp_noalloc", "fsops_mlp_workspace_bytes", "fsops_set_workspace",
    "fsops_read_kernel_status", "fsops_set_wait_timeout_ns", "fsops_debug_set_extra_arrivals",
    "fsops_debug_set_knob", "KNOBS", "fsops_read_noalloc_status", "fsops_quantize_fp8_blockscale",
    "fsops_blockscale_scale_count", "fsops_fp8_blockscale_gemm", "fsops_blockscale_gemm_workspace_bytes",
    "fsops_status_string", "fsops_version", "fsops_last_cuda_error", "fsops_rmsnorm_quantize_mxfp8",
    "fsops_mxfp8_swiglu_mlp_block", "fsops_mxfp8_paged_decode_attention", "fsops_paged_attention_workspace_bytes",
    "quantize_weight", "MLPWeights", "prepare_mlp_weights", "quantize_blockscale",
    "Workspace", "pair_gate_up",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_CUDA, ERR_TIMEOUT, ERR_NO_DEVICE = range(7)
SCALES_ROWMAJOR, SCALES_TCGEN05 = 0, 1
# fsops_knob values (include/fsops.h)
KNOBS = {"TR0": 0, "TR1": 1, "WHOLE_TILES": 2, "PAIRS": 3, "GEMM_FORM": 4, "PRIME": 5, "MAX_INFLIGHT": 6,
         "LOCAL_XQ": 7, "DECODE_PATH": 8, "COOPERATIVE": 9,
         "EARLY_W": 10, "ALIGNED": 11, "ATTN_CHUNKS": 12}
DTYPE_BF16, DTYPE_F32, DTYPE_MXFP8 = 0, 1, 2

if not os.path.exists(_build.LIB):
    raise ImportError("libfsops.so is not built (%s); run python mxfp8_swiglu_mlp_gb300/build.py" % _build.LIB)

lib = ctypes.CDLL(_build.LIB)

_vp, _i, _u32, _u64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t


class _MlpScales(ctypes.Structure):
    _fields_ = [("gateup", _vp), ("down", _vp)]


_SIGS = {
    "fsops_quantize_mxfp8": ([_vp, _i, _i, _i, _vp, _vp, _i, _vp], _i),
    "fsops_scale_bytes": ([_i, _i, _i], _sz),
    "fsops_quantize_mxfp8_gateup": ([_vp, _vp, _i, _i, _i, _vp, _vp, _vp], _i),
    "fsops_quantize_fp8_blockscale": ([_vp, _i, _i, _i, _i, _vp, _vp, _vp], _i),
    "fsops_blockscale_scale_count": ([_i, _i, _i], _sz),
    "fsops_fp8_blockscale_gemm": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "fsops_blockscale_gemm_workspace_bytes": ([_i, _i, _i], _sz),
    "fsops_mxfp8_gemm": ([_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _sz, _vp], _i),
    "fsops_mxfp8_gemm_ex": ([_vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "fsops_gemm_workspace_bytes": ([_i, _i, _i], _sz),
    "fsops_swiglu_quantize_mxfp8": ([_vp, _i, _i, _vp, _vp, _vp], _i),
    "fsops_mxfp8_swiglu_mlp": ([_vp, _vp, _vp, ctypes.POINTER(_MlpScales), _vp, _i, _i, _i, _vp], _i),
    "fsops_mxfp8_swiglu_mlp_unfused": ([_vp, _vp, _vp, ctypes.POINTER(_MlpScales), _vp, _i, _i, _i, _vp], _i),
    "fsops_mxfp8_swiglu_mlp_noalloc": ([_vp, _vp, _vp, ctypes.POINTER(_MlpScales), _vp, _i, _i, _i, _vp], _i),
    "fsops_rmsnorm_quantize_mxfp8": ([_vp, _vp, ctypes.c_float, _i, _i, _i, _vp, _vp, _i, _vp], _i),
    "fsops_mxfp8_swiglu_mlp_block": ([_vp, _vp, ctypes.c_float, _i, _vp, _vp, ctypes.POINTER(_MlpScales), _vp, _i, _i,
                                      _i, _vp], _i),
    "fsops_mxfp8_paged_decode_attention": ([_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i,
                                            ctypes.c_float, _vp, _sz, _vp], _i),
    "fsops_paged_attention_workspace_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "fsops_mlp_workspace_bytes": ([_i, _i, _i], _sz),
    "fsops_set_workspace": ([_vp, _sz], _i),
    "fsops_read_kernel_status": ([_vp, ctypes.POINTER(_u32)], _i),
    "fsops_read_noalloc_status": ([ctypes.POINTER(_u32)], _i),
    "fsops_set_wait_timeout_ns": ([_u64], _i),
    "fsops_debug_set_extra_arrivals": ([_u32], _i),
    "fsops_debug_set_knob": ([_i, _i], _i),
    "fsops_status_string": ([_i], ctypes.c_char_p),
    "fsops_version": ([], _i),
    "fsops_last_cuda_error": ([], _i),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class FsopsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.cuda_error = lib.fsops_last_cuda_error() if status == ERR_CUDA else 0
        msg = "%s: %s (status %d)" % (where, lib.fsops_status_string(status).decode(), status)
        if self.cuda_error:
            msg += ", cudaError %d" % self.cuda_error
        super().__init__(msg)


def _check(status: int, where: str) -> None:
    if status != OK:
        raise FsopsError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- same-name wrappers
def fsops_quantize_mxfp8(x, rows: int, K: int, ld: int, codes, scales, layout: int, stream=None) -> None:
    _check(lib.fsops_quantize_mxfp8(_ptr(x), rows, K, ld, _ptr(codes), _ptr(scales), layout, _stream(stream)),
           "fsops_quantize_mxfp8")


def fsops_quantize_mxfp8_gateup(w_gate, w_up, I: int, H: int, ld: int, codes, scales, stream=None) -> None:
    _check(lib.fsops_quantize_mxfp8_gateup(_ptr(w_gate), _ptr(w_up), I, H, ld, _ptr(codes), _ptr(scales),
                                           _stream(stream)), "fsops_quantize_mxfp8_gateup")


def fsops_quantize_fp8_blockscale(x, rows: int, K: int, ld: int, block_rows: int, codes, scales,
                                  stream=None) -> None:
    _check(lib.fsops_quantize_fp8_blockscale(_ptr(x), rows, K, ld, block_rows, _ptr(codes), _ptr(scales),
                                             _stream(stream)), "fsops_quantize_fp8_blockscale")


def fsops_blockscale_scale_count(rows: int, K: int, block_rows: int) -> int:
    return lib.fsops_blockscale_scale_count(rows, K, block_rows)


def fsops_fp8_blockscale_gemm(a_codes, a_scales, w_codes, w_scales, c, c_dtype: int, M: int, N: int, K: int,
                              workspace, ws_bytes: int, stream=None) -> None:
    _check(lib.fsops_fp8_blockscale_gemm(_ptr(a_codes), _ptr(a_scales), _ptr(w_codes), _ptr(w_scales), _ptr(c),
                                         c_dtype, M, N, K, _ptr(workspace), ws_bytes, _stream(stream)),
           "fsops_fp8_blockscale_gemm")


def fsops_blockscale_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib.fsops_blockscale_gemm_workspace_bytes(M, N, K)


def quantize_blockscale(x_bf16, block_rows: int, stream=None):
    """bf16 CUDA tensor [rows, K] -> (E4M3 codes uint8 [rows, K], fp32 scales
    [ceil(rows / block_rows), K / 128]) in blocks of block_rows x 128."""
    import torch

    rows, K = x_bf16.shape
    codes = torch.empty((rows, K), dtype=torch.uint8, device=x_bf16.device)
    scales = torch.empty(((rows + block_rows - 1) // block_rows, K // 128), dtype=torch.float32,
                         device=x_bf16.device)
    fsops_quantize_fp8_blockscale(x_bf16, rows, K, x_bf16.stride(0), block_rows, codes, scales, stream)
    return codes, scales


def fsops_rmsnorm_quantize_mxfp8(x, gamma, eps: float, rows: int, K: int, ld: int, codes, scales, layout: int,
                                 stream=None) -> None:
    _check(lib.fsops_rmsnorm_quantize_mxfp8(_ptr(x), _ptr(gamma), eps, rows, K, ld, _ptr(codes), _ptr(scales), layout,
                                            _stream(stream)), "fsops_rmsnorm_quantize_mxfp8")


def fsops_scale_bytes(rows: int, K: int, layout: int) -> int:
    return lib.fsops_scale_bytes(rows, K, layout)


def fsops_mxfp8_gemm(a_bf16, b_codes, b_scales, c_bf16, M: int, N: int, K: int, workspace, ws_bytes: int,
                     stream=None) -> None:
    _check(lib.fsops_mxfp8_gemm(_ptr(a_bf16), _ptr(b_codes), _ptr(b_scales), _ptr(c_bf16), M, N, K,
                                _ptr(workspace), ws_bytes, _stream(stream)), "fsops_mxfp8_gemm")


def fsops_mxfp8_gemm_ex(a, a_scales, a_dtype: int, b_codes, b_scales, c, c_dtype: int, M: int, N: int, K: int,
                        workspace, ws_bytes: int, stream=None) -> None:
    _check(lib.fsops_mxfp8_gemm_ex(_ptr(a), _ptr(a_scales), a_dtype, _ptr(b_codes), _ptr(b_scales), _ptr(c),
                                   c_dtype, M, N, K, _ptr(workspace), ws_bytes, _stream(stream)),
           "fsops_mxfp8_gemm_ex")


def fsops_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib.fsops_gemm_workspace_bytes(M, N, K)


def fsops_swiglu_quantize_mxfp8(gu, M: int, I: int, h_codes, h_scales, stream=None) -> None:
    _check(lib.fsops_swiglu_quantize_mxfp8(_ptr(gu), M, I, _ptr(h_codes), _ptr(h_scales), _stream(stream)),
           "fsops_swiglu_quantize_mxfp8")


def _mlp_scales(scales) -> _MlpScales:
    gateup, down = scales
    return _MlpScales(_ptr(gateup), _ptr(down))


def fsops_mxfp8_swiglu_mlp(x_bf16, w_gateup, w_down, scales, y_bf16, M: int, H: int, I: int, stream=None) -> None:
    """``scales`` is (gateup_scales, down_scales)."""
    sc = _mlp_scales(scales)
    _check(lib.fsops_mxfp8_swiglu_mlp(_ptr(x_bf16), _ptr(w_gateup), _ptr(w_down), ctypes.byref(sc), _ptr(y_bf16),
                                      M, H, I, _stream(stream)), "fsops_mxfp8_swiglu_mlp")


def fsops_paged_attention_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, page_size: int, max_pages: int) -> int:
    return lib.fsops_paged_attention_workspace_bytes(B, Hq, Hkv, D, page_size, max_pages)


def fsops_mxfp8_paged_decode_attention(q, k_codes, k_scales, v_codes, v_scales, num_pages: int, block_table,
                                       max_pages: int, seq_lens, out, B: int, Hq: int, Hkv: int, D: int, page_size: int,
                                       sm_scale: float, workspace, ws_bytes: int, stream=None) -> None:
    """One decode step of attention over the paged MXFP8 KV cache (see fsops.h)."""
    _check(lib.fsops_mxfp8_paged_decode_attention(_ptr(q), _ptr(k_codes), _ptr(k_scales), _ptr(v_codes),
                                                  _ptr(v_scales), num_pages, _ptr(block_table), max_pages,
                                                  _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, page_size, sm_scale,
                                                  _ptr(workspace), ws_bytes, _stream(stream)),
           "fsops_mxfp8_paged_decode_attention")


def fsops_mxfp8_swiglu_mlp_block(x_bf16, gamma_bf16, eps: float, residual: bool, w_gateup, w_down, scales, y_bf16,
                                 M: int, H: int, I: int, stream=None) -> None:
    """y = x + MLP(RMSNorm(x) * gamma) (``residual``) or the MLP alone."""
    sc = _mlp_scales(scales)
    _check(lib.fsops_mxfp8_swiglu_mlp_block(_ptr(x_bf16), _ptr(gamma_bf16), eps, 1 if residual else 0, _ptr(w_gateup),
                                            _ptr(w_down), ctypes.byref(sc), _ptr(y_bf16), M, H, I, _stream(stream)),
           "fsops_mxfp8_swiglu_mlp_block")


def fsops_mxfp8_swiglu_mlp_unfused(x_bf16, w_gateup, w_down, scales, y_bf16, M: int, H: int, I: int,
                                   stream=None) -> None:
    sc = _mlp_scales(scales)
    _check(lib.fsops_mxfp8_swiglu_mlp_unfused(_ptr(x_bf16), _ptr(w_gateup), _ptr(w_down), ctypes.byref(sc),
                                              _ptr(y_bf16), M, H, I, _stream(stream)),
           "fsops_mxfp8_swiglu_mlp_unfused")


def fsops_mxfp8_swiglu_mlp_noalloc(x_bf16, w_gateup, w_down, scales, y_bf16, M: int, H: int, I: int,
                                   stream=None) -> None:
    """The fused MLP without a workspace: for callers that cannot allocate
    device memory (its scratch is a fixed 8 MiB buffer inside the library)."""
    sc = _mlp_scales(scales)
    _check(lib.fsops_mxfp8_swiglu_mlp_noalloc(_ptr(x_bf16), _ptr(w_gateup), _ptr(w_down), ctypes.byref(sc),
                                              _ptr(y_bf16), M, H, I, _stream(stream)),
           "fsops_mxfp8_swiglu_mlp_noalloc")


def fsops_mlp_workspace_bytes(M: int, H: int, I: int) -> int:
    return lib.fsops_mlp_workspace_bytes(M, H, I)


def fsops_set_workspace(ws, nbytes: int) -> None:
    _check(lib.fsops_set_workspace(_ptr(ws), nbytes), "fsops_set_workspace")


def fsops_read_kernel_status(workspace=None) -> int:
    w = _u32(0)
    _check(lib.fsops_read_kernel_status(_ptr(workspace), ctypes.byref(w)), "fsops_read_kernel_status")
    return w.value


def fsops_read_noalloc_status() -> int:
    w = _u32(0)
    _check(lib.fsops_read_noalloc_status(ctypes.byref(w)), "fsops_read_noalloc_status")
    return w.value


def fsops_set_wait_timeout_ns(ns: int) -> None:
    _check(lib.fsops_set_wait_timeout_ns(ns), "fsops_set_wait_timeout_ns")


def fsops_debug_set_extra_arrivals(n: int) -> None:
    _check(lib.fsops_debug_set_extra_arrivals(n), "fsops_debug_set_extra_arrivals")


def fsops_debug_set_knob(knob, value: int) -> None:
    """Force a plan knob (a name of ``KNOBS`` or its number); -1 restores the default."""
    k = KNOBS[knob] if isinstance(knob, str) else int(knob)
    _check(lib.fsops_debug_set_knob(k, int(value)), "fsops_debug_set_knob")


def fsops_status_string(s: int) -> str:
    return lib.fsops_status_string(s).decode()


def fsops_version() -> int:
    return lib.fsops_version()


def fsops_last_cuda_error() -> int:
    return lib.fsops_last_cuda_error()


# ---------------------------------------------------------------- tensor helpers
def quantize_weight(w_bf16, layout: int = SCALES_TCGEN05, stream=None) -> Tuple["object", "object"]:
    """Quantise a bf16 CUDA tensor [rows, K] -> (codes uint8 [rows, K], scales uint8)."""
    import torch

    rows, K = w_bf16.shape
    codes = torch.empty((rows, K), dtype=torch.uint8, device=w_bf16.device)
    scales = torch.empty(fsops_scale_bytes(rows, K, layout), dtype=torch.uint8, device=w_bf16.device)
    fsops_quantize_mxfp8(w_bf16, rows, K, w_bf16.stride(0), codes, scales, layout, stream)
    return codes, scales


class MLPWeights:
    """Quantised MLP weights: W_gateup ([2I, H], gate/up rows paired in blocks
    of 64, see ``pair_gate_up``) and W_down ([H, I])."""

    def __init__(self, gateup_codes, gateup_scales, down_codes, down_scales, H: int, I: int):
        self.gateup_codes, self.gateup_scales = gateup_codes, gateup_scales
        self.down_codes, self.down_scales = down_codes, down_scales
        self.H, self.I = H, I

    @property
    def scales(self):
        return (self.gateup_scales, self.down_scales)


PAIR_ROWS = 64


def pair_gate_up(w_gate, w_up):
    """The row order of W_gateup as a bf16 tensor (for inspection and tests;
    ``prepare_mlp_weights`` quantises straight into this order on the device):
    128-row block j holds W_gate rows 64j..64j+63 followed by W_up rows
    64j..64j+63."""
    import torch

    I, H = w_gate.shape
    return torch.stack([w_gate.reshape(I // PAIR_ROWS, PAIR_ROWS, H), w_up.reshape(I // PAIR_ROWS, PAIR_ROWS, H)],
                       dim=1).reshape(2 * I, H).contiguous()


def prepare_mlp_weights(w_gate, w_up, w_down, stream=None) -> MLPWeights:
    """bf16 CUDA tensors W_gate [I, H], W_up [I, H], W_down [H, I] -> MLPWeights
    (W_gateup quantised into the paired row order by fsops_quantize_mxfp8_gateup)."""
    import torch

    I, H = w_gate.shape
    if w_up.shape != (I, H) or w_down.shape != (H, I):
        raise ValueError("W_gate, W_up must be [I, H] and W_down [H, I]")
    if w_gate.stride(1) != 1 or w_up.stride(1) != 1 or w_gate.stride(0) != w_up.stride(0):
        w_gate, w_up = w_gate.contiguous(), w_up.contiguous()
    gc = torch.empty((2 * I, H), dtype=torch.uint8, device=w_gate.device)
    gs = torch.empty(fsops_scale_bytes(2 * I, H, SCALES_TCGEN05), dtype=torch.uint8, device=w_gate.device)
    fsops_quantize_mxfp8_gateup(w_gate, w_up, I, H, w_gate.stride(0), gc, gs, stream)
    dc, ds = quantize_weight(w_down.contiguous(), SCALES_TCGEN05, stream)
    return MLPWeights(gc, gs, dc, ds, H, I)


class Workspace:
    """Device workspace registered for the MLP entry points of the current device."""

    def __init__(self, M: int, H: int, I: int, device=None):
        import torch

        n = fsops_mlp_workspace_bytes(M, H, I)
        if n == 0:
            raise FsopsError(ERR_UNSUPPORTED_SHAPE, "fsops_mlp_workspace_bytes")
        self.nbytes = n
        self.buf = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        fsops_set_workspace(self.ptr, n)
