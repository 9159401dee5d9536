"""CPU oracle for the decode-shape MXFP8 SwiGLU MLP (fp64, plain, slow).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA library and never loads it.

What it computes, step by step, and where the step comes from:

1. MXFP8 quantisation (``quantize_bf16`` / ``quantize_f64``): 1x32 blocks
   along K, OCP UE8M0 scale, OCP E4M3 elements (Fish Audio post p2,
   "Estrategia de cuantizacion FP8"; X copy, "Custom kernels for the shapes
   TTS actually uses").  The rule itself (floor(log2 amax) - 8,
   round-to-nearest-even, saturate to +-448) is the OCP MX rule; the element
   loops are in ``mx_quant.c``.
2. Dequantisation: code value * 2^(scale - 127), exact.
3. SwiGLU MLP forward (X copy, "Custom kernels ...": activation, gate
   multiplication, down projection; p2 "Por que cuBLAS no era suficiente"):
   g = x^ W_g^T, u = x^ W_u^T, h = SiLU(g) * u, y = h^ W_d^T.  The matrix
   products are numpy float64 matmuls of the dequantised operands.
4. The intermediate h is requantised to MXFP8 along I before the down
   projection (p2 "Resultados de benchmark del kernel": the SwiGLU prologue is
   fused into the activation quantisation of the down GEMM), so the oracle
   mirrors that quantisation point: h^ = dequant(quant(h)).
5. The output is rounded once from fp64 to bf16 (round-to-nearest-even); the
   pages do not name the output type, bf16 matches the input activations.
6. The decoder block around the MLP (``rmsnorm``, ``mlp_block``): the pages
   name the MLP as Qwen3-4B's (p2, "Resultados de benchmark del kernel"), a
   pre-norm decoder layer, but never write the norm or the residual out.  The
   plainest reading, used here: the MLP's input is RMSNorm(x) * gamma =
   x / sqrt(mean(x^2) + eps) * gamma per token row, in float64, quantised to
   MXFP8 straight from float64; the block's output is x + MLP(...), rounded
   once to bf16.

7. Paged decode attention over an MXFP8 KV cache
   (``paged_decode_attention``): the pages list MXFP8 FlashAttention with
   paged decode and GQA through a stride-0 K/V broadcast (p2, "Ya esta
   disponible") without writing it out.  Read plainly: K and V are cached
   as MXFP8 (1x32 blocks along the head dimension, the rule of step 1), q
   and the probabilities stay in full precision, query head h reads KV head
   h // (Hq / Hkv), scores = sm_scale * q . k, softmax over the sequence,
   out = p . v, rounded once to bf16.

8. The second scale format of the same library, "bsgemm" (p1 "Custom
   kernels for the shapes TTS actually uses"; p2 "Estrategia de
   cuantizacion FP8": FP8 with 128x128 block scales, for Hopper), read
   plainly: weights in 128x128 blocks, activations in 1x128 groups along K
   (one token's block), each with an fp32 scale s = amax / 448 (1 for an
   all-zero block) and E4M3 codes RNE-satfinite of v / s.  s and v / s are
   computed in IEEE fp32, the precision a kernel takes that decision in, so
   the codes are defined bit for bit (``quantize_blockscale``); the GEMM
   (``gemm_blockscale``) is then exact up to float64 rounding.

Weight scales may be returned in the row-major layout or in the tiled layout
the library consumes (``scales_rowmajor_to_tiled``): 128-row x 4-block tiles
of 512 bytes, tile (rt, kg) at byte (rt * ceil(K/128) + kg) * 512, entry
(r, kb) at (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4 inside it.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c_long, c_void = ctypes.c_long, ctypes.c_void_p
        lib.mxo_e4m3_value.argtypes = [ctypes.c_int]
        lib.mxo_e4m3_value.restype = ctypes.c_double
        lib.mxo_e4m3_round.argtypes = [ctypes.c_double]
        lib.mxo_e4m3_round.restype = ctypes.c_int
        lib.mxo_block_exponent.argtypes = [ctypes.c_double]
        lib.mxo_block_exponent.restype = ctypes.c_int
        for name in ("mxo_quantize_f64", "mxo_quantize_bf16"):
            getattr(lib, name).argtypes = [c_void, c_long, c_long, c_void, c_void]
            getattr(lib, name).restype = None
        lib.mxo_dequantize.argtypes = [c_void, c_void, c_long, c_long, c_void]
        lib.mxo_dequantize.restype = None
        lib.mxo_round_bf16.argtypes = [c_void, c_long, c_void]
        lib.mxo_round_bf16.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- E4M3 / UE8M0
def e4m3_table() -> np.ndarray:
    """The 127 non-negative finite E4M3 values, indexed by magnitude code."""
    lib = _load()
    return np.array([lib.mxo_e4m3_value(c) for c in range(127)], dtype=np.float64)


def e4m3_round_code(t: float) -> int:
    """Magnitude code of the E4M3 value nearest to t >= 0 (ties to even, saturating)."""
    return int(_load().mxo_e4m3_round(float(t)))


def block_exponent(amax: float) -> int:
    return int(_load().mxo_block_exponent(float(amax)))


# ---------------------------------------------------------------- quantisation
def quantize_f64(v: np.ndarray):
    """v [rows, K] float64 -> (codes uint8 [rows, K], scales uint8 [rows, K/32] row-major)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, K = v.shape
    assert K % 32 == 0
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    _load().mxo_quantize_f64(_ptr(v), rows, K, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_bf16(bits: np.ndarray):
    """bf16 bit patterns [rows, K] -> (codes, row-major scales)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    rows, K = bits.shape
    assert K % 32 == 0
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    _load().mxo_quantize_bf16(_ptr(bits), rows, K, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, K = codes.shape
    assert scales.shape == (rows, K // 32)
    out = np.empty((rows, K), np.float64)
    _load().mxo_dequantize(_ptr(codes), _ptr(scales), rows, K, _ptr(out))
    return out


def round_bf16_bits(y: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 (ties to even), as uint16 bit patterns."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty(y.shape, np.uint16)
    _load().mxo_round_bf16(_ptr(y), y.size, _ptr(out))
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- scale layouts
def _tiled_offsets(rows: int, nb: int) -> np.ndarray:
    """Byte offset of every (row, block) entry in the tiled layout, shape [rows, nb]."""
    n_kg = -(-nb // 4)
    r = np.arange(rows, dtype=np.int64)[:, None]
    kb = np.arange(nb, dtype=np.int64)[None, :]
    rt, rr = r // 128, r % 128
    kg, kk = kb // 4, kb % 4
    return (rt * n_kg + kg) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + kk


def scales_rowmajor_to_tiled(scales: np.ndarray) -> np.ndarray:
    """Row-major [rows, K/32] UE8M0 bytes -> the tiled byte layout (flat uint8).

    Rows are padded to a multiple of 128 and blocks to a multiple of 4 with
    byte 0.  Tile (rt, kg) covers rows 128rt..128rt+127 and blocks
    4kg..4kg+3; it starts at byte (rt * n_kg + kg) * 512, and entry (r, kb)
    sits at (r % 32) * 16 + ((r % 128) // 32) * 4 + (kb % 4) inside it.
    """
    rows, nb = scales.shape
    out = np.zeros((-(-rows // 128)) * (-(-nb // 4)) * 512, np.uint8)
    out[_tiled_offsets(rows, nb)] = scales
    return out


def scales_tiled_to_rowmajor(tiled: np.ndarray, rows: int, K: int) -> np.ndarray:
    return np.asarray(tiled, np.uint8)[_tiled_offsets(rows, K // 32)]


def tiled_scale_bytes(rows: int, K: int) -> int:
    return (-(-rows // 128)) * (-(-(K // 32) // 4)) * 512


# ---------------------------------------------------------------- the MLP
def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g)), in float64."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def quant_dequant(v: np.ndarray) -> np.ndarray:
    return dequantize(*quantize_f64(v))


def quantize_weights(wg_bits, wu_bits, wd_bits) -> Dict[str, np.ndarray]:
    """Quantise the three bf16 weight matrices; W_gateup is [gate; up] stacked."""
    gu_bits = np.concatenate([wg_bits, wu_bits], axis=0)
    gu_codes, gu_scales = quantize_bf16(gu_bits)
    d_codes, d_scales = quantize_bf16(wd_bits)
    return {"gateup_codes": gu_codes, "gateup_scales": gu_scales,
            "down_codes": d_codes, "down_scales": d_scales}


def swiglu_mlp(x_bits: np.ndarray, qw: Dict[str, np.ndarray],
               rows_down: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Forward of the MXFP8 SwiGLU MLP for bf16 x [M, H] and quantised weights.

    ``rows_down`` restricts the down projection to those output features (for
    sampled checks at full size); y then has shape [M, len(rows_down)].
    Returns x^ (dequantised), g, u, h, h^ (dequantised), y (fp64) and
    y_bf16 (uint16 bits).
    """
    xc, xs = quantize_bf16(x_bits)
    return _mlp_from_quantised(xc, xs, qw, rows_down)


def _mlp_from_quantised(xc: np.ndarray, xs: np.ndarray, qw: Dict[str, np.ndarray],
                        rows_down: Optional[np.ndarray]) -> Dict[str, np.ndarray]:
    """The MLP from MXFP8 x^ (codes, row-major scales) on: steps 2-5."""
    I = qw["gateup_codes"].shape[0] // 2
    xd = dequantize(xc, xs)
    wgu = dequantize(qw["gateup_codes"], qw["gateup_scales"])
    g = xd @ wgu[:I].T
    u = xd @ wgu[I:].T
    del wgu
    h = silu(g) * u
    hc, hs = quantize_f64(h)
    hd = dequantize(hc, hs)
    dc, ds = qw["down_codes"], qw["down_scales"]
    if rows_down is not None:
        dc, ds = dc[rows_down], ds[rows_down]
    wd = dequantize(dc, ds)
    y = hd @ wd.T
    return {"x_codes": xc, "x_scales": xs, "xd": xd, "g": g, "u": u, "h": h,
            "h_codes": hc, "h_scales": hs, "hd": hd, "y": y,
            "y_bf16": round_bf16_bits(y)}


# ---------------------------------------------------------------- the decoder block
def rmsnorm(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of bf16 rows x [M, H] with bf16 gain gamma [H], in float64:
    x[m, k] / sqrt(mean_j x[m, j]^2 + eps) * gamma[k]."""
    x = bf16_bits_to_f64(x_bits)
    g = bf16_bits_to_f64(np.asarray(gamma_bits, np.uint16))
    mean_sq = np.mean(x * x, axis=1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * g[None, :]


def mlp_block(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float, qw: Dict[str, np.ndarray],
              residual: bool = True, rows_down: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """y = x + MLP(RMSNorm(x) * gamma) (``residual``) or the MLP alone.  The
    normalised rows are quantised from float64; ``rows_down`` restricts the
    output features as in ``swiglu_mlp``."""
    n = rmsnorm(x_bits, gamma_bits, eps)
    xc, xs = quantize_f64(n)
    res = _mlp_from_quantised(xc, xs, qw, rows_down)
    y = res["y"]
    if residual:
        x = bf16_bits_to_f64(x_bits)
        y = y + (x if rows_down is None else x[:, rows_down])
    res.update({"norm": n, "y": y, "y_bf16": round_bf16_bits(y)})
    return res


# ---------------------------------------------------------------- paged decode attention
def paged_decode_attention(q_bits: np.ndarray, k_codes: np.ndarray, k_scales: np.ndarray, v_codes: np.ndarray,
                           v_scales: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray,
                           sm_scale: float) -> Dict[str, np.ndarray]:
    """One decode step of attention over a paged MXFP8 KV cache, in float64.

    q_bits [B, Hq, D] bf16; k_codes / v_codes [num_pages, Hkv, P, D] E4M3;
    k_scales / v_scales [num_pages, Hkv, P, D / 32] UE8M0 (row-major per
    token); block_table [B, max_pages] page ids; seq_lens [B] (>= 1).  Token
    t of sequence b is slot t % P of page block_table[b, t // P].
    Returns out (float64 [B, Hq, D]) and out_bf16 (uint16 bits).
    """
    q = bf16_bits_to_f64(q_bits)
    B, Hq, D = q.shape
    _, Hkv, P, _ = k_codes.shape
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(seq_lens[b])
        pages = [int(block_table[b, i]) for i in range(-(-n // P))]
        for hk in range(Hkv):
            kc = np.concatenate([k_codes[p, hk] for p in pages])[:n]
            ks = np.concatenate([k_scales[p, hk] for p in pages])[:n]
            vc = np.concatenate([v_codes[p, hk] for p in pages])[:n]
            vs = np.concatenate([v_scales[p, hk] for p in pages])[:n]
            k = dequantize(kc, ks)
            v = dequantize(vc, vs)
            for g in range(G):
                h = hk * G + g
                s = sm_scale * (k @ q[b, h])
                w = np.exp(s - s.max())
                out[b, h] = (w / w.sum()) @ v
    return {"out": out, "out_bf16": round_bf16_bits(out)}


# ---------------------------------------------------------------- 128x128 block scales
def quantize_blockscale(bits: np.ndarray, block_rows: int, block_cols: int = 128):
    """bf16 bit patterns [rows, K] -> (E4M3 codes [rows, K], fp32 scales
    [ceil(rows / block_rows), K / block_cols]).  Each block's scale is
    fl32(amax / 448) (1 when the block is all zero); each element's code is
    the E4M3 round-to-nearest-even, saturated at 448, of fl32(v / scale)."""
    v = bf16_bits_to_f64(np.asarray(bits, np.uint16)).astype(np.float32)
    rows, K = v.shape
    assert K % block_cols == 0
    rb = -(-rows // block_rows)
    scales = np.ones((rb, K // block_cols), np.float32)
    codes = np.empty((rows, K), np.uint8)
    for i in range(rb):
        for j in range(K // block_cols):
            blk = v[i * block_rows:(i + 1) * block_rows, j * block_cols:(j + 1) * block_cols]
            amax = np.float32(np.abs(blk).max())
            if amax > 0:
                scales[i, j] = np.float32(amax / np.float32(448.0))
            t = (blk / scales[i, j]).astype(np.float32)
            mag = np.vectorize(e4m3_round_code, otypes=[np.uint8])(np.abs(t).astype(np.float64))
            # the sign bit is kept, also where the magnitude rounds to zero
            codes[i * block_rows:(i + 1) * block_rows, j * block_cols:(j + 1) * block_cols] = \
                mag | np.where(np.signbit(t), 0x80, 0).astype(np.uint8)
    return codes, scales


def dequantize_blockscale(codes: np.ndarray, scales: np.ndarray, block_rows: int, block_cols: int = 128) -> np.ndarray:
    """codes [rows, K] times their blocks' fp32 scales, in float64."""
    codes = np.asarray(codes, np.uint8)
    vals = e4m3_table()[codes & 0x7F] * np.where(codes & 0x80, -1.0, 1.0)
    s = np.repeat(np.repeat(scales.astype(np.float64), block_rows, axis=0), block_cols, axis=1)
    return vals * s[: codes.shape[0], : codes.shape[1]]


def gemm_blockscale(a_bits: np.ndarray, w_bits: np.ndarray) -> Dict[str, np.ndarray]:
    """C [M, N] = A^ W^^T with A [M, K] in 1x128 groups and W [N, K] in 128x128
    blocks (both bf16 in, quantised here)."""
    ac, as_ = quantize_blockscale(a_bits, 1)
    wc, ws = quantize_blockscale(w_bits, 128)
    c = dequantize_blockscale(ac, as_, 1) @ dequantize_blockscale(wc, ws, 128).T
    return {"a_codes": ac, "a_scales": as_, "w_codes": wc, "w_scales": ws, "c": c, "c_bf16": round_bf16_bits(c)}


def gemm(a_bits: np.ndarray, b_codes: np.ndarray, b_scales: np.ndarray,
         a_prequant: Optional[tuple] = None) -> Dict[str, np.ndarray]:
    """C [M, N] = A^ B^^T for bf16 A [M, K] (quantised here) and MXFP8 B [N, K]."""
    if a_prequant is None:
        ac, as_ = quantize_bf16(a_bits)
    else:
        ac, as_ = a_prequant
    c = dequantize(ac, as_) @ dequantize(b_codes, b_scales).T
    return {"a_codes": ac, "a_scales": as_, "c": c, "c_bf16": round_bf16_bits(c)}


def swiglu_quantize(gu: np.ndarray):
    """gu [M, 2I] (gate columns first) -> MXFP8 codes/scales of SiLU(g) * u."""
    I = gu.shape[1] // 2
    h = silu(gu[:, :I]) * gu[:, I:]
    return quantize_f64(h)


# ---------------------------------------------------------------- metrics
def rel_l2(a: np.ndarray, ref: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / den) if den > 0 else float(np.linalg.norm(a))


def max_abs_normalized(a: np.ndarray, ref: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(a - ref)) / den) if den > 0 else float(np.max(np.abs(a)))


def per_row_rel_l2(a: np.ndarray, ref: np.ndarray) -> np.ndarray:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.linalg.norm(a - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)
