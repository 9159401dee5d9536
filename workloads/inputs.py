"""Seeded synthetic inputs for the decode-shape MXFP8 SwiGLU MLP.

This module draws random bf16 tensors and nothing else: it holds none of the
MXFP8 arithmetic, so the oracle and the CUDA path can both be fed from it
without sharing any of the method's code.

Workloads (shapes follow the decode problem of the Fish Audio post, p1
"The GPU problem you're paying for": M <= 128 tokens per step; the sizes
themselves are synthetic stand-ins, there is no dataset or checkpoint):

========  ====  =====  =====  ======  ==============================================
name      M     H      I      layers  structure
========  ====  =====  =====  ======  ==============================================
m1        1     1024   2816   1       x ~ N(0,1); W ~ N(0, 1/sqrt(K)) + 0.1% x20
m16       16    2560   9728   1       same
m64       64    4096   12288  32      same, one x for every layer
m128      128   4096   12288  32      x[m,:] = s_m * z, log10 s_m ~ U(-2, 2)
sweep     1..128 5120  17408  16      W as m1 plus 1% of 32-blocks zeroed
========  ====  =====  =====  ======  ==============================================

Recipe (all draws in float32, then rounded to bf16 with round-to-nearest-even):

* The config's base seed s gives ``SeedSequence(s).spawn(1 + layers)``; child 0
  draws x, child 1 + l draws the weights of layer l, in the order W_gate
  [I, H], W_up [I, H], W_down [H, I].
* A weight matrix [rows, K] is ``standard_normal / sqrt(K)`` (sigma = 1/sqrt(K)),
  then exactly ``round(0.001 * rows * K)`` entries, drawn without replacement,
  are multiplied by 20 (outliers).
* ``zero_block_frac`` > 0 then zeroes that fraction of the 32-element blocks
  along K (drawn without replacement).
* x is [M, H] standard normal; for ``token_scale_log10`` = (a, b) each row m is
  multiplied by 10**u_m with u_m ~ U(a, b).
* The RMSNorm gain of the decoder block (``make_norm_gain``) is [H],
  1 + 0.1 * standard normal, from ``SeedSequence(s).spawn(1 + layers + 1)``'s
  last child (the streams above are unchanged); its eps is ``NORM_EPS``.

``backend="torch-cuda"`` draws the same distributions with a seeded
``torch.Generator`` on the GPU (a different random stream); it exists only so
that the benchmark can build the 32-layer workloads (5 GB of weights) in
seconds. Every oracle comparison uses the numpy backend.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np

__all__ = ["Workload", "WORKLOADS", "bf16_bits_from_f32", "bf16_bits_to_f32",
           "make_activations", "make_layer", "make_workload_small", "make_norm_gain", "NORM_EPS",
           "AttnWorkload", "ATTN_WORKLOADS", "make_attention"]

# eps of the decoder block's RMSNorm (the value Qwen3-family configs use)
NORM_EPS = 1e-6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    I: int
    layers: int
    seed: int
    outlier_frac: float = 0.001
    outlier_mult: float = 20.0
    zero_block_frac: float = 0.0
    token_scale_log10: Optional[Tuple[float, float]] = None
    M_sweep: Tuple[int, ...] = ()

    def with_M(self, M: int) -> "Workload":
        return dataclasses.replace(self, M=M)

    @property
    def weight_bytes(self) -> int:
        """E4M3 codes plus UE8M0 scales of the three weight matrices."""
        return 3 * self.H * self.I + 3 * self.H * self.I // 32


WORKLOADS: Dict[str, Workload] = {
    "m1": Workload("m1", 1, 1024, 2816, 1, 0),
    "m16": Workload("m16", 16, 2560, 9728, 1, 1),
    "m64": Workload("m64", 64, 4096, 12288, 32, 2),
    "m128": Workload("m128", 128, 4096, 12288, 32, 34, token_scale_log10=(-2.0, 2.0)),
    "sweep": Workload("sweep", 128, 5120, 17408, 16, 35, zero_block_frac=0.01,
                      M_sweep=(1, 2, 4, 8, 16, 32, 64, 128)),
}


def make_workload_small(name: str, M: int, H: int, I: int, seed: int, **kw) -> Workload:
    """A workload with the same recipe at a size the oracle finishes in seconds."""
    return Workload(name, M, H, I, 1, seed, **kw)


# ---------------------------------------------------------------- bf16 helpers
def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns, round-to-nearest-even.

    Inputs here are finite; the conversion is done by torch (a library routine).
    """
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exactly equal float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- numpy draws
def _children(wl: Workload) -> List[np.random.SeedSequence]:
    return np.random.SeedSequence(wl.seed).spawn(1 + wl.layers)


def _weight_numpy(rng: np.random.Generator, rows: int, K: int, wl: Workload) -> np.ndarray:
    w = rng.standard_normal((rows, K), dtype=np.float32)
    w *= np.float32(1.0 / math.sqrt(K))
    n = rows * K
    n_out = int(round(wl.outlier_frac * n))
    if n_out:
        pos = rng.choice(n, size=n_out, replace=False)
        w.reshape(-1)[pos] *= np.float32(wl.outlier_mult)
    if wl.zero_block_frac > 0:
        nb = n // 32
        nz = int(round(wl.zero_block_frac * nb))
        blocks = rng.choice(nb, size=nz, replace=False)
        w.reshape(nb, 32)[blocks, :] = 0.0
    return bf16_bits_from_f32(w)


def make_layer(wl: Workload, layer: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) as uint16 bf16 bits."""
    rng = np.random.Generator(np.random.PCG64(_children(wl)[1 + layer]))
    wg = _weight_numpy(rng, wl.I, wl.H, wl)
    wu = _weight_numpy(rng, wl.I, wl.H, wl)
    wd = _weight_numpy(rng, wl.H, wl.I, wl)
    return wg, wu, wd


def make_activations(wl: Workload, M: Optional[int] = None) -> np.ndarray:
    """x [M, H] as uint16 bf16 bits."""
    M = wl.M if M is None else M
    rng = np.random.Generator(np.random.PCG64(_children(wl)[0]))
    x = rng.standard_normal((M, wl.H), dtype=np.float32)
    if wl.token_scale_log10 is not None:
        lo, hi = wl.token_scale_log10
        u = rng.uniform(lo, hi, size=(M, 1))
        x = (x * np.power(10.0, u)).astype(np.float32)
    return bf16_bits_from_f32(x)


def make_norm_gain(wl: Workload) -> np.ndarray:
    """RMSNorm gain gamma [H] as uint16 bf16 bits: 1 + 0.1 * N(0, 1)."""
    ss = np.random.SeedSequence(wl.seed).spawn(1 + wl.layers + 1)[-1]
    rng = np.random.Generator(np.random.PCG64(ss))
    g = 1.0 + 0.1 * rng.standard_normal(wl.H, dtype=np.float32)
    return bf16_bits_from_f32(g.astype(np.float32))


# ---------------------------------------------------------------- torch draws
def make_layer_torch(wl: Workload, layer: int, device) -> tuple:
    """Same recipe drawn with a seeded torch.Generator on ``device`` (bf16 tensors).

    Used for the multi-layer benchmark workloads only.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 1000003 + 7919 * (layer + 1))

    def draw(rows, K):
        w = torch.randn(rows, K, generator=g, device=device, dtype=torch.float32)
        w *= 1.0 / math.sqrt(K)
        n = rows * K
        n_out = int(round(wl.outlier_frac * n))
        if n_out:
            pos = torch.randperm(n, generator=g, device=device)[:n_out]
            w.view(-1)[pos] *= wl.outlier_mult
        if wl.zero_block_frac > 0:
            nb = n // 32
            nz = int(round(wl.zero_block_frac * nb))
            blocks = torch.randperm(nb, generator=g, device=device)[:nz]
            w.view(nb, 32)[blocks] = 0.0
        return w.to(torch.bfloat16)

    return draw(wl.I, wl.H), draw(wl.I, wl.H), draw(wl.H, wl.I)


def make_activations_torch(wl: Workload, M: int, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 1000003 + 1)
    x = torch.randn(M, wl.H, generator=g, device=device, dtype=torch.float32)
    if wl.token_scale_log10 is not None:
        lo, hi = wl.token_scale_log10
        u = torch.rand(M, 1, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo
        x = x * torch.pow(10.0, u)
    return x.to(torch.bfloat16)


# ---------------------------------------------------------------- paged decode attention
@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """One decode step over a paged KV cache: B sequences of lengths drawn
    uniformly in [len_lo, len_hi], Hq query heads sharing Hkv KV heads (GQA),
    head dimension D, pages of P tokens."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    len_lo: int
    len_hi: int
    seed: int


# a64: Qwen3-4B's attention geometry (32 query heads, 8 KV heads, D = 128)
# at 64 sequences of 2k-6k tokens, pages of 16 tokens
ATTN_WORKLOADS: Dict[str, AttnWorkload] = {
    "a64": AttnWorkload("a64", 64, 32, 8, 128, 16, 2048, 6144, 90),
}


def make_attention(wl: AttnWorkload) -> dict:
    """q [B, Hq, D], the cache's K and V [num_pages, Hkv, P, D] (bf16 bits,
    standard normal, every slot drawn, also past a sequence's end), seq_lens
    [B] and block_table [B, max_pages] (int32; each sequence's pages are a
    random set of the physical pages; unused entries are -1)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(wl.seed)))
    lens = rng.integers(wl.len_lo, wl.len_hi + 1, size=wl.B).astype(np.int32)
    npg = [(int(n) + wl.P - 1) // wl.P for n in lens]
    total = int(sum(npg))
    perm = rng.permutation(total).astype(np.int32)
    table = np.full((wl.B, max(npg)), -1, np.int32)
    o = 0
    for b, n in enumerate(npg):
        table[b, :n] = perm[o:o + n]
        o += n
    q = rng.standard_normal((wl.B, wl.Hq, wl.D), dtype=np.float32)
    k = rng.standard_normal((total, wl.Hkv, wl.P, wl.D), dtype=np.float32)
    v = rng.standard_normal((total, wl.Hkv, wl.P, wl.D), dtype=np.float32)
    return {"q": bf16_bits_from_f32(q), "k": bf16_bits_from_f32(k), "v": bf16_bits_from_f32(v),
            "seq_lens": lens, "block_table": table}
