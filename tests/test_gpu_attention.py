"""Paged decode attention over an MXFP8 KV cache (fsops_mxfp8_paged_decode_attention)
against the oracle's paged_decode_attention, on seeded paged caches."""
import math

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


class Cache:
    """A workload's paged cache on the device, quantised by the library."""

    def __init__(self, fs, wl, mutate=None):
        import torch

        self.wl = wl
        self.d = inputs.make_attention(wl)
        if mutate is not None:
            mutate(self.d)
        npages = self.d["k"].shape[0]
        self.npages = npages
        rows = npages * wl.Hkv * wl.P
        self.dev = {}
        for name in ("k", "v"):
            x = to_dev_u16(self.d[name].reshape(rows, wl.D))
            codes = torch.empty(rows, wl.D, dtype=torch.uint8, device="cuda")
            scales = torch.empty(rows * wl.D // 32, dtype=torch.uint8, device="cuda")
            fs.fsops_quantize_mxfp8(x, rows, wl.D, wl.D, codes, scales, fs.SCALES_ROWMAJOR)
            self.dev[name] = (codes, scales)
        self.q = to_dev_u16(self.d["q"])
        self.table = torch.from_numpy(self.d["block_table"]).cuda()
        self.lens = torch.from_numpy(self.d["seq_lens"]).cuda()
        self.max_pages = self.d["block_table"].shape[1]
        self.ws_n = fs.fsops_paged_attention_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, wl.P, self.max_pages)
        assert self.ws_n > 0
        self.ws = torch.zeros(self.ws_n + 256, dtype=torch.uint8, device="cuda")
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr = self.ws.data_ptr() + off
        torch.cuda.synchronize()

    def run(self, fs, out=None, stream=None, sm_scale=None):
        import torch

        wl = self.wl
        if out is None:
            out = torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.bfloat16, device="cuda")
        sm = 1.0 / math.sqrt(wl.D) if sm_scale is None else sm_scale
        (kc, ks), (vc, vs) = self.dev["k"], self.dev["v"]
        fs.fsops_mxfp8_paged_decode_attention(self.q, kc, ks, vc, vs, self.npages, self.table, self.max_pages,
                                              self.lens, out, wl.B, wl.Hq, wl.Hkv, wl.D, wl.P, sm, self.ws_ptr,
                                              self.ws_n, stream)
        return out

    def oracle(self, seqs=None, sm_scale=None):
        wl, d = self.wl, self.d
        rows = self.npages * wl.Hkv * wl.P
        kc, ks = oracle.quantize_bf16(d["k"].reshape(rows, wl.D))
        vc, vs = oracle.quantize_bf16(d["v"].reshape(rows, wl.D))
        shp, sshp = (self.npages, wl.Hkv, wl.P, wl.D), (self.npages, wl.Hkv, wl.P, wl.D // 32)
        sel = np.arange(wl.B) if seqs is None else np.asarray(seqs)
        sm = 1.0 / math.sqrt(wl.D) if sm_scale is None else sm_scale
        return oracle.paged_decode_attention(d["q"][sel], kc.reshape(shp), ks.reshape(sshp), vc.reshape(shp),
                                             vs.reshape(sshp), d["block_table"][sel], d["seq_lens"][sel], sm)


def _check(got_bits, ref):
    got = bf16_bits_to_f64(got_bits).reshape(ref["out"].shape)
    want = bf16_bits_to_f64(ref["out_bf16"])
    assert rel_l2(got, want) <= REL_L2_TOL, rel_l2(got, want)
    assert max_abs_norm(got, want) <= MAX_ABS_TOL, max_abs_norm(got, want)
    # fp32 against fp64 softmax: almost every bf16 output is the same
    assert np.mean(got == want) > 0.99


# (B, Hq, Hkv, P, len_lo, len_hi, seed): group sizes 4, 1, 8, 2; page sizes
# 16..128; lengths from 1 token to several 128-token chunks
SHAPES = [(3, 8, 2, 16, 1, 300, 1), (4, 4, 4, 32, 100, 700, 2), (2, 16, 2, 64, 128, 128, 3),
          (3, 8, 4, 128, 200, 1000, 4), (5, 32, 8, 16, 1, 40, 5)]


@pytest.mark.parametrize("B,Hq,Hkv,P,lo,hi,seed", SHAPES)
def test_attention_matches_oracle(fs, B, Hq, Hkv, P, lo, hi, seed):
    import torch

    wl = inputs.AttnWorkload("t", B, Hq, Hkv, 128, P, lo, hi, seed)
    c = Cache(fs, wl)
    out = c.run(fs)
    torch.cuda.synchronize()
    assert fs.fsops_read_kernel_status(c.ws_ptr) == 0
    _check(from_dev_bf16(out), c.oracle())


@pytest.mark.parametrize("chunks", [1, 3, 64])
def test_attention_chunks_per_block(fs, knob, chunks):
    """Blocks of 1, 3 and up to 64 chunks (splits past a short sequence's end
    run no chunk and leave an empty partial result), on a mix of lengths."""
    import torch

    knob("ATTN_CHUNKS", chunks)  # before the workspace is sized
    wl = inputs.AttnWorkload("t", 4, 8, 2, 128, 16, 90, 2100, 7)
    c = Cache(fs, wl)
    out = c.run(fs)
    torch.cuda.synchronize()
    assert fs.fsops_read_kernel_status(c.ws_ptr) == 0
    _check(from_dev_bf16(out), c.oracle())


def _pow2(bits, k):
    """bf16 bit patterns times 2^k (exact while the result stays normal)."""
    return inputs.bf16_bits_from_f32(bf16_bits_to_f64(bits).astype(np.float32) * np.float32(2.0 ** k))


def _spread_v(d):
    """Every third token's V 2^-20 times smaller (its block scales 2^20 below
    its neighbours'), and a few all-zero 32-element V blocks (scale byte 0)."""
    v = d["v"]
    v[:, :, 1::3, :] = _pow2(v[:, :, 1::3, :], -20)
    v[::2, 0, 5, 32:64] = 0
    v[1::3, -1, 12, 96:128] = 0


def _q_range(d):
    """Query heads far from unit size: one 2^40 times larger (a one-hot
    softmax), one 2^-40 times smaller (uniform weights), one with a single
    large element."""
    q = d["q"]
    q[:, 0, :] = _pow2(q[:, 0, :], 40)
    q[:, 1, :] = _pow2(q[:, 1, :], -40)
    q[:, 2, 7] = _pow2(q[:, 2, 7], 20)


def _k_spread(d):
    """Every fifth token's K 2^-12 times smaller, every seventh 2^6 larger."""
    k = d["k"]
    k[:, :, 0::5, :] = _pow2(k[:, :, 0::5, :], -12)
    k[:, :, 3::7, :] = _pow2(k[:, :, 3::7, :], 6)


@pytest.mark.parametrize("mutate", [_spread_v, _q_range, _k_spread], ids=["v_spread", "q_range", "k_spread"])
def test_attention_scale_ranges(fs, mutate):
    """Scales far apart within one tensor-core step: V block scales 2^15 and
    more apart among 16 neighbouring tokens (and zero blocks), which the
    kernel adds with fp32 FMAs; query heads of very different size (the
    power-of-two prescale of q); K scales spread over 2^18."""
    import torch

    wl = inputs.AttnWorkload("t", 3, 8, 2, 128, 16, 100, 700, 11)
    c = Cache(fs, wl, mutate)
    out = c.run(fs)
    torch.cuda.synchronize()
    assert fs.fsops_read_kernel_status(c.ws_ptr) == 0
    _check(from_dev_bf16(out), c.oracle())


def test_attention_long_sequences_split(fs):
    """Sequences long enough to be split over several blocks (partial results
    merged by the second launch), and a zero softmax scale (uniform weights)."""
    import torch

    wl = inputs.AttnWorkload("t", 2, 8, 2, 128, 16, 5000, 9000, 6)
    c = Cache(fs, wl)
    out = c.run(fs)
    torch.cuda.synchronize()
    _check(from_dev_bf16(out), c.oracle())
    out0 = c.run(fs, sm_scale=0.0)
    torch.cuda.synchronize()
    _check(from_dev_bf16(out0), c.oracle(sm_scale=0.0))


def test_attention_full_workload_sampled(fs):
    """The a64 workload (Qwen3-4B attention geometry, 64 sequences of 2k-6k
    tokens): 8 sampled sequences checked against the oracle."""
    import torch

    wl = inputs.ATTN_WORKLOADS["a64"]
    c = Cache(fs, wl)
    out = c.run(fs)
    torch.cuda.synchronize()
    assert fs.fsops_read_kernel_status(c.ws_ptr) == 0
    seqs = np.sort(np.random.default_rng(2).choice(wl.B, 8, replace=False))
    got = from_dev_bf16(out)[seqs]
    _check(got, c.oracle(seqs))


def test_attention_graph_replay(fs):
    import torch

    wl = inputs.AttnWorkload("t", 4, 8, 2, 128, 16, 50, 900, 7)
    c = Cache(fs, wl)
    ref = from_dev_bf16(c.run(fs))
    out = torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            c.run(fs, out=out, stream=s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(from_dev_bf16(out), ref)


def test_attention_bad_page_id_is_reported(fs):
    """A block-table entry outside [0, num_pages) is caught by the kernel's own
    bounds check: reported in the status word, never read."""
    import torch

    wl = inputs.AttnWorkload("t", 2, 8, 2, 128, 16, 40, 60, 8)
    c = Cache(fs, wl)
    bad = c.d["block_table"].copy()
    bad[1, 0] = c.npages + 5
    c.table = torch.from_numpy(bad).cuda()
    c.run(fs)
    torch.cuda.synchronize()
    word = fs.fsops_read_kernel_status(c.ws_ptr)
    assert word >> 24 == fs.ERR_INVALID_ARG, hex(word)
    assert fs.fsops_read_kernel_status(c.ws_ptr) == 0  # read and cleared
    # sequence 0 (all of its pages valid) is still right
    got = from_dev_bf16(c.run(fs))
    torch.cuda.synchronize()
    fs.fsops_read_kernel_status(c.ws_ptr)
    _check(got[:1], c.oracle([0]))
