"""Helpers shared by the GPU tests: host <-> device marshalling and metrics."""
import numpy as np


def to_dev_u16(bits: np.ndarray):
    """uint16 bf16 bit patterns -> torch.bfloat16 CUDA tensor with the same bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16)


def from_dev_bf16(t) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 bit patterns (numpy)."""
    import torch

    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_l2(a, ref) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs_norm(a, ref) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-300))


def per_row_rel_l2(a, ref) -> np.ndarray:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.linalg.norm(a - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-300)


# The output gate of the MLP: rel-L2 <= 2e-3 and max-abs-normalised <= 1e-2
# against the oracle's bf16-rounded y.
REL_L2_TOL = 2e-3
MAX_ABS_TOL = 1e-2
# Per-row rel-L2 bound.  The kernel computes h = SiLU(g) * u in fp32 and the
# oracle in fp64; where the two straddle an E4M3 rounding boundary (about
# 3e-5 of the elements) one intermediate code differs by one step (1/16..1/8
# of |h_k|), which moves that token's row by up to ~|dh_k| / ||h|| -- a few
# 1e-3 for a large h_k.  Whole-output rel-L2 stays far below 2e-3; a single
# row may not, so rows get the max-abs bound.
PER_ROW_TOL = 1e-2


def assert_repeat_close(a_bits: np.ndarray, b_bits: np.ndarray, max_diff_frac: float = 1e-3) -> None:
    """Two runs of a kernel whose split-K partial sums are added in arrival
    order: every element agrees to one bf16 step (fp32 reassociation can move
    a value across one rounding boundary, no further), and few elements differ
    at all.  A race that loses or doubles a partial sum moves an element by a
    whole partial sum, far more than one step."""
    a = bf16_bits_to_f64(a_bits)
    b = bf16_bits_to_f64(b_bits)
    mag = np.maximum(np.abs(a), np.abs(b))
    _, e = np.frexp(np.where(mag > 0, mag, 1.0))
    step = np.ldexp(1.0, e - 8)  # spacing of bf16 values (8 significant bits) at that magnitude
    # an element near zero is a sum whose partials nearly cancel; fp32
    # reassociation error there is relative to the partials, so it gets an
    # absolute floor of 2^-16 of the output's largest magnitude
    floor = np.ldexp(float(np.max(mag)), -16) if mag.size else 0.0
    bad = np.abs(a - b) > np.maximum(step, floor)
    assert not np.any(bad), (np.argwhere(bad)[:5], a[bad][:5], b[bad][:5])
    assert np.mean(a != b) <= max_diff_frac, np.mean(a != b)


def control_words_clear(ctl_u8) -> bool:
    """Whether a workspace's control region (a uint8 device tensor) is back at
    zero between launches.  Bytes 8-15 are left out: they hold the 64-bit
    count of grid-wide kernel blocks that have left, over all launches."""
    c = ctl_u8.clone()
    c[8:16] = 0
    return int(c.count_nonzero()) == 0
