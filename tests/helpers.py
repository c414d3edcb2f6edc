"""Shared test helpers: oracle inputs from torch tensors, parity metrics and
running the CUDA path through the C ABI."""

import numpy as np
import torch

# Tolerances for bf16-input / fp32-accumulate outputs and gradients, and for
# d(topk weights): the parity bar of the layer, derived from its bf16 arithmetic.
REL_FROB = 5e-3
MAX_ABS_RMS = 3e-2
DW_REL = 1e-2


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_frob(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / n) if n > 0 else float(np.linalg.norm(got))


def assert_close(name, got, ref, rel=REL_FROB, max_abs_rms=MAX_ABS_RMS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite values" % name
    rf = rel_frob(got, ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    mx = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert rf <= rel, "%s: relative Frobenius error %.3e > %.1e" % (name, rf, rel)
    assert mx <= max_abs_rms * rms + 1e-30, "%s: max abs error %.3e > %.1e * rms %.3e" % (
        name, mx, max_abs_rms, rms)
    return rf, mx / rms if rms > 0 else 0.0


def bf16_step(v):
    """Spacing of the bf16 values at |v| (2^(e-7) for |v| in [2^e, 2^(e+1)))."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7)


def assert_close_bf16_output(name, got, ref):
    """For a bf16 output whose largest elements are many times its rms: the
    relative Frobenius bound, and max abs error <= 3e-2 rms plus one bf16
    step of the reference element.  Where |ref| reaches 8-12x rms, one step
    of the output format is 0.03-0.09 rms by itself, and an exact value near a
    rounding midpoint lands on either neighbour after any fp32 evaluation."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rf = rel_frob(got, ref)
    assert rf <= REL_FROB, "%s: relative Frobenius error %.3e > %.1e" % (name, rf, REL_FROB)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = np.abs(got - ref) - (MAX_ABS_RMS * rms + bf16_step(ref))
    assert np.all(excess <= 0), "%s: error beyond 3e-2 rms + one bf16 step by %.3e rms" % (
        name, float(excess.max()) / rms)


def assert_dw_close(got, ref):
    rf = rel_frob(got, ref)
    assert rf <= DW_REL, "d_topk_w relative error %.3e > %.1e" % (rf, DW_REL)
    return rf


def oracle_inputs(case):
    return (f64(case.x), case.topk_idx.cpu().numpy().astype(np.int64), f64(case.topk_w),
            f64(case.w_gate_up), f64(case.w_down), f64(case.dy) if case.dy is not None else None)


def to_device(case, device="cuda"):
    import copy
    c = copy.copy(case)
    for f in ("x", "topk_idx", "topk_w", "w_gate_up", "w_down", "dy"):
        v = getattr(case, f)
        if v is not None:
            setattr(c, f, v.to(device).contiguous())
    return c
