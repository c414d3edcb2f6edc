"""GPU parity on seeded random shapes (the second test adds a random gate_up
layout and a random choice of biases): H and I any multiple of 8 from 8 up
(below one 64-element k-block, below one 128-feature tile, ragged against
both), 1 to 40 experts, k up to 8, 1 to 700 tokens, both activations, both
storage dtypes and all four routing kinds.  Every output against the fp64
oracle: y and dx (bf16 outputs: relative Frobenius and max abs <= 3e-2 rms
plus one bf16 step of the reference element), d(topk w), and every expert's
gate, up and down weight gradients, with exact zeros for experts without a
token; the backward that recomputes the saved context must match the one
that reads it bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import ACT_CLAMPED_GLU, ACT_SWIGLU, Recipe
from tests.helpers import (assert_close, assert_close_bf16_output, assert_dw_close,
                           oracle_inputs, to_device)

pytestmark = pytest.mark.gpu

ROUTINGS = ("softmax_topk_renorm", "uniform_topk_softmax", "zipf", "uniform_ids")


def _cases(n=40, seed=2024):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        H = int(8 * g.integers(1, 70))
        I = int(8 * g.integers(1, 50))
        E = int(g.integers(1, 41))
        k = int(g.integers(1, min(E, 8) + 1))
        T = int(g.integers(1, 701))
        act = ACT_SWIGLU if g.random() < 0.5 else ACT_CLAMPED_GLU
        dtype = "fp32" if g.random() < 0.2 else "bf16"
        routing = ROUTINGS[int(g.integers(0, len(ROUTINGS)))]
        if routing == "zipf" and E < 4:
            routing = "softmax_topk_renorm"
        out.append((i, T, H, I, E, k, act, dtype, routing))
    return out


@pytest.mark.parametrize("i,T,H,I,E,k,act,dtype,routing", _cases())
def test_random_shape_parity(i, T, H, I, E, k, act, dtype, routing):
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("rand", T=T, H=H, I=I, E=E, k=k, act=act, dtype=dtype, weight_std="fan_in",
               routing=routing, seed=7000 + i)
    case = synth.make_case(r)
    d = to_device(case)
    run = LayerRunner(T, H, I, E, k, act, MOE_FP32 if dtype == "fp32" else MOE_BF16, r.limit,
                      r.alpha)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down).clone()
    dx, dtw, dwgu, dwd = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w,
                                                          d.w_gate_up, d.w_down)]
    # the backward without the saved context recomputes it: bit for bit the same
    again = run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, recompute=True)
    torch.cuda.synchronize()
    run.check()
    for a, b in zip((dx, dtw, dwgu, dwd), again):
        assert torch.equal(a, b)
    x, idx, w, wgu, wd, dy = oracle_inputs(case)
    y_ref = oracle.moe_forward(x, idx, w, wgu, wd, act)
    dx_ref, dw_ref, dgu_ref, dd_ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    if dtype == "bf16":
        assert_close_bf16_output("y", y.double().cpu().numpy(), y_ref)
        assert_close_bf16_output("dx", dx.double().cpu().numpy(), dx_ref)
    else:
        assert_close("y", y.double().cpu().numpy(), y_ref)
        assert_close("dx", dx.double().cpu().numpy(), dx_ref)
    assert_dw_close(dtw.cpu().numpy(), dw_ref)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    for e in range(E):
        if counts[e] == 0:
            assert torch.all(dwgu[e] == 0) and torch.all(dwd[e] == 0), e
            continue
        got = dwgu[e].double().cpu().numpy()
        assert_close("d_gate[%d]" % e, got[:, :I], dgu_ref[e][:, :I])
        assert_close("d_up[%d]" % e, got[:, I:], dgu_ref[e][:, I:])
        assert_close("d_down[%d]" % e, dwd[e].double().cpu().numpy(), dd_ref[e])


def _layout_bias_cases(n=24, seed=2025):
    """The first n random shapes again, each with a random gate_up layout and
    a random choice of biases (none, gate_up, down, both)."""
    g = np.random.default_rng(seed)
    return [c + (int(g.integers(0, 2)), ("none", "gate_up", "down", "both")[int(g.integers(0, 4))])
            for c in _cases()[:n]]


@pytest.mark.parametrize("i,T,H,I,E,k,act,dtype,routing,layout,biases", _layout_bias_cases())
def test_random_shape_layout_and_bias_parity(i, T, H, I, E, k, act, dtype, routing, layout,
                                             biases):
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    from tests.helpers import f64
    r = Recipe("rand", T=T, H=H, I=I, E=E, k=k, act=act, dtype=dtype, weight_std="fan_in",
               routing=routing, seed=7000 + i)
    case = synth.make_case(r)
    use_gu, use_d = biases in ("both", "gate_up"), biases in ("both", "down")
    bgu_t, bd_t = synth.make_biases(r) if biases != "none" else (None, None)
    x, idx, w, wgu_l, wd, dy = oracle_inputs(case)
    wgu = oracle.gate_up_concatenated(wgu_l, layout)
    bgu = oracle.gate_up_concatenated(f64(bgu_t), layout) if use_gu else None
    bd = f64(bd_t) if use_d else None
    d = to_device(case)
    bkw = dict(b_gate_up=bgu_t.cuda() if use_gu else None, b_down=bd_t.cuda() if use_d else None)
    run = LayerRunner(T, H, I, E, k, act, MOE_FP32 if dtype == "fp32" else MOE_BF16, r.limit,
                      r.alpha, gate_up_layout=layout)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, **bkw).clone()
    grads = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                             d.w_down, **bkw)]
    torch.cuda.synchronize()
    run.check()
    okw = dict(b_gate_up=bgu, b_down=bd)
    y_ref = oracle.moe_forward(x, idx, w, wgu, wd, act, **okw)
    ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, act, **okw)
    check = assert_close_bf16_output if dtype == "bf16" else assert_close
    check("y", y.double().cpu().numpy(), y_ref)
    check("dx", grads[0].double().cpu().numpy(), ref[0])
    assert_dw_close(grads[1].cpu().numpy(), ref[1])
    counts = np.bincount(idx.reshape(-1), minlength=E)
    for e in range(E):
        got = oracle.gate_up_concatenated(grads[2][e].double().cpu().numpy(), layout)
        if counts[e] == 0:
            assert not got.any() and torch.all(grads[3][e] == 0), e
        else:
            assert_close("d_gate[%d]" % e, got[:, :I], ref[2][e][:, :I])
            assert_close("d_up[%d]" % e, got[:, I:], ref[2][e][:, I:])
            assert_close("d_down[%d]" % e, grads[3][e].double().cpu().numpy(), ref[3][e])
    if biases != "none":
        dbgu = oracle.gate_up_concatenated(grads[4].double().cpu().numpy(), layout)
        assert_close("db_gate_up", dbgu, ref[4])
        assert_close("db_down", grads[5].double().cpu().numpy(), ref[5])
