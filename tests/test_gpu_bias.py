"""GPU parity of the optional per-expert biases (h = x Wgu[e] + b_gate_up[e],
o = act(h) Wd[e] + b_down[e]) against the fp64 oracle: the forward, every
gradient including db_gate_up / db_down and the bias term of d(topk
weights), in both gate_up layouts and both dtypes, with one bias or both,
and with empty experts.  The backward without a saved context must give
bit-identical results, and an inference forward (no saved context) the same
y as the training one."""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import ACT_CLAMPED_GLU, ACT_SWIGLU, Recipe
from tests.helpers import assert_close, assert_dw_close, f64, oracle_inputs, to_device

pytestmark = pytest.mark.gpu

BIAS_CASES = [
    # T, H, I, E, k, act, dtype, std, layout, biases, routing
    (512, 384, 320, 8, 4, ACT_SWIGLU, "bf16", None, 0, "both", "softmax_topk_renorm"),
    (600, 256, 200, 6, 4, ACT_CLAMPED_GLU, "bf16", 0.2, 1, "both", "softmax_topk_renorm"),
    (300, 136, 200, 6, 2, ACT_SWIGLU, "bf16", None, 0, "down", "uniform_ids"),
    (300, 136, 264, 5, 3, ACT_CLAMPED_GLU, "bf16", 0.2, 0, "gate_up", "uniform_topk_softmax"),
    (64, 128, 128, 8, 2, ACT_SWIGLU, "fp32", None, 0, "both", "softmax_topk_renorm"),
    (200, 128, 136, 5, 3, ACT_CLAMPED_GLU, "fp32", 0.2, 1, "both", "uniform_ids"),
    (700, 256, 256, 40, 8, ACT_SWIGLU, "bf16", None, 0, "both", "zipf"),   # empty experts
]


def _halves(a, layout):
    """(gate, up) column sets of a [..., 2I] array in the given layout."""
    if layout == 1:
        return a[..., 0::2], a[..., 1::2]
    I = a.shape[-1] // 2
    return a[..., :I], a[..., I:]


@pytest.mark.parametrize("T,H,I,E,k,act,dtype,std,layout,biases,routing", BIAS_CASES)
def test_bias_parity(T, H, I, E, k, act, dtype, std, layout, biases, routing):
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("bias", T=T, H=H, I=I, E=E, k=k, act=act, dtype=dtype,
               weight_std=std if std is not None else "fan_in", routing=routing, seed=500 + T)
    case = synth.make_case(r)
    bgu_t, bd_t = synth.make_biases(r)
    use_gu, use_d = biases in ("both", "gate_up"), biases in ("both", "down")
    x, idx, w, wgu_l, wd, dy = oracle_inputs(case)
    wgu = oracle.gate_up_concatenated(wgu_l, layout)
    bgu = oracle.gate_up_concatenated(f64(bgu_t), layout) if use_gu else None
    bd = f64(bd_t) if use_d else None

    d = to_device(case)
    bgu_d = bgu_t.cuda() if use_gu else None
    bd_d = bd_t.cuda() if use_d else None
    mdt = MOE_FP32 if dtype == "fp32" else MOE_BF16
    run = LayerRunner(T, H, I, E, k, act, mdt, r.limit, r.alpha, gate_up_layout=layout)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down,
                    b_gate_up=bgu_d, b_down=bd_d).clone()
    grads = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                             d.w_down, b_gate_up=bgu_d, b_down=bd_d)]
    again = run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, recompute=True,
                         b_gate_up=bgu_d, b_down=bd_d)
    inf = LayerRunner(T, H, I, E, k, act, mdt, r.limit, r.alpha, gate_up_layout=layout,
                      training=False, backward=False)
    y_inf = inf.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, use_plan=False,
                        b_gate_up=bgu_d, b_down=bd_d)
    torch.cuda.synchronize()
    run.check()
    inf.check()

    assert_close("y", y.float().cpu().numpy(),
                 oracle.moe_forward(x, idx, w, wgu, wd, act, b_gate_up=bgu, b_down=bd))
    assert torch.equal(y, y_inf)
    dx_ref, dw_ref, dwgu_ref, dwd_ref, dbgu_ref, dbd_ref = oracle.moe_backward(
        dy, x, idx, w, wgu, wd, act, b_gate_up=bgu, b_down=bd)
    dx, dtw, dwgu, dwd, dbgu, dbd = grads
    assert_close("dx", dx.float().cpu().numpy(), dx_ref)
    assert_dw_close(dtw.cpu().numpy(), dw_ref)
    gate, up = _halves(dwgu.cpu().numpy(), layout)
    gate_ref, up_ref = _halves(oracle.gate_up_in_layout(dwgu_ref, layout), layout)
    assert_close("d_gate", gate, gate_ref)
    assert_close("d_up", up, up_ref)
    assert_close("d_down", dwd.cpu().numpy(), dwd_ref)
    bgate, bup = _halves(dbgu.cpu().numpy(), layout)
    bgate_ref, bup_ref = _halves(oracle.gate_up_in_layout(dbgu_ref, layout), layout)
    assert_close("db_gate", bgate, bgate_ref)
    assert_close("db_up", bup, bup_ref)
    assert_close("db_down", dbd.cpu().numpy(), dbd_ref)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    for e in np.nonzero(counts == 0)[0]:
        assert torch.all(dbgu[e] == 0) and torch.all(dbd[e] == 0)
    names = ("dx", "d_topk_w", "dw_gate_up", "dw_down", "db_gate_up", "db_down")
    for name, a, b in zip(names, grads, again):
        assert torch.equal(a, b), name


def test_bias_changes_only_what_it_should():
    """A zero bias gives bit-for-bit the layer without biases; the bias
    gradients do not depend on the bias values (they are sums of dh and
    w * dy), only the other outputs do."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("bias0", T=400, H=256, I=192, E=8, k=4, act=ACT_SWIGLU, dtype="bf16",
               weight_std="fan_in", routing="softmax_topk_renorm", seed=3)
    d = to_device(synth.make_case(r))
    bgu, bd = (t.cuda() for t in synth.make_biases(r))
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, r.limit, r.alpha)
    run.plan(d.topk_idx)
    args = (d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down)
    y0 = run.forward(*args).clone()
    g0 = [t.clone() for t in run.backward(d.dy, *args)]
    z_gu, z_d = torch.zeros_like(bgu), torch.zeros_like(bd)
    yz = run.forward(*args, b_gate_up=z_gu, b_down=z_d).clone()
    gz = [t.clone() for t in run.backward(d.dy, *args, b_gate_up=z_gu, b_down=z_d)]
    torch.cuda.synchronize()
    run.check()
    assert torch.equal(y0, yz)
    for name, a, b in zip(("dx", "d_topk_w", "dw_gate_up", "dw_down"), g0, gz):
        assert torch.equal(a, b), name
    # db_down is sum w * dy whatever the bias values; with b_down only the
    # d(topk weights) term and y change, not dx or the weight gradients
    run.forward(*args, b_down=bd)
    gd = [t.clone() for t in run.backward(d.dy, *args, b_down=bd)]
    torch.cuda.synchronize()
    assert torch.equal(gd[5], gz[5])
    for name, a, b in zip(("dx", "dw_gate_up", "dw_down"), (g0[0], g0[2], g0[3]),
                          (gd[0], gd[2], gd[3])):
        assert torch.equal(a, b), name
    assert not torch.equal(gd[1], g0[1])
