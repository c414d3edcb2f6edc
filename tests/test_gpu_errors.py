"""Device-side error reporting without faulting the GPU.

* An expert id outside [0, E) is counted by the plan kernel into the
  workspace error word; the call returns, the host reads MOE_ERR_BAD_INDEX,
  and the context stays usable.
* The pipeline waits inside the GEMM kernels are bounded: with the limit
  set to 1 ns, waits that are not satisfied at once give up, every warp role
  unwinds (draining copies and MMAs already in flight with a separate fixed
  limit), MOE_ERR_TIMEOUT is reported, and the next call with the normal
  limit is correct.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import ACT_SWIGLU, Recipe
from tests.helpers import assert_close, oracle_inputs, to_device

pytestmark = pytest.mark.gpu


def _runner(r):
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    return LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16)


def test_bad_expert_index_reported():
    from dispatch_gemm_combine_gb300 import MOE_ERR_BAD_INDEX, MoeError
    r = Recipe("t", T=100, H=64, I=64, E=4, k=2, act=ACT_SWIGLU, weight_std="fan_in",
               routing="uniform_ids", seed=1)
    case = to_device(synth.make_case(r))
    idx = case.topk_idx.clone()
    idx[17, 1] = 4          # == E: out of range
    idx[50, 0] = -3
    run = _runner(r)
    run.plan(idx)
    with pytest.raises(MoeError) as ei:
        run.check()
    assert ei.value.status == MOE_ERR_BAD_INDEX
    # the forward with its own plan reports it as well and does not fault
    run.forward(case.x, idx, case.topk_w, case.w_gate_up, case.w_down, use_plan=False)
    with pytest.raises(MoeError):
        run.check()
    # context still usable: a valid call afterwards is correct
    run.plan(case.topk_idx)
    y = run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
    run.check()
    x, i, w, wgu, wd, _ = oracle_inputs(case)
    assert_close("y", y.float().cpu().numpy(), oracle.moe_forward(x, i, w, wgu, wd, ACT_SWIGLU))


def test_pipeline_wait_timeout_unwinds():
    from dispatch_gemm_combine_gb300 import MOE_ERR_TIMEOUT, MoeError, moe_set_wait_timeout_ns
    r = Recipe("t", T=2048, H=512, I=512, E=8, k=4, act=ACT_SWIGLU, weight_std="fan_in",
               routing="softmax_topk_renorm", seed=2)
    case = to_device(synth.make_case(r))
    run = _runner(r)
    run.plan(case.topk_idx)
    run.check()
    old = moe_set_wait_timeout_ns(1)
    try:
        run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
        torch.cuda.synchronize()
    finally:
        moe_set_wait_timeout_ns(old)
    with pytest.raises(MoeError) as ei:
        run.check()
    assert ei.value.status == MOE_ERR_TIMEOUT
    y = run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
    run.check()
    x, i, w, wgu, wd, _ = oracle_inputs(case)
    assert_close("y", y.float().cpu().numpy(), oracle.moe_forward(x, i, w, wgu, wd, ACT_SWIGLU))


def test_backward_wait_timeout_unwinds():
    """The same for the backward's GEMMs (down dgrad, both weight gradients,
    gate_up dgrad): a 1 ns limit reports MOE_ERR_TIMEOUT, and the next
    backward with the normal limit matches the oracle."""
    from dispatch_gemm_combine_gb300 import MOE_ERR_TIMEOUT, MoeError, moe_set_wait_timeout_ns
    r = Recipe("t", T=1024, H=256, I=256, E=8, k=2, act=ACT_SWIGLU, weight_std="fan_in",
               routing="softmax_topk_renorm", seed=3)
    case = to_device(synth.make_case(r))
    run = _runner(r)
    run.plan(case.topk_idx)
    run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
    run.check()
    args = (case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
    old = moe_set_wait_timeout_ns(1)
    try:
        run.backward(*args)
        torch.cuda.synchronize()
    finally:
        moe_set_wait_timeout_ns(old)
    with pytest.raises(MoeError) as ei:
        run.check()
    assert ei.value.status == MOE_ERR_TIMEOUT
    dx = run.backward(*args)[0]
    run.check()
    x, i, w, wgu, wd, dy = oracle_inputs(case)
    dx_ref = oracle.moe_backward(dy, x, i, w, wgu, wd, ACT_SWIGLU)[0]
    assert_close("dx", dx.float().cpu().numpy(), dx_ref)
