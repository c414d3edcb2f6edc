"""The layer as a CUDA graph: one training step (plan, forward with the saved
context, backward) captured from the C-ABI calls and replayed.

The calls enqueue only kernels on the caller's stream (no allocation, no
host synchronisation), so a captured step is a valid graph.  The kernels are
deterministic, so a replay must reproduce an eager step bit for bit, also
after the input buffers were refilled with new values in place (the graph
reads its inputs when it runs, not when it was captured)."""

import pytest
import torch

import synth
from synth import ACT_CLAMPED_GLU, ACT_SWIGLU, Recipe

pytestmark = pytest.mark.gpu


def _outputs(run):
    return [t.clone() for t in (run.y, run.dx, run.d_topk_w, run.dw_gate_up, run.dw_down)]


@pytest.mark.parametrize("act,dtype", [(ACT_CLAMPED_GLU, "bf16"), (ACT_SWIGLU, "fp32")])
def test_captured_step_replays_like_eager(act, dtype):
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("graph", T=600, H=256, I=192, E=8, k=4, act=act, dtype=dtype, weight_std="fan_in",
               routing="softmax_topk_renorm", seed=11)
    case = synth.make_case(r, device="cuda")
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_FP32 if dtype == "fp32" else MOE_BF16,
                      r.limit, r.alpha)
    stream = torch.cuda.Stream()

    def step():
        run.plan(case.topk_idx)
        run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
        run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)

    with torch.cuda.stream(stream):
        step()                                   # first calls configure the kernels
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()

    # new values in the same buffers: a different routing and new activations
    r2 = Recipe("graph2", T=r.T, H=r.H, I=r.I, E=r.E, k=r.k, act=act, dtype=dtype,
                weight_std="fan_in", routing="uniform_topk_softmax", seed=12)
    new = synth.make_case(r2, device="cuda")
    for name in ("x", "topk_idx", "topk_w", "dy"):
        getattr(case, name).copy_(getattr(new, name))
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    eager = _outputs(run)
    for t in (run.y, run.dx, run.d_topk_w, run.dw_gate_up, run.dw_down):
        t.fill_(float("nan"))
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    run.check()
    for name, a, b in zip(("y", "dx", "d_topk_w", "dw_gate_up", "dw_down"), eager, _outputs(run)):
        assert torch.equal(a, b), name
