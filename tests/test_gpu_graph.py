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


def test_captured_step_with_router_and_biases():
    """The same for a step that starts from router logits (moe_route builds
    the ids, weights and plan) and carries per-expert biases: every kernel
    the step launches is captured and replayed bit for bit."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("graphb", T=500, H=256, I=200, E=12, k=3, act=ACT_CLAMPED_GLU, dtype="bf16",
               weight_std=0.2, routing="softmax_topk_renorm", seed=21)
    case = synth.make_case(r, device="cuda")
    bgu, bd = synth.make_biases(r, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(22)
    logits = torch.randn((r.T, r.E), generator=g, device="cuda", dtype=torch.float32)
    idx = torch.empty((r.T, r.k), dtype=torch.int32, device="cuda")
    w = torch.empty((r.T, r.k), dtype=torch.float32, device="cuda")
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, r.limit, r.alpha)
    stream = torch.cuda.Stream()
    outs = lambda: [t.clone() for t in (idx, w, run.y, run.dx, run.d_topk_w, run.dw_gate_up,
                                        run.dw_down, run.db_gate_up, run.db_down)]

    def step():
        run.route(logits, idx, w)
        run.forward(case.x, idx, w, case.w_gate_up, case.w_down, b_gate_up=bgu, b_down=bd)
        run.backward(case.dy, case.x, idx, w, case.w_gate_up, case.w_down, b_gate_up=bgu,
                     b_down=bd)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    logits.copy_(torch.randn((r.T, r.E), generator=g, device="cuda", dtype=torch.float32))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    eager = outs()
    for t in (idx, run.y, run.dx, run.dw_gate_up, run.db_down):
        t.fill_(-1)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    run.check()
    names = ("topk_idx", "topk_w", "y", "dx", "d_topk_w", "dw_gate_up", "dw_down", "db_gate_up",
             "db_down")
    for name, a, b in zip(names, eager, outs()):
        assert torch.equal(a, b), name


def test_two_streams_concurrently_match_alone():
    """Two layers of different shapes, each with its own workspaces, enqueued
    interleaved on two streams (their kernels may overlap on the GPU): every
    output equals the same step run alone, bit for bit (the library keeps no
    state that two calls with separate workspaces could share)."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    recipes = [Recipe("s1", T=700, H=256, I=192, E=10, k=3, act=ACT_SWIGLU, dtype="bf16",
                      weight_std="fan_in", routing="softmax_topk_renorm", seed=31),
               Recipe("s2", T=400, H=384, I=320, E=6, k=2, act=ACT_CLAMPED_GLU, dtype="bf16",
                      weight_std=0.2, routing="uniform_ids", seed=32)]
    cases = [synth.make_case(r, device="cuda") for r in recipes]
    runs = [LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, r.limit, r.alpha)
            for r in recipes]

    def step(run, c):
        run.plan(c.topk_idx)
        run.forward(c.x, c.topk_idx, c.topk_w, c.w_gate_up, c.w_down)
        run.backward(c.dy, c.x, c.topk_idx, c.topk_w, c.w_gate_up, c.w_down)

    def outs(run):
        return [t.clone() for t in (run.y, run.dx, run.d_topk_w, run.dw_gate_up, run.dw_down)]

    alone = []
    for run, c in zip(runs, cases):
        step(run, c)
        torch.cuda.synchronize()
        alone.append(outs(run))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for run, c, st in zip(runs, cases, streams):
            with torch.cuda.stream(st):
                step(run, c)
    torch.cuda.synchronize()
    for run, ref in zip(runs, alone):
        run.check()
        for name, a, b in zip(("y", "dx", "d_topk_w", "dw_gate_up", "dw_down"), ref, outs(run)):
            assert torch.equal(a, b), name
