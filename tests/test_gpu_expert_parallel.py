"""GPU side of the expert-parallel exchange: the two row primitives of the C
ABI (moe_gather_rows, moe_combine_rows) against plain torch on the same
values, and the expert-parallel layer on one rank (its exchanges are then
identities, every kernel step runs) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import ACT_CLAMPED_GLU, ACT_SWIGLU, Recipe
from tests.helpers import assert_close, assert_dw_close, oracle_inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,cols", [(torch.bfloat16, 136), (torch.float32, 1), (torch.int32, 3)])
def test_gather_rows_exact(dtype, cols):
    import dispatch_gemm_combine_gb300 as m
    g = torch.Generator().manual_seed(5)
    src = (torch.randn(50, cols, generator=g) * 100).to(dtype).cuda()
    index = torch.randint(-3, 160, (300,), generator=g, dtype=torch.int32).cuda()
    for div in (1, 3):
        dst = torch.full((300, cols), 7, dtype=dtype, device="cuda")
        m.gather_rows(index, div, src, dst)
        torch.cuda.synchronize()
        want = torch.zeros_like(dst)
        i = index.long()
        ok = (i >= 0) & (i < 50 * div)
        want[ok] = src[i[ok] // div]
        assert torch.equal(dst, want)


@pytest.mark.parametrize("src_dtype,out_fp32", [(torch.bfloat16, 0), (torch.float32, 0),
                                                (torch.float32, 1)])
def test_combine_rows_matches_fixed_order_sum(src_dtype, out_fp32):
    import dispatch_gemm_combine_gb300 as m
    T, k, H = 257, 3, 200
    g = torch.Generator().manual_seed(9)
    src = torch.randn(T * k, H, generator=g).to(src_dtype).cuda()
    inv = torch.randperm(T * k, generator=g).to(torch.int32).cuda()
    shape = m.Shape(T, H, 64, 8, k, out_fp32=out_fp32)
    dst = torch.empty(T, H, dtype=torch.float32 if out_fp32 else torch.bfloat16, device="cuda")
    m.combine_rows(shape, inv, src, dst)
    torch.cuda.synchronize()
    rows = src.float()[inv.long()].reshape(T, k, H)
    acc = torch.zeros(T, H, device="cuda")
    for j in range(k):                     # fp32, j ascending: the kernel's order
        acc = acc + rows[:, j]
    assert torch.equal(dst, acc.to(dst.dtype))
    # weighted: fused multiply-adds in the same order, within one fp32 step
    w = torch.rand(T, k, generator=g).cuda()
    dst2 = torch.empty_like(dst)
    m.combine_rows(shape, inv, src, dst2, topk_w=w)
    torch.cuda.synchronize()
    ref = (rows.double() * w.double()[:, :, None]).sum(1)
    assert torch.allclose(dst2.double(), ref, rtol=1e-2 if not out_fp32 else 1e-6, atol=1e-6)


@pytest.mark.parametrize("act,E", [(ACT_CLAMPED_GLU, 8), (ACT_SWIGLU, 5)])
def test_expert_parallel_single_rank(act, E):
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.expert_parallel import CudaOps, ExpertParallelMoE
    r = Recipe("ep", T=300, H=128, I=96, E=E, k=2, act=act, weight_std="fan_in",
               routing="softmax_topk_renorm", seed=23 + E)
    case = synth.make_case(r)
    d = to_device(case)
    ep = ExpertParallelMoE(E, r.k, CudaOps(r.H, r.I, act, MOE_BF16, r.limit, r.alpha))
    y = ep.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down)
    dx, dtw, dwgu, dwd = ep.backward(d.dy)
    torch.cuda.synchronize()
    x, idx, w, wgu, wd, dy = oracle_inputs(case)
    assert_close("y", y.float().cpu().numpy(), oracle.moe_forward(x, idx, w, wgu, wd, act))
    ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    assert_close("dx", dx.float().cpu().numpy(), ref[0])
    assert_dw_close(dtw.cpu().numpy(), ref[1])
    assert_close("dw_gate_up", dwgu.cpu().numpy(), ref[2])
    assert_close("dw_down", dwd.cpu().numpy(), ref[3])


def test_expert_parallel_single_rank_is_the_layer_bit_for_bit():
    """On one rank every exchange is an identity and the owner's plan sees the
    rows in the layer's own expert-grouped order, so the owner runs the same
    tiles on the same rows; with fp32 owner outputs and the same fixed-order
    combine, y, dx, d(topk w), the weight gradients and the bias gradients
    equal the fused layer's bit for bit."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.expert_parallel import CudaOps, ExpertParallelMoE
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("ep", T=1024, H=512, I=384, E=16, k=4, act=ACT_CLAMPED_GLU, weight_std=0.05,
               routing="uniform_topk_softmax", seed=31)
    case = synth.make_case(r)
    d = to_device(case)
    bgu, bd = (t.cuda() for t in synth.make_biases(r))
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, r.limit, r.alpha)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, b_gate_up=bgu,
                    b_down=bd).clone()
    ref = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                           d.w_down, b_gate_up=bgu, b_down=bd)]
    ep = ExpertParallelMoE(r.E, r.k, CudaOps(r.H, r.I, r.act, MOE_BF16, r.limit, r.alpha))
    for _ in range(2):   # twice: the owner's buffers are reused
        y2 = ep.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, bgu, bd)
        got = ep.backward(d.dy)
        torch.cuda.synchronize()
        run.check()
        assert torch.equal(y2, y)
        for name, a, b in zip(("dx", "d_topk_w", "dw_gate_up", "dw_down", "db_gate_up",
                               "db_down"), got, ref):
            assert torch.equal(a, b), name
