"""GPU parity of the top-k router (moe_route) against the fp64 oracle: the
chosen ids and the plan bit-exact, the weights within fp32 rounding of a
k-term softmax.  Logits include exact ties (integer values, equal rows),
expert counts that are not multiples of 32, and the limits E = 1024, k = 32."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # T, E, k, kind
    (1, 1, 1, "normal"),
    (100, 8, 2, "normal"),
    (1000, 128, 4, "uniform"),
    (777, 256, 8, "normal"),
    (513, 37, 5, "ties"),
    (300, 1024, 32, "normal"),
    (256, 64, 64 // 2, "ties"),
    (40, 16, 16, "equal"),
]


def _logits(T, E, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "uniform":
        z = torch.rand(T, E, generator=g)
    elif kind == "ties":
        z = torch.round(torch.randn(T, E, generator=g) * 2.0)
    elif kind == "equal":
        z = torch.full((T, E), 0.5)
    else:
        z = torch.randn(T, E, generator=g) * 3.0
    return z.float()


@pytest.mark.parametrize("T,E,k,kind", CASES)
def test_route_matches_oracle(T, E, k, kind):
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    z = _logits(T, E, kind, seed=T + E + k)
    run = LayerRunner(T, 64, 64, E, k, 0, MOE_BF16, training=False, backward=False)
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    run.route(z.cuda(), idx, w)
    run.check()
    idx_ref, w_ref = oracle.route(z.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    np.testing.assert_allclose(w.cpu().double().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    counts, offsets, perm, inv = oracle.dispatch_plan(idx_ref, E)
    assert np.array_equal(run.plan_t["counts"].cpu().numpy(), counts)
    assert np.array_equal(run.plan_t["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(run.plan_t["perm"].cpu().numpy()[:T * k], perm)
    assert np.array_equal(run.plan_t["inv"].cpu().numpy()[:T * k], inv)


def test_route_without_plan_and_empty():
    import dispatch_gemm_combine_gb300 as m
    T, E, k = 333, 48, 3
    z = _logits(T, E, "normal", seed=9)
    shape = m.Shape(T, 64, 64, E, k)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    m.route(shape, z.cuda(), idx, w)
    torch.cuda.synchronize()
    idx_ref, w_ref = oracle.route(z.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    np.testing.assert_allclose(w.cpu().double().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    m.route(m.Shape(0, 64, 64, E, k), None, None, None)   # T = 0: nothing to do
    torch.cuda.synchronize()
