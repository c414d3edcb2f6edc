"""Parity at the full workload sizes, in the launch configuration bench.py
times (same C-ABI calls, persistent grids of one CTA per SM).

The oracle cannot redo a whole full-size layer in fp64 within a test, so it
computes sampled outputs one by one:
  * y, dx, d(topk weights) of sampled tokens (each depends only on the
    token's own k slots: the oracle runs on those tokens alone);
  * the complete gate / up / down weight gradients of sampled experts (the
    oracle runs on exactly the tokens routed to them);
  * exact zeros for experts that received no token.
Two identities that hold at any size check the whole tensors:
  sum_{t,j} w[t,j] d_w[t,j] = <dy, y>   and   sum_e <dWd_e, Wd_e> = <dy, y>
(y is linear in the routing weights and in the down weights).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import assert_close, assert_dw_close

pytestmark = pytest.mark.gpu


class LazyExperts:
    """Expert weights fetched from the device one expert at a time."""

    def __init__(self, t):
        self.t = t

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        # widened on the device (exact), so the host receives fp64 directly
        return self.t[int(e)].double().cpu().numpy()


def _run(r, backward, biases=None):
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    case = synth.make_case(r, device="cuda", with_dy=backward)
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, r.limit, r.alpha,
                      training=backward, backward=backward)
    bkw = {} if biases is None else dict(b_gate_up=biases[0], b_down=biases[1])
    run.plan(case.topk_idx)
    y = run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down, **bkw)
    grads = None
    if backward:
        grads = run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up,
                             case.w_down, **bkw)
    torch.cuda.synchronize()
    run.check()
    return case, run, y, grads


def _host(case, toks):
    f = lambda t: t[toks].double().cpu().numpy()
    x, w = f(case.x), f(case.topk_w)
    idx = case.topk_idx[toks].cpu().numpy().astype(np.int64)
    dy = f(case.dy) if case.dy is not None else None
    return x, idx, w, dy


def _check_tokens(case, y, grads, n_tok, seed):
    r = case.recipe
    g = np.random.default_rng(seed)
    toks = torch.from_numpy(np.sort(g.choice(r.T, size=min(n_tok, r.T), replace=False)))
    x, idx, w, dy = _host(case, toks)
    wgu, wd = LazyExperts(case.w_gate_up), LazyExperts(case.w_down)
    y_ref = oracle.moe_forward(x, idx, w, wgu, wd, r.act, r.limit, r.alpha)
    assert_close("y[sample]", y[toks].double().cpu().numpy(), y_ref)
    if grads is not None:
        dx, dtw = grads[0], grads[1]
        used = sorted(set(idx.reshape(-1).tolist()))
        dx_ref, dw_ref, _, _ = oracle.moe_backward(dy, x, idx, w, wgu, wd, r.act, r.limit,
                                                   r.alpha, experts=used)
        assert_close("dx[sample]", dx[toks].double().cpu().numpy(), dx_ref)
        assert_dw_close(dtw[toks].cpu().numpy(), dw_ref)


def _check_expert_grads(case, run, grads, n_exp, seed, max_rows=4096, hottest=False):
    """Weight gradients of n_exp sampled experts (among those with at most
    max_rows rows), and with hottest=True also of the expert holding the most
    rows, element by element against the oracle on exactly their tokens."""
    r = case.recipe
    counts = run.plan_t["counts"].cpu().numpy()
    live = [e for e in range(r.E) if 0 < counts[e] <= max_rows]
    g = np.random.default_rng(seed)
    picks = [int(e) for e in g.choice(live, size=min(n_exp, len(live)), replace=False)]
    if hottest:
        picks.append(int(np.argmax(counts)))
    for e in picks:
        toks = torch.nonzero((case.topk_idx == e).any(dim=1)).flatten().cpu()
        x, idx, w, dy = _host(case, toks)
        wgu, wd = LazyExperts(case.w_gate_up), LazyExperts(case.w_down)
        _, _, dgu, dd = oracle.moe_backward(dy, x, idx, w, wgu, wd, r.act, r.limit, r.alpha,
                                            experts=[e])
        got_gu = grads[2][e].double().cpu().numpy()
        assert_close("d_gate[%d]" % e, got_gu[:, :r.I], dgu[e][:, :r.I])
        assert_close("d_up[%d]" % e, got_gu[:, r.I:], dgu[e][:, r.I:])
        assert_close("d_down[%d]" % e, grads[3][e].double().cpu().numpy(), dd[e])
    for e in np.nonzero(counts == 0)[0]:
        assert torch.all(grads[2][int(e)] == 0) and torch.all(grads[3][int(e)] == 0)


# Relative agreement of the two gradient sides of <dy, y> (below).  An expert
# whose weight gradients take w*a as one bf16 value (those with many
# effectively weighted rows) adds sum_{r,i} x_ri d_ri to <dWd, Wd>, with x_ri =
# w_r a_ri dA'_ri and d_ri the relative rounding error (|d| <= 2^-8, about
# uniform): a random-sign sum of standard deviation ~ 2^-8 / sqrt(3) (2.3e-3)
# of the sum it perturbs, itself of random sign.  1e-2 allows about four
# standard deviations; with hi + lo operands the sides agree to ~1e-5.
IDENTITY_REL = 1e-2


def _check_identities(case, y, grads):
    # Both gradient sides equal <dy, y_exact> up to the rounding of the
    # weight gradients' operands (IDENTITY_REL) and carry no bf16 output
    # rounding.  <dy, y> with the GPU's bf16 y differs from <dy, y_exact> by
    # at most ||dy|| ||y - y_exact|| (Cauchy-Schwarz), i.e. by at most
    # 5e-3 ||dy|| ||y|| under the relative Frobenius tolerance; <dy, y> itself
    # is a sum of random-sign terms, so a relative bound on it would be
    # meaningless.
    dy, yd = case.dy.double(), y.double()
    ly = float((dy * yd).sum())
    sw = float((case.topk_w.double() * grads[1].double()).sum())
    sd = float((case.w_down.double() * grads[3].double()).sum())
    assert abs(sw - sd) <= IDENTITY_REL * abs(sd), (sw, sd)
    bound = 5e-3 * float(dy.norm()) * float(yd.norm())
    assert abs(sw - ly) <= bound, (sw, ly, bound)


def test_clamped_glu_workload_fwd_bwd():
    """T=8192, H=I=2880, 128 experts, top-4, clamped GLU: the bench step."""
    case, run, y, grads = _run(synth.RECIPES["clamped_glu_fwd"], backward=True)
    _check_tokens(case, y, grads, n_tok=24, seed=1)
    _check_expert_grads(case, run, grads, n_exp=2, seed=2)
    _check_identities(case, y, grads)


def test_swiglu_forward_workload():
    """T=4096, H=8192, I=2048, 256 experts, top-8 (26 GB of weights)."""
    case, run, y, _ = _run(synth.RECIPES["swiglu_fwd"], backward=False)
    _check_tokens(case, y, None, n_tok=32, seed=3)


def test_swiglu_backward_workload():
    """T=4096, H=4096, I=2048, 256 experts, top-8, fp32 weight gradients."""
    case, run, y, grads = _run(synth.RECIPES["swiglu_bwd"], backward=True)
    _check_tokens(case, y, grads, n_tok=8, seed=4)
    _check_expert_grads(case, run, grads, n_exp=2, seed=5)
    _check_identities(case, y, grads)


@pytest.mark.parametrize("T", synth.ZIPF_TOKENS)
def test_zipf_sweep(T):
    """Load imbalance on the backward-workload shape: ~30% of experts empty,
    the hottest expert over 10x the mean."""
    r = synth.RECIPES["zipf_sweep"].scaled(T=T)
    case, run, y, grads = _run(r, backward=True)
    zero, ratio = synth.routing_stats(case.topk_idx, r.E)
    assert zero >= 0.25 and ratio > 10.0, (zero, ratio)
    _check_tokens(case, y, grads, n_tok=6, seed=T)
    # a sampled expert plus the hottest one (about 0.9 T rows at this routing:
    # the longest weight-gradient contraction of the sweep)
    _check_expert_grads(case, run, grads, n_exp=1, seed=T + 1, max_rows=2048, hottest=True)
    _check_identities(case, y, grads)


def test_clamped_glu_workload_with_biases():
    """The bench step with per-expert biases on both projections: sampled
    tokens and experts (their bias gradients included) against the oracle,
    and, over every expert, y being linear in (Wd, b_down) jointly:
    sum_e <dWd_e, Wd_e> + <db_down_e, b_down_e> = <dy, y>."""
    r = synth.RECIPES["clamped_glu_fwd"]
    bgu, bd = synth.make_biases(r, device="cuda")
    case, run, y, grads = _run(r, backward=True, biases=(bgu, bd))
    bgu_h, bd_h = bgu.double().cpu().numpy(), bd.double().cpu().numpy()
    kw = dict(b_gate_up=bgu_h, b_down=bd_h)
    g = np.random.default_rng(11)
    toks = torch.from_numpy(np.sort(g.choice(r.T, size=16, replace=False)))
    x, idx, w, dy = _host(case, toks)
    wgu, wd = LazyExperts(case.w_gate_up), LazyExperts(case.w_down)
    y_ref = oracle.moe_forward(x, idx, w, wgu, wd, r.act, r.limit, r.alpha, **kw)
    assert_close("y[sample]", y[toks].double().cpu().numpy(), y_ref)
    used = sorted(set(idx.reshape(-1).tolist()))
    dx_ref, dw_ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, r.act, r.limit, r.alpha,
                                         experts=used, **kw)[:2]
    assert_close("dx[sample]", grads[0][toks].double().cpu().numpy(), dx_ref)
    assert_dw_close(grads[1][toks].cpu().numpy(), dw_ref)
    for e in (int(v) for v in g.choice(r.E, size=2, replace=False)):
        etoks = torch.nonzero((case.topk_idx == e).any(dim=1)).flatten().cpu()
        x, idx, w, dy = _host(case, etoks)
        _, _, dgu, dd, dbgu, dbd = oracle.moe_backward(dy, x, idx, w, wgu, wd, r.act, r.limit,
                                                       r.alpha, experts=[e], **kw)
        got_gu = grads[2][e].double().cpu().numpy()
        assert_close("d_gate[%d]" % e, got_gu[:, :r.I], dgu[e][:, :r.I])
        assert_close("d_up[%d]" % e, got_gu[:, r.I:], dgu[e][:, r.I:])
        assert_close("d_down[%d]" % e, grads[3][e].double().cpu().numpy(), dd[e])
        assert_close("db_gate_up[%d]" % e, grads[4][e].double().cpu().numpy(), dbgu[e])
        assert_close("db_down[%d]" % e, grads[5][e].double().cpu().numpy(), dbd[e])
    dyd, yd = case.dy.double(), y.double()
    ly = float((dyd * yd).sum())
    sw = float((case.topk_w.double() * grads[1].double()).sum())
    sd = float((case.w_down.double() * grads[3].double()).sum() + (bd.double() * grads[5].double()).sum())
    assert abs(sw - sd) <= IDENTITY_REL * abs(sd), (sw, sd)
    assert abs(sw - ly) <= 5e-3 * float(dyd.norm()) * float(yd.norm()), (sw, ly)
