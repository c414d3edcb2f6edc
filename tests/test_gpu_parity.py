"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs, element by element.  Sizes span several 128-row tiles
per expert, several column tiles, k-block tails (H, I not multiples of 64 or
256) and the degenerate cases of the layer."""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import ACT_CLAMPED_GLU, ACT_SWIGLU, Recipe
from tests.helpers import assert_close, assert_dw_close, oracle_inputs, to_device

pytestmark = pytest.mark.gpu


def _runner(r, training=True, backward=True):
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    return LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act,
                       MOE_FP32 if r.dtype == "fp32" else MOE_BF16, r.limit, r.alpha,
                       training=training, backward=backward)


def _recipe(T, H, I, E, k, act, seed, dtype="bf16", routing="softmax_topk_renorm", std=None):
    return Recipe("t", T=T, H=H, I=I, E=E, k=k, act=act, dtype=dtype,
                  weight_std=std if std is not None else "fan_in", routing=routing, seed=seed)


# ------------------------------------------------------------------- plan
PLAN_CASES = [
    # T, k, E, routing
    (1, 1, 1, "uniform_ids"),
    (7, 2, 5, "uniform_ids"),
    (300, 4, 8, "softmax_topk_renorm"),
    (1000, 8, 256, "softmax_topk_renorm"),      # several 1024-slot chunks
    (2500, 3, 16, "uniform_ids"),                # duplicates within a token allowed
    (3000, 8, 256, "zipf"),                      # skewed, ~30% experts empty
    (4096, 8, 1024, "uniform_ids"),
]


@pytest.mark.parametrize("T,k,E,routing", PLAN_CASES)
def test_plan_bit_exact(T, k, E, routing):
    r = _recipe(T, 64, 64, E, k, ACT_SWIGLU, seed=T + E, routing=routing)
    case = synth.make_case(r, with_dy=False)
    run = _runner(r, training=False, backward=False)
    idx = case.topk_idx.cuda()
    run.plan(idx)
    run.check()
    counts, offsets, perm, inv = oracle.dispatch_plan(case.topk_idx.numpy(), E)
    assert np.array_equal(run.plan_t["counts"].cpu().numpy(), counts)
    assert np.array_equal(run.plan_t["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(run.plan_t["perm"].cpu().numpy()[:T * k], perm)
    assert np.array_equal(run.plan_t["inv"].cpu().numpy()[:T * k], inv)


def test_plan_all_tokens_one_expert():
    T, k, E = 2000, 1, 16
    idx = torch.full((T, k), 11, dtype=torch.int32)
    r = _recipe(T, 64, 64, E, k, ACT_SWIGLU, seed=0)
    run = _runner(r, training=False, backward=False)
    run.plan(idx.cuda())
    run.check()
    counts, offsets, perm, inv = oracle.dispatch_plan(idx.numpy(), E)
    assert np.array_equal(run.plan_t["counts"].cpu().numpy(), counts)
    assert np.array_equal(run.plan_t["perm"].cpu().numpy(), perm)
    assert np.array_equal(run.plan_t["inv"].cpu().numpy(), inv)


# ------------------------------------------------------------------- forward / backward
FB_CASES = [
    # T, H, I, E, k, act, dtype, std, routing
    (512, 384, 320, 8, 4, ACT_SWIGLU, "bf16", None, "softmax_topk_renorm"),
    (512, 384, 320, 8, 4, ACT_CLAMPED_GLU, "bf16", 0.2, "uniform_topk_softmax"),
    (300, 136, 200, 6, 2, ACT_SWIGLU, "bf16", None, "uniform_ids"),   # K tails, N tails
    (64, 128, 128, 8, 2, ACT_SWIGLU, "fp32", None, "softmax_topk_renorm"),  # tiny fp32 recipe
    (200, 264, 136, 5, 3, ACT_CLAMPED_GLU, "fp32", 0.2, "uniform_ids"),
    (1, 64, 64, 4, 1, ACT_SWIGLU, "bf16", None, "uniform_ids"),       # a single token
    (700, 256, 256, 40, 8, ACT_SWIGLU, "bf16", None, "zipf"),         # empty experts, hot expert
]


def _run_case(r, with_bwd=True, use_plan=True):
    case = synth.make_case(r, with_dy=with_bwd)
    d = to_device(case)
    run = _runner(r, training=with_bwd, backward=with_bwd)
    if use_plan:
        run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, use_plan=use_plan)
    grads = None
    if with_bwd:
        if not use_plan:
            run.plan(d.topk_idx)
        grads = run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down)
    torch.cuda.synchronize()
    run.check()
    return case, y, grads


@pytest.mark.parametrize("T,H,I,E,k,act,dtype,std,routing", FB_CASES)
def test_forward_backward_parity(T, H, I, E, k, act, dtype, std, routing):
    r = _recipe(T, H, I, E, k, act, seed=1000 + T, dtype=dtype, routing=routing, std=std)
    case, y, grads = _run_case(r)
    x, idx, w, wgu, wd, dy = oracle_inputs(case)
    y_ref = oracle.moe_forward(x, idx, w, wgu, wd, act)
    assert_close("y", y.float().cpu().numpy(), y_ref)
    dx_ref, dw_ref, dwgu_ref, dwd_ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    dx, dtw, dwgu, dwd = grads
    assert_close("dx", dx.float().cpu().numpy(), dx_ref)
    assert_dw_close(dtw.cpu().numpy(), dw_ref)
    assert_close("d_gate", dwgu[:, :, :I].cpu().numpy(), dwgu_ref[:, :, :I])
    assert_close("d_up", dwgu[:, :, I:].cpu().numpy(), dwgu_ref[:, :, I:])
    assert_close("d_down", dwd.cpu().numpy(), dwd_ref)
    # experts that received no token get exactly zero weight gradients
    counts = np.bincount(idx.reshape(-1), minlength=E)
    for e in np.nonzero(counts == 0)[0]:
        assert torch.all(dwgu[e] == 0) and torch.all(dwd[e] == 0)


def test_forward_internal_plan_matches_external():
    r = _recipe(333, 128, 192, 6, 3, ACT_CLAMPED_GLU, seed=5, std=0.2, routing="uniform_ids")
    _, y1, _ = _run_case(r, with_bwd=False, use_plan=True)
    _, y2, _ = _run_case(r, with_bwd=False, use_plan=False)
    assert torch.equal(y1, y2)


def test_forward_is_deterministic():
    r = _recipe(1024, 256, 256, 16, 4, ACT_SWIGLU, seed=9)
    case = synth.make_case(r)
    d = to_device(case)
    run = _runner(r)
    run.plan(d.topk_idx)
    outs = []
    for _ in range(3):
        y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down).clone()
        g = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                             d.w_down)]
        outs.append((y, g))
    run.check()
    for y, g in outs[1:]:
        assert torch.equal(y, outs[0][0])
        for a, b in zip(g, outs[0][1]):
            assert torch.equal(a, b)


def test_zero_tokens():
    from dispatch_gemm_combine_gb300 import MOE_BF16, Shape, alloc_plan, ffn_bwd, ffn_fwd, workspace
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    run = LayerRunner(0, 64, 64, 4, 2, ACT_SWIGLU, MOE_BF16)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    wgu = torch.randn((4, 64, 128), device="cuda").bfloat16()
    wd = torch.randn((4, 64, 64), device="cuda").bfloat16()
    run.dw_gate_up.fill_(1.0)
    run.dw_down.fill_(1.0)
    run.plan(idx)
    run.forward(x, idx, w, wgu, wd)
    run.backward(x, x, idx, w, wgu, wd)
    torch.cuda.synchronize()
    run.check()
    assert torch.all(run.dw_gate_up == 0) and torch.all(run.dw_down == 0)


@pytest.mark.parametrize("act,dtype", [(ACT_CLAMPED_GLU, "bf16"), (ACT_SWIGLU, "fp32")])
def test_backward_recompute_is_bit_identical(act, dtype):
    """Without the saved context the backward recomputes it with the same
    kernels on the same inputs, so every gradient must match bit for bit."""
    r = _recipe(700, 136, 200, 8, 3, act, seed=21, dtype=dtype)
    case = to_device(synth.make_case(r))
    run = _runner(r)
    run.plan(case.topk_idx)
    run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
    saved = [t.clone() for t in run.backward(case.dy, case.x, case.topk_idx, case.topk_w,
                                             case.w_gate_up, case.w_down)]
    again = run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up,
                         case.w_down, recompute=True)
    torch.cuda.synchronize()
    run.check()
    for name, a, b in zip(("dx", "d_topk_w", "dw_gate_up", "dw_down"), saved, again):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("T,H,I,E,k,act,dtype,std", [
    (600, 256, 200, 6, 4, ACT_CLAMPED_GLU, "bf16", 0.2),   # odd m-tiles (half units), N tail
    (300, 136, 264, 5, 3, ACT_SWIGLU, "bf16", None),
    (200, 128, 136, 5, 3, ACT_CLAMPED_GLU, "fp32", 0.2),
])
def test_interleaved_gate_up_parity(T, H, I, E, k, act, dtype, std):
    """gate_up weights with interleaved gate/up columns: the layer equals the
    oracle on the same weights taken apart into [gate | up], and dw_gate_up
    comes back interleaved; the backward without a saved context too."""
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32, MOE_GATE_UP_INTERLEAVED
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = _recipe(T, H, I, E, k, act, seed=77 + T, dtype=dtype, std=std)
    case = synth.make_case(r)
    x, idx, w, wgu_il, wd, dy = oracle_inputs(case)       # the recipe's weights, read as interleaved
    wgu = oracle.gate_up_concatenated(wgu_il, 1)
    d = to_device(case)
    run = LayerRunner(T, H, I, E, k, act, MOE_FP32 if dtype == "fp32" else MOE_BF16, r.limit,
                      r.alpha, gate_up_layout=MOE_GATE_UP_INTERLEAVED)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down)
    grads = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                             d.w_down)]
    again = run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, recompute=True)
    torch.cuda.synchronize()
    run.check()
    assert_close("y", y.float().cpu().numpy(), oracle.moe_forward(x, idx, w, wgu, wd, act))
    dx_ref, dw_ref, dwgu_ref, dwd_ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    dwgu_ref_il = oracle.gate_up_in_layout(dwgu_ref, 1)
    dx, dtw, dwgu, dwd = grads
    assert_close("dx", dx.float().cpu().numpy(), dx_ref)
    assert_dw_close(dtw.cpu().numpy(), dw_ref)
    assert_close("d_gate", dwgu[:, :, 0::2].cpu().numpy(), dwgu_ref_il[:, :, 0::2])
    assert_close("d_up", dwgu[:, :, 1::2].cpu().numpy(), dwgu_ref_il[:, :, 1::2])
    assert_close("d_down", dwd.cpu().numpy(), dwd_ref)
    for name, a, b in zip(("dx", "d_topk_w", "dw_gate_up", "dw_down"), grads, again):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("T,H,I,E,k,act,dtype,layout,bias", [
    (37, 8, 8, 3, 2, ACT_SWIGLU, "bf16", 0, False),           # one 16-byte row per token
    (50, 16, 24, 1, 1, ACT_CLAMPED_GLU, "bf16", 1, True),     # a single expert
    (65, 64, 8, 64, 32, ACT_SWIGLU, "bf16", 0, True),         # top-32, I of one row
    (129, 8, 72, 5, 3, ACT_CLAMPED_GLU, "fp32", 1, True),     # fp32, H of one row
    (300, 200, 8, 7, 7, ACT_SWIGLU, "fp32", 0, False),        # k = E: every expert per token
])
def test_extreme_shapes(T, H, I, E, k, act, dtype, layout, bias):
    """The declared limits of the shape (H, I multiples of 8 from 8 up, any
    T, 1 <= k <= E, one expert): boxes wider than the tensor, single-chunk
    epilogues, every row of a tile padding but one."""
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = _recipe(T, H, I, E, k, act, seed=900 + T, dtype=dtype, routing="uniform_ids", std=0.3)
    case = synth.make_case(r)
    x, idx, w, wgu_l, wd, dy = oracle_inputs(case)
    wgu = oracle.gate_up_concatenated(wgu_l, layout)
    kw, bkw = {}, {}
    if bias:
        bgu_t, bd_t = synth.make_biases(r)
        kw = dict(b_gate_up=oracle.gate_up_concatenated(bgu_t.double().numpy(), layout),
                  b_down=bd_t.double().numpy())
        bkw = dict(b_gate_up=bgu_t.cuda(), b_down=bd_t.cuda())
    d = to_device(case)
    run = LayerRunner(T, H, I, E, k, act, MOE_FP32 if dtype == "fp32" else MOE_BF16, r.limit,
                      r.alpha, gate_up_layout=layout)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, **bkw).clone()
    grads = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                             d.w_down, **bkw)]
    torch.cuda.synchronize()
    run.check()
    assert_close("y", y.float().cpu().numpy(), oracle.moe_forward(x, idx, w, wgu, wd, act, **kw))
    ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, act, **kw)
    assert_close("dx", grads[0].float().cpu().numpy(), ref[0])
    assert_dw_close(grads[1].cpu().numpy(), ref[1])
    assert_close("dw_gate_up", grads[2].cpu().numpy(), oracle.gate_up_in_layout(ref[2], layout))
    assert_close("dw_down", grads[3].cpu().numpy(), ref[3])
    if bias:
        assert_close("db_gate_up", grads[4].cpu().numpy(), oracle.gate_up_in_layout(ref[4], layout))
        assert_close("db_down", grads[5].cpu().numpy(), ref[5])


@pytest.mark.parametrize("k", [1, 2])
def test_expert_counts_at_tile_boundaries(k):
    """Experts holding exactly 0, 1, 15-17, 64-65, 255-257, 271-273 and 511-513
    rows: every edge of the 16-row token units, the 32-row warps, the
    128-row tiles (half units) and the 256-row pairs, against the oracle."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    counts = [1, 15, 16, 17, 255, 256, 257, 271, 272, 273, 511, 512, 513, 0, 64, 65]
    E, H, I = len(counts), 128, 96
    slots = np.repeat(np.arange(E), counts)               # each expert's rows, k per token
    g = np.random.default_rng(41 + k)
    slots = slots[g.permutation(slots.size)]
    T = slots.size // k
    idx = torch.from_numpy(slots[:T * k].reshape(T, k).astype(np.int32))
    # fan-in weights: the structure is under test here; the heavy-tailed std-0.3
    # draw of the same counts is the next test
    r = _recipe(T, H, I, E, k, ACT_CLAMPED_GLU, seed=60 + k, routing="uniform_ids")
    case = synth.make_case(r)
    case.topk_idx = idx
    x, idx_np, w, wgu, wd, dy = oracle_inputs(case)
    d = to_device(case)
    run = LayerRunner(T, H, I, E, k, r.act, MOE_BF16, r.limit, r.alpha)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down).clone()
    dx, dtw, dwgu, dwd = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w,
                                                          d.w_gate_up, d.w_down)]
    torch.cuda.synchronize()
    run.check()
    got = np.bincount(idx_np.reshape(-1), minlength=E)
    assert np.array_equal(run.plan_t["counts"].cpu().numpy(), got)
    assert_close("y", y.float().cpu().numpy(), oracle.moe_forward(x, idx_np, w, wgu, wd, r.act))
    ref = oracle.moe_backward(dy, x, idx_np, w, wgu, wd, r.act)
    assert_close("dx", dx.float().cpu().numpy(), ref[0])
    assert_dw_close(dtw.cpu().numpy(), ref[1])
    for e in range(E):   # per expert: each boundary case on its own
        if got[e]:
            assert_close("dw_gate_up[%d]" % e, dwgu[e].cpu().numpy(), ref[2][e])
            assert_close("dw_down[%d]" % e, dwd[e].cpu().numpy(), ref[3][e])
        else:
            assert torch.all(dwgu[e] == 0) and torch.all(dwd[e] == 0)


@pytest.mark.parametrize("k", [1, 2])
def test_expert_counts_at_tile_boundaries_heavy_tailed(k):
    """The tile-boundary counts with std-0.3 weights, where |y| and |dx| reach
    7-10x their rms.  The bf16 outputs y and dx then carry two errors at their
    largest elements: the arithmetic's (chiefly the bf16 rounding of the
    activation before the down GEMM, ~1e-2 rms at the tails) and their own
    rounding to bf16, one step of which is 2^-7 of the value, up to 0.055 rms
    here.  Where the exact value lies near a rounding midpoint, the first
    error moves the second to the neighbouring bf16 value, so no bf16-output
    evaluation that is not correctly rounded can promise 3e-2 rms there.  y
    and dx are held to the relative Frobenius bound and to max abs error
    <= 3e-2 rms plus one bf16 step of the reference element; the fp32 outputs
    (d(topk w), every expert's weight gradients) keep the usual bounds."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    from tests.helpers import assert_close_bf16_output
    counts = [1, 15, 16, 17, 255, 256, 257, 271, 272, 273, 511, 512, 513, 0, 64, 65]
    E, H, I = len(counts), 128, 96
    slots = np.repeat(np.arange(E), counts)
    g = np.random.default_rng(41 + k)
    slots = slots[g.permutation(slots.size)]
    T = slots.size // k
    idx = torch.from_numpy(slots[:T * k].reshape(T, k).astype(np.int32))
    r = _recipe(T, H, I, E, k, ACT_CLAMPED_GLU, seed=60 + k, routing="uniform_ids", std=0.3)
    case = synth.make_case(r)
    case.topk_idx = idx
    x, idx_np, w, wgu, wd, dy = oracle_inputs(case)
    d = to_device(case)
    run = LayerRunner(T, H, I, E, k, r.act, MOE_BF16, r.limit, r.alpha)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down).clone()
    dx, dtw, dwgu, dwd = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w,
                                                          d.w_gate_up, d.w_down)]
    torch.cuda.synchronize()
    run.check()
    ref = oracle.moe_backward(dy, x, idx_np, w, wgu, wd, r.act)
    assert_close_bf16_output("y", y.double().cpu().numpy(),
                             oracle.moe_forward(x, idx_np, w, wgu, wd, r.act))
    assert_close_bf16_output("dx", dx.double().cpu().numpy(), ref[0])
    assert_dw_close(dtw.cpu().numpy(), ref[1])
    for e in range(E):
        if counts[e]:
            assert_close("dw_gate_up[%d]" % e, dwgu[e].cpu().numpy(), ref[2][e])
            assert_close("dw_down[%d]" % e, dwd[e].cpu().numpy(), ref[3][e])
        else:
            assert torch.all(dwgu[e] == 0) and torch.all(dwd[e] == 0)


@pytest.mark.parametrize("limit", [3.0, 5.3])
def test_clamped_glu_limits_and_saved_context(limit):
    """The clamped GLU at other limits: 3.0, an fp16 value (the saved
    pre-activations are fp16, many of them past the clamp and kept as
    markers), and 5.3, which fp16 does not represent (fp32 context).  Both
    against the oracle at the same limit, the recompute backward bit for bit."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    r = Recipe("lim", T=400, H=192, I=136, E=6, k=3, act=ACT_CLAMPED_GLU, weight_std=0.2,
               routing="softmax_topk_renorm", seed=88, limit=limit)
    case = synth.make_case(r)
    x, idx, w, wgu, wd, dy = oracle_inputs(case)
    d = to_device(case)
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, limit, r.alpha)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down).clone()
    grads = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up,
                                             d.w_down)]
    again = run.backward(d.dy, d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down, recompute=True)
    torch.cuda.synchronize()
    run.check()
    assert_close("y", y.float().cpu().numpy(),
                 oracle.moe_forward(x, idx, w, wgu, wd, r.act, limit, r.alpha))
    ref = oracle.moe_backward(dy, x, idx, w, wgu, wd, r.act, limit, r.alpha)
    assert_close("dx", grads[0].float().cpu().numpy(), ref[0])
    assert_dw_close(grads[1].cpu().numpy(), ref[1])
    assert_close("dw_gate_up", grads[2].cpu().numpy(), ref[2])
    assert_close("dw_down", grads[3].cpu().numpy(), ref[3])
    for name, a, b in zip(("dx", "d_topk_w", "dw_gate_up", "dw_down"), grads, again):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("act", [ACT_SWIGLU, ACT_CLAMPED_GLU])
def test_weight_gradients_long_and_short_contractions(act):
    """Two experts with 1100 and 1500 rows (contractions of 18 and 24 k-blocks,
    one bf16 operand after the split selection) among 98 with 0-30 rows (hi +
    lo operands, or zeros), several tiles per expert: every expert's weight
    gradients against the oracle, and the layer's other outputs."""
    from dispatch_gemm_combine_gb300 import MOE_BF16
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    g = np.random.default_rng(71)
    E, H, I = 100, 512, 256
    counts = np.concatenate([[1100, 1500], g.integers(0, 31, E - 2)])
    slots = np.repeat(np.arange(E), counts)
    slots = slots[g.permutation(slots.size)]
    T = slots.size
    idx = torch.from_numpy(slots.reshape(T, 1).astype(np.int32))
    r = _recipe(T, H, I, E, 1, act, seed=72, routing="uniform_ids", std=None)
    case = synth.make_case(r)
    case.topk_idx = idx
    x, idx_np, w, wgu, wd, dy = oracle_inputs(case)
    d = to_device(case)
    run = LayerRunner(T, H, I, E, 1, act, MOE_BF16, r.limit, r.alpha)
    run.plan(d.topk_idx)
    y = run.forward(d.x, d.topk_idx, d.topk_w, d.w_gate_up, d.w_down).clone()
    dx, dtw, dwgu, dwd = [t.clone() for t in run.backward(d.dy, d.x, d.topk_idx, d.topk_w,
                                                          d.w_gate_up, d.w_down)]
    torch.cuda.synchronize()
    run.check()
    # y and dx reach 11x their rms here (k = 1, weights U(0,1)): bf16 outputs
    # are held to the bound with one bf16 step of headroom
    from tests.helpers import assert_close_bf16_output
    assert_close_bf16_output("y", y.double().cpu().numpy(),
                             oracle.moe_forward(x, idx_np, w, wgu, wd, act))
    ref = oracle.moe_backward(dy, x, idx_np, w, wgu, wd, act)
    assert_close_bf16_output("dx", dx.double().cpu().numpy(), ref[0])
    assert_dw_close(dtw.cpu().numpy(), ref[1])
    for e in range(E):
        if counts[e]:
            assert_close("dw_gate_up[%d]" % e, dwgu[e].cpu().numpy(), ref[2][e])
            assert_close("dw_down[%d]" % e, dwd[e].cpu().numpy(), ref[3][e])
        else:
            assert torch.all(dwgu[e] == 0) and torch.all(dwd[e] == 0)
