"""Expert-parallel exchange on two and three CPU ranks (gloo): every rank's outputs and
its experts' weight gradients equal the single-process layer on all ranks'
tokens.

The exchange logic under test is the product's (ExpertParallelMoE: expert
ranges, the counts exchange, split sizes, the received rows' expert ids, the
return exchange, the combine and the slot-order return of d(topk w)).  The
per-step arithmetic that runs in the CUDA kernels on a GPU (plan, row
gathers, combine, the per-expert layer) is stood in for by the fp64 oracle
behind the same interface, so the comparison is exact up to fp64 rounding.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from synth import ACT_CLAMPED_GLU, ACT_SWIGLU, Recipe


class OracleOps:
    """fp64 stand-ins for the kernel steps (CPU tensors, float64 rows)."""

    def __init__(self, act):
        self.act = act

    def to_comm(self, t):
        return t

    def to_device(self, t):
        return t

    def to_host(self, t):
        return t.numpy().astype(np.int64)

    def plan(self, topk_idx, E):
        counts, offsets, perm, inv = oracle.dispatch_plan(topk_idx.numpy(), E)
        return {"counts_host": counts, "perm": torch.from_numpy(perm), "inv": torch.from_numpy(inv)}

    def gather(self, index, div, src, n):
        return src[index[:n].long() // div].clone()

    def combine(self, inv, src, T, k, like):
        return src[inv.long()].reshape(T, k, src.shape[1]).sum(dim=1)

    def expert_forward(self, x_rows, ids, w_rows, E_loc, w_gate_up, w_down, b_gate_up=None,
                       b_down=None):
        w = w_rows.reshape(-1, 1).numpy()
        y = oracle.moe_forward(x_rows.numpy(), ids.numpy(), w, w_gate_up, w_down, self.act)
        return torch.from_numpy(np.ascontiguousarray(y)), (x_rows.numpy(), ids.numpy(), w,
                                                           w_gate_up, w_down)

    def expert_backward(self, ctx, dy_rows):
        x, ids, w, wgu, wd = ctx
        dx, dw, dgu, dd = oracle.moe_backward(dy_rows.numpy(), x, ids, w, wgu, wd, self.act)
        return torch.from_numpy(dx), torch.from_numpy(dw).reshape(-1), dgu, dd


def _rank_tokens(case_args, rank):
    """This rank's tokens: (x, idx, w, dy) as float64 / int32 CPU tensors."""
    T_per, H, I, E, k, act, routing, skew = case_args
    r = Recipe("ep", T=T_per[rank], H=H, I=I, E=E, k=k, act=act, weight_std="fan_in",
               routing=routing, seed=500 + rank)
    c = synth.make_case(r)
    idx = c.topk_idx
    if skew:   # every token to the first rank's experts only
        idx = idx % (E // 2)
    return c.x.double(), idx, c.topk_w.double(), c.dy.double()


def _weights(case_args):
    T_per, H, I, E, k, act, routing, skew = case_args
    r = Recipe("ep_w", T=1, H=H, I=I, E=E, k=k, act=act, weight_std="fan_in", seed=77)
    c = synth.make_case(r)
    return c.w_gate_up.double().numpy(), c.w_down.double().numpy()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, case_args, out):
    from dispatch_gemm_combine_gb300.expert_parallel import ExpertParallelMoE, expert_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T_per, H, I, E, k, act, routing, skew = case_args
        wgu, wd = _weights(case_args)
        lo, hi = expert_range(E, world, rank)
        x, idx, w, dy = _rank_tokens(case_args, rank)
        ep = ExpertParallelMoE(E, k, OracleOps(act), group=dist.group.WORLD)
        y = ep.forward(x, idx, w, wgu[lo:hi], wd[lo:hi])
        dx, dtw, dgu, dd = ep.backward(dy)
        # the single-process layer: this rank's tokens for y / dx / d(topk w);
        # every rank's tokens for this rank's experts' weight gradients
        xn, idn, wn, dyn = x.numpy(), idx.numpy(), w.numpy(), dy.numpy()
        y_ref = oracle.moe_forward(xn, idn, wn, wgu, wd, act)
        dx_ref, dw_ref, _, _ = oracle.moe_backward(dyn, xn, idn, wn, wgu, wd, act)
        all_t = [_rank_tokens(case_args, q) for q in range(world)]
        X = np.concatenate([t[0].numpy() for t in all_t])
        IDX = np.concatenate([t[1].numpy() for t in all_t])
        W = np.concatenate([t[2].numpy() for t in all_t])
        DY = np.concatenate([t[3].numpy() for t in all_t])
        _, _, dgu_ref, dd_ref = oracle.moe_backward(DY, X, IDX, W, wgu, wd, act)

        def rel(a, b):
            a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
            n = np.linalg.norm(b)
            return float(np.linalg.norm(a - b) / n) if n > 0 else float(np.linalg.norm(a))

        out[rank] = {"y": rel(y.numpy(), y_ref), "dx": rel(dx.numpy(), dx_ref),
                     "d_topk_w": rel(dtw.numpy(), dw_ref),
                     "d_gate_up": rel(np.asarray(dgu), dgu_ref[lo:hi]),
                     "d_down": rel(np.asarray(dd), dd_ref[lo:hi]), "lo": lo, "hi": hi}
    finally:
        dist.destroy_process_group()


CASES = [
    # T per rank, H, I, E, k, act, routing, skew
    ((40, 37), 16, 24, 6, 2, ACT_SWIGLU, "softmax_topk_renorm", False),
    ((33, 50), 24, 16, 5, 3, ACT_CLAMPED_GLU, "uniform_ids", False),   # uneven ranges (2 / 3)
    ((20, 25), 16, 16, 4, 2, ACT_SWIGLU, "uniform_ids", True),          # rank 1 receives nothing
]


@pytest.mark.parametrize("case_args", CASES)
def test_expert_parallel_two_ranks_equals_single_process(case_args):
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, case_args, out), nprocs=world,
                       start_method="spawn")
    for r in range(world):
        errs = {k: v for k, v in out[r].items() if k in ("y", "dx", "d_topk_w", "d_gate_up",
                                                          "d_down")}
        assert all(v <= 1e-12 for v in errs.values()), (r, errs)
    assert out[0]["hi"] == out[1]["lo"] and out[0]["lo"] == 0 and out[1]["hi"] == case_args[3]


def test_expert_parallel_three_ranks_one_without_tokens():
    """Three ranks with uneven expert ranges (2 / 2 / 3 of 7); the middle rank
    has no tokens of its own but still owns experts that receive rows."""
    world = 3
    case_args = ((23, 0, 31), 16, 16, 7, 2, ACT_SWIGLU, "softmax_topk_renorm", False)
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, case_args, out), nprocs=world,
                       start_method="spawn")
    for r in range(world):
        errs = {k: v for k, v in out[r].items() if k in ("y", "dx", "d_topk_w", "d_gate_up",
                                                          "d_down")}
        assert all(v <= 1e-12 for v in errs.values()), (r, errs)
    assert [(out[r]["lo"], out[r]["hi"]) for r in range(world)] == [(0, 2), (2, 4), (4, 7)]


def test_expert_ranges_cover_all_experts():
    from dispatch_gemm_combine_gb300.expert_parallel import expert_range
    for E in (1, 5, 8, 128, 257):
        for world in range(1, min(E, 9) + 1):
            r = [expert_range(E, world, q) for q in range(world)]
            assert r[0][0] == 0 and r[-1][1] == E
            assert all(r[q][1] == r[q + 1][0] for q in range(world - 1))
            sizes = [b - a for a, b in r]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
