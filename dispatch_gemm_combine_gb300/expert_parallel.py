"""Expert-parallel execution of the MoE expert layer across ranks.

The backward page ("MoE expert parallel execution backward", title) names
expert-parallel execution: the experts are spread over devices, every
device keeps its own tokens, and a token's rows travel to the devices that
hold its experts and back.  Here every rank owns a contiguous range of
experts, [E r / R, E (r+1) / R) on rank r of R, and holds those experts'
weights and weight gradients only.

Forward on each rank:
  1. dispatch plan of the local tokens over all E experts (moe_plan);
  2. dispatch: gather the token rows and routing weights into the plan's
     expert-grouped order (moe_gather_rows); the rows bound for rank q are
     then the one contiguous segment of q's experts;
  3. all-to-all of the per-expert counts, then of the row segments and the
     routing weights: every rank receives, from every rank, the rows of its
     own experts, in (source rank, expert, slot) order;
  4. expert computation on the received rows: the layer itself with one
     choice per row (k = 1), the received routing weight scaling each row's
     output, fp32 results (moe_ffn_fwd with out_fp32);
  5. the mirrored all-to-all brings the scaled expert outputs back into the
     source's expert-grouped order;
  6. combine: y[t] = sum_j rows[inv[t k + j]] in fp32, j ascending
     (moe_combine_rows): deterministic, no atomics.
Backward mirrors it: dy is dispatched like x, the owners run the layer's
backward on their rows (dx rows, d(topk w) per row, their experts' weight
gradients), the dx rows and d(topk w) values come back and are combined
(dx) or put back in slot order (d(topk w)).  Exchanged row data lands in
ordinary local buffers before any kernel reads it; no kernel reads another
device's memory.

The arithmetic runs in the library's kernels through `CudaOps`; the
exchange is torch.distributed's all_to_all_single (NCCL between GPUs).  The
split sizes of a collective must be known on the host, so the per-expert
counts come to the host once per call; the small index bookkeeping on them
(split sizes, each received row's local expert id) runs there.  `ops` may
be any object with CudaOps's methods (the CPU tests of the exchange logic
pass one built on the fp64 reference).
"""

import numpy as np
import torch

from . import (MOE_BF16, Shape, alloc_plan, combine_rows, gather_rows, plan, workspace,
               check_device_error)
from .runner import LayerRunner


def expert_range(E, world, rank):
    """Experts [lo, hi) owned by `rank` of `world`: contiguous, sizes differing
    by at most one."""
    return rank * E // world, (rank + 1) * E // world


class _Exchange:
    """all_to_all of row blocks over a process group (group None: one rank,
    the exchange is the identity)."""

    def __init__(self, group):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        if group is None:
            self.rank, self.world = 0, 1
        else:
            self.rank = dist.get_rank(group)
            self.world = dist.get_world_size(group)

    def rows(self, send, send_splits, recv_splits):
        """Rows [sum(send_splits), ...] -> rows [sum(recv_splits), ...]."""
        if self.world == 1:
            return send
        out = send.new_empty((int(sum(recv_splits)),) + tuple(send.shape[1:]))
        self.dist.all_to_all_single(out, send.contiguous(), [int(v) for v in recv_splits],
                                    [int(v) for v in send_splits], group=self.group)
        return out


class ExpertParallelMoE:
    """The MoE expert layer with the experts spread over the ranks of `group`.

    E experts in all, k choices per token.  forward() takes this rank's tokens
    (x [T,H], topk_idx [T,k] of global expert ids, topk_w [T,k]) and this
    rank's experts' weights (w_gate_up [E_loc,H,2I], w_down [E_loc,I,H]);
    backward() returns (dx, d_topk_w, dw_gate_up, dw_down) with the weight
    gradients of this rank's experts, summed over every rank's tokens."""

    def __init__(self, E, k, ops, group=None):
        self.E, self.k, self.ops = E, k, ops
        self.x = _Exchange(group)
        self.rank, self.world = self.x.rank, self.x.world
        if E < self.world:
            raise ValueError("expert parallelism needs at least one expert per rank "
                             "(E=%d, %d ranks)" % (E, self.world))
        self.lo, self.hi = expert_range(E, self.world, self.rank)
        self.E_loc = self.hi - self.lo
        self._ctx = None

    def _bounds(self):
        return [expert_range(self.E, self.world, q) for q in range(self.world)]

    def forward(self, x, topk_idx, topk_w, w_gate_up, w_down, b_gate_up=None, b_down=None):
        """y [T,H] for this rank's tokens.  b_gate_up [E_loc,2I] / b_down
        [E_loc,H]: the optional per-expert biases of this rank's experts."""
        ops, k = self.ops, self.k
        T = topk_idx.shape[0]
        Tk = T * k
        p = ops.plan(topk_idx, self.E)
        counts = np.asarray(p["counts_host"], dtype=np.int64)
        # dispatch into the expert-grouped order: token rows and routing weights
        xs = ops.gather(p["perm"], k, x, Tk)
        ws = ops.gather(p["perm"], 1, topk_w.reshape(-1, 1), Tk)
        send = [int(counts[a:b].sum()) for a, b in self._bounds()]
        # every rank's counts of this rank's experts: rank p sends its whole
        # count vector, split by the owners' expert ranges
        cnt = ops.to_comm(torch.from_numpy(counts))
        rc = self.x.rows(cnt, [b - a for a, b in self._bounds()], [self.E_loc] * self.world)
        recv_counts = ops.to_host(rc).reshape(self.world, self.E_loc)
        recv = recv_counts.sum(axis=1)
        xr = self.x.rows(xs, send, recv)
        wr = self.x.rows(ws, send, recv)
        # local expert id of every received row: (source, expert, slot) order
        ids = np.repeat(np.tile(np.arange(self.E_loc, dtype=np.int32), self.world),
                        recv_counts.reshape(-1))
        ids = ops.to_device(torch.from_numpy(ids.reshape(-1, 1)))
        yr, ctx = ops.expert_forward(xr, ids, wr, self.E_loc, w_gate_up, w_down, b_gate_up,
                                     b_down)
        ys = self.x.rows(yr, recv, send)
        y = ops.combine(p["inv"], ys, T, k, like=x)
        self._ctx = (p, send, recv, ctx, T)
        return y

    def backward(self, dy):
        """(dx, d_topk_w, dw_gate_up, dw_down) and, with biases, (db_gate_up,
        db_down) of this rank's experts."""
        if self._ctx is None:
            raise RuntimeError("backward() needs a forward() first")
        ops, k = self.ops, self.k
        p, send, recv, ctx, T = self._ctx
        Tk = T * k
        dys = ops.gather(p["perm"], k, dy, Tk)
        dyr = self.x.rows(dys, send, recv)
        g = ops.expert_backward(ctx, dyr)
        dxr, dwr = g[0], g[1]
        dxs = self.x.rows(dxr, recv, send)
        dws = self.x.rows(dwr.reshape(-1, 1), recv, send)
        dx = ops.combine(p["inv"], dxs, T, k, like=dy)
        d_topk_w = ops.gather(p["inv"], 1, dws, Tk).reshape(T, k)
        self._ctx = None
        return (dx, d_topk_w) + tuple(g[2:])


class CudaOps:
    """The steps of the expert-parallel layer on the GPU, through the C ABI.
    Tensors live on `device`; the collectives run on the same device (NCCL)."""

    def __init__(self, H, I, act, dtype=MOE_BF16, clamp_limit=7.0, alpha=1.702, device="cuda",
                 gate_up_layout=0):
        self.H, self.I, self.act, self.dtype = H, I, act, dtype
        self.limit, self.alpha, self.device = clamp_limit, alpha, device
        self.layout = gate_up_layout
        self._run = None   # the owner-side buffers, kept while the row count repeats

    def to_comm(self, t):
        return t.to(self.device)

    def to_device(self, t):
        return t.to(self.device)

    def to_host(self, t):
        return t.cpu().numpy().astype(np.int64)

    def plan(self, topk_idx, E):
        T, k = topk_idx.shape
        shape = Shape(T, self.H, self.I, E, k, self.act, self.dtype, self.limit, self.alpha)
        pt, ps = alloc_plan(shape, self.device)
        ws = workspace(shape, 0, self.device)
        plan(shape, topk_idx, ps, ws)
        check_device_error(ws)
        pt["counts_host"] = pt["counts"].cpu().numpy()
        return pt

    def gather(self, index, div, src, n):
        dst = torch.empty((n,) + tuple(src.shape[1:]), dtype=src.dtype, device=self.device)
        if n:
            gather_rows(index[:n], div, src.contiguous(), dst)
        return dst

    def combine(self, inv, src, T, k, like):
        # (only T, H, k, the storage dtype and out_fp32 matter to the combine)
        shape = Shape(T, self.H, self.I, k, k, self.act, self.dtype, self.limit, self.alpha,
                      out_fp32=like.dtype == torch.float32)
        dst = torch.empty((T, self.H), dtype=like.dtype, device=self.device)
        if T:
            combine_rows(shape, inv, src.contiguous(), dst)
        return dst

    def expert_forward(self, x_rows, ids, w_rows, E_loc, w_gate_up, w_down, b_gate_up=None,
                       b_down=None):
        n = x_rows.shape[0]
        key = (n, max(E_loc, 1))
        if self._run is None or self._run[0] != key:
            self._run = (key, LayerRunner(n, self.H, self.I, key[1], 1, self.act, self.dtype,
                                          self.limit, self.alpha, device=self.device,
                                          gate_up_layout=self.layout, out_fp32=True))
        run = self._run[1]
        ctx = (run, x_rows, ids, w_rows.reshape(-1, 1).contiguous(), w_gate_up, w_down, b_gate_up,
               b_down)
        if n:
            run.plan(ids)
            run.forward(x_rows, ids, ctx[3], w_gate_up, w_down, b_gate_up=b_gate_up,
                        b_down=b_down)
        return run.y, ctx

    def expert_backward(self, ctx, dy_rows):
        run, x_rows, ids, w_rows, w_gate_up, w_down, b_gate_up, b_down = ctx
        g = run.backward(dy_rows.contiguous(), x_rows, ids, w_rows, w_gate_up, w_down,
                         b_gate_up=b_gate_up, b_down=b_down)
        run.check()
        return (g[0], g[1].reshape(-1)) + tuple(g[2:])
