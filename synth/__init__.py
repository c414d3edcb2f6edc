"""Seeded synthetic inputs for the MoE expert layer.

This module only draws random inputs: hidden states, routing (expert ids and
weights), expert weights and the upstream gradient.  It holds none of the
layer's arithmetic and is shared by the tests, the benchmark and the oracle
checks so that both sides see identical values.

Routing is input generation (the router sits above the layer): the pages take
the top-k expert ids and weights as given.  Recipes follow the workloads of
the three kernel-records pages (model dimensions from each page's workload
line); the pages do not publish their 16-case suites, so these seeded cases
stand in for them.

All random values are drawn in float32 from a torch.Generator on `device`
and then cast to the case dtype; draws happen in a fixed order (x, routing,
w_gate_up, w_down, dy) so a case is a pure function of (recipe, seed, device
type).
"""

from dataclasses import dataclass, field
import math

import torch

ACT_SWIGLU = 0
ACT_CLAMPED_GLU = 1

_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


@dataclass
class Recipe:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    act: int
    dtype: str = "bf16"
    weight_std: object = 0.02          # float, or "fan_in" for N(0, 1/sqrt(fan_in))
    routing: str = "softmax_topk_renorm"
    seed: int = 0
    limit: float = 7.0
    alpha: float = 1.702
    notes: str = ""

    def scaled(self, **kw):
        d = dict(self.__dict__)
        d.update(kw)
        return Recipe(**d)

    @property
    def Tk(self):
        return self.T * self.k


# The five workloads.  Sizes and distributions are the pages' model
# dimensions plus the value recipes stated for each case.
RECIPES = {
    "tiny_fp32": Recipe("tiny_fp32", T=64, H=128, I=128, E=8, k=2, act=ACT_SWIGLU,
                        dtype="fp32", weight_std="fan_in",
                        routing="softmax_topk_renorm", seed=0,
                        notes="tiny correctness case, fwd+bwd, finite differences"),
    "clamped_glu_fwd": Recipe("clamped_glu_fwd", T=8192, H=2880, I=2880, E=128, k=4,
                              act=ACT_CLAMPED_GLU, dtype="bf16", weight_std=0.02,
                              routing="uniform_topk_softmax", seed=1,
                              notes="dispatch-and-combine page dims (H=I=2880, 128 experts, top-4)"),
    "swiglu_fwd": Recipe("swiglu_fwd", T=4096, H=8192, I=2048, E=256, k=8,
                         act=ACT_SWIGLU, dtype="bf16", weight_std=0.02,
                         routing="softmax_topk_renorm", seed=2,
                         notes="token-repeat page dims (H=8192, 256 experts, top-8, I=2048)"),
    "swiglu_bwd": Recipe("swiglu_bwd", T=4096, H=4096, I=2048, E=256, k=8,
                         act=ACT_SWIGLU, dtype="bf16", weight_std=0.02,
                         routing="softmax_topk_renorm", seed=3,
                         notes="backward page dims (H=4096, 256 experts, top-8, I=2048)"),
    "zipf_sweep": Recipe("zipf_sweep", T=2048, H=4096, I=2048, E=256, k=8,
                         act=ACT_SWIGLU, dtype="bf16", weight_std=0.02,
                         routing="zipf", seed=4,
                         notes="load-imbalance sweep, T in {512, 2048, 8192, 16384}"),
}
ZIPF_TOKENS = (512, 2048, 8192, 16384)


@dataclass
class Case:
    recipe: Recipe
    x: torch.Tensor           # [T, H] dtype
    topk_idx: torch.Tensor    # [T, k] int32
    topk_w: torch.Tensor      # [T, k] float32
    w_gate_up: torch.Tensor   # [E, H, 2I] dtype
    w_down: torch.Tensor      # [E, I, H] dtype
    dy: torch.Tensor = None   # [T, H] dtype
    extra: dict = field(default_factory=dict)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, out_dtype):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(out_dtype)


def _routing(r, g, device):
    """Expert ids [T,k] (int32) and weights [T,k] (float32) for recipe r."""
    T, E, k = r.T, r.E, r.k
    if r.routing == "softmax_topk_renorm":
        logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
        probs = torch.softmax(logits, dim=-1)
        vals, ids = torch.topk(probs, k, dim=-1)
        w = vals / vals.sum(dim=-1, keepdim=True)
    elif r.routing == "uniform_topk_softmax":
        logits = torch.rand((T, E), generator=g, device=device, dtype=torch.float32)
        vals, ids = torch.topk(logits, k, dim=-1)
        w = torch.softmax(vals, dim=-1)
    elif r.routing == "zipf":
        # Experts are randomly ranked; rank r (1-based) has popularity
        # r^-1.2 for the first E - round(0.3 E) ranks and 0 for the rest, so
        # about 30% of experts receive no token.  Each token draws k distinct
        # experts without replacement in proportion to popularity
        # (Gumbel-top-k on log p); weights are a softmax of k N(0,1) logits.
        rank_of = torch.randperm(E, generator=g, device=device)
        n_live = E - int(round(0.3 * E))
        ranks = torch.arange(1, E + 1, device=device, dtype=torch.float32)
        logp = torch.where(ranks <= n_live, -1.2 * torch.log(ranks),
                           torch.full_like(ranks, -float("inf")))
        logp_e = logp[rank_of]                         # popularity of expert e
        u = torch.rand((T, E), generator=g, device=device, dtype=torch.float32)
        u = u.clamp_(min=1e-12, max=1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        _, ids = torch.topk(logp_e[None, :] + gumbel, k, dim=-1)
        wl = torch.randn((T, k), generator=g, device=device, dtype=torch.float32)
        w = torch.softmax(wl, dim=-1)
    elif r.routing == "uniform_ids":
        # ids uniform over experts (may repeat within a token), weights U(0,1).
        ids = torch.randint(0, E, (T, k), generator=g, device=device)
        w = torch.rand((T, k), generator=g, device=device, dtype=torch.float32)
    else:
        raise ValueError(r.routing)
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def make_case(r: Recipe, device="cpu", with_dy=True, weight_chunk=8):
    """Draw one case.  Weights are drawn expert by expert (chunks of
    `weight_chunk` experts) so that huge weight tensors need little scratch."""
    dt = _DTYPES[r.dtype]
    g = _gen(r.seed, device)
    x = _normal((r.T, r.H), 1.0, g, device, dt)
    ids, w = _routing(r, g, device)
    if r.weight_std == "fan_in":
        std_gu, std_d = 1.0 / math.sqrt(r.H), 1.0 / math.sqrt(r.I)
    else:
        std_gu = std_d = float(r.weight_std)
    wgu = torch.empty((r.E, r.H, 2 * r.I), dtype=dt, device=device)
    wd = torch.empty((r.E, r.I, r.H), dtype=dt, device=device)
    for e0 in range(0, r.E, weight_chunk):
        e1 = min(r.E, e0 + weight_chunk)
        wgu[e0:e1] = _normal((e1 - e0, r.H, 2 * r.I), std_gu, g, device, dt)
    for e0 in range(0, r.E, weight_chunk):
        e1 = min(r.E, e0 + weight_chunk)
        wd[e0:e1] = _normal((e1 - e0, r.I, r.H), std_d, g, device, dt)
    dy = _normal((r.T, r.H), 1.0, g, device, dt) if with_dy else None
    return Case(r, x, ids, w, wgu, wd, dy)


def make_biases(r: Recipe, device="cpu", std=0.5):
    """Optional per-expert biases of recipe r: (b_gate_up [E, 2I], b_down
    [E, H]) in the case dtype, N(0, std^2).  They come from their own
    generator (seed r.seed + 1000003), so drawing them leaves make_case's
    values unchanged.  b_gate_up's columns are in whatever layout the caller
    reads the gate_up weight in."""
    dt = _DTYPES[r.dtype]
    g = _gen(r.seed + 1000003, device)
    b_gate_up = _normal((r.E, 2 * r.I), std, g, device, dt)
    b_down = _normal((r.E, r.H), std, g, device, dt)
    return b_gate_up, b_down


def routing_stats(topk_idx, E):
    """(fraction of experts with no token, max count / mean count)."""
    counts = torch.bincount(topk_idx.reshape(-1).long().cpu(), minlength=E).double()
    zero = float((counts == 0).double().mean())
    mean = float(counts.mean())
    return zero, (float(counts.max()) / mean if mean > 0 else 0.0)
