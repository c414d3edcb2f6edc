"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: values
worked by hand (tests/golden), brute force over every expert, library
routines in special cases (torch float64 functions and autograd), closed
forms, invariants, and central finite differences.  A plausible mistake in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a
missed routing weight) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import ACT_SWIGLU, ACT_CLAMPED_GLU

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def _rand_case(T, H, I, E, k, act, seed, distinct=True, scale=None):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    if distinct:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
    else:
        idx = rng.integers(0, E, size=(T, k))
    w = rng.random((T, k))
    sgu = scale if scale is not None else 1.0 / math.sqrt(H)
    sd = 1.0 / math.sqrt(I)
    wgu = rng.standard_normal((E, H, 2 * I)) * sgu
    wd = rng.standard_normal((E, I, H)) * sd
    dy = rng.standard_normal((T, H))
    return x, idx, w, wgu, wd, dy


# --------------------------------------------------------------------------
# hand-worked examples
# --------------------------------------------------------------------------

def _load_golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = [s.strip() for s in line.split("=", 1)]
        ex, name = key.split(".", 1)
        out.setdefault(ex, {})[name] = np.array([float(v) for v in val.split()])
    return out


@pytest.mark.parametrize("ex", ["ex1", "ex2"])
def test_worked_examples(ex):
    d = _load_golden()[ex]
    T, H, I, E, k = [int(v) for v in d["shape"]]
    act = int(d["act"][0])
    x = d["x"].reshape(T, H)
    idx = d["topk_idx"].astype(np.int64).reshape(T, k)
    w = d["topk_w"].reshape(T, k)
    wgu = d["w_gate_up"].reshape(E, H, 2 * I)
    wd = d["w_down"].reshape(E, I, H)
    dy = d["dy"].reshape(T, H)
    y = oracle.moe_forward(x, idx, w, wgu, wd, act)
    np.testing.assert_allclose(y.reshape(-1), d["y"], rtol=1e-14, atol=1e-14)
    if "counts" in d:
        counts, offsets, perm, inv = oracle.dispatch_plan(idx, E)
        assert list(counts) == list(d["counts"].astype(int))
        assert list(offsets) == list(d["offsets"].astype(int))
        assert list(perm) == list(d["perm"].astype(int))
        assert list(inv) == list(d["inv"].astype(int))
    dx, dw, dwgu, dwd = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    np.testing.assert_allclose(dw.reshape(-1), d["d_topk_w"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dwd.reshape(-1), d["dw_down"], rtol=1e-14, atol=1e-14)
    if "dw_gate_up" in d:
        np.testing.assert_allclose(dwgu.reshape(-1), d["dw_gate_up"], atol=0)
    if "dx" in d:
        np.testing.assert_allclose(dx.reshape(-1), d["dx"], atol=0)


# --------------------------------------------------------------------------
# dispatch plan
# --------------------------------------------------------------------------

def _plan_by_counting(idx, E):
    """Position of every slot by counting, written independently: a slot's
    row is the number of slots of smaller expert id plus the number of
    earlier slots of the same expert."""
    flat = [int(v) for v in np.asarray(idx).reshape(-1)]
    n = len(flat)
    inv = []
    for s in range(n):
        before = sum(1 for q in range(n) if flat[q] < flat[s])
        same_earlier = sum(1 for q in range(s) if flat[q] == flat[s])
        inv.append(before + same_earlier)
    perm = [0] * n
    for s, r in enumerate(inv):
        perm[r] = s
    counts = [flat.count(e) for e in range(E)]
    return counts, perm, inv


@pytest.mark.parametrize("T,k,E,seed,distinct", [
    (13, 3, 5, 0, True), (20, 2, 7, 1, False), (1, 1, 1, 2, True),
    (9, 4, 4, 3, True), (30, 1, 16, 4, False), (0, 2, 3, 5, True)])
def test_plan_matches_counting(T, k, E, seed, distinct):
    rng = np.random.default_rng(seed)
    if distinct:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
    else:
        idx = rng.integers(0, E, size=(T, k))
    counts, offsets, perm, inv = oracle.dispatch_plan(idx, E)
    c2, p2, i2 = _plan_by_counting(idx, E)
    assert list(counts) == c2
    assert list(perm) == p2
    assert list(inv) == i2
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert list(np.diff(offsets)) == c2


def test_plan_invariants_skewed():
    rng = np.random.default_rng(7)
    E, T, k = 64, 500, 6
    # heavily skewed: most slots on expert 3, many experts empty
    idx = np.where(rng.random((T, k)) < 0.7, 3, rng.integers(0, 10, size=(T, k)))
    counts, offsets, perm, inv = oracle.dispatch_plan(idx, E)
    flat = idx.reshape(-1)
    assert counts.sum() == T * k
    assert sorted(perm.tolist()) == list(range(T * k))
    assert np.all(inv[perm] == np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)
    assert (counts == 0).sum() >= E - 10


def test_plan_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.dispatch_plan(np.array([[0, 5]]), 5)
    with pytest.raises(ValueError):
        oracle.dispatch_plan(np.array([[-1, 0]]), 5)


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------

def test_swiglu_matches_torch_silu():
    rng = np.random.default_rng(0)
    g = rng.standard_normal(1000) * 4
    u = rng.standard_normal(1000) * 4
    ref = (F.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(oracle.activation(g, u, ACT_SWIGLU), ref, rtol=1e-14, atol=1e-15)


def test_clamped_glu_closed_forms():
    L, al = 7.0, 1.702
    # g = 0 gives zero whatever u is
    assert oracle.activation(0.0, 123.0, ACT_CLAMPED_GLU) == 0.0
    # both clamps active from above: (7+1) * 7 * sigmoid(11.914)
    sig = 1.0 / (1.0 + math.exp(-11.914))
    for g, u in [(7.0, 7.0), (9.0, 50.0), (1e6, 7.5)]:
        assert abs(oracle.activation(g, u, ACT_CLAMPED_GLU) - 56.0 * sig) < 1e-12
    # up clamped from below: (-7+1) * g * sigmoid(alpha g)
    for g in [-3.0, 0.5, 2.0]:
        ref = -6.0 * g / (1.0 + math.exp(-al * g))
        assert abs(oracle.activation(g, -9.0, ACT_CLAMPED_GLU) - ref) < 1e-12
    # unclamped region equals torch's clamp/sigmoid composition (library)
    rng = np.random.default_rng(1)
    g = rng.standard_normal(500) * 5
    u = rng.standard_normal(500) * 5
    tg, tu = torch.from_numpy(g), torch.from_numpy(u)
    gate = torch.clamp(tg, max=L)
    ref = (torch.clamp(tu, -L, L) + 1) * gate * torch.sigmoid(al * gate)
    np.testing.assert_allclose(oracle.activation(g, u, ACT_CLAMPED_GLU), ref.numpy(),
                               rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("act", [ACT_SWIGLU, ACT_CLAMPED_GLU])
def test_activation_grad_vs_autograd(act):
    rng = np.random.default_rng(2)
    g = rng.standard_normal(2000) * 6
    u = rng.standard_normal(2000) * 6
    # stay away from the clamp kinks, where the derivative is one-sided
    keep = (np.abs(g - 7) > 1e-3) & (np.abs(np.abs(u) - 7) > 1e-3)
    g, u = g[keep], u[keep]
    tg = torch.tensor(g, requires_grad=True)
    tu = torch.tensor(u, requires_grad=True)
    if act == ACT_SWIGLU:
        a = F.silu(tg) * tu
    else:
        gate = torch.clamp(tg, max=7.0)
        a = (torch.clamp(tu, -7.0, 7.0) + 1) * gate * torch.sigmoid(1.702 * gate)
    a.sum().backward()
    dg, du = oracle.activation_grad(g, u, act)
    np.testing.assert_allclose(dg, tg.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(du, tu.grad.numpy(), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

def _torch_act(g, u, act):
    if act == ACT_SWIGLU:
        return F.silu(g) * u
    gate = torch.clamp(g, max=7.0)
    return (torch.clamp(u, -7.0, 7.0) + 1) * gate * torch.sigmoid(1.702 * gate)


def _dense_bruteforce(x, idx, w, wgu, wd, act):
    """Every expert applied to every token, masked by routing, token by token
    (torch float64, no grouping)."""
    T, H = x.shape
    E, _, I2 = wgu.shape
    I = I2 // 2
    y = torch.zeros((T, H), dtype=torch.float64)
    tx, twgu, twd = map(torch.from_numpy, (x, wgu, wd))
    for t in range(T):
        for e in range(E):
            c = sum(w[t, j] for j in range(idx.shape[1]) if idx[t, j] == e)
            h = tx[t] @ twgu[e]
            a = _torch_act(h[:I], h[I:], act)
            y[t] += float(c) * (a @ twd[e])
    return y.numpy()


@pytest.mark.parametrize("act", [ACT_SWIGLU, ACT_CLAMPED_GLU])
@pytest.mark.parametrize("distinct", [True, False])
def test_forward_dense_bruteforce(act, distinct):
    x, idx, w, wgu, wd, _ = _rand_case(9, 12, 8, 5, 3, act, seed=3, distinct=distinct,
                                       scale=1.5 if act == ACT_CLAMPED_GLU else None)
    y = oracle.moe_forward(x, idx, w, wgu, wd, act)
    yb = _dense_bruteforce(x, idx, w, wgu, wd, act)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max())


@pytest.mark.parametrize("act", [ACT_SWIGLU, ACT_CLAMPED_GLU])
def test_k1_w1_reduces_to_single_ffn(act):
    x, idx, w, wgu, wd, _ = _rand_case(17, 10, 6, 4, 1, act, seed=4)
    w = np.ones_like(w)
    y = oracle.moe_forward(x, idx, w, wgu, wd, act)
    tx = torch.from_numpy(x)
    for t in range(17):
        e = int(idx[t, 0])
        lin_g = F.linear(tx[t:t + 1], torch.from_numpy(wgu[e][:, :6].T.copy()))
        lin_u = F.linear(tx[t:t + 1], torch.from_numpy(wgu[e][:, 6:].T.copy()))
        ref = F.linear(_torch_act(lin_g, lin_u, act), torch.from_numpy(wd[e].T.copy()))
        np.testing.assert_allclose(y[t], ref.numpy()[0], rtol=1e-12, atol=1e-13)


def test_linearity_in_routing_weights():
    x, idx, w, wgu, wd, _ = _rand_case(11, 8, 6, 6, 3, ACT_SWIGLU, seed=5)
    w2 = np.random.default_rng(9).random(w.shape)
    a, b = 0.7, -1.3
    lhs = oracle.moe_forward(x, idx, a * w + b * w2, wgu, wd, ACT_SWIGLU)
    rhs = a * oracle.moe_forward(x, idx, w, wgu, wd, ACT_SWIGLU) + \
        b * oracle.moe_forward(x, idx, w2, wgu, wd, ACT_SWIGLU)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    zero = oracle.moe_forward(x, idx, 0 * w, wgu, wd, ACT_SWIGLU)
    assert np.all(zero == 0)


def test_relabel_and_token_permutation_equivariance():
    x, idx, w, wgu, wd, _ = _rand_case(10, 8, 5, 6, 2, ACT_CLAMPED_GLU, seed=6, scale=1.0)
    y = oracle.moe_forward(x, idx, w, wgu, wd, ACT_CLAMPED_GLU)
    rng = np.random.default_rng(11)
    sigma = rng.permutation(6)              # new id of old expert e is sigma[e]
    wgu2 = np.empty_like(wgu)
    wd2 = np.empty_like(wd)
    wgu2[sigma] = wgu
    wd2[sigma] = wd
    y2 = oracle.moe_forward(x, sigma[idx], w, wgu2, wd2, ACT_CLAMPED_GLU)
    np.testing.assert_allclose(y2, y, rtol=1e-13, atol=1e-13)
    pt = rng.permutation(10)
    y3 = oracle.moe_forward(x[pt], idx[pt], w[pt], wgu, wd, ACT_CLAMPED_GLU)
    np.testing.assert_allclose(y3, y[pt], rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def _autograd_dense(x, idx, w, wgu, wd, dy, act):
    """torch float64 autograd through the dense masked formulation."""
    T, H = x.shape
    E = wgu.shape[0]
    I = wd.shape[1]
    tx = torch.tensor(x, requires_grad=True)
    tw = torch.tensor(w, requires_grad=True)
    tgu = torch.tensor(wgu, requires_grad=True)
    td = torch.tensor(wd, requires_grad=True)
    onehot = F.one_hot(torch.from_numpy(idx).long(), E).double()       # [T,k,E]
    coef = (onehot * tw[:, :, None]).sum(1)                            # [T,E]
    y = torch.zeros((T, H), dtype=torch.float64)
    for e in range(E):
        h = tx @ tgu[e]
        y = y + coef[:, e:e + 1] * (_torch_act(h[:, :I], h[:, I:], act) @ td[e])
    (y * torch.from_numpy(dy)).sum().backward()
    return tx.grad.numpy(), tw.grad.numpy(), tgu.grad.numpy(), td.grad.numpy()


@pytest.mark.parametrize("act", [ACT_SWIGLU, ACT_CLAMPED_GLU])
def test_backward_vs_autograd_dense(act):
    x, idx, w, wgu, wd, dy = _rand_case(12, 10, 7, 5, 2, act, seed=8,
                                        scale=2.0 if act == ACT_CLAMPED_GLU else None)
    dx, dw, dwgu, dwd = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    rx, rw, rgu, rd = _autograd_dense(x, idx, w, wgu, wd, dy, act)
    for a, b in [(dx, rx), (dw, rw), (dwgu, rgu), (dwd, rd)]:
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11 * max(1.0, np.abs(b).max()))


def _fd_check(f, arr, coords, analytic, h=1e-5, tol=1e-6):
    scale = np.sqrt(np.mean(analytic ** 2)) + 1e-300
    for c in coords:
        old = arr[c]
        arr[c] = old + h
        fp = f()
        arr[c] = old - h
        fm = f()
        arr[c] = old
        fd = (fp - fm) / (2 * h)
        an = analytic[c]
        assert abs(fd - an) <= tol * max(abs(an), scale), (c, fd, an)


def _fd_direction(f, arr, analytic, rng, h=1e-5, tol=1e-6):
    d = rng.standard_normal(arr.shape)
    d /= np.linalg.norm(d)
    old = arr.copy()
    arr += h * d
    fp = f()
    arr[...] = old - h * d
    fm = f()
    arr[...] = old
    fd = (fp - fm) / (2 * h)
    an = float(np.sum(analytic * d))
    assert abs(fd - an) <= tol * max(abs(an), np.linalg.norm(analytic) * 1e-3), (fd, an)


def _random_coords(shape, n, rng):
    return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(n)]


def test_backward_finite_differences_tiny_fp32_recipe():
    """fp64 central differences at the tiny case's size (T=64, H=I=128, E=8,
    top-2, SwiGLU): all 128 routing weights, 64 random coordinates of each
    other tensor, and 8 random unit directions per tensor."""
    x, idx, w, wgu, wd, dy = _rand_case(64, 128, 128, 8, 2, ACT_SWIGLU, seed=0)
    act = ACT_SWIGLU
    dx, dw, dwgu, dwd = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    L = lambda: float(np.sum(dy * oracle.moe_forward(x, idx, w, wgu, wd, act)))
    rng = np.random.default_rng(1)
    _fd_check(L, w, [(t, j) for t in range(64) for j in range(2)], dw)
    _fd_check(L, x, _random_coords(x.shape, 64, rng), dx)
    _fd_check(L, wgu, _random_coords(wgu.shape, 64, rng), dwgu)
    _fd_check(L, wd, _random_coords(wd.shape, 64, rng), dwd)
    for arr, an in [(w, dw), (x, dx), (wgu, dwgu), (wd, dwd)]:
        for _ in range(8):
            _fd_direction(L, arr, an, rng)


def test_backward_finite_differences_clamped():
    """Clamped GLU with weights scaled so both clamps bind on many entries;
    coordinates whose pre-activations sit within 1e-4 of a kink are skipped
    (the central difference straddles the kink there)."""
    act = ACT_CLAMPED_GLU
    x, idx, w, wgu, wd, dy = _rand_case(16, 12, 10, 4, 2, act, seed=2, scale=3.0)
    h1 = np.stack([x[t] @ wgu[idx[t, j]] for t in range(16) for j in range(2)])
    assert (h1[:, :10] > 7).mean() > 0.05 and (np.abs(h1[:, 10:]) > 7).mean() > 0.05
    dx, dw, dwgu, dwd = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    L = lambda: float(np.sum(dy * oracle.moe_forward(x, idx, w, wgu, wd, act)))
    h = 1e-6
    # a perturbation of size h moves pre-activations by at most h * max|coef|;
    # check that none of them is within that distance of a kink
    margin = np.min(np.concatenate([np.abs(h1[:, :10] - 7).ravel(),
                                    np.abs(np.abs(h1[:, 10:]) - 7).ravel()]))
    assert margin > 1e-4
    rng = np.random.default_rng(3)
    _fd_check(L, w, [(t, j) for t in range(16) for j in range(2)], dw, h=h, tol=1e-5)
    _fd_check(L, wd, _random_coords(wd.shape, 64, rng), dwd, h=h, tol=1e-5)
    _fd_check(L, wgu, _random_coords(wgu.shape, 64, rng), dwgu, h=h, tol=1e-5)
    _fd_check(L, x, _random_coords(x.shape, 64, rng), dx, h=h, tol=1e-5)


@pytest.mark.parametrize("act", [ACT_SWIGLU, ACT_CLAMPED_GLU])
def test_backward_exact_identities(act):
    x, idx, w, wgu, wd, dy = _rand_case(40, 16, 12, 6, 3, act, seed=12)
    y = oracle.moe_forward(x, idx, w, wgu, wd, act)
    dx, dw, dwgu, dwd = oracle.moe_backward(dy, x, idx, w, wgu, wd, act)
    ly = float(np.sum(dy * y))
    # y is linear in the routing weights and in the down weights
    assert abs(float(np.sum(w * dw)) - ly) < 1e-11 * max(1, abs(ly))
    assert abs(float(np.sum(wd * dwd)) - ly) < 1e-11 * max(1, abs(ly))
    if act == ACT_SWIGLU:
        # a = silu(g) * u is linear in u, hence in the up weights
        I = wd.shape[1]
        assert abs(float(np.sum(wgu[:, :, I:] * dwgu[:, :, I:])) - ly) < 1e-11 * max(1, abs(ly))


def test_backward_empty_experts_and_subset():
    x, idx, w, wgu, wd, dy = _rand_case(8, 6, 4, 10, 2, ACT_SWIGLU, seed=13)
    idx = idx % 3                                  # experts 3..9 receive nothing
    dx, dw, dwgu, dwd = oracle.moe_backward(dy, x, idx, w, wgu, wd, ACT_SWIGLU)
    assert np.all(dwgu[3:] == 0) and np.all(dwd[3:] == 0)
    sx, sw, sgu, sd = oracle.moe_backward(dy, x, idx, w, wgu, wd, ACT_SWIGLU, experts=[1, 5])
    np.testing.assert_array_equal(sgu[1], dwgu[1])
    np.testing.assert_array_equal(sd[5], dwd[5])


# ------------------------------------------------------------------- router
def _route_by_selection(z, k):
    """Top-k by k passes of 'largest remaining logit, lowest id on ties'."""
    T, E = z.shape
    idx = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        taken = set()
        for j in range(k):
            best = None
            for e in range(E):
                if e in taken:
                    continue
                if best is None or z[t, e] > z[t, best]:
                    best = e
            idx[t, j] = best
            taken.add(best)
    return idx


@pytest.mark.parametrize("T,E,k,seed", [(40, 8, 2, 0), (25, 16, 5, 1), (12, 7, 7, 2), (30, 32, 8, 3)])
def test_route_selection_bruteforce(T, E, k, seed):
    rng = np.random.default_rng(seed)
    z = rng.normal(size=(T, E)).astype(np.float32)
    z[:, : E // 2] = np.round(z[:, : E // 2])          # many exact ties
    idx, w = oracle.route(z, k)
    assert np.array_equal(idx, _route_by_selection(z.astype(np.float64), k))


def test_route_weights_are_renormalised_full_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(4)
    z = rng.normal(size=(50, 64)) * 3.0
    idx, w = oracle.route(z, 6)
    p = softmax(z, axis=1)
    sel = np.take_along_axis(p, idx, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)
    # weights follow the order of the logits and sum to one
    assert np.all(np.diff(w, axis=1) <= 0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)


def test_route_special_cases():
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    z = rng.normal(size=(9, 12))
    idx, w = oracle.route(z, 12)                        # k = E: every expert, full softmax
    assert all(sorted(r.tolist()) == list(range(12)) for r in idx)
    np.testing.assert_allclose(w, np.take_along_axis(softmax(z, axis=1), idx, axis=1), rtol=1e-12)
    i2, w2 = oracle.route(z + 123.25, 4)                # shift invariance
    i1, w1 = oracle.route(z, 4)
    assert np.array_equal(i1, i2)
    np.testing.assert_allclose(w1, w2, rtol=1e-12)
    ie, we = oracle.route(np.zeros((3, 10)), 4)         # all equal: lowest ids, equal weights
    assert np.array_equal(ie, np.tile(np.arange(4), (3, 1)))
    np.testing.assert_allclose(we, 0.25)
    i0, w0 = oracle.route(np.zeros((2, 1)), 1)          # one expert
    assert np.array_equal(i0, [[0], [0]]) and np.all(w0 == 1.0)
    counts, _, _, _ = oracle.dispatch_plan(i1, 12)      # routed ids feed the plan
    assert counts.sum() == 9 * 4


def test_gate_up_layouts():
    # interleaved [g0 u0 g1 u1 g2 u2] -> concatenated [g0 g1 g2 u0 u1 u2]
    w = np.array([[10., 20., 11., 21., 12., 22.]])
    assert np.array_equal(oracle.gate_up_concatenated(w, 1), [[10., 11., 12., 20., 21., 22.]])
    assert np.array_equal(oracle.gate_up_concatenated(w, 0), w)
    rng = np.random.default_rng(6)
    c = rng.normal(size=(3, 5, 8))
    assert np.array_equal(oracle.gate_up_concatenated(oracle.gate_up_in_layout(c, 1), 1), c)
    assert np.array_equal(oracle.gate_up_in_layout(oracle.gate_up_concatenated(c, 1), 1), c)


def test_biases_finite_differences_and_identities():
    """Per-expert biases: fp64 central differences for every gradient the
    biases add or change, the exact identity <db_down, b_down> = <dy, y> -
    <dy, y without b_down> (y is affine in b_down), and zero biases giving
    the bias-free layer."""
    x, idx, w, wgu, wd, dy = _rand_case(12, 16, 10, 4, 2, ACT_CLAMPED_GLU, seed=8)
    rng = np.random.default_rng(9)
    E, I, H = wd.shape
    bgu = rng.normal(size=(E, 2 * I)) * 0.5
    bd = rng.normal(size=(E, H)) * 0.5
    act = ACT_CLAMPED_GLU
    dx, dw, dwgu, dwd, dbgu, dbd = oracle.moe_backward(dy, x, idx, w, wgu, wd, act,
                                                         b_gate_up=bgu, b_down=bd)
    L = lambda: float(np.sum(dy * oracle.moe_forward(x, idx, w, wgu, wd, act,
                                                      b_gate_up=bgu, b_down=bd)))
    _fd_check(L, bgu, [(e, c) for e in range(E) for c in range(2 * I)], dbgu)
    _fd_check(L, bd, [(e, c) for e in range(E) for c in range(H)], dbd)
    _fd_check(L, w, [(t, j) for t in range(12) for j in range(2)], dw)
    _fd_check(L, x, _random_coords(x.shape, 24, rng), dx)
    _fd_check(L, wgu, _random_coords(wgu.shape, 24, rng), dwgu)
    y_b = oracle.moe_forward(x, idx, w, wgu, wd, act, b_gate_up=bgu, b_down=bd)
    y_nob = oracle.moe_forward(x, idx, w, wgu, wd, act, b_gate_up=bgu)
    assert np.isclose(np.sum(dbd * bd), np.sum(dy * (y_b - y_nob)), rtol=1e-12)
    y0 = oracle.moe_forward(x, idx, w, wgu, wd, act, b_gate_up=0 * bgu, b_down=0 * bd)
    assert np.array_equal(y0, oracle.moe_forward(x, idx, w, wgu, wd, act))
