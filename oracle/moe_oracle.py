"""fp64 CPU oracle for the MoE expert layer (dispatch -> expert FFN -> combine).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test suite, the package smoke check and the
CPU-baseline leg of the benchmark use it.  It shares no code, table or helper
with the CUDA library; it imports numpy and nothing else.

Sources (kernel-records pages on the subject):
  * "Sparse expert dispatch and combine", description: experts are processed
    one after another; the tokens routed to an expert are extracted, passed
    through a gate_up projection, a gated GLU with clamping and a down
    projection, and scattered back with an accumulating index add.
  * "MoE training token repeat and expert computation", description: each
    token is repeated num_experts_per_tok times, each expert picks its rows by
    masked indexing and applies a SwiGLU FFN, the routing weights scale the
    expert outputs, and the k outputs of a token are summed.
  * "MoE expert parallel execution backward", description: gradients for
    hidden_states, topk_weights, gate_weights, up_weights and down_weights.

Conventions (readings where the pages are silent):
  * fused gate_up weight Wgu[e] has shape [H, 2I]; gate = columns [0, I),
    up = columns [I, 2I); down weight Wd[e] has shape [I, H]; y = x @ W.
  * slot s = t*k + j is the j-th routing choice of token t.
  * clamped GLU (the pages name the clamp but no constants): gate = min(g, L),
    up = clamp(u, -L, L), a = (up + 1) * gate * sigmoid(alpha * gate), with
    L = 7.0 and alpha = 1.702.  Its derivative at the clamp boundaries is
    taken with inclusive masks (g <= L, -L <= u <= L).
  * SwiGLU: a = silu(g) * u.
  * the routing weight scales the expert output after the down projection.

The router step (route) turns logits into top-k ids and weights; the layer
itself takes ids and weights as given.

Every computation is carried out in float64 on values converted exactly from
the caller's inputs.  Parity status: every function below is pinned by the
CPU tests (brute force, closed forms, library special cases, finite
differences, exact identities); none is "parity unpinned".
"""

import numpy as np

ACT_SWIGLU = 0
ACT_CLAMPED_GLU = 1

CLAMP_LIMIT = 7.0
CLAMP_ALPHA = 1.702


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def sigmoid(z):
    """Logistic function 1 / (1 + exp(-z)) in float64."""
    z = _f64(z)
    return 1.0 / (1.0 + np.exp(-z))


def activation(g, u, act, limit=CLAMP_LIMIT, alpha=CLAMP_ALPHA):
    """Gated activation a(g, u).

    SwiGLU (the token-repeat page's "SwiGLU FFN"): a = g * sigmoid(g) * u.
    Clamped GLU (the dispatch-and-combine page's "gated GLU with clamping"):
    gate = min(g, limit), up = clamp(u, -limit, limit),
    a = (up + 1) * gate * sigmoid(alpha * gate).
    """
    g = _f64(g)
    u = _f64(u)
    if act == ACT_SWIGLU:
        return g * sigmoid(g) * u
    if act == ACT_CLAMPED_GLU:
        gate = np.minimum(g, limit)
        up = np.clip(u, -limit, limit)
        return (up + 1.0) * gate * sigmoid(alpha * gate)
    raise ValueError("unknown activation %r" % (act,))


def activation_grad(g, u, act, limit=CLAMP_LIMIT, alpha=CLAMP_ALPHA):
    """Partial derivatives (da/dg, da/du) of `activation`, by calculus.

    SwiGLU: da/dg = u * s * (1 + g * (1 - s)) with s = sigmoid(g);
            da/du = g * s.
    Clamped GLU: with gc = min(g, L), uc = clamp(u, -L, L), s = sigmoid(alpha*gc),
            da/dg = [g <= L] * (uc + 1) * (s + alpha * gc * s * (1 - s));
            da/du = [-L <= u <= L] * gc * s.
    """
    g = _f64(g)
    u = _f64(u)
    if act == ACT_SWIGLU:
        s = sigmoid(g)
        return u * s * (1.0 + g * (1.0 - s)), g * s
    if act == ACT_CLAMPED_GLU:
        gc = np.minimum(g, limit)
        uc = np.clip(u, -limit, limit)
        s = sigmoid(alpha * gc)
        dg = np.where(g <= limit, (uc + 1.0) * (s + alpha * gc * s * (1.0 - s)), 0.0)
        du = np.where((u >= -limit) & (u <= limit), gc * s, 0.0)
        return dg, du
    raise ValueError("unknown activation %r" % (act,))


def gate_up_concatenated(w_gate_up, layout):
    """The fused gate_up weight [..., 2I] in the concatenated layout (gate =
    columns [0, I), up = [I, 2I)), the layout every function here takes.
    layout 0 is that layout already; layout 1 interleaves the two (gate =
    the even columns, up = the odd ones).  The pages fix neither."""
    w = _f64(w_gate_up)
    if layout == 0:
        return w
    return np.concatenate([w[..., 0::2], w[..., 1::2]], axis=-1)


def gate_up_in_layout(w_concat, layout):
    """Inverse of gate_up_concatenated: a concatenated [..., 2I] array (a
    weight or its gradient) in the given layout."""
    w = _f64(w_concat)
    if layout == 0:
        return w
    I = w.shape[-1] // 2
    out = np.empty_like(w)
    out[..., 0::2] = w[..., :I]
    out[..., 1::2] = w[..., I:]
    return out


def route(logits, k):
    """Top-k routing of router logits [T, E] (the step before the layer).

    The workload specifications route each token to the k experts with the
    largest router logits and weight them by a softmax over those k logits;
    the alternative wording (top-k of the full softmax, renormalised to sum
    to one) gives the same weights, since the softmax is monotonic and its
    normaliser cancels.  Readings where the sources are silent: equal logits
    are ordered by ascending expert id (so the selection is unique), the k
    choices of a token are listed by descending logit, and the logits are
    finite.

    Returns topk_idx [T, k] int64 and topk_w [T, k] float64.
    """
    z = _f64(logits)
    T, E = z.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # stable sort of the negated logits: descending, equal values by id
    order = np.argsort(-z, axis=1, kind="stable")[:, :k]
    top = np.take_along_axis(z, order, axis=1)
    e = np.exp(top - top[:, :1])
    return order.astype(np.int64), e / e.sum(axis=1, keepdims=True)


def dispatch_plan(topk_idx, E):
    """Dispatch plan by masked indexing (token-repeat page, description).

    The flattened index array lists slot s = t*k + j.  For expert e = 0..E-1
    in order, the rows whose expert id equals e are taken in increasing slot
    order; concatenating them gives `perm` (row r of the expert-grouped order
    holds slot perm[r]).  counts[e] is the number of such rows, offsets is the
    exclusive prefix sum of counts (length E+1) and inv is the inverse
    permutation (inv[perm[r]] = r).  All results are int64 numpy arrays.
    """
    flat = np.asarray(topk_idx).reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    groups = [np.nonzero(flat == e)[0] for e in range(E)]
    counts = np.array([g.size for g in groups], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.concatenate(groups) if flat.size else np.zeros(0, dtype=np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int64)
    return counts, offsets, perm.astype(np.int64), inv


def moe_forward(x, topk_idx, topk_w, w_gate_up, w_down, act,
                limit=CLAMP_LIMIT, alpha=CLAMP_ALPHA, return_slots=False,
                b_gate_up=None, b_down=None):
    """Forward pass of the expert layer, in the token-repeat page's order.

    1. repeat each token k times: x_rep[s] = x[s // k]  (slot s = t*k + j);
    2. for each expert e, pick its rows by masked indexing, h = x_rep @ Wgu[e]
       (+ b_gate_up[e]), a = act(h[:, :I], h[:, I:]), o = a @ Wd[e]
       (+ b_down[e]);
    3. scale each slot's output by its routing weight;
    4. sum the k scaled outputs of each token.

    Returns y [T, H] (float64); with return_slots also the unscaled slot
    outputs o [T*k, H].
    """
    x = _f64(x)
    T, H = x.shape
    idx = np.asarray(topk_idx).astype(np.int64)
    k = idx.shape[1]
    w = _f64(topk_w).reshape(-1)
    Wgu = w_gate_up
    Wd = w_down
    flat = idx.reshape(-1)
    x_rep = np.repeat(x, k, axis=0)
    o = np.zeros((T * k, H), dtype=np.float64)
    # Experts are visited in increasing id; an expert no row selects does no
    # work.  Wgu / Wd may be arrays or mappings keyed by expert id.
    for e in np.unique(flat):
        e = int(e)
        mask = flat == e
        I = np.shape(Wd[e])[0]
        h1 = x_rep[mask] @ _f64(Wgu[e])
        if b_gate_up is not None:
            h1 = h1 + _f64(b_gate_up[e])
        a = activation(h1[:, :I], h1[:, I:], act, limit, alpha)
        o[mask] = a @ _f64(Wd[e])
        if b_down is not None:
            o[mask] = o[mask] + _f64(b_down[e])
    y = (o * w[:, None]).reshape(T, k, H).sum(axis=1)
    if return_slots:
        return y, o
    return y


def moe_backward(dy, x, topk_idx, topk_w, w_gate_up, w_down, act,
                 limit=CLAMP_LIMIT, alpha=CLAMP_ALPHA, experts=None,
                 b_gate_up=None, b_down=None):
    """Exact gradients of L = <dy, y> for the layer (backward page).

    Per expert e, over its rows (slots s with idx[s] == e, in slot order):
      h = x_s Wgu[e], a = act(g, u), o_s = a Wd[e];
      d_topk_w[s] = <dy_t, o_s>                       (y is linear in w)
      do_s        = w_s dy_t
      dWd[e]      = sum_s a_s^T do_s
      da_s        = do_s Wd[e]^T
      dh_s        = [da_s * da/dg , da_s * da/du]
      dWgu[e]     = sum_s x_t^T dh_s                   (d_gate = [:, :I], d_up = [:, I:])
      dx_t       += dh_s Wgu[e]^T                      (summed over the k slots of t)
    Experts with no rows get zero weight gradients.

    With per-expert biases (h = x_s Wgu[e] + b_gate_up[e], o_s = a Wd[e] +
    b_down[e]) the same formulas hold with these h and o, and the biases'
    gradients are db_gate_up[e] = sum_s dh_s and db_down[e] = sum_s do_s.

    Returns (dx [T,H], d_topk_w [T,k], dWgu [E,H,2I], dWd [E,I,H]) in float64,
    and, when either bias is given, also (db_gate_up [E,2I], db_down [E,H]).
    With `experts` (an iterable of expert ids) only those experts' weight
    gradients are formed and the returned dWgu / dWd are dicts keyed by id;
    dx and d_topk_w are then complete only for tokens whose experts are all
    in the set.
    """
    x = _f64(x)
    dy = _f64(dy)
    T, H = x.shape
    idx = np.asarray(topk_idx).astype(np.int64)
    k = idx.shape[1]
    w = _f64(topk_w).reshape(-1)
    flat = idx.reshape(-1)
    x_rep = np.repeat(x, k, axis=0)
    dy_rep = np.repeat(dy, k, axis=0)
    d_w = np.zeros(T * k, dtype=np.float64)
    dx_rep = np.zeros((T * k, H), dtype=np.float64)
    subset = experts is not None
    ids = sorted(set(int(e) for e in experts)) if subset else list(range(len(w_gate_up)))
    E = len(w_gate_up)
    I = np.shape(w_down[ids[0]])[0] if ids else 0
    dWgu = {} if subset else np.zeros((E, H, 2 * I), dtype=np.float64)
    dWd = {} if subset else np.zeros((E, I, H), dtype=np.float64)
    with_bias = b_gate_up is not None or b_down is not None
    dbgu = np.zeros((E, 2 * I), dtype=np.float64)
    dbd = np.zeros((E, H), dtype=np.float64)
    for e in ids:
        rows = np.nonzero(flat == e)[0]
        Wg = _f64(w_gate_up[e])
        Wde = _f64(w_down[e])
        if rows.size == 0:
            if subset:
                dWgu[e] = np.zeros((H, 2 * I))
                dWd[e] = np.zeros((I, H))
            continue
        xe = x_rep[rows]
        dye = dy_rep[rows]
        we = w[rows]
        h1 = xe @ Wg
        if b_gate_up is not None:
            h1 = h1 + _f64(b_gate_up[e])
        g, u = h1[:, :I], h1[:, I:]
        a = activation(g, u, act, limit, alpha)
        o = a @ Wde
        if b_down is not None:
            o = o + _f64(b_down[e])
        d_w[rows] = np.sum(dye * o, axis=1)
        do = we[:, None] * dye
        dWd[e] = a.T @ do
        da = do @ Wde.T
        dadg, dadu = activation_grad(g, u, act, limit, alpha)
        dh = np.concatenate([da * dadg, da * dadu], axis=1)
        dWgu[e] = xe.T @ dh
        dx_rep[rows] = dh @ Wg.T
        dbgu[e] = dh.sum(axis=0)
        dbd[e] = do.sum(axis=0)
    dx = dx_rep.reshape(T, k, H).sum(axis=1)
    if with_bias:
        return dx, d_w.reshape(T, k), dWgu, dWd, dbgu, dbd
    return dx, d_w.reshape(T, k), dWgu, dWd


def forward_rows(x_rows, e_rows, w_rows, w_gate_up, w_down, act,
                 limit=CLAMP_LIMIT, alpha=CLAMP_ALPHA):
    """y for a handful of tokens, given each token's k (expert, weight) pairs.

    x_rows [n, H]; e_rows, w_rows [n, k].  Used to check sampled outputs of
    large workloads; it is moe_forward restricted to the given tokens.
    """
    return moe_forward(x_rows, e_rows, w_rows, w_gate_up, w_down, act, limit, alpha)
