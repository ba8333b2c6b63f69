"""Full GDN layer decode step over a draft tree -- TEST INFRASTRUCTURE ONLY.

The oracle for one Gated DeltaNet layer that scores a whole draft tree, in
fp64: numpy for the dense parts, the C path-walk oracle (``tree_verify``,
``commit``) for the recurrence.  Only the tests, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import it.  It shares no code with
the CUDA library.

Sources: "Pith review of SpecLA: Efficient Speculative Decoding for
Linear-Attention Models" (pith.science 7ERME3HB), "Referee Report", major
comment 1 (one GDN layer: h_v = 8 heads, d_k = d_v = 256, causal depthwise
convolution of kernel size 4, SiLU gating), and "Core claim" (every node sees
the recurrence along its own root-to-node path only).

Steps, in the order the layer applies them, for every draft node t:

1. projections          Y_t = W_in x_t, split into pre-convolution q | k | v,
                        the output gate z, and the gate pre-activations a, b
                        (W_in rows in that order: H d_k, H d_k, H d_v, H d_v, H, H)
2. causal depthwise conv c_t = sum_i w[:, i] * u_i over the window
                        u_0..u_3 = pre-conv rows of (great-grandparent,
                        grandparent, parent, t); window positions above a root
                        take the committed convolution history (3 pre-conv
                        rows, oldest first).  No bias, no activation.
3. q, k                 L2-normalised per head
4. gates                alpha = exp(-softplus(a)), beta = sigmoid(b)
5. recurrence           o_t = S_t q_t with the gated delta rule along path(t)
6. output               out_t = W_o (o_t * SiLU(z_t))

Commit of an accepted root-first path p_0 .. p_{L-1}: the recurrent state of
p_{L-1} (``commit``) and the new convolution history, the last three rows of
[history rows; pre-conv rows of p_0 .. p_{L-1}].

``sequential_chain`` is a second, independent formulation used to pin this
one: a plain token-by-token decode loop with a rolling convolution buffer and
an explicitly updated state matrix.
"""
from __future__ import annotations

import numpy as np

from . import commit as _commit
from . import tree_verify as _tree_verify

KCONV = 4


def split_sizes(H, dk, dv):
    """Row counts of W_in's blocks: q, k, v, z (gate), a, b."""
    return [H * dk, H * dk, H * dv, H * dv, H, H]


def conv_window(parent_row, t):
    """Sources of the 4 window positions of node t, oldest first.

    Each entry is ("node", j) for a draft node or ("hist", r) for row r (0 =
    oldest) of the committed convolution history.
    """
    chain = [("node", int(t))]
    cur = ("node", int(t))
    hist = 2
    for _ in range(KCONV - 1):
        if cur[0] == "node" and parent_row[cur[1]] >= 0:
            cur = ("node", int(parent_row[cur[1]]))
        else:
            cur = ("hist", hist)
            hist -= 1
        chain.append(cur)
    return chain[::-1]


def _silu(x):
    return x / (1.0 + np.exp(-x))


def _softplus(x):
    return np.logaddexp(0.0, x)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def project(X, W_in, H, dk, dv):
    """Step 1: Y = X W_in^T split into (pre-conv q|k|v, z, a, b)."""
    Y = np.asarray(X, np.float64) @ np.asarray(W_in, np.float64).T
    s = np.cumsum([0] + split_sizes(H, dk, dv))
    return Y[..., s[0]:s[3]], Y[..., s[3]:s[4]], Y[..., s[4]:s[5]], Y[..., s[5]:s[6]]


def tree_conv(pre, conv_w, conv_state, parent):
    """Step 2: depthwise causal conv over each node's ancestor window.

    pre [B, N, C] pre-conv rows; conv_w [C, 4] (tap 0 = oldest); conv_state
    [B, 3, C] committed history (oldest first); parent [B, N].
    """
    B, N, C = pre.shape
    w = np.asarray(conv_w, np.float64)
    out = np.zeros((B, N, C))
    for b in range(B):
        for t in range(N):
            for i, (kind, j) in enumerate(conv_window(parent[b], t)):
                row = pre[b, j] if kind == "node" else conv_state[b, j]
                out[b, t] += w[:, i] * row
    return out


def heads_l2norm(x, H, d):
    """Step 3: L2-normalise each head's d-vector; x [B, N, H*d] -> [B, N, H, d]."""
    x = x.reshape(x.shape[0], x.shape[1], H, d)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def layer_step(X, W_in, conv_w, conv_state, W_o, parent, S0, H, dk, dv, nthreads=None):
    """One layer decode step over a draft tree.  Returns a dict of fp64 arrays.

    X [B, N, hidden]; W_in [4*H*d + 2H, hidden]; conv_w [H*(2dk+dv), 4];
    conv_state [B, 3, H*(2dk+dv)]; W_o [hidden, H*dv]; parent [B, N];
    S0 [B, H, dv, dk].
    """
    B, N, _ = np.shape(X)
    pre, z, a, bpre = project(X, W_in, H, dk, dv)
    c = tree_conv(pre, conv_w, np.asarray(conv_state, np.float64), parent)
    q = heads_l2norm(c[..., : H * dk], H, dk)
    k = heads_l2norm(c[..., H * dk: 2 * H * dk], H, dk)
    v = c[..., 2 * H * dk:].reshape(B, N, H, dv)
    alpha = np.exp(-_softplus(a))
    beta = _sigmoid(bpre)
    o, delta, g = _tree_verify(q, k, v, alpha, beta, parent, S0, nthreads=nthreads)
    y = o.reshape(B, N, H * dv) * _silu(z)
    out = y @ np.asarray(W_o, np.float64).T
    return dict(pre=pre, z=z, q=q, k=k, v=v, alpha=alpha, beta=beta, o=o, delta=delta, g=g, y=y, out=out)


def commit_conv_state(conv_state, pre, path):
    """New convolution history after accepting ``path`` ([B, Lmax], root first, -1 padded)."""
    conv_state = np.asarray(conv_state, np.float64)
    B = conv_state.shape[0]
    new = np.zeros_like(conv_state)
    for b in range(B):
        rows = [conv_state[b, r] for r in range(KCONV - 1)]
        rows += [pre[b, j] for j in path[b] if j >= 0]
        new[b] = np.stack(rows[-(KCONV - 1):])
    return new


def layer_commit(r, parent, S0, conv_state, path, nthreads=None):
    """Recurrent state and convolution history after the accepted path of a layer_step result ``r``."""
    S_new = _commit(r["k"], r["v"], r["alpha"], r["beta"], parent, S0, path, nthreads=nthreads)
    return S_new, commit_conv_state(conv_state, r["pre"], path)


def sequential_chain(X, W_in, conv_w, conv_state, W_o, S0, H, dk, dv):
    """Decode the tokens of one sequence one by one (a linear chain), fp64.

    X [T, hidden]; conv_state [3, C]; S0 [H, dv, dk].  A rolling buffer holds
    the last three pre-conv rows; the state is a matrix updated in place by
    S <- alpha S (I - beta k k^T) + beta v k^T.  Returns (out [T, hidden],
    final state [H, dv, dk], final conv history [3, C]).
    """
    X = np.asarray(X, np.float64)
    W_in = np.asarray(W_in, np.float64)
    W_o = np.asarray(W_o, np.float64)
    w = np.asarray(conv_w, np.float64)
    sizes = split_sizes(H, dk, dv)
    C = sizes[0] + sizes[1] + sizes[2]
    buf = [np.asarray(conv_state[i], np.float64).copy() for i in range(KCONV - 1)]
    S = np.asarray(S0, np.float64).copy()
    outs = []
    eye = np.eye(dk)
    for x in X:
        y = W_in @ x
        u = y[:C]
        zg = y[C:C + sizes[3]]
        a = y[C + sizes[3]:C + sizes[3] + H]
        bb = y[C + sizes[3] + H:]
        window = buf + [u]
        c = sum(w[:, i] * window[i] for i in range(KCONV))
        buf = window[1:]
        o = np.zeros(H * dv)
        for h in range(H):
            qh = c[h * dk:(h + 1) * dk]
            kh = c[H * dk + h * dk:H * dk + (h + 1) * dk]
            vh = c[2 * H * dk + h * dv:2 * H * dk + (h + 1) * dv]
            qh = qh / np.sqrt(qh @ qh)
            kh = kh / np.sqrt(kh @ kh)
            al = 1.0 / (1.0 + np.exp(a[h]))          # exp(-softplus(a)) = 1 / (1 + e^a)
            be = 1.0 / (1.0 + np.exp(-bb[h]))
            S[h] = al * S[h] @ (eye - be * np.outer(kh, kh)) + be * np.outer(vh, kh)
            o[h * dv:(h + 1) * dv] = S[h] @ qh
        gate = zg / (1.0 + np.exp(-zg))
        outs.append(W_o @ (o * gate))
    out = np.stack(outs) if outs else np.zeros((0, W_o.shape[0]))
    return out, S, np.stack(buf)


def model_step(X, layers, parent, H, dk, dv, nthreads=None):
    """L layers on a residual stream: h_0 = X, h_(l+1) = h_l + out_l (fp64).  ``layers`` is a list of
    dicts with W_in, conv_w, conv_state, W_o, S0.  Returns (list of layer_step results, h_L)."""
    res = []
    h = np.asarray(X, np.float64)
    for lay in layers:
        r = layer_step(h, lay["W_in"], lay["conv_w"], lay["conv_state"], lay["W_o"], parent, lay["S0"], H, dk, dv,
                       nthreads=nthreads)
        res.append(r)
        h = h + r["out"]
    return res, h
