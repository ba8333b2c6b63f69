"""Pins for the full-layer oracle (oracle/layer.py), CPU only.

What fixes each check, other than the oracle itself:
* a linear chain decoded token by token with a rolling conv buffer and an
  explicit state matrix (a different algorithm) gives the same outputs,
  state and conv history;
* convolution taps picked one at a time select the window rows written out by
  hand for a small tree (ancestors, then the committed history above a root);
* sibling isolation: perturbing one node's input leaves every non-descendant's
  output bit-identical;
* closed forms of the gates: a = 0 gives alpha = 1/2, a = ln(e - 1) gives
  alpha = 1/e, b = 0 gives beta = 1/2, z = 0 silences the output, W_o = I
  returns o * SiLU(z) itself;
* q and k leave the normalisation with unit norm per head;
* two decode steps (a tree step, its accepted path committed, then a chain
  step) equal one sequential decode over the accepted tokens and the new ones.
"""
import numpy as np
import pytest

from speculative_decoding_linear_gb300 import workloads as wl

H, DK, DV, HID = 2, 16, 16, 32


@pytest.fixture(scope="module")
def layer(oracle_mod):
    from oracle import layer as L
    return L


def small(seed, N=8, B=2, tree=None, maxdepth=None):
    return wl.make_layer_workload(4, seed=seed, B=B, N=N, H=H, dk=DK, dv=DV, hidden=HID, tree=tree,
                                  maxdepth=maxdepth)


def run(layer, w, **over):
    x = dict(X=w.widened("X"), W_in=w.widened("W_in"), conv_w=w.widened("conv_w"),
             conv_state=w.widened("conv_state"), W_o=w.widened("W_o"), parent=w.parent,
             S0=w.widened("S0"))
    x.update(over)
    return layer.layer_step(H=w.H, dk=w.dk, dv=w.dv, nthreads=1, **x), x


def test_chain_equals_sequential_decode(layer):
    w = small(11, N=6, tree="chain")
    r, x = run(layer, w)
    path = np.tile(np.arange(6, dtype=np.int32), (w.B, 1))
    S_new, hist_new = layer.layer_commit(r, w.parent, x["S0"], x["conv_state"], path, nthreads=1)
    for b in range(w.B):
        out, S, hist = layer.sequential_chain(x["X"][b], x["W_in"], x["conv_w"], x["conv_state"][b],
                                              x["W_o"], x["S0"][b], H, DK, DV)
        np.testing.assert_allclose(r["out"][b], out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(S_new[b], S, rtol=0, atol=1e-12)
        np.testing.assert_allclose(hist_new[b], hist, rtol=0, atol=0)


def test_partial_chain_commit_equals_shorter_decode(layer):
    w = small(12, N=5, tree="chain")
    r, x = run(layer, w)
    for L in (0, 1, 2, 4):
        path = np.full((w.B, 5), -1, np.int32)
        path[:, :L] = np.arange(L)
        S_new, hist_new = layer.layer_commit(r, w.parent, x["S0"], x["conv_state"], path, nthreads=1)
        for b in range(w.B):
            _, S, hist = layer.sequential_chain(x["X"][b, :L], x["W_in"], x["conv_w"], x["conv_state"][b],
                                                x["W_o"], x["S0"][b], H, DK, DV)
            np.testing.assert_allclose(S_new[b], S, rtol=0, atol=1e-12)
            np.testing.assert_array_equal(hist_new[b], hist)


def test_conv_taps_select_the_hand_written_window(layer):
    parent = np.array([[-1, 0, 1, 2, 0, 4]], np.int32)
    C = 3
    pre = np.arange(6 * C, dtype=np.float64).reshape(1, 6, C) + 1.0
    hist = -np.arange(3 * C, dtype=np.float64).reshape(1, 3, C) - 100.0
    # oldest .. newest sources of each node's window, written out by hand
    expect = {0: ["h0", "h1", "h2", 0], 1: ["h1", "h2", 0, 1], 2: ["h2", 0, 1, 2], 3: [0, 1, 2, 3],
              4: ["h1", "h2", 0, 4], 5: ["h2", 0, 4, 5]}
    for tap in range(4):
        cw = np.zeros((C, 4))
        cw[:, tap] = 1.0
        c = layer.tree_conv(pre, cw, hist, parent)
        for t, src in expect.items():
            s = src[tap]
            want = hist[0, int(s[1])] if isinstance(s, str) else pre[0, s]
            np.testing.assert_array_equal(c[0, t], want)


def test_identity_tap_gives_normalised_projection(layer):
    w = small(13)
    cw = np.zeros_like(w.widened("conv_w"))
    cw[:, 3] = 1.0
    r, x = run(layer, w, conv_w=cw)
    pre = x["X"] @ x["W_in"].T
    qn = pre[..., :H * DK].reshape(w.B, w.N, H, DK)
    np.testing.assert_allclose(r["q"], qn / np.linalg.norm(qn, axis=-1, keepdims=True), rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["v"].reshape(w.B, w.N, -1), pre[..., 2 * H * DK:2 * H * DK + H * DV],
                               rtol=0, atol=1e-14)


def test_unit_norm_q_k(layer):
    r, _ = run(layer, small(14))
    np.testing.assert_allclose(np.linalg.norm(r["q"], axis=-1), 1.0, atol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(r["k"], axis=-1), 1.0, atol=1e-13)


def test_sibling_isolation(layer):
    w = small(15, N=12, B=1)
    r0, x = run(layer, w)
    par = w.parent[0]
    j = 3
    X2 = x["X"].copy()
    X2[0, j] += 0.5
    r1, _ = run(layer, w, X=X2)
    desc = {j}
    for t in range(w.N):
        if par[t] in desc:
            desc.add(t)
    for t in range(w.N):
        if t in desc:
            assert not np.array_equal(r0["out"][0, t], r1["out"][0, t])
        else:
            np.testing.assert_array_equal(r0["out"][0, t], r1["out"][0, t])


def _rows(w):
    s = np.cumsum([0] + [H * DK, H * DK, H * DV, H * DV, H, H])
    return {n: slice(s[i], s[i + 1]) for i, n in enumerate("qkvzab")}


def test_gate_closed_forms(layer):
    w = small(16)
    rs = _rows(w)
    W = w.widened("W_in").copy()
    W[rs["a"]] = 0.0
    W[rs["b"]] = 0.0
    r, _ = run(layer, w, W_in=W)
    assert np.all(r["alpha"] == 0.5) and np.all(r["beta"] == 0.5)
    # a = ln(e - 1) on every node: hidden unit 0 carries 1, every other input is 0
    X = np.zeros_like(w.widened("X"))
    X[..., 0] = 1.0
    W2 = W.copy()
    W2[rs["a"], 0] = np.log(np.e - 1.0)
    r2, _ = run(layer, w, W_in=W2, X=X)
    np.testing.assert_allclose(r2["alpha"], np.exp(-1.0), rtol=1e-15)
    # z = 0 silences every output
    W3 = w.widened("W_in").copy()
    W3[rs["z"]] = 0.0
    r3, _ = run(layer, w, W_in=W3)
    assert np.all(r3["out"] == 0.0)


def test_identity_o_proj_returns_gated_recurrence(layer):
    w = small(17)
    r, _ = run(layer, w, W_o=np.eye(HID))
    z = r["z"]
    np.testing.assert_allclose(r["out"], r["o"].reshape(w.B, w.N, -1) * z * (1 / (1 + np.exp(-z))),
                               rtol=1e-15, atol=0)


def test_two_steps_equal_sequential_decode(layer):
    w1 = small(18, N=10, B=2)
    r1, x1 = run(layer, w1)
    S1, hist1 = layer.layer_commit(r1, w1.parent, x1["S0"], x1["conv_state"], w1.path, nthreads=1)
    w2 = small(19, N=4, B=2, tree="chain")
    r2, _ = run(layer, w2, W_in=x1["W_in"], conv_w=x1["conv_w"], W_o=x1["W_o"], S0=S1, conv_state=hist1)
    for b in range(w1.B):
        acc = [j for j in w1.path[b] if j >= 0]
        toks = np.concatenate([x1["X"][b, acc], w2.widened("X")[b]])
        out, _, _ = layer.sequential_chain(toks, x1["W_in"], x1["conv_w"], x1["conv_state"][b], x1["W_o"],
                                           x1["S0"][b], H, DK, DV)
        np.testing.assert_allclose(r1["out"][b, acc], out[:len(acc)], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r2["out"][b], out[len(acc):], rtol=0, atol=1e-12)


def test_model_step_of_one_layer_is_the_layer_step(layer):
    w = small(21)
    r, x = run(layer, w)
    lay = dict(W_in=x["W_in"], conv_w=x["conv_w"], conv_state=x["conv_state"], W_o=x["W_o"], S0=x["S0"])
    (m,), h = layer.model_step(x["X"], [lay], w.parent, H, DK, DV, nthreads=1)
    np.testing.assert_array_equal(m["out"], r["out"])
    np.testing.assert_array_equal(h, x["X"] + r["out"])
