"""Full GDN layer decode step on the GPU against the fp64 layer oracle.

Every intermediate the library keeps (projections, normalised q/k, v, gates,
recurrence outputs, factor record) and the layer output are compared element
by element; two consecutive steps check the fused commit of the recurrent
state and of the convolution history.  Shapes span several GEMM tiles with
ragged tails; the last case is the full 64 x 64-node, hidden-2048 workload.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, assert_close
from speculative_decoding_linear_gb300 import gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def bf16(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


class LayerRun:
    """Device buffers of one layer instance; ping-pong records across steps."""

    def __init__(self, w):
        self.w = w
        self.W_in, self.W_o = bf16(w.W_in), bf16(w.W_o)
        self.conv_w = f32(w.conv_w)
        self.S = f32(w.S0)
        self.conv_state = f32(w.conv_state)
        self.recs = []

    def step(self, X, parent, prev_path=None, N_prev=0):
        w = self.w
        B, N = parent.shape
        rec = torch.empty(gdnspec.gdn_layer_record_bytes(B, N, w.H, w.hidden, w.dk, w.dv), dtype=torch.uint8,
                          device="cuda")
        ws = torch.empty(gdnspec.gdn_layer_workspace_bytes(B, N, w.H, w.hidden, w.dk, w.dv), dtype=torch.uint8,
                         device="cuda")
        out = torch.empty((B, N, w.hidden), dtype=torch.float32, device="cuda")
        prev = self.recs[-1] if prev_path is not None else None
        gdnspec.gdn_layer_tree_step(bf16(X), self.W_in, self.conv_w, self.W_o, torch.from_numpy(parent.astype(np.int32)).cuda(),
                                    self.S, self.conv_state, prev, N_prev,
                                    None if prev_path is None else torch.from_numpy(prev_path).cuda(),
                                    out, rec, ws, w.H, w.dk, w.dv)
        assert gdnspec.gdn_last_error() == gdnspec.OK
        self.recs.append(rec)
        Y, fac = gdnspec.layer_record_views(rec, B, N, w.H, w.hidden, w.dk, w.dv)
        views = gdnspec.layer_workspace_views(ws, B, N, w.H, w.hidden, w.dk, w.dv)
        return out, Y, fac, views


def oracle_step(layer, w, X, parent, S0, conv_state):
    return layer.layer_step(wl.bf16_bits_to_f64(X), w.widened("W_in"), w.widened("conv_w"), conv_state,
                            w.widened("W_o"), parent, S0, w.H, w.dk, w.dv)


def compare(w, r, out, Y, fac, views, parent):
    B, N = parent.shape
    H, dk, dv = w.H, w.dk, w.dv
    Yh = Y.cpu().numpy().reshape(B, N, -1)
    C = H * (2 * dk + dv)
    assert_close(Yh[..., :C], r["pre"], "projections (q|k|v)", tol=1e-4)
    assert_close(Yh[..., C:C + H * dv], r["z"], "projections (gate)", tol=1e-4)
    delta, key, g, par = gdnspec.factor_views(fac, B, N, H, dk, dv, "f32")
    if dk == 256 and dv == 256:
        # single-kernel verifier: q lives as bf16 hi + lo terms, the keys only in the factor record
        q = views["qhi"].float() + views["qlo"].float()
        assert_close(q.cpu().numpy(), r["q"], "q (hi + lo)")
        assert_close((views["khi"].float() + views["klo"].float()).cpu().numpy(), r["k"], "k (hi + lo)")
        assert_close(np.transpose(key.cpu().numpy(), (0, 2, 1, 3)), r["k"], "k (factor record)")
    else:
        assert_close(views["q"].cpu().numpy(), r["q"], "q")
        assert_close(views["k"].cpu().numpy(), r["k"], "k")
    assert_close(views["v"].cpu().numpy(), r["v"], "v")
    np.testing.assert_allclose(views["alpha"].cpu().numpy(), r["alpha"], rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(views["beta"].cpu().numpy(), r["beta"], rtol=2e-5, atol=1e-6)
    assert_close(views["o"].cpu().numpy(), r["o"], "o")
    y = (views["yhi"].float() + views["ylo"].float()).cpu().numpy().reshape(B, N, H * dv)
    assert_close(y, r["y"], "gated output y (hi + lo)")
    assert_close(delta.cpu().numpy(), r["delta"], "delta")
    assert np.array_equal(par.cpu().numpy(), parent)
    return assert_close(out.cpu().numpy(), r["out"], "layer output")


SMALL = [  # (B, N, H, dk, dv, hidden, maxdepth): ragged GEMM tiles in M, N and K
    (2, 16, 2, 64, 64, 128, 4),
    (3, 37, 2, 32, 64, 192, 8),
    (5, 64, 1, 128, 128, 256, 8),
    (3, 64, 2, 256, 256, 256, 8),      # d_k = 256: tensor-core verification with split fp32 q/k
    (4, 23, 1, 256, 128, 128, 3),
]


@pytest.mark.parametrize("shape", SMALL)
def test_layer_step_matches_oracle(oracle_mod, shape):
    from oracle import layer
    B, N, H, dk, dv, hid, md = shape
    w = wl.make_layer_workload(4, seed=41 + B, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
    run = LayerRun(w)
    out, Y, fac, views = run.step(w.X, w.parent)
    r = oracle_step(layer, w, w.X, w.parent, w.widened("S0"), w.widened("conv_state"))
    compare(w, r, out, Y, fac, views, w.parent)
    # no pending commit: state and conv history untouched
    assert torch.equal(run.S.cpu(), torch.from_numpy(w.S0))
    assert torch.equal(run.conv_state.cpu(), torch.from_numpy(w.conv_state))


def test_two_steps_sixteen_node_path(oracle_mod):
    """A 16-node accepted path (d = 256, fp32 q/k as bf16 hi + lo): the single-kernel verifier then
    has room for one q/k buffer only and streams the four slabs' copies through it."""
    from oracle import layer
    B, N, H, dk, dv, hid = 2, 24, 2, 256, 256, 256
    w = wl.make_layer_workload(4, seed=301, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=6)
    w2 = wl.make_layer_workload(4, seed=302, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=6)
    chain = np.tile(wl.chain_tree(N), (B, 1))          # first step: a chain, 16 of its nodes accepted
    paths = np.tile(np.arange(16, dtype=np.int32), (B, 1))
    run = LayerRun(w)
    run.step(w.X, chain)
    r1 = oracle_step(layer, w, w.X, chain, w.widened("S0"), w.widened("conv_state"))
    S1, hist1 = layer.layer_commit(r1, chain, w.widened("S0"), w.widened("conv_state"), paths)
    out, Y, fac, views = run.step(w2.X, w2.parent, prev_path=paths, N_prev=N)
    assert_close(run.S.cpu().numpy(), S1, "committed state")
    assert_close(run.conv_state.cpu().numpy(), hist1, "committed conv history", tol=1e-5)
    r2 = oracle_step(layer, w, w2.X, w2.parent, S1, hist1)
    compare(w, r2, out, Y, fac, views, w2.parent)


@pytest.mark.parametrize("shape", SMALL[:2] + SMALL[3:])
def test_two_steps_commit_state_and_conv_history(oracle_mod, shape):
    from oracle import layer
    B, N, H, dk, dv, hid, md = shape
    w = wl.make_layer_workload(4, seed=77 + B, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
    w2 = wl.make_layer_workload(4, seed=78 + B, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
    run = LayerRun(w)
    run.step(w.X, w.parent)
    r1 = oracle_step(layer, w, w.X, w.parent, w.widened("S0"), w.widened("conv_state"))
    S1, hist1 = layer.layer_commit(r1, w.parent, w.widened("S0"), w.widened("conv_state"), w.path)
    out, Y, fac, views = run.step(w2.X, w2.parent, prev_path=w.path, N_prev=N)
    assert_close(run.S.cpu().numpy(), S1, "committed state")
    assert_close(run.conv_state.cpu().numpy(), hist1, "committed conv history", tol=1e-5)
    r2 = oracle_step(layer, w, w2.X, w2.parent, S1, hist1)
    compare(w, r2, out, Y, fac, views, w2.parent)


def test_layer_full_size(oracle_mod):
    """64 sequences x 64-node trees (depth <= 8), hidden 2048, 8 heads of 256: every element."""
    from oracle import layer
    w = wl.make_layer_workload(4)
    run = LayerRun(w)
    out, Y, fac, views = run.step(w.X, w.parent)
    r = oracle_step(layer, w, w.X, w.parent, w.widened("S0"), w.widened("conv_state"))
    compare(w, r, out, Y, fac, views, w.parent)


@pytest.mark.parametrize("shape", SMALL[:2])
def test_per_token_decode_matches_oracle(oracle_mod, shape):
    """Node-by-node decoding from materialised parent states gives the tree step's outputs."""
    from oracle import layer
    B, N, H, dk, dv, hid, md = shape
    w = wl.make_layer_workload(4, seed=91 + B, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
    X = bf16(w.X)
    W_in, W_o, cw = bf16(w.W_in), bf16(w.W_o), f32(w.conv_w)
    S0, cs = f32(w.S0), f32(w.conv_state)
    parent = torch.from_numpy(w.parent).cuda()
    rec = torch.empty(gdnspec.gdn_layer_record_bytes(B, N, H, hid, dk, dv), dtype=torch.uint8, device="cuda")
    ws = torch.empty(gdnspec.gdn_layer_workspace_bytes(B, N, H, hid, dk, dv), dtype=torch.uint8, device="cuda")
    S_nodes = torch.empty((N, B, H, dv, dk), dtype=torch.float32, device="cuda")
    out = torch.empty((B, N, hid), dtype=torch.float32, device="cuda")
    for t in range(N):
        gdnspec.gdn_layer_token_step(X, W_in, cw, W_o, parent, S0, cs, S_nodes, t, out, rec, ws, H, dk, dv)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    r = oracle_step(layer, w, w.X, w.parent, w.widened("S0"), w.widened("conv_state"))
    views = gdnspec.layer_workspace_views(ws, B, N, H, hid, dk, dv)
    assert_close(views["o"].cpu().numpy(), r["o"], "o")
    assert_close(out.cpu().numpy(), r["out"], "layer output")
    # the materialised state of each accepted end node equals the oracle's commit of its path
    S_ref = oracle_mod.commit(r["k"], r["v"], r["alpha"], r["beta"], w.parent, w.widened("S0"), w.path)
    ends = [int(p[p >= 0][-1]) for p in w.path]
    got = np.stack([S_nodes[ends[b], b].cpu().numpy() for b in range(B)])
    assert_close(got, S_ref, "node state")
    assert torch.equal(cs.cpu(), torch.from_numpy(w.conv_state))


@pytest.mark.parametrize("shape", [SMALL[0], SMALL[3]])
def test_model_step_layers_back_to_back(oracle_mod, shape):
    """Three layers on a residual stream (h_{l+1} = h_l + out_l), then a second step committing every layer."""
    from oracle import layer
    B, N, H, dk, dv, hid, md = shape
    L = 3
    ws_ = [wl.make_layer_workload(4, seed=300 + 7 * l + B, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
           for l in range(L)]
    w0 = ws_[0]
    runs = [LayerRun(w) for w in ws_]
    X = bf16(w0.X)
    parent = torch.from_numpy(w0.parent.astype(np.int32)).cuda()
    rec_bytes = gdnspec.gdn_layer_record_bytes(B, N, H, hid, dk, dv)
    recs = [[torch.empty(rec_bytes, dtype=torch.uint8, device="cuda") for _ in range(L)] for _ in range(2)]
    ws = torch.empty(gdnspec.gdn_model_workspace_bytes(L, B, N, H, hid, dk, dv), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, N, hid), dtype=torch.float32, device="cuda")
    args = dict(W_in=[r.W_in for r in runs], conv_w=[r.conv_w for r in runs], W_o=[r.W_o for r in runs],
                S=[r.S for r in runs], conv_state=[r.conv_state for r in runs])
    gdnspec.gdn_model_tree_step(X, args["W_in"], args["conv_w"], args["W_o"], parent, args["S"], args["conv_state"],
                                None, 0, None, out, recs[0], ws, H, dk, dv)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    lays = [dict(W_in=w.widened("W_in"), conv_w=w.widened("conv_w"), conv_state=w.widened("conv_state"),
                 W_o=w.widened("W_o"), S0=w.widened("S0")) for w in ws_]
    res, h = layer.model_step(w0.widened("X"), lays, w0.parent, H, dk, dv)
    assert_close(out.cpu().numpy(), h, "residual stream after the last layer")
    # second step: every layer commits the first step's accepted path, then verifies a new tree
    w2 = wl.make_layer_workload(4, seed=399 + B, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
    parent2 = torch.from_numpy(w2.parent.astype(np.int32)).cuda()
    path = torch.from_numpy(w0.path).cuda()
    gdnspec.gdn_model_tree_step(bf16(w2.X), args["W_in"], args["conv_w"], args["W_o"], parent2, args["S"],
                                args["conv_state"], recs[0], N, path, out, recs[1], ws, H, dk, dv)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    for l in range(L):
        S1, hist1 = layer.layer_commit(res[l], w0.parent, lays[l]["S0"], lays[l]["conv_state"], w0.path)
        assert_close(runs[l].S.cpu().numpy(), S1, "committed state, layer %d" % l)
        assert_close(runs[l].conv_state.cpu().numpy(), hist1, "committed conv history, layer %d" % l, tol=1e-4)
        lays[l]["S0"], lays[l]["conv_state"] = S1, hist1
    _, h2 = layer.model_step(w2.widened("X"), lays, w2.parent, H, dk, dv)
    assert_close(out.cpu().numpy(), h2, "residual stream, second step")


@pytest.mark.parametrize("shape", [SMALL[0], SMALL[3]])
def test_invalid_prev_path_leaves_state_and_conv_history_uncommitted(shape):
    """A previous accepted path that is not a root-first parent chain: the step reports
    GDN_ERR_PATH and neither the recurrent state nor the conv history moves (the verifier's
    commit and the conv kernel's history commit reject the same paths)."""
    B, N, H, dk, dv, hid, md = shape
    w = wl.make_layer_workload(4, seed=909, B=B, N=N, H=H, dk=dk, dv=dv, hidden=hid, maxdepth=md)
    run = LayerRun(w)
    run.step(w.X, w.parent)
    bad = np.full((B, 3), -1, dtype=np.int32)
    for b in range(B):                         # root, then a node that is not the root's child
        kids = set(np.nonzero(w.parent[b] == 0)[0].tolist())
        bad[b, :2] = [0, next(t for t in range(1, N) if t not in kids)]
    S_before, hist_before = run.S.clone(), run.conv_state.clone()
    rec = torch.empty(gdnspec.gdn_layer_record_bytes(B, N, H, hid, dk, dv), dtype=torch.uint8, device="cuda")
    ws = torch.empty(gdnspec.gdn_layer_workspace_bytes(B, N, H, hid, dk, dv), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, N, hid), dtype=torch.float32, device="cuda")
    gdnspec.gdn_layer_tree_step(bf16(w.X), run.W_in, run.conv_w, run.W_o, torch.from_numpy(w.parent).cuda(), run.S,
                                run.conv_state, run.recs[-1], N, torch.from_numpy(bad).cuda(), out, rec, ws, H, dk, dv)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_PATH
    assert torch.equal(run.S, S_before)
    assert torch.equal(run.conv_state, hist_before)
