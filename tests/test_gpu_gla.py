"""Gated linear attention (per-channel gates) on the GPU against the fp64 oracle (oracle/gla.py).

Verification outputs and the GLA factor record (innovations, per-channel log
gates, key and parent copies) element by element, then the commit from that
record: in place and out of place, the empty path (bit-identical), an invalid
path (rejected, state untouched).  Shapes cover the SIMT contraction (small
d), the tensor-core contraction (d_k = 256, d_v a multiple of 128, bf16 and
fp32 inputs), ragged node counts, a 64-deep chain, a forest and the full
16 x 64-node, 8-head, d = 256 batch (checked on sampled sequences).
"""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import TOL, assert_close, dev_inputs
from oracle import gla as GLA
from speculative_decoding_linear_gb300 import gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def gla_workload(B, N, H, dk, dv, tree, seed, dtype=wl.BF16):
    rng = np.random.default_rng(seed)
    if tree == "chain":
        parent = np.tile(wl.chain_tree(N), (B, 1))
    elif tree == "forest":
        parent = np.full((B, N), -1, np.int32)
    else:
        parent = np.stack([wl.random_tree(rng, N, tree) for _ in range(B)])
    return wl.make_gla_workload(3, seed=seed, B=B, parent=parent, N=N, H=H, dk=dk, dv=dv, dtype=dtype)


def run_gla(w):
    d = dev_inputs(w)
    out = torch.full((w.B, w.N, w.H, w.dv), float("nan"), dtype=torch.float32, device="cuda")
    fac = torch.zeros(gdnspec.gdn_gla_factors_bytes(w.B, w.N, w.H, w.dk, w.dv, w.dtype), dtype=torch.uint8,
                      device="cuda")
    ws = torch.empty(gdnspec.gdn_gla_workspace_bytes(w.B, w.N, w.H, w.dk, w.dv), dtype=torch.uint8, device="cuda")
    gdnspec.gdn_gla_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, fac, ws)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    return d, out, fac


def oracle_of(w):
    x = [w.widened(n) for n in ("q", "k", "v", "alpha", "beta", "S0")]
    return x, GLA.tree_verify(x[0], x[1], x[2], x[3], x[4], w.parent, x[5])


def check_record(w, out, fac, ref, seqs=None):
    o_ref, d_ref, g_ref = ref
    delta, key, g, par = gdnspec.gla_factor_views(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    o, dl, gg = out.cpu().numpy(), delta.cpu().numpy(), g.cpu().numpy()
    kk = key.cpu()
    kk = kk.view(torch.int16).numpy() if kk.dtype == torch.bfloat16 else kk.numpy()
    kin = w.k.view(np.int16) if w.k.dtype == np.uint16 else w.k
    pp = par.cpu().numpy()
    if seqs is not None:
        o, dl, gg, kk, pp, kin = o[seqs], dl[seqs], gg[seqs], kk[seqs], pp[seqs], kin[seqs]
    assert_close(o, o_ref, "out")
    assert_close(dl, d_ref, "delta")
    np.testing.assert_allclose(gg, g_ref, rtol=1e-5, atol=2e-5)
    assert np.array_equal(kk, np.transpose(kin, (0, 2, 1, 3))), "key copy"
    assert np.array_equal(pp, w.parent if seqs is None else w.parent[seqs]), "parent copy"


CASES = [  # (B, N, H, dk, dv, tree, dtype): tree = max depth, "chain" or "forest"
    (1, 7, 1, 16, 16, 2, wl.F32),                  # SIMT contraction, tiny
    (3, 37, 2, 128, 64, 6, wl.BF16),               # SIMT, ragged N
    (2, 21, 3, 64, 48, 4, wl.F32),                 # SIMT, d_v not a multiple of 32
    (4, 64, 8, 256, 256, 8, wl.BF16),              # tensor-core contraction
    (2, 33, 2, 256, 128, 5, wl.F32),               # tensor-core, fp32 inputs, ragged N
    (2, 64, 2, 256, 256, "chain", wl.BF16),        # 64-deep chain: gate differences down to ~ -70
    (2, 40, 2, 256, 256, "forest", wl.BF16),       # every node a root
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_gla_verify_matches_oracle(case):
    B, N, H, dk, dv, tree, dtype = case
    w = gla_workload(B, N, H, dk, dv, tree, seed=100 + N + dk, dtype=dtype)
    _, out, fac = run_gla(w)
    _, ref = oracle_of(w)
    check_record(w, out, fac, ref)


@pytest.mark.parametrize("case", [CASES[1], CASES[3], CASES[4], CASES[5]], ids=["simt", "tc", "tc_f32", "chain"])
def test_gla_commit_matches_oracle(case):
    B, N, H, dk, dv, tree, dtype = case
    w = gla_workload(B, N, H, dk, dv, tree, seed=300 + N, dtype=dtype)
    d, out, fac = run_gla(w)
    x, _ = oracle_of(w)
    S_ref = GLA.commit(x[1], x[2], x[3], x[4], w.parent, x[5], w.path)
    S_new = torch.full_like(d["S0"], float("nan"))
    gdnspec.gdn_gla_commit(d["S0"], fac, d["path"], S_new, N, w.dtype)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    assert_close(S_new.cpu().numpy(), S_ref, "committed state")
    S = d["S0"].clone()                                     # in place
    gdnspec.gdn_gla_commit(S, fac, d["path"], S, N, w.dtype)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    assert torch.equal(S, S_new)


def test_gla_commit_empty_and_invalid_paths():
    w = gla_workload(3, 24, 2, 128, 64, 5, seed=41)
    d, out, fac = run_gla(w)
    empty = torch.full((w.B, 4), -1, dtype=torch.int32, device="cuda")
    S_new = torch.full_like(d["S0"], float("nan"))
    gdnspec.gdn_gla_commit(d["S0"], fac, empty, S_new, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    assert torch.equal(S_new, d["S0"])
    bad = np.full((w.B, 4), -1, np.int32)
    for b in range(w.B):                                    # root, then a node that is not its child
        kids = set(np.nonzero(w.parent[b] == 0)[0].tolist())
        bad[b, :2] = [0, next(t for t in range(1, w.N) if t not in kids)]
    S_bad = torch.full_like(d["S0"], 7.0)
    gdnspec.gdn_gla_commit(d["S0"], fac, torch.from_numpy(bad).cuda(), S_bad, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_PATH
    assert torch.all(S_bad == 7.0)


def test_gla_rejects_an_invalid_tree():
    w = gla_workload(2, 16, 2, 64, 64, 4, seed=43)
    w.parent[1, 5] = 9                                      # parent after the node
    d = dev_inputs(w)
    out = torch.zeros((w.B, w.N, w.H, w.dv), dtype=torch.float32, device="cuda")
    fac = torch.zeros(gdnspec.gdn_gla_factors_bytes(w.B, w.N, w.H, w.dk, w.dv, w.dtype), dtype=torch.uint8,
                      device="cuda")
    ws = torch.empty(gdnspec.gdn_gla_workspace_bytes(w.B, w.N, w.H, w.dk, w.dv), dtype=torch.uint8, device="cuda")
    gdnspec.gdn_gla_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, fac, ws)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_TREE


def test_gla_full_batch_sampled_sequences():
    """16 sequences x 64-node trees (depth <= 8), 8 heads of d = 256, bf16 -- the batched tree workload's
    shape with per-channel gates; the oracle checks every output of sequences 0, 7 and 15."""
    w = wl.make_gla_workload(3)
    _, out, fac = run_gla(w)
    seqs = [0, 7, 15]
    sub = dataclasses.replace(w, B=len(seqs), q=w.q[seqs], k=w.k[seqs], v=w.v[seqs], alpha=w.alpha[seqs],
                              beta=w.beta[seqs], parent=w.parent[seqs], S0=w.S0[seqs], path=w.path[seqs])
    _, ref = oracle_of(sub)
    check_record(w, out, fac, ref, seqs=seqs)
