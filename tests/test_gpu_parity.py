"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Indices and masks are compared bit for bit; floating-point outputs, buffered
innovations and committed states within max|err| <= 2e-3 x RMS of the oracle
(fp32 state, bf16 inputs).
"""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import (TOL, alloc_outputs, assert_close, check_verify, dev_inputs, oracle_inputs,
                     run_chain_verify, run_tree_verify)
from speculative_decoding_linear_gb300 import gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    gdnspec.gdn_last_error()
    yield
    assert gdnspec.gdn_last_error() == 0


# ---------------------------------------------------------------------------
# ancestor mask (bit-exact)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [0, 1, 2, 3, "chain64", "forest"])
def test_tree_mask_bit_exact(oracle_mod, cfg):
    if cfg == "chain64":
        parent = wl.chain_tree(64)[None]
    elif cfg == "forest":
        parent = np.array([[-1, -1, 0, 1, 3, -1, 5, 2]], np.int32)
    else:
        parent = wl.make_workload(cfg).parent
    B, N = parent.shape
    p = torch.from_numpy(parent).cuda()
    mask = torch.empty((B, N), dtype=torch.int64, device="cuda")
    depth = torch.empty((B, N), dtype=torch.int32, device="cuda")
    gdnspec.gdn_tree_mask(p, mask, depth)
    m_ref, d_ref = oracle_mod.tree_meta(parent)
    assert np.array_equal(mask.cpu().numpy().view(np.uint64), m_ref)
    assert np.array_equal(depth.cpu().numpy(), d_ref)


# ---------------------------------------------------------------------------
# tree verify
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_tree_verify_configs(oracle_mod, cfg):
    w = wl.make_workload(cfg)
    _, out, fac = run_tree_verify(w)
    check_verify(w, out, fac, oracle_mod)


@pytest.mark.parametrize("seed", range(12))
def test_tree_verify_fuzz(oracle_mod, seed):
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.choice([1, 2, 5, 17, 33, 64]))
    dk = int(rng.choice([16, 32, 64, 128, 256]))
    dv = int(rng.choice([16, 48, 96, 256]))
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    maxdepth = int(rng.integers(0, N))
    parent = np.stack([wl.random_tree(rng, N, maxdepth) for _ in range(B)])
    if seed % 3 == 0 and N > 2:      # forests: extra roots
        parent[:, N // 2] = -1
    dtype = wl.F32 if seed % 4 == 1 else wl.BF16
    w = wl.custom_workload(B, N, H, dk, dv, parent, seed=seed, dtype=dtype)
    _, out, fac = run_tree_verify(w)
    check_verify(w, out, fac, oracle_mod)


def test_tree_verify_chain_topology_deep(oracle_mod):
    """A 64-node chain through the tree path: 64 depth levels."""
    w = wl.custom_workload(2, 64, 2, 256, 256, wl.chain_tree(64), seed=5)
    _, out, fac = run_tree_verify(w)
    check_verify(w, out, fac, oracle_mod)


def test_sibling_isolation_on_gpu():
    """Perturbing one node leaves every non-descendant's GPU output bit-identical."""
    w = wl.make_workload(2)
    d = dev_inputs(w)
    _, out0, _ = run_tree_verify(w, d)
    victim = 5
    desc = {victim}
    for t in range(victim + 1, w.N):
        if w.parent[0, t] in desc:
            desc.add(t)
    d2 = {k: v.clone() for k, v in d.items()}
    d2["k"][0, victim] = torch.flip(d2["k"][0, victim], dims=[-1])
    d2["v"][0, victim] = -d2["v"][0, victim]
    d2["beta"][0, victim] = 0.95
    _, out1, _ = run_tree_verify(w, d2)
    o0, o1 = out0.cpu().numpy(), out1.cpu().numpy()
    for t in range(w.N):
        if t in desc:
            assert not np.array_equal(o0[0, t], o1[0, t])
        else:
            assert np.array_equal(o0[0, t], o1[0, t]), t


# ---------------------------------------------------------------------------
# chain verify (state-resident serial path)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["cfg1", "n1", "n64", "d16_f32", "b3_h5", "n5_f32_d32", "n8_b4", "n7_dv48",
                                  "n9_d256", "n16_f32_d256"])
def test_chain_verify(oracle_mod, case):
    """Chain verification (the serial token loop: 8-lane rows for d_k = 256, 32-lane rows otherwise)."""
    if case == "n9_d256":
        w = wl.custom_workload(2, 9, 4, 256, 256, wl.chain_tree(9), seed=12)
    elif case == "n16_f32_d256":
        w = wl.custom_workload(1, 16, 3, 256, 256, wl.chain_tree(16), seed=13, dtype=wl.F32)
    elif case == "cfg1":
        w = wl.make_workload(1)
    elif case == "n5_f32_d32":
        w = wl.custom_workload(2, 5, 3, 32, 32, wl.chain_tree(5), seed=8, dtype=wl.F32)
    elif case == "n8_b4":
        w = wl.custom_workload(4, 8, 8, 256, 256, wl.chain_tree(8), seed=10)
    elif case == "n7_dv48":
        w = wl.custom_workload(1, 7, 2, 256, 48, wl.chain_tree(7), seed=11)
    elif case == "n1":
        w = wl.custom_workload(1, 1, 8, 256, 256, wl.chain_tree(1), seed=3)
    elif case == "n64":
        w = wl.custom_workload(1, 64, 4, 256, 256, wl.chain_tree(64), seed=4)
    elif case == "d16_f32":
        w = wl.custom_workload(2, 9, 3, 16, 16, wl.chain_tree(9), seed=6, dtype=wl.F32)
    else:
        w = wl.custom_workload(3, 13, 5, 128, 64, wl.chain_tree(13), seed=7)
    _, out, fac = run_chain_verify(w)
    check_verify(w, out, fac, oracle_mod)


# ---------------------------------------------------------------------------
# commit
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
@pytest.mark.parametrize("inplace", [False, True])
def test_commit(oracle_mod, cfg, inplace):
    w = wl.make_workload(cfg)
    d, out, fac = run_tree_verify(w)
    S = d["S0"].clone() if inplace else d["S0"]
    S_new = S if inplace else torch.empty_like(S)
    gdnspec.gdn_commit(S, fac, d["path"], S_new, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == 0
    x = oracle_inputs(w)
    ref = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    assert_close(S_new.cpu().numpy(), ref, "S_new")
    # rows whose path is empty keep S0 bit for bit
    for b in range(w.B):
        if w.path[b, 0] < 0:
            assert torch.equal(S_new[b], d["S0"][b])


def test_commit_empty_path_bit_identical():
    w = wl.make_workload(3)
    d, _, fac = run_tree_verify(w)
    path = torch.full_like(d["path"], -1)
    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_commit(d["S0"], fac, path, S_new, w.N, w.dtype)
    assert torch.equal(S_new, d["S0"])


def test_commit_full_chain_64(oracle_mod):
    w = wl.custom_workload(1, 64, 2, 256, 256, wl.chain_tree(64), seed=9,
                           path=np.arange(64, dtype=np.int32)[None], lmax=64)
    d, _, fac = run_chain_verify(w)
    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_commit(d["S0"], fac, d["path"], S_new, w.N, w.dtype)
    x = oracle_inputs(w)
    ref = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    assert_close(S_new.cpu().numpy(), ref, "S_new")


# ---------------------------------------------------------------------------
# fused commit + verify (delayed state update)
# ---------------------------------------------------------------------------
def _second_tree(w, seed, chain=False):
    N2 = w.N if chain else max(1, w.N - 3)
    parent = wl.chain_tree(N2) if chain else None
    if parent is None:
        rng = np.random.default_rng(seed)
        parent = np.stack([wl.random_tree(rng, N2, 5) for _ in range(w.B)])
    return wl.custom_workload(w.B, N2, w.H, w.dk, w.dv, parent, seed=seed, dtype=w.dtype)


@pytest.mark.parametrize("cfg", [0, 2, 3])
def test_fused_commit_tree_verify(oracle_mod, cfg):
    w1 = wl.make_workload(cfg)
    d1, _, fac1 = run_tree_verify(w1)
    w2 = _second_tree(w1, seed=77 + cfg)
    d2 = dev_inputs(w2)
    S = d1["S0"].clone()
    out2, fac2, ws2 = alloc_outputs(w2)
    gdnspec.gdn_commit_tree_verify(S, fac1, w1.N, d1["path"], d2["q"], d2["k"], d2["v"], d2["alpha"],
                                   d2["beta"], d2["parent"], out2, fac2, ws2)
    assert gdnspec.gdn_last_error() == 0
    # committed state == oracle commit of tree 1's accepted path
    x1 = oracle_inputs(w1)
    S_ref = oracle_mod.commit(x1["k"], x1["v"], x1["alpha"], x1["beta"], w1.parent, x1["S0"], w1.path)
    assert_close(S.cpu().numpy(), S_ref, "committed S")
    # fused == unfused commit, bit for bit
    S_unf = torch.empty_like(S)
    gdnspec.gdn_commit(d1["S0"], fac1, d1["path"], S_unf, w1.N, w1.dtype)
    assert torch.equal(S, S_unf)
    # tree 2 verified from the committed state
    w2.S0 = S.cpu().numpy()
    check_verify(w2, out2, fac2, oracle_mod)


def test_split_launch_verify_and_fused_commit(oracle_mod):
    """More (sequence, head) pairs than SMs with a remainder that fits one wave as two CTAs per pair:
    the single-kernel verifier covers whole waves in one launch and the rest in a second launch of
    half-tile CTAs.  22 sequences x 8 heads = 176 pairs (on 152 SMs: 152 + 24 x 2)."""
    rng = np.random.default_rng(808)
    B, N, H = 22, 40, 8
    parent = np.stack([wl.random_tree(rng, N, 8) for _ in range(B)])
    w1 = wl.custom_workload(B, N, H, 256, 256, parent, seed=808)
    d1, out1, fac1 = run_tree_verify(w1)
    check_verify(w1, out1, fac1, oracle_mod)
    w2 = _second_tree(w1, seed=809)
    d2 = dev_inputs(w2)
    S = d1["S0"].clone()
    out2, fac2, ws2 = alloc_outputs(w2)
    gdnspec.gdn_commit_tree_verify(S, fac1, w1.N, d1["path"], d2["q"], d2["k"], d2["v"], d2["alpha"],
                                   d2["beta"], d2["parent"], out2, fac2, ws2)
    assert gdnspec.gdn_last_error() == 0
    S_unf = torch.empty_like(S)
    gdnspec.gdn_commit(d1["S0"], fac1, d1["path"], S_unf, w1.N, w1.dtype)
    assert torch.equal(S, S_unf)
    x1 = oracle_inputs(w1)
    S_ref = oracle_mod.commit(x1["k"], x1["v"], x1["alpha"], x1["beta"], w1.parent, x1["S0"], w1.path)
    assert_close(S.cpu().numpy(), S_ref, "committed S")
    w2.S0 = S.cpu().numpy()
    check_verify(w2, out2, fac2, oracle_mod)


@pytest.mark.parametrize("cfg", [1, "b2"])
def test_fused_commit_chain_verify(oracle_mod, cfg):
    w1 = wl.make_workload(1) if cfg == 1 else wl.custom_workload(2, 8, 3, 64, 128, wl.chain_tree(8), seed=8)
    d1, _, fac1 = run_chain_verify(w1)
    w2 = _second_tree(w1, seed=91, chain=True)
    d2 = dev_inputs(w2)
    S = d1["S0"].clone()
    out2, fac2, _ = alloc_outputs(w2)
    gdnspec.gdn_commit_chain_verify(S, fac1, w1.N, d1["path"], d2["q"], d2["k"], d2["v"], d2["alpha"],
                                    d2["beta"], out2, fac2)
    assert gdnspec.gdn_last_error() == 0
    S_unf = torch.empty_like(S)
    gdnspec.gdn_commit(d1["S0"], fac1, d1["path"], S_unf, w1.N, w1.dtype)
    assert torch.equal(S, S_unf)
    x1 = oracle_inputs(w1)
    S_ref = oracle_mod.commit(x1["k"], x1["v"], x1["alpha"], x1["beta"], w1.parent, x1["S0"], w1.path)
    assert_close(S.cpu().numpy(), S_ref, "committed S")
    w2.S0 = S.cpu().numpy()
    check_verify(w2, out2, fac2, oracle_mod)


def test_chain_and_tree_paths_agree():
    """The chain kernel and the tree kernel on a chain topology give close results."""
    w = wl.make_workload(1)
    d = dev_inputs(w)
    _, o_c, f_c = run_chain_verify(w, d)
    _, o_t, f_t = run_tree_verify(w, d)
    assert_close(o_c.cpu().numpy(), o_t.cpu().numpy(), "chain vs tree", tol=1e-3)


# ---------------------------------------------------------------------------
# device-detected errors
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bad", [[-1, 0, 2, 1], [-1, 0, 1, 7], [-1, -3, 0, 1]])
def test_invalid_parent_reported(bad):
    w = wl.custom_workload(1, 4, 2, 32, 32, [-1, 0, 1, 2], seed=1)
    d = dev_inputs(w)
    d["parent"] = torch.tensor([bad], dtype=torch.int32, device="cuda")
    out, fac, ws = alloc_outputs(w)
    gdnspec.gdn_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"],
                            out, fac, ws)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_TREE
    assert gdnspec.gdn_last_error() == 0          # cleared by the read
    mask = torch.empty((1, 4), dtype=torch.int64, device="cuda")
    depth = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    gdnspec.gdn_tree_mask(d["parent"], mask, depth)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_TREE


@pytest.mark.parametrize("bad", [[1, -1, -1], [0, 3, -1], [0, -1, 1], [0, 1, 5], [-2, -1, -1]])
def test_invalid_path_reported(bad):
    w = wl.custom_workload(1, 4, 2, 32, 32, [-1, 0, 0, 1], seed=2)
    d, _, fac = run_tree_verify(w)
    path = torch.tensor([bad], dtype=torch.int32, device="cuda")
    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_commit(d["S0"], fac, path, S_new, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_PATH
    out, fac2, ws = alloc_outputs(w)
    S = d["S0"].clone()
    gdnspec.gdn_commit_tree_verify(S, fac, w.N, path, d["q"], d["k"], d["v"], d["alpha"], d["beta"],
                                   d["parent"], out, fac2, ws)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_PATH


# ---------------------------------------------------------------------------
# layer-major sweep with launch overlap (programmatic dependent launch)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_overlapped_layer_sweep_matches_serial(cfg):
    """Several layers back to back with launch overlap on give the same bits as with it off."""
    chain = cfg == 1
    results = []
    for overlap in (False, True):
        prev = gdnspec.gdn_set_launch_overlap(overlap)
        try:
            layers = []
            for r in range(4):
                w = wl.make_workload(cfg, seed=100 + r)
                d = dev_inputs(w)
                out, fac0, ws = alloc_outputs(w)
                fac1 = gdnspec.empty_factors(w.B, w.N, w.H, w.dk, w.dv, w.dtype)
                layers.append((w, d, out, fac0, fac1, ws))
            for step in range(3):
                for (w, d, out, fac0, fac1, ws) in layers:
                    prevf, nextf = (fac0, fac1) if step % 2 == 0 else (fac1, fac0)
                    if step == 0:
                        if chain:
                            gdnspec.gdn_chain_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                                     out, fac1)
                        else:
                            gdnspec.gdn_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"],
                                                    d["S0"], out, fac1, ws)
                    elif chain:
                        gdnspec.gdn_commit_chain_verify(d["S0"], prevf, w.N, d["path"], d["q"], d["k"], d["v"],
                                                        d["alpha"], d["beta"], out, nextf)
                    else:
                        gdnspec.gdn_commit_tree_verify(d["S0"], prevf, w.N, d["path"], d["q"], d["k"], d["v"],
                                                       d["alpha"], d["beta"], d["parent"], out, nextf, ws)
            torch.cuda.synchronize()
            assert gdnspec.gdn_last_error() == 0
            results.append([(l[1]["S0"].clone(), l[2].clone()) for l in layers])
        finally:
            gdnspec.gdn_set_launch_overlap(prev)
    for (s0, o0), (s1, o1) in zip(*results):
        assert torch.equal(s0, s1) and torch.equal(o0, o1)


# ---------------------------------------------------------------------------
# tensor-core contraction (bf16, d_k = 256, >= 120 (b, h, 128-row) tiles)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["b8_n37", "b15_n64_lastrows_oob", "b60_n1", "forest_b8", "deep_chain"])
def test_tensor_core_contraction(oracle_mod, case):
    rng = np.random.default_rng(hash(case) % 2 ** 32)
    if case == "b8_n37":
        B, N, md = 8, 37, 6
    elif case == "b15_n64_lastrows_oob":
        B, N, md = 15, 64, 8
    elif case == "b60_n1":
        B, N, md = 60, 1, 0
    elif case == "forest_b8":
        B, N, md = 8, 20, 0
    else:
        B, N, md = 8, 64, 63
    parent = np.stack([wl.chain_tree(N) if case == "deep_chain" else wl.random_tree(rng, N, md)
                       for _ in range(B)])
    w = wl.custom_workload(B, N, 8, 256, 256, parent, seed=len(case))
    _, out, fac = run_tree_verify(w)
    check_verify(w, out, fac, oracle_mod)


@pytest.mark.parametrize("L", [0, 1, 9, 16])
def test_tensor_core_fused_commit(oracle_mod, L):
    """Fused commit on the tensor-core path: paths of length 0..16 into a 16-deep chain tree."""
    B, N = 8, 16
    w1 = wl.custom_workload(B, N, 8, 256, 256, wl.chain_tree(N), seed=40 + L,
                            path=np.tile(np.r_[np.arange(L), -np.ones(16 - L)].astype(np.int32), (B, 1)), lmax=16)
    d1, _, fac1 = run_tree_verify(w1)
    rng = np.random.default_rng(L)
    w2 = wl.custom_workload(B, 48, 8, 256, 256, np.stack([wl.random_tree(rng, 48, 7) for _ in range(B)]),
                            seed=60 + L)
    d2 = dev_inputs(w2)
    S = d1["S0"].clone()
    out2, fac2, ws2 = alloc_outputs(w2)
    gdnspec.gdn_commit_tree_verify(S, fac1, N, d1["path"], d2["q"], d2["k"], d2["v"], d2["alpha"],
                                   d2["beta"], d2["parent"], out2, fac2, ws2)
    assert gdnspec.gdn_last_error() == 0
    S_unf = torch.empty_like(S)
    gdnspec.gdn_commit(d1["S0"], fac1, d1["path"], S_unf, N, w1.dtype)
    assert torch.equal(S, S_unf)
    x1 = oracle_inputs(w1)
    S_ref = oracle_mod.commit(x1["k"], x1["v"], x1["alpha"], x1["beta"], w1.parent, x1["S0"], w1.path)
    assert_close(S.cpu().numpy(), S_ref, "committed S")
    w2.S0 = S.cpu().numpy()
    check_verify(w2, out2, fac2, oracle_mod)


@pytest.mark.parametrize("L", [0, 7])
def test_tensor_core_two_kernel_path(oracle_mod, L):
    """d_v = 128 takes the prologue + contraction kernel pair (d_v = 256 takes the single kernel):
    verification, then a fused commit of a path of length L, against the oracle."""
    B, N, H = 6, 40, 4
    rng = np.random.default_rng(70 + L)
    parent = np.stack([wl.random_tree(rng, N, 7) for _ in range(B)])
    w1 = wl.custom_workload(B, N, H, 256, 128, parent, seed=80 + L)
    d1, out1, fac1 = run_tree_verify(w1)
    check_verify(w1, out1, fac1, oracle_mod)
    paths = np.full((B, 16), -1, np.int32)
    for b in range(B):
        p = wl.root_path(parent[b], int(rng.integers(0, N)))[:L]
        paths[b, :len(p)] = p
    w2 = wl.custom_workload(B, 33, H, 256, 128, np.stack([wl.random_tree(rng, 33, 6) for _ in range(B)]),
                            seed=90 + L)
    d2 = dev_inputs(w2)
    S = d1["S0"].clone()
    out2, fac2, ws2 = alloc_outputs(w2)
    path_dev = torch.from_numpy(paths).cuda()
    gdnspec.gdn_commit_tree_verify(S, fac1, N, path_dev, d2["q"], d2["k"], d2["v"], d2["alpha"], d2["beta"],
                                   d2["parent"], out2, fac2, ws2)
    assert gdnspec.gdn_last_error() == 0
    x1 = oracle_inputs(w1)
    S_ref = oracle_mod.commit(x1["k"], x1["v"], x1["alpha"], x1["beta"], parent, x1["S0"], paths)
    assert_close(S.cpu().numpy(), S_ref, "committed S")
    w2.S0 = S.cpu().numpy()
    check_verify(w2, out2, fac2, oracle_mod)


# ---------------------------------------------------------------------------
# replay baselines (what the tree verifier and the factor commit replace)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [0, 2, 3])
def test_replay_baselines_match_oracle(oracle_mod, cfg):
    w = wl.make_workload(cfg)
    d = dev_inputs(w)
    out = torch.full((w.B, w.N, w.H, w.dv), float("nan"), dtype=torch.float32, device="cuda")
    gdnspec.gdn_replay_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out)
    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_replay_commit(d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], d["path"], S_new)
    assert gdnspec.gdn_last_error() == 0
    x = oracle_inputs(w)
    o_ref, _, _ = oracle_mod.tree_verify(**x)
    assert_close(out.cpu().numpy(), o_ref, "replay verify")
    S_ref = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    assert_close(S_new.cpu().numpy(), S_ref, "replay commit")


def test_replay_commit_rejects_bad_path():
    w = wl.make_workload(2)
    d = dev_inputs(w)
    bad = d["path"].clone()
    bad[0, 0] = 5 if int(w.parent[0, 5]) >= 0 else 6      # not a root
    S_new = torch.zeros_like(d["S0"])
    gdnspec.gdn_replay_commit(d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], bad, S_new)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_PATH


# ---------------------------------------------------------------------------
# chain-decomposed (hybrid) verification
# ---------------------------------------------------------------------------
def _random_trees(B, N, depth, seed):
    rng = np.random.default_rng(seed)
    return np.stack([wl.random_tree(rng, N, depth) for _ in range(B)])


def _wide_two_level():
    """A root with 21 children, each with two leaf children: 22 branching nodes, all live at once."""
    return np.array([-1] + [0] * 21 + [1 + i // 2 for i in range(42)], dtype=np.int32)


def _hybrid_cases():
    full_binary = np.array([-1] + [(t - 1) // 2 for t in range(1, 63)], dtype=np.int32)   # 31 branching nodes
    return [
        ("tiny_binary7", lambda: wl.make_workload(0)),
        ("chain8", lambda: wl.make_workload(1)),
        ("two_level_narrow", lambda: wl.custom_workload(
            2, 28, 8, 256, 256, np.concatenate([wl.narrow_tree(20, 3, 4), [9, 20, 21, 22, 9, 24, 25, 26]]), seed=60)),
        ("narrow_b4_n64", lambda: wl.custom_workload(4, 64, 8, 256, 256, wl.narrow_tree(64, 4, 8), seed=61)),
        ("narrow_b3_n37_f32", lambda: wl.custom_workload(3, 37, 2, 64, 128, wl.narrow_tree(37, 3, 5), seed=62,
                                                         dtype=wl.F32)),
        ("forest_b2", lambda: wl.custom_workload(2, 16, 4, 256, 256, np.full(16, -1, np.int32), seed=63)),
        # more branch states than the on-chip slots: the rest go through the workspace
        ("full_binary63", lambda: wl.custom_workload(1, 63, 2, 64, 64, full_binary, seed=64)),
        ("wide_two_level_n64", lambda: wl.custom_workload(2, 64, 2, 256, 256, _wide_two_level(), seed=65)),
        ("random_depth8_n64", lambda: wl.custom_workload(4, 64, 4, 256, 256, _random_trees(4, 64, 8, 66), seed=66)),
        ("random_depth4_n50_f32", lambda: wl.custom_workload(3, 50, 2, 128, 64, _random_trees(3, 50, 4, 67),
                                                             seed=67, dtype=wl.F32)),
    ]


def hybrid_workspace(w):
    n = gdnspec.gdn_hybrid_workspace_bytes(w.B, w.N, w.H, w.dk, w.dv)
    return torch.empty(n, dtype=torch.uint8, device="cuda") if n else None


@pytest.mark.parametrize("name,make", _hybrid_cases())
def test_hybrid_verify_matches_oracle(oracle_mod, name, make):
    w = make()
    d = dev_inputs(w)
    out, fac, _ = alloc_outputs(w)
    ws = hybrid_workspace(w)
    for _ in range(2):                                   # the second call reuses the workspace's slots
        out.fill_(float("nan"))
        gdnspec.gdn_hybrid_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out,
                                       fac, ws)
        assert gdnspec.gdn_last_error() == 0
        check_verify(w, out, fac, oracle_mod)
    # its factor record commits like the tree verifier's
    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_commit(d["S0"], fac, d["path"], S_new, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == 0
    x = oracle_inputs(w)
    S_ref = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    assert_close(S_new.cpu().numpy(), S_ref, "commit of hybrid factors")


def test_hybrid_full_batch_sampled_sequences(oracle_mod):
    """The batched tree workload (16 x 64-node random trees of depth <= 8, 8 heads, d = 256, bf16): every
    sequence's record against the tree verifier's, three sequences against the oracle."""
    w = wl.make_workload(3)
    d = dev_inputs(w)
    out, fac, ws = alloc_outputs(w)
    gdnspec.gdn_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, fac, ws)
    out_h, fac_h, _ = alloc_outputs(w)
    gdnspec.gdn_hybrid_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out_h,
                                   fac_h, hybrid_workspace(w))
    assert gdnspec.gdn_last_error() == 0
    assert_close(out_h.cpu().numpy(), out.cpu().numpy(), "hybrid vs tree verifier out")
    dt, _, _, _ = gdnspec.factor_views(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    dh, _, _, _ = gdnspec.factor_views(fac_h, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    assert_close(dh.cpu().numpy(), dt.cpu().numpy(), "hybrid vs tree verifier delta")
    seqs = [0, 9, 15]
    sub = dataclasses.replace(w, B=len(seqs), q=w.q[seqs], k=w.k[seqs], v=w.v[seqs], alpha=w.alpha[seqs],
                              beta=w.beta[seqs], parent=w.parent[seqs], S0=w.S0[seqs], path=w.path[seqs])
    x = oracle_inputs(sub)
    o_ref, d_ref, _ = oracle_mod.tree_verify(**x)
    assert_close(out_h.cpu().numpy()[seqs], o_ref, "hybrid out, sampled sequences")
    assert_close(dh.cpu().numpy()[seqs], d_ref, "hybrid delta, sampled sequences")


def test_hybrid_argument_and_tree_errors():
    w = wl.custom_workload(2, 40, 2, 64, 64, _random_trees(2, 40, 5, 68), seed=68)
    d = dev_inputs(w)
    out, fac, _ = alloc_outputs(w)
    assert gdnspec.gdn_hybrid_workspace_bytes(w.B, 18, w.H, w.dk, w.dv) == 0
    assert gdnspec.gdn_hybrid_workspace_bytes(w.B, 19, w.H, w.dk, w.dv) > 0
    with pytest.raises(gdnspec.GdnError) as e:            # this size needs a workspace: nothing launched
        gdnspec.gdn_hybrid_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out,
                                       fac, None)
    assert e.value.code == gdnspec.ERR_ARG
    bad = d["parent"].clone()
    bad[1, 7] = 30                                        # parent after the node
    gdnspec.gdn_hybrid_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], bad, d["S0"], out, fac,
                                   hybrid_workspace(w))
    assert gdnspec.gdn_last_error() == gdnspec.ERR_TREE


# ---------------------------------------------------------------------------
# confidence-guided pruning (index work: bit-exact against the oracle)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_prune_matches_oracle(seed):
    from oracle import prune as P
    rng = np.random.default_rng(700 + seed)
    B, N = 12, [64, 37, 7, 64][seed]
    parent = np.stack([wl.random_tree(rng, N, int(rng.integers(0, 9))) for _ in range(B)])
    logp = (-rng.exponential(1.0, (B, N))).astype(np.float32)
    logp[:, ::5] = 0.0                                   # exact ties
    for tau, budget in [(np.inf, 64), (0.0, 64), (0.7, 20), (2.0, 5), (1.0, 0)]:
        d_par = torch.from_numpy(parent).cuda()
        d_lp = torch.from_numpy(logp).cuda()
        idx = torch.empty((B, N), dtype=torch.int32, device="cuda")
        npar = torch.empty((B, N), dtype=torch.int32, device="cuda")
        nk = torch.empty(B, dtype=torch.int32, device="cuda")
        gdnspec.gdn_prune_tree(d_par, d_lp, tau, budget, idx, npar, nk)
        assert gdnspec.gdn_last_error() == 0
        for b in range(B):
            ri, rp, rn = P.prune(parent[b], logp[b], tau, budget)
            assert int(nk[b]) == rn
            assert np.array_equal(idx[b].cpu().numpy(), ri)
            got = npar[b].cpu().numpy()
            assert np.array_equal(got[:rn], rp) and np.all(got[rn:] == -1)


def test_prune_rejects_invalid_tree():
    parent = torch.tensor([[-1, 0, 3, 1]], dtype=torch.int32, device="cuda")
    lp = torch.zeros((1, 4), dtype=torch.float32, device="cuda")
    out = [torch.empty((1, 4), dtype=torch.int32, device="cuda") for _ in range(2)] + \
          [torch.empty(1, dtype=torch.int32, device="cuda")]
    gdnspec.gdn_prune_tree(parent, lp, 1.0, 4, *out)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_TREE


# ---------------------------------------------------------------------------
# decay-gated linear attention and DeltaNet through the same kernels and commit
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["tiny", "tree32_h2", "b3_n64_tc", "chain8"])
def test_linear_attention_verify_and_commit(case):
    from oracle import linear as LA
    if case == "tiny":
        w = wl.make_workload(0)
    elif case == "tree32_h2":
        w = wl.custom_workload(1, 32, 2, 256, 256, wl.random_tree(np.random.default_rng(31), 32, 6), seed=31)
    elif case == "b3_n64_tc":
        w = wl.custom_workload(3, 64, 2, 256, 256, wl.random_tree(np.random.default_rng(32), 64, 8), seed=32)
    else:
        w = wl.custom_workload(2, 8, 2, 64, 64, wl.chain_tree(8), seed=33)
    d = dev_inputs(w)
    out, fac, ws = alloc_outputs(w)
    gdnspec.gdn_linear_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, fac, ws)
    assert gdnspec.gdn_last_error() == 0
    x = oracle_inputs(w)
    o_ref, d_ref, g_ref = LA.tree_verify(x["q"], x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"])
    delta, key, g, par = gdnspec.factor_views(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    assert_close(out.cpu().numpy(), o_ref, "linear-attention output")
    assert_close(delta.cpu().numpy(), d_ref, "factor delta = beta v")
    np.testing.assert_allclose(g.cpu().numpy(), g_ref, rtol=1e-5, atol=1e-5)
    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_commit(d["S0"], fac, d["path"], S_new, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == 0
    S_ref = LA.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    assert_close(S_new.cpu().numpy(), S_ref, "commit of linear-attention factors")


def test_deltanet_is_gdn_with_unit_gates(oracle_mod):
    w = wl.make_workload(2)
    w.alpha[:] = 1.0
    d, out, fac = run_tree_verify(w)
    check_verify(w, out, fac, oracle_mod)
