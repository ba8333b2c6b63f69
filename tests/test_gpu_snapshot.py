"""Snapshot baseline (every draft node's state stored, the accepted one copied) against the fp64 oracle.

The snapshot verifier's outputs and its stored node states, and the snapshot
commit, must equal the path walk; the commit of an empty path returns S0
bit-identical and an invalid path is rejected with the state untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, dev_inputs, oracle_inputs
from speculative_decoding_linear_gb300 import gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run(w):
    d = dev_inputs(w)
    out = torch.full((w.B, w.N, w.H, w.dv), float("nan"), dtype=torch.float32, device="cuda")
    S_nodes = torch.empty((w.N, w.B, w.H, w.dv, w.dk), dtype=torch.float32, device="cuda")
    gdnspec.gdn_snapshot_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, S_nodes)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    return d, out, S_nodes


CASES = [
    ("config0", lambda: wl.make_workload(0)),
    ("config2", lambda: wl.make_workload(2)),
    ("b3_ragged", lambda: wl.custom_workload(3, 37, 2, 128, 48, np.stack([wl.random_tree(np.random.default_rng(s), 37, 6)
                                                                          for s in range(3)]), seed=5)),
    ("chain16_f32", lambda: wl.custom_workload(2, 16, 2, 64, 64, wl.chain_tree(16), seed=6, dtype=wl.F32)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_snapshot_verify_and_commit_match_oracle(name, make):
    w = make()
    d, out, S_nodes = run(w)
    x = oracle_inputs(w)
    o_ref, _, _ = oracle.tree_verify(**x)
    assert_close(out.cpu().numpy(), o_ref, "out")
    S_ref = oracle.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    S_new = torch.full_like(d["S0"], float("nan"))
    gdnspec.gdn_snapshot_commit(S_nodes, d["S0"], d["parent"], d["path"], S_new)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    assert_close(S_new.cpu().numpy(), S_ref, "committed state")
    S = d["S0"].clone()                                  # in place
    gdnspec.gdn_snapshot_commit(S_nodes, S, d["parent"], d["path"], S)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    assert torch.equal(S, S_new)


def test_snapshot_commit_empty_and_invalid_paths():
    w = wl.make_workload(3, seed=12, B=4)
    d, out, S_nodes = run(w)
    empty = torch.full((w.B, 3), -1, dtype=torch.int32, device="cuda")
    S_new = torch.full_like(d["S0"], float("nan"))
    gdnspec.gdn_snapshot_commit(S_nodes, d["S0"], d["parent"], empty, S_new)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    assert torch.equal(S_new, d["S0"])
    bad = np.full((w.B, 3), -1, np.int32)
    for b in range(w.B):
        kids = set(np.nonzero(w.parent[b] == 0)[0].tolist())
        bad[b, :2] = [0, next(t for t in range(1, w.N) if t not in kids)]
    S_bad = torch.full_like(d["S0"], 3.0)
    gdnspec.gdn_snapshot_commit(S_nodes, d["S0"], d["parent"], torch.from_numpy(bad).cuda(), S_bad)
    assert gdnspec.gdn_last_error() == gdnspec.ERR_PATH
    assert torch.all(S_bad == 3.0)
