"""Failure detection and resume on the GPU, in forms that fault, trap or hang nothing.

* A bounded wait that runs out: a self-test kernel waits, through the kernels'
  own bounded wait, on an mbarrier that nothing arrives on (no copy or MMA in
  flight); with the wait limit set to one millisecond it records
  GDN_ERR_TIMEOUT and returns, and the next call works normally.
* A corrupted factor record: one innovation row is changed on the host before
  the commit; parity against the fp64 oracle must fail for exactly that
  (sequence, head), by exactly the rank-1 amount the commit formula predicts.
* Resume: the committed state plus the pending (factors, accepted path)
  record, saved to a file and loaded back, must give a bit-identical next step.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, alloc_outputs, dev_inputs, oracle_inputs, rel_err, run_tree_verify
from speculative_decoding_linear_gb300 import checkpoint, faults, gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_stuck_wait_runs_out_and_the_context_survives():
    gdnspec.gdn_last_error()                       # start from a clear error word
    gdnspec.gdn_set_wait_limit_ns(1_000_000)       # 1 ms
    try:
        gdnspec.gdn_selftest_stuck_wait()
        assert gdnspec.gdn_last_error() == gdnspec.ERR_TIMEOUT
        assert gdnspec.gdn_last_error() == gdnspec.OK   # read and cleared
    finally:
        gdnspec.gdn_set_wait_limit_ns(1_000_000_000)
    w = wl.make_workload(2)                        # the next call runs and is right
    _, out, fac = run_tree_verify(w)
    o_ref, _, _ = oracle.tree_verify(**oracle_inputs(w))
    assert rel_err(out.cpu().numpy(), o_ref) <= TOL


def test_wait_limit_rejects_out_of_range_values():
    for ns in (0, 999, 60_000_000_001):
        with pytest.raises(gdnspec.GdnError):
            gdnspec.gdn_set_wait_limit_ns(ns)


def test_corrupted_factor_row_is_caught_by_parity():
    w = wl.make_workload(3, seed=77)
    d, out, fac = run_tree_verify(w)
    x = oracle_inputs(w)
    _, _, g_ref = oracle.tree_verify(**x)
    S_ref = oracle.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)

    # plant the fault: head 3 of the first sequence whose accepted path has >= 2 nodes, at the
    # path's second node
    b = next(i for i in range(w.B) if np.sum(w.path[i] >= 0) >= 2)
    h = 3
    path_b = [int(t) for t in w.path[b] if t >= 0]
    j, a = path_b[1], path_b[-1]
    c = 0.75
    faults.corrupt_delta_row(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype, b, h, j, c)

    S_new = torch.empty_like(d["S0"])
    gdnspec.gdn_commit(d["S0"], fac, d["path"], S_new, w.N, w.dtype)
    assert gdnspec.gdn_last_error() == 0
    S = S_new.cpu().numpy().astype(np.float64)

    assert rel_err(S, S_ref) > 10 * TOL                     # parity fails
    other = np.ones((w.B, w.H), bool)
    other[b, h] = False
    assert rel_err(S[other], S_ref[other]) <= TOL           # everywhere else it still holds
    # by exactly the rank-1 amount e^{g_a - g_j} c 1 k_j^T
    expect = np.exp(g_ref[b, h, a] - g_ref[b, h, j]) * c * np.outer(np.ones(w.dv), x["k"][b, j, h])
    scale = np.sqrt(np.mean(S_ref ** 2))
    assert np.max(np.abs((S[b, h] - S_ref[b, h]) - expect)) <= TOL * scale


def test_persist_and_reload_gives_a_bit_identical_next_step(tmp_path):
    w1 = wl.make_workload(3, seed=91)
    w2 = wl.make_workload(3, seed=92)              # the next step's drafts, same batch
    d1 = dev_inputs(w1)
    d2 = dev_inputs(w2)
    out1, fac1, ws = alloc_outputs(w1)
    gdnspec.gdn_tree_verify(d1["q"], d1["k"], d1["v"], d1["alpha"], d1["beta"], d1["parent"], d1["S0"], out1, fac1,
                            ws)
    assert gdnspec.gdn_last_error() == 0
    ck = tmp_path / "layer0.npz"
    checkpoint.save(ck, d1["S0"], fac1, d1["path"], w1.B, w1.N, w1.H, w1.dk, w1.dv, w1.dtype)

    def next_step(S, fac_prev, path_prev):
        out, fac, ws2 = alloc_outputs(w2)
        gdnspec.gdn_commit_tree_verify(S, fac_prev, w1.N, path_prev, d2["q"], d2["k"], d2["v"], d2["alpha"],
                                       d2["beta"], d2["parent"], out, fac, ws2)
        assert gdnspec.gdn_last_error() == 0
        return S, out, fac

    S_a, out_a, fac_a = next_step(d1["S0"].clone(), fac1, d1["path"])
    S_r, fac_r, path_r, meta = checkpoint.load(ck, "cuda")
    assert meta["N"] == w1.N and meta["dtype"] == w1.dtype
    S_b, out_b, fac_b = next_step(S_r, fac_r, path_r)
    assert torch.equal(S_a, S_b)
    assert torch.equal(out_a, out_b)
    assert torch.equal(fac_a, fac_b)
    # and the resumed step is the right one
    x = oracle_inputs(w1)
    S_ref = oracle.commit(x["k"], x["v"], x["alpha"], x["beta"], w1.parent, x["S0"], w1.path)
    assert rel_err(S_b.cpu().numpy(), S_ref) <= TOL
