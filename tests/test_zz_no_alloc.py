"""gdn_tree_verify_noalloc: tree verification for callers that cannot allocate device memory.

Callers inside a host framework that owns all device memory (no raw
cudaMalloc allowed), or in a decode loop that must not allocate, cannot hand
gdn_tree_verify a workspace.  The allocation-free entry point keeps that
workspace in a fixed scratch array inside the library.

These tests call it through the C ABI (raw pointers and sizes) on the shapes
whose kernels do pass tables through the workspace -- the two-kernel
tensor-core form (d_v = 128) and the SIMT prologue/contraction pair (d_k =
128, and fp32 q/k/v) -- each twice in a row, a larger batch and tree first,
then a smaller ragged one, so that the second call runs over the first call's
leftover scratch contents.  Outputs, innovations, gates, key copies and
parents are checked against the fp64 oracle and against the workspace-taking
entry point.  The single-kernel verifier (bf16, d_k = d_v = 256) uses no
workspace, so it runs at batch sizes beyond the scratch array; requests that
do need more scratch than the array holds are refused before any launch.

This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, alloc_outputs, check_verify, dev_inputs, rel_err
from speculative_decoding_linear_gb300 import gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(d, w, out, fac):
    L = gdnspec.lib()
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.gdn_tree_verify_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                   gdnspec.dtype_code(d["q"].dtype), d["alpha"].data_ptr(),
                                   d["beta"].data_ptr(), d["parent"].data_ptr(), d["S0"].data_ptr(),
                                   out.data_ptr(), fac.data_ptr(), w.B, w.N, w.H, w.dk, w.dv, stream)
    assert rc == gdnspec.OK, gdnspec.strerror(rc)
    assert L.gdn_last_error(stream) == gdnspec.OK


def _with_workspace(d, w):
    out, fac, ws = alloc_outputs(w)
    gdnspec.gdn_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, fac, ws)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    return out, fac


def _same_as_workspace_call(w, out, fac, out_ref, fac_ref):
    assert rel_err(out.cpu().numpy(), out_ref.cpu().numpy()) <= TOL
    dl, key, g, par = gdnspec.factor_views(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    dl_r, key_r, g_r, par_r = gdnspec.factor_views(fac_ref, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    assert rel_err(dl.cpu().numpy(), dl_r.cpu().numpy()) <= TOL
    assert torch.equal(key, key_r) and torch.equal(par, par_r)
    np.testing.assert_allclose(g.cpu().numpy(), g_r.cpu().numpy(), rtol=1e-6, atol=1e-6)


def _trees(rng, B, N, maxdepth):
    return np.stack([wl.random_tree(rng, N, maxdepth) for _ in range(B)]).astype(np.int32)


# (label, dtype, d_k, d_v): shapes whose kernels write and read the workspace
WORKSPACE_PATHS = [
    ("tensor_core_two_kernel", wl.BF16, 256, 128),
    ("simt_bf16", wl.BF16, 128, 128),
    ("simt_f32", wl.F32, 64, 64),
]


@pytest.mark.parametrize("label,dtype,dk,dv", WORKSPACE_PATHS, ids=[p[0] for p in WORKSPACE_PATHS])
def test_noalloc_workspace_paths_match_oracle(label, dtype, dk, dv):
    oracle.build()
    rng = np.random.default_rng(4242)
    # two calls in a row: more (sequence, head) pairs and a full 64-node tree first, then a ragged
    # 37-node batch with other trees -- the second call runs over the first call's scratch contents
    for call, (B, N, H, depth) in enumerate(((6, 64, 4, 8), (3, 37, 2, 5))):
        w = wl.custom_workload(B, N, H, dk, dv, _trees(rng, B, N, depth), seed=700 + call, dtype=dtype)
        d = dev_inputs(w)
        out = torch.full((w.B, w.N, w.H, w.dv), float("nan"), dtype=torch.float32, device="cuda")
        fac = torch.zeros(gdnspec.gdn_factors_bytes(w.B, w.N, w.H, w.dk, w.dv, w.dtype), dtype=torch.uint8,
                          device="cuda")
        _noalloc(d, w, out, fac)
        torch.cuda.synchronize()
        check_verify(w, out, fac, oracle)
        _same_as_workspace_call(w, out, fac, *_with_workspace(d, w))


def test_noalloc_single_kernel_path_needs_no_scratch():
    """bf16, d_k = d_v = 256 runs the single-kernel verifier, which uses no workspace: 128 sequences x
    8 heads of 64-node trees (more than the scratch array would hold) run and match gdn_tree_verify."""
    w = wl.make_workload(3, seed=811, B=128)
    d = dev_inputs(w)
    out_ref, fac_ref = _with_workspace(d, w)
    out = torch.full_like(out_ref, float("nan"))
    fac = torch.zeros_like(fac_ref)
    _noalloc(d, w, out, fac)
    torch.cuda.synchronize()
    _same_as_workspace_call(w, out, fac, out_ref, fac_ref)


def test_noalloc_rejects_requests_beyond_its_scratch():
    """A shape that passes tables through the workspace (d_k = 128: the SIMT pair) with more (sequence,
    head) records than the fixed scratch holds: a clear error, returned before any launch."""
    L = gdnspec.lib()
    p = torch.empty(16, dtype=torch.uint8, device="cuda").data_ptr()   # never dereferenced
    out, fac = p, p + (1 << 30)          # 16-byte aligned, non-overlapping address ranges
    rc = L.gdn_tree_verify_noalloc(p, p, p, 0, p, p, p, p, out, fac, 200, 64, 8, 128, 128,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == gdnspec.ERR_CAPACITY
    assert "scratch" in gdnspec.strerror(rc)
