"""gdn_tree_verify_noalloc: tree verification for callers that cannot allocate device memory.

Callers inside a host framework that owns all device memory (no raw
cudaMalloc allowed), or in a decode loop that must not allocate, cannot hand
gdn_tree_verify a workspace.  The allocation-free entry point keeps that
workspace in a fixed scratch array inside the library.  These tests call it
through the C ABI (raw pointers and sizes) and compare it with the
workspace-taking entry point on the same inputs, twice in a row (the second
call sees the first call's leftover scratch contents), on both contraction
kernels (the SIMT one for one sequence, the tensor-core one for 16).

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import TOL, alloc_outputs, dev_inputs, rel_err
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


def _reference(d, w):
    out, fac, ws = alloc_outputs(w)
    gdnspec.gdn_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"], out, fac, ws)
    assert gdnspec.gdn_last_error() == gdnspec.OK
    return out, fac


@pytest.mark.parametrize("cfgs", [(3, 2), (2, 3)])
def test_noalloc_matches_workspace_entry_point(cfgs):
    for call, cfg in enumerate(cfgs):          # two calls in a row, different trees and sizes
        w = wl.make_workload(cfg, seed=500 + call)
        d = dev_inputs(w)
        out_ref, fac_ref = _reference(d, w)
        out = torch.full_like(out_ref, float("nan"))
        fac = torch.zeros_like(fac_ref)
        _noalloc(d, w, out, fac)
        torch.cuda.synchronize()
        assert rel_err(out.cpu().numpy(), out_ref.cpu().numpy()) <= TOL
        dl, key, g, par = gdnspec.factor_views(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
        dl_r, key_r, g_r, par_r = gdnspec.factor_views(fac_ref, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
        assert rel_err(dl.cpu().numpy(), dl_r.cpu().numpy()) <= TOL
        assert torch.equal(key, key_r) and torch.equal(par, par_r)
        np.testing.assert_allclose(g.cpu().numpy(), g_r.cpu().numpy(), rtol=1e-6, atol=1e-6)


def test_noalloc_rejects_requests_beyond_its_scratch():
    """B * H (sequence, head) workspace records beyond the fixed scratch: a clear error, no launch."""
    L = gdnspec.lib()
    p = torch.empty(16, dtype=torch.uint8, device="cuda").data_ptr()   # never dereferenced
    out, fac = p, p + (1 << 30)          # 16-byte aligned, non-overlapping address ranges
    rc = L.gdn_tree_verify_noalloc(p, p, p, 0, p, p, p, p, out, fac, 200, 64, 8, 256, 256,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == gdnspec.ERR_CAPACITY
    assert "scratch" in gdnspec.strerror(rc)
