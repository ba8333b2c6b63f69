"""Shared helpers for the GPU parity tests: move a seeded workload to the
device, run the library through its C ABI, and compare with the oracle."""
import numpy as np
import torch

from speculative_decoding_linear_gb300 import gdnspec
from speculative_decoding_linear_gb300 import workloads as wl

# max |err| <= TOL x RMS(reference), per output tensor (fp32 state, bf16 inputs)
TOL = 2e-3


def dev_inputs(w, device="cuda"):
    """Torch device tensors holding exactly the workload's stored bits."""
    def qkv(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).to(device)
        return torch.from_numpy(x.copy()).to(device)
    return dict(
        q=qkv(w.q), k=qkv(w.k), v=qkv(w.v),
        alpha=torch.from_numpy(w.alpha.copy()).to(device),
        beta=torch.from_numpy(w.beta.copy()).to(device),
        parent=torch.from_numpy(w.parent.copy()).to(device),
        S0=torch.from_numpy(w.S0.copy()).to(device),
        path=torch.from_numpy(w.path.copy()).to(device),
    )


def oracle_inputs(w):
    return dict(q=w.widened("q"), k=w.widened("k"), v=w.widened("v"),
                alpha=w.alpha.astype(np.float64), beta=w.beta.astype(np.float64),
                parent=w.parent, S0=w.S0.astype(np.float64))


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-30))


def assert_close(got, ref, what, tol=TOL):
    e = rel_err(got, ref)
    assert np.all(np.isfinite(got)), "%s: non-finite values" % what
    assert e <= tol, "%s: max|err| = %.3g x RMS > %.3g" % (what, e, tol)
    return e


def alloc_outputs(w, device="cuda"):
    out = torch.empty((w.B, w.N, w.H, w.dv), dtype=torch.float32, device=device)
    fac = gdnspec.empty_factors(w.B, w.N, w.H, w.dk, w.dv, w.dtype, device)
    ws = gdnspec.empty_workspace(w.B, w.N, w.H, w.dk, w.dv, device)
    return out, fac, ws


def run_tree_verify(w, d=None):
    d = d or dev_inputs(w)
    out, fac, ws = alloc_outputs(w)
    gdnspec.gdn_tree_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["S0"],
                            out, fac, ws)
    assert gdnspec.gdn_last_error() == 0
    return d, out, fac


def run_chain_verify(w, d=None):
    d = d or dev_inputs(w)
    out, fac, _ = alloc_outputs(w)
    gdnspec.gdn_chain_verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], out, fac)
    assert gdnspec.gdn_last_error() == 0
    return d, out, fac


def check_verify(w, out, fac, oracle_mod, want=None):
    """Compare outputs and the factor record with the oracle; returns the errors."""
    x = oracle_inputs(w)
    o_ref, d_ref, g_ref = oracle_mod.tree_verify(**x, want=want)
    delta, key, g, par = gdnspec.factor_views(fac, w.B, w.N, w.H, w.dk, w.dv, w.dtype)
    o = out.cpu().numpy()
    dl = delta.cpu().numpy()
    gg = g.cpu().numpy()
    if want is not None:
        sel = np.asarray(want, bool)
        o, o_ref = o[sel], o_ref[sel]
        selh = np.broadcast_to(sel[:, None, :], (w.B, w.H, w.N))
        dl, d_ref = dl[selh], d_ref[selh]
        gg, g_ref = gg[selh], g_ref[selh]
    errs = dict(out=assert_close(o, o_ref, "out"),
                delta=assert_close(dl, d_ref, "delta"))
    np.testing.assert_allclose(gg, g_ref, rtol=1e-5, atol=1e-5)
    assert np.array_equal(par.cpu().numpy(), w.parent), "factor parent copy"
    kin = w.k if w.k.dtype != np.uint16 else w.k.view(np.int16)
    kk = key.cpu()
    kk = kk.view(torch.int16).numpy() if kk.dtype == torch.bfloat16 else kk.numpy()
    assert np.array_equal(kk, np.transpose(kin, (0, 2, 1, 3))), "factor key copy"
    return errs
