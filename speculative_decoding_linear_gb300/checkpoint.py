"""Persist and reload the resumable state of a speculative decode stream.

Between two decode steps of a layer the only state that carries over is the
committed recurrent state S and the pending commit: the previous step's
factor record (delta, k, g, parent per draft node) and its accepted path
(review of SpecLA, pith.science 7ERME3HB, "Core claim": the accepted path is
applied from the buffered factors by the next verification).  Saving those
three and loading them back must reproduce the next step bit for bit.

Host-side file handling only: tensors are copied to host memory and written
with numpy; loading copies them back to the device.
"""
from __future__ import annotations

import json

import numpy as np


def save(path, S, factors, accepted_path, B, N, H, dk, dv, dtype):
    """Write S (fp32 [B,H,dv,dk]), the factor buffer (bytes) and the accepted path (int32 [B,Lmax]) of
    one layer, with the factor record's shape, to an .npz file."""
    meta = dict(B=int(B), N=int(N), H=int(H), dk=int(dk), dv=int(dv), dtype=str(dtype))
    np.savez(path, S=S.detach().cpu().numpy(), factors=factors.detach().cpu().numpy(),
             path=accepted_path.detach().cpu().numpy(), meta=np.frombuffer(json.dumps(meta).encode(), np.uint8))


def load(path, device):
    """(S, factors, accepted_path, meta) as tensors on `device`, exactly the bytes that were saved."""
    import torch
    with np.load(path) as z:
        meta = json.loads(bytes(z["meta"]).decode())
        S = torch.from_numpy(z["S"].copy()).to(device)
        fac = torch.from_numpy(z["factors"].copy()).to(device)
        acc = torch.from_numpy(z["path"].copy()).to(device)
    return S, fac, acc, meta
