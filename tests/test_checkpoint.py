"""Checkpoint files round-trip the resumable state exactly (CPU only; the bit-identical next step
after a reload is checked on the GPU in test_gpu_failure.py)."""
import numpy as np
import torch

from speculative_decoding_linear_gb300 import checkpoint


def test_checkpoint_round_trip_is_exact(tmp_path):
    rng = np.random.default_rng(3)
    S = torch.from_numpy(rng.standard_normal((2, 3, 16, 16)).astype(np.float32))
    fac = torch.from_numpy(rng.integers(0, 256, 4096, dtype=np.uint8))
    path = torch.tensor([[0, 2, -1], [0, -1, -1]], dtype=torch.int32)
    f = tmp_path / "layer.npz"
    checkpoint.save(f, S, fac, path, 2, 5, 3, 16, 16, "bf16")
    S2, fac2, path2, meta = checkpoint.load(f, "cpu")
    assert torch.equal(S, S2) and torch.equal(fac, fac2) and torch.equal(path, path2)
    assert S2.dtype == torch.float32 and fac2.dtype == torch.uint8 and path2.dtype == torch.int32
    assert meta == dict(B=2, N=5, H=3, dk=16, dv=16, dtype="bf16")
