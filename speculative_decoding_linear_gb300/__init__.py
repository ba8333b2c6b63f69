"""GB300-native tree verification and factor-buffer commit for Gated DeltaNet layers.

The compute path is the C-ABI library ``libgdnspec.so`` (hand-written sm_103a
CUDA kernels); :mod:`.gdnspec` is its thin Python binding and
:mod:`.workloads` draws the seeded synthetic inputs.
"""
__all__ = ["gdnspec", "workloads"]
