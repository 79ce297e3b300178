"""GB300-native gated delta rule (GatedDeltaNet): forward pass and full VJP.

The compute path is the C-ABI library built from ``csrc/`` (hand-written
sm_103a CUDA kernels); ``ops`` is a thin ctypes binding over it.  Nothing in
this package falls back to a CPU or PyTorch implementation: calling an op
without the compiled library raises.
"""

__all__ = ["ops", "workloads"]
