"""libssd: the Mamba-2 SSD layer and its multi-step verification decode as
hand-written sm_103a CUDA kernels behind a C ABI (libssd.so), with a thin
ctypes binding.  PyTorch supplies device memory and streams only."""
__all__ = ["synth"]
