"""Fused SwiGLU MLP forward and backward for GB300 (sm_103a).

Y = (SiLU(X Wg^T) * (X Wu^T)) Wd^T with the gradients dX, dWg, dWu, dWd, as
hand-written tcgen05/TMEM/TMA CUDA kernels behind a C ABI
(``include/swiglu_mlp.h``).  ``backward_tcgen05_tma_gb300.api`` is the thin
ctypes binding; importing this package does not load the CUDA library.
"""
__all__ = ["api", "module", "synthetic", "metrics"]
