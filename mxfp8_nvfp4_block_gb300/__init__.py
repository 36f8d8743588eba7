"""Fused grouped-MLP forward for MoE layers with MXFP8 / NVFP4 block quantisation
on GB300 (sm_103a).

The compute path is the C-ABI library ``libgmlp.so`` (hand-written CUDA with
inline PTX: TMA, tcgen05 block-scaled MMA, TMEM), declared in
``include/gmlp.h``.  ``gmlp`` is its thin ctypes binding; ``inputs`` draws the
seeded synthetic workloads.  Importing this package loads nothing: the binding
loads the library on first use and raises if it is missing.
"""
__all__ = ["gmlp", "inputs"]
