"""Tile-wise mixed-precision CG for GB300 (sm_103a).

The GPU library (``libevocg.so``, C ABI in ``include/evocg.h``) holds the whole hot path:
the tile builder, the mixed-precision SpMV, the fused CG vector kernels, the precision
controllers and the CUDA-graph loop driver. ``evocg`` is a thin ctypes binding over it;
``workloads`` draws the seeded synthetic inputs.
"""
__all__ = ["evocg", "workloads"]
