"""Purlin-style collective datapath (copy and N-to-1 reduce Atoms driven by a
layout-derived Stage, Notify And Consume schedule) for one GB300 GPU.

The N ranks of a collective are N separate buffers in the GPU's HBM.  The
compute path is a C-ABI shared library built from `csrc/` (hand-written
sm_103a CUDA); `purlin.py` is the thin ctypes binding over it.
"""
