"""GB300 MoE expert-parallel dispatch / combine.

The compute path is the C-ABI library built from ``csrc/`` (hand-written
sm_103a CUDA); :mod:`.ep` binds it with ctypes under the same names as
``include/ep.h``.  :mod:`.workloads` draws the seeded synthetic inputs.
"""
