"""combine_fp8_quant_gb300 -- single-GPU MoE permute / FP8 group quantisation /
combine / requantisation for GB300 (sm_103a).

The compute lives in ``libmoeperm.so`` (hand-written CUDA, C ABI declared in
``include/moeperm.h``); this package is its Python binding. Build the library
with ``__graft_entry__.build()`` (or ``python -m combine_fp8_quant_gb300.build``).
"""
from .moeperm import *  # noqa: F401,F403
from .moeperm import load, lib, Workspace, MoePermError  # noqa: F401
