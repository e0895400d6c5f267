"""top_sparse_decode_gqa_gb300 -- top-k sparse decode attention with GQA on GB300 (sm_103a).

The compute path is the C-ABI library ``libsdgqa.so`` (hand-written CUDA kernels, see
``include/sd.h``); ``binding`` marshals torch tensors into its calls.  The library is
loaded on first use and its absence is an error: there is no CPU fallback.
``workloads`` draws the seeded synthetic inputs.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "binding", "build"]
