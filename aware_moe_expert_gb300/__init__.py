"""k-aware Mixture-of-Experts layer forward for GB300 (sm_103a).

The compute path is the CUDA library ``libmoe.so`` built from ``csrc/``; the
Python side only marshals arguments (see ``binding``).  The library is loaded
on first use and its absence is an error: there is no CPU fallback.
"""
__all__ = ["binding", "inputs", "workloads"]
