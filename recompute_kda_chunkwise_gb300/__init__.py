"""GB300-native chunk-parallel Kimi Delta Attention (KDA) forward and backward.

The compute lives in a C-ABI CUDA library (``include/kda.h``); this package is
its thin Python binding. Importing the package does not load the library;
the first call does, and it fails loudly if the library has not been built.
"""
from .inputs import WORKLOADS, HEADLINE, Workload, make_inputs, make_states, cu_seqlens_of  # noqa: F401

__all__ = ["WORKLOADS", "HEADLINE", "Workload", "make_inputs", "make_states", "cu_seqlens_of"]
