"""GB300-native verify step of speculative decoding.

The compute lives in ``libspec_verify.so`` (CUDA kernels for sm_103a behind
the C-ABI in include/spec_verify.h).  This package only loads it and
marshals PyTorch tensors into its calls.
"""
from . import _native
from ._native import SVError, lib
from .verify import (build_t2d, d2t_scatter, sample, softmax_topp, topk, verify_chain, verify_tree,
                     verify_tree_sample, workspace)

__all__ = ["SVError", "lib", "build_t2d", "d2t_scatter", "sample", "softmax_topp", "topk", "verify_chain",
           "verify_tree", "verify_tree_sample", "workspace", "_native"]
