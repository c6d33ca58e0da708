"""GB300-native tree verification for tree speculative decoding.

The product is libtreeverify.so (C ABI in include/treeverify.h, CUDA kernels
for sm_103a in csrc/).  This package builds it (build.py) and exposes a thin
ctypes binding (binding.py) that the tests and the benchmark call.
"""
from .binding import (EXPORTED, AttnArgs, TVError, accept, accept_fused, accept_fused_workspace_size, accept_noalloc,
                      accept_workspace_size, attn, attn_args, attn_launches,
                      attn_workspace_size, build_mask, build_tree, gdn_commit, gdn_tree, kv_commit, lib, selftest_wait,
                      status_str)

__all__ = ["EXPORTED", "AttnArgs", "TVError", "accept", "accept_fused", "accept_fused_workspace_size", "accept_noalloc", "accept_workspace_size", "attn", "attn_args", "attn_launches",
           "attn_workspace_size", "build_mask", "build_tree", "gdn_commit", "gdn_tree", "kv_commit", "lib", "selftest_wait",
           "status_str"]
