"""GB300-native target-side verify step of speculative decoding.

The compute path is the C-ABI library ``libspecdec.so`` (hand-written CUDA for
sm_103a, built from ``csrc/`` by ``build.py``); ``binding`` is its thin ctypes
binding and ``workloads`` holds the seeded synthetic input generators.
"""
from .binding import (LinearOut, SpecdecError, TreeOut, alloc_workspace, linear_finalize,
                      load_library, row_stats, status_string, tree_finalize, verify_linear,
                      verify_tree, workspace_size)

__all__ = ["LinearOut", "TreeOut", "SpecdecError", "alloc_workspace", "linear_finalize",
           "load_library", "row_stats", "status_string", "tree_finalize", "verify_linear",
           "verify_tree", "workspace_size"]
