"""GB300-native Graft hot path (prune-then-graft hybrid draft trees, arXiv 2605.20104).

The compute path is libgraft.so (hand-written CUDA for sm_103a behind the C
ABI in include/graft.h); ``graft`` is its thin ctypes binding.
"""
from .graft import (EXPORTS, GRAFT_BF16, GRAFT_F32, GRAFT_MODE_CHECKPOINT, GRAFT_MODE_STATIC, GRAFT_MODE_TAIL, Graft,
                    GraftError, TreeBuffers, calibrate_thresholds, graft_config, graft_default_config, library_path,
                    load, template)

__all__ = ["EXPORTS", "GRAFT_BF16", "GRAFT_F32", "GRAFT_MODE_CHECKPOINT", "GRAFT_MODE_STATIC", "GRAFT_MODE_TAIL",
           "Graft", "GraftError", "TreeBuffers", "calibrate_thresholds", "graft_config", "graft_default_config",
           "library_path", "load", "template"]
