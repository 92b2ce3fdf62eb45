"""GB300-native RNN-T joint network + output layer + transducer loss (fwd + bwd).

The computation runs in the CUDA kernels of ``librnnt_gb300.so`` behind the C
ABI of ``include/rnnt.h``; this package is its thin Python binding.
"""
from .binding import (EXPORTS, RNNT_BF16, RNNT_BF16_E4M3, RNNT_F32, RNNT_TILED, RNNT_UNTILED,
                      Rnnt, RnntBwdOpts, RnntDims, RnntError, RnntParams, RnntSavedOffsets,
                      load, make_dims, make_params, rnnt_bwd, rnnt_bwd_ex, rnnt_device_status,
                      rnnt_fwd, rnnt_fwd_bwd, rnnt_fwd_noalloc, rnnt_graph_capturable, rnnt_profile_start,
                      rnnt_profile_stop, rnnt_saved_bytes, rnnt_saved_layout,
                      rnnt_status_string, rnnt_tile_cells_for_budget, rnnt_workspace_bytes)

__all__ = ["EXPORTS", "RNNT_BF16", "RNNT_BF16_E4M3", "RNNT_F32", "RNNT_TILED", "RNNT_UNTILED",
           "Rnnt", "RnntBwdOpts", "RnntDims", "RnntError", "RnntParams", "RnntSavedOffsets",
           "load", "make_dims", "make_params", "rnnt_bwd", "rnnt_bwd_ex", "rnnt_device_status",
           "rnnt_fwd", "rnnt_fwd_bwd", "rnnt_fwd_noalloc", "rnnt_graph_capturable", "rnnt_profile_start",
           "rnnt_profile_stop", "rnnt_saved_bytes", "rnnt_saved_layout", "rnnt_status_string",
           "rnnt_tile_cells_for_budget", "rnnt_workspace_bytes"]
