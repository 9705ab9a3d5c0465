"""GB300-native chunkwise Gated DeltaNet forward.

The computation lives in ``libgdn.so`` (CUDA kernels for sm_103a behind the C ABI
of include/gdn.h); this package is its Python binding.
"""
from .gdn import (GDN_OK, GDN_EINVAL, GDN_EDTYPE, GDN_ELAUNCH, GDN_ETIMEOUT, GDN_ECUDA,
                  GDN_BF16, GDN_BWD_AUTO, GDN_BWD_CHUNKED, GDN_BWD_TOKENS, GDN_F32, GDN_PATH_NONE, GDN_PATH_SIMT, GDN_PATH_TCGEN05, GDN_PATH_TF32, GdnError,
                  GatedDeltaNetFunction, gated_delta_rule,
                  chunk_bwd, chunk_fwd, gdn_bwd_select_path, gdn_chunk_bwd, gdn_chunk_bwd_noalloc, gdn_chunk_bwd_workspace_bytes, decode_step, gdn_check_status, gdn_chunk_fwd, gdn_decode_step,
                  gdn_launches_per_call, gdn_linear_chunk_fwd, gdn_linear_split_segments,
                  gdn_linear_segment_map, gdn_linear_state_correct, gdn_linear_state_correct_supported, gdn_select_path, gdn_state_fold,
                  gdn_version,
                  linear_chunk_fwd, load_library)

__all__ = ["gated_delta_rule", "GatedDeltaNetFunction", "chunk_fwd", "gdn_chunk_fwd", "chunk_bwd", "gdn_chunk_bwd",
           "gdn_chunk_bwd_noalloc", "gdn_chunk_bwd_workspace_bytes", "linear_chunk_fwd", "gdn_linear_chunk_fwd", "decode_step", "gdn_decode_step", "gdn_state_fold", "gdn_select_path", "gdn_launches_per_call",
           "gdn_linear_split_segments", "gdn_linear_segment_map", "gdn_linear_state_correct", "gdn_linear_state_correct_supported",
           "gdn_check_status", "gdn_version", "load_library", "GdnError", "GDN_F32", "GDN_BF16",
           "GDN_OK", "GDN_EINVAL", "GDN_EDTYPE", "GDN_ELAUNCH", "GDN_ETIMEOUT", "GDN_ECUDA",
           "GDN_PATH_NONE", "GDN_PATH_SIMT", "GDN_PATH_TCGEN05", "GDN_PATH_TF32", "GDN_BWD_AUTO",
           "GDN_BWD_TOKENS",
           "GDN_BWD_CHUNKED", "gdn_bwd_select_path"]
