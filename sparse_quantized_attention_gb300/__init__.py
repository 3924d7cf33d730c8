"""FFD (Faster Flash Decoding) sparse decode attention for NVIDIA GB300 (sm_103a).

The compute path is libffd.so (hand-written CUDA, C ABI in include/ffd.h); this package is its
ctypes binding. See ``ffd`` for the entry points.
"""
from .ffd import (CacheDesc, DecodeParams, FFDError, QuantizedCache, alloc_quantized_cache,
                  alloc_workspace, ffd_append_kv, ffd_decode_attention, ffd_decode_attention_static,
                  ffd_decode_workspace_size,
                  ffd_dense_decode, ffd_dense_workspace_size, ffd_get_error, ffd_quantize_keys,
                  ffd_set_profile_events, ffd_status_string, ffd_version, lib, library_path,
                  make_params, SELECT_TOPK, SELECT_TOPP, alloc_select_workspace,
                  ffd_select_workspace_size, ffd_select_blocks, ffd_decode_attention_masked,
                  ffd_art_workspace_size, alloc_art_workspace, ffd_art_attention,
                  ffd_suggest_schedule, ffd_last_cuda_error, SCHEDULE_FUSED,
                  SCHEDULE_SCAN_REFINE)

__all__ = ["CacheDesc", "DecodeParams", "FFDError", "QuantizedCache", "alloc_quantized_cache",
           "alloc_workspace", "ffd_append_kv", "ffd_decode_attention", "ffd_decode_attention_static",
           "ffd_decode_workspace_size",
           "ffd_dense_decode", "ffd_dense_workspace_size", "ffd_get_error",
           "ffd_quantize_keys", "ffd_set_profile_events", "ffd_status_string", "ffd_version",
           "lib", "library_path", "make_params", "SELECT_TOPK", "SELECT_TOPP",
           "alloc_select_workspace", "ffd_select_workspace_size", "ffd_select_blocks",
           "ffd_decode_attention_masked", "ffd_art_workspace_size", "alloc_art_workspace",
           "ffd_art_attention", "ffd_suggest_schedule", "ffd_last_cuda_error", "SCHEDULE_FUSED",
           "SCHEDULE_SCAN_REFINE"]
