"""ChunkKV chunk-level KV-cache compression on one GB300: Python binding of libchunkkv.so."""
from .api import (ChunkKVError, CompressResult, Params, chunkkv_compress_layers, chunkkv_compress_tail,
                  chunkkv_tail_sizes, compress_tail, chunkkv_gather,
                  chunkkv_launch_count, chunkkv_set_phase_events, PHASES, chunkkv_selftest_wait_timeout,
                  chunkkv_layer_overlap, chunkkv_probe_ex2,
                  chunkkv_out_capacity, chunkkv_score, chunkkv_score_noalloc, chunkkv_score_path, chunkkv_select,
                  chunkkv_status_check, chunkkv_workspace_size, compress_layers, make_params,
                  params_for)

__all__ = [
    "ChunkKVError", "CompressResult", "Params", "chunkkv_compress_layers", "chunkkv_compress_tail",
    "chunkkv_tail_sizes", "compress_tail", "chunkkv_gather", "chunkkv_launch_count",
    "chunkkv_set_phase_events", "PHASES", "chunkkv_selftest_wait_timeout", "chunkkv_layer_overlap",
    "chunkkv_probe_ex2",
    "chunkkv_out_capacity", "chunkkv_score", "chunkkv_score_noalloc", "chunkkv_score_path", "chunkkv_select",
    "chunkkv_status_check", "chunkkv_workspace_size", "compress_layers", "make_params", "params_for",
]
