"""CPU oracle (test infrastructure only; never imported by the library)."""
from .chunkkv_oracle import (chunk_scores, chunkkv_head, compress_layers, compress_tail_head, gather,
                             group_window_rows, kept_indices, key_scores, layer_jaccard, layer_overlap, n_select,
                             scoring_layer, tail_key_scores, top_chunks, window_limits)

__all__ = ["chunk_scores", "chunkkv_head", "compress_layers", "compress_tail_head", "gather", "group_window_rows",
           "kept_indices", "key_scores", "layer_jaccard", "layer_overlap", "n_select", "scoring_layer", "tail_key_scores", "top_chunks",
           "window_limits"]
