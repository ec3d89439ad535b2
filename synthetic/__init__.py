"""Seeded synthetic workloads shared by the tests, the benchmark and the smoke run."""
from .generator import (HostStream, NeedleSpec, Workload, gen_kv_raw, gen_q_window,
                        make_all_layers, make_layer, needle_spans, needle_vectors,
                        normal_f32, splitmix64_int, splitmix64_torch, stream_key)
from . import configs

__all__ = [
    "HostStream", "NeedleSpec", "Workload", "gen_kv_raw", "gen_q_window", "make_all_layers",
    "make_layer", "needle_spans", "needle_vectors", "normal_f32", "splitmix64_int",
    "splitmix64_torch", "stream_key", "configs",
]
