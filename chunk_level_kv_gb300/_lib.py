"""ctypes view of libchunkkv.so (the C-ABI declared in include/chunkkv.h)."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libchunkkv.so")

MAX_BATCH = 1024
MAX_GATHER_LAYERS = 64
PROBE_THREADS, PROBE_CHAINS = 256, 16          # CHUNKKV_PROBE_THREADS, CHUNKKV_PROBE_CHAINS

STATUS = {
    0: "CHUNKKV_OK",
    1: "CHUNKKV_ERR_INVALID_ARG",
    2: "CHUNKKV_ERR_UNSUPPORTED",
    3: "CHUNKKV_ERR_WORKSPACE_TOO_SMALL",
    4: "CHUNKKV_ERR_CUDA",
    5: "CHUNKKV_ERR_TIMEOUT",
}
F32, BF16 = 0, 1


class Params(ctypes.Structure):
    """chunkkv_params."""
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("w", ctypes.c_int32), ("c", ctypes.c_int32), ("L_max", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("q_stride_b", ctypes.c_int64), ("q_stride_w", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
        ("kv_stride_t", ctypes.c_int64), ("kv_stride_h", ctypes.c_int64),
        ("causal_window", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                          f"g.build()'` (the library has no non-CUDA fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(Params)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    pp = ctypes.POINTER(ctypes.c_void_p)
    sigs = {
        "chunkkv_out_capacity": [P, ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "chunkkv_workspace_size": [P, i32, i32, ctypes.POINTER(sz)],
        "chunkkv_score": [P, vp, vp, vp, vp, sz, vp],
        "chunkkv_select": [P, vp, vp, vp, vp],
        "chunkkv_gather": [P, i32, vp, vp, pp, pp, pp, pp, vp],
        "chunkkv_compress_layers": [P, i32, i32, pp, pp, pp, pp, pp, vp, vp, vp, vp, sz, vp],
        "chunkkv_tail_sizes": [P, ctypes.POINTER(i32), i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                               ctypes.POINTER(sz)],
        "chunkkv_compress_tail": [P, ctypes.POINTER(i32), i32, i32, pp, pp, pp, pp, pp, vp, vp, vp, vp, sz, vp],
        "chunkkv_status_check": [vp, vp, ctypes.POINTER(i32)],
        "chunkkv_score_path": [P],
        "chunkkv_score_noalloc": [P, vp, vp, vp, vp],
        "chunkkv_set_phase_events": [pp, i32],
        "chunkkv_selftest_wait_timeout": [vp, sz, vp],
        "chunkkv_layer_overlap": [P, i32, vp, vp, vp, vp, vp],
        "chunkkv_probe_ex2": [vp, i32, i32, vp],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int32
    lib.chunkkv_status_string.argtypes = [ctypes.c_int32]
    lib.chunkkv_status_string.restype = ctypes.c_char_p
    lib.chunkkv_launch_count.argtypes = []
    lib.chunkkv_launch_count.restype = ctypes.c_uint64
    return lib


LIB = _load()
