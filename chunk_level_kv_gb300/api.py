"""Python binding of the ChunkKV C-ABI: argument marshalling only.

Every step of the compression runs in the library's CUDA kernels; this module
only turns torch tensors into the pointers, strides and host tables the C
calls take, and uses torch for device memory and the current CUDA stream.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from ._lib import BF16, F32, LIB, MAX_GATHER_LAYERS, PROBE_CHAINS, PROBE_THREADS, STATUS, Params

_DT = {torch.float32: F32, torch.bfloat16: BF16}


class ChunkKVError(RuntimeError):
    def __init__(self, where: str, code: int):
        self.code = code
        msg = LIB.chunkkv_status_string(code).decode()
        super().__init__(f"{where}: {STATUS.get(code, code)} ({msg})")


def _check(where: str, code: int) -> None:
    if code != 0:
        raise ChunkKVError(where, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None else t.data_ptr()
    return arr


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def make_params(*, cu_seqlens, Hq: int, Hkv: int, d: int, w: int, c: int, L_max: int,
                dtype: torch.dtype, q_strides=None, kv_strides=None, causal_window: bool = False):
    """chunkkv_params from sizes; q_strides = (b, w, head), kv_strides = (token, head) in elements.

    Returns (params, keepalive): keepalive owns the host cu_seqlens array.
    """
    cu = (ctypes.c_int32 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    B = len(cu_seqlens) - 1
    if q_strides is None:
        q_strides = (w * Hq * d, Hq * d, d)
    if kv_strides is None:
        kv_strides = (Hkv * d, d)
    p = Params(B=B, Hq=Hq, Hkv=Hkv, d=d, w=w, c=c, L_max=L_max, dtype=_DT[dtype],
               cu_seqlens=ctypes.cast(cu, ctypes.POINTER(ctypes.c_int32)),
               q_stride_b=q_strides[0], q_stride_w=q_strides[1], q_stride_h=q_strides[2],
               kv_stride_t=kv_strides[0], kv_stride_h=kv_strides[1], causal_window=int(bool(causal_window)))
    return p, cu


def params_for(q_win, k, cu_seqlens, *, Hkv: int, w: int, c: int, L_max: int, causal_window: bool = False):
    """chunkkv_params describing q_win [B, w, Hq, d] and k [T_total, Hkv, d] as laid out in memory."""
    Hq, d = q_win.shape[2], q_win.shape[3]
    assert q_win.stride(3) == 1 and k.stride(2) == 1, "the head dimension must be contiguous"
    return make_params(cu_seqlens=cu_seqlens, Hq=Hq, Hkv=Hkv, d=d, w=w, c=c, L_max=L_max,
                       dtype=k.dtype, q_strides=(q_win.stride(0), q_win.stride(1), q_win.stride(2)),
                       kv_strides=(k.stride(0), k.stride(1)), causal_window=causal_window)


def chunkkv_out_capacity(p: Params):
    n_cap, c_max = ctypes.c_int32(), ctypes.c_int32()
    _check("chunkkv_out_capacity", LIB.chunkkv_out_capacity(ctypes.byref(p), ctypes.byref(n_cap),
                                                            ctypes.byref(c_max)))
    return n_cap.value, c_max.value


def chunkkv_workspace_size(p: Params, n_layers: int = 1, n_reuse: int = 1) -> int:
    n = ctypes.c_size_t()
    _check("chunkkv_workspace_size", LIB.chunkkv_workspace_size(ctypes.byref(p), n_layers, n_reuse,
                                                                ctypes.byref(n)))
    return n.value


def chunkkv_score_path(p: Params) -> int:
    return int(LIB.chunkkv_score_path(ctypes.byref(p)))


def chunkkv_launch_count() -> int:
    return int(LIB.chunkkv_launch_count())


PHASE_EVENTS = 7          # CHUNKKV_PHASE_EVENTS
PHASES = ("pack", "score", "lse", "finalize", "select", "gather")


def chunkkv_set_phase_events(events) -> None:
    """None (off) or PHASE_EVENTS torch.cuda.Event objects that later compress calls of this
    thread record at their phase boundaries (each event is recorded once here so that it exists)."""
    if events is None:
        _check("chunkkv_set_phase_events", LIB.chunkkv_set_phase_events(None, 0))
        return
    for e in events:
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("chunkkv_set_phase_events", LIB.chunkkv_set_phase_events(arr, len(events)))


def chunkkv_score(p: Params, q_win, k, chunk_scores, ws) -> None:
    _check("chunkkv_score", LIB.chunkkv_score(ctypes.byref(p), _ptr(q_win), _ptr(k), _ptr(chunk_scores),
                                              _ptr(ws), ws.numel() * ws.element_size(), _stream(k.device)))


def chunkkv_score_noalloc(p: Params, q_win, k, chunk_scores) -> None:
    """chunkkv_score without a workspace: for callers that cannot allocate device memory.

    The scratch lives in one fixed-size device array inside the library (shared
    by every call, so calls must not overlap on the GPU); shapes that need more
    raise ChunkKVError with CHUNKKV_ERR_WORKSPACE_TOO_SMALL.
    """
    _check("chunkkv_score_noalloc", LIB.chunkkv_score_noalloc(ctypes.byref(p), _ptr(q_win), _ptr(k),
                                                              _ptr(chunk_scores), _stream(k.device)))


def chunkkv_select(p: Params, chunk_scores, indices, counts) -> None:
    _check("chunkkv_select", LIB.chunkkv_select(ctypes.byref(p), _ptr(chunk_scores), _ptr(indices),
                                                _ptr(counts), _stream(counts.device)))


def chunkkv_gather(p: Params, indices, counts, k, v, k_out, v_out) -> None:
    """k, v, k_out, v_out: lists of per-layer tensors sharing one index list."""
    n = len(k)
    _check("chunkkv_gather", LIB.chunkkv_gather(ctypes.byref(p), n, _ptr(indices), _ptr(counts),
                                                _ptr_array(k), _ptr_array(v), _ptr_array(k_out),
                                                _ptr_array(v_out), _stream(counts.device)))


def chunkkv_compress_layers(p: Params, n_reuse: int, q_win, k, v, k_out, v_out, indices, counts,
                            chunk_scores, ws) -> None:
    """Lists of per-layer tensors q_win (None for reuse layers), k, v, k_out, v_out."""
    n = len(k)
    _check("chunkkv_compress_layers",
           LIB.chunkkv_compress_layers(ctypes.byref(p), n, n_reuse, _ptr_array(q_win), _ptr_array(k),
                                       _ptr_array(v), _ptr_array(k_out), _ptr_array(v_out),
                                       _ptr(indices), _ptr(counts), _ptr(chunk_scores), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(counts.device)))


def _n_prev_array(n_prev):
    return (ctypes.c_int32 * max(len(n_prev), 1))(*[int(x) for x in n_prev])


def chunkkv_tail_sizes(p: Params, n_prev, n_layers: int = 1, n_reuse: int = 1):
    """(n_cap_max, C_max, workspace bytes) of an incremental pass (chunkkv_compress_tail)."""
    n_cap, c_max, ws = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    _check("chunkkv_tail_sizes", LIB.chunkkv_tail_sizes(ctypes.byref(p), _n_prev_array(n_prev), n_layers, n_reuse,
                                                        ctypes.byref(n_cap), ctypes.byref(c_max), ctypes.byref(ws)))
    return n_cap.value, c_max.value, ws.value


def chunkkv_compress_tail(p: Params, n_prev, n_reuse: int, q_win, k, v, k_out, v_out, indices, counts,
                          chunk_scores, ws) -> None:
    """One incremental pass during decoding over the layers in the lists q_win (None for reuse layers), k,
    v, k_out, v_out: n_prev (host ints, one per sequence) positions of each cache are kept as they are,
    the rest is the new tail to compress (tail positions in indices)."""
    n = len(k)
    _check("chunkkv_compress_tail",
           LIB.chunkkv_compress_tail(ctypes.byref(p), _n_prev_array(n_prev), n, n_reuse, _ptr_array(q_win),
                                     _ptr_array(k), _ptr_array(v), _ptr_array(k_out), _ptr_array(v_out),
                                     _ptr(indices), _ptr(counts), _ptr(chunk_scores), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(counts.device)))


def chunkkv_layer_overlap(p: Params, indices, counts):
    """(inter, union) int32 [n_lists - 1, B, Hkv]: overlap counts of adjacent kept index lists
    (indices [n_lists, B, Hkv, n_cap], counts [n_lists, B, Hkv] as chunkkv_compress_layers writes)."""
    n = indices.shape[0]
    inter = torch.empty((max(n - 1, 0),) + tuple(counts.shape[1:]), dtype=torch.int32, device=counts.device)
    uni = torch.empty_like(inter)
    _check("chunkkv_layer_overlap", LIB.chunkkv_layer_overlap(ctypes.byref(p), n, _ptr(indices), _ptr(counts),
                                                              _ptr(inter), _ptr(uni), _stream(counts.device)))
    return inter, uni


def chunkkv_selftest_wait_timeout(ws) -> None:
    """Failure-path self test: a bounded device wait that nothing completes gives up after about a
    millisecond and records code 0x1FF in ws's error word (read it with chunkkv_status_check)."""
    _check("chunkkv_selftest_wait_timeout",
           LIB.chunkkv_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), _stream(ws.device)))


def chunkkv_probe_ex2(sink, blocks: int, iters: int) -> int:
    """Exponential-unit throughput probe on the current stream: launches `blocks` CTAs whose threads
    evaluate `iters` rounds of independent base-2 exponentials (the scoring kernels' instruction).
    sink: float32 device tensor of at least blocks * PROBE_THREADS elements.  Returns the number of
    exponentials the launch evaluates (time it with events)."""
    assert sink.numel() >= blocks * PROBE_THREADS and sink.dtype == torch.float32
    _check("chunkkv_probe_ex2", LIB.chunkkv_probe_ex2(_ptr(sink), blocks, iters, _stream(sink.device)))
    return blocks * PROBE_THREADS * PROBE_CHAINS * iters


def chunkkv_status_check(ws) -> int:
    """Synchronises the current stream and reports a device-side wait that gave up (raises)."""
    code = ctypes.c_int32()
    st = LIB.chunkkv_status_check(_ptr(ws), _stream(ws.device), ctypes.byref(code))
    _check("chunkkv_status_check", st)
    return code.value


@dataclass
class CompressResult:
    k_out: list              # per layer [B, Hkv, n_cap_max, d]
    v_out: list
    indices: torch.Tensor    # [groups, B, Hkv, n_cap_max] int32
    counts: torch.Tensor     # [groups, B, Hkv] int32
    chunk_scores: torch.Tensor | None   # [groups, B, Hkv, C_max] fp32
    workspace: torch.Tensor


def compress_layers(q_win, k, v, cu_seqlens, *, Hq: int, Hkv: int, w: int, c: int, L_max: int,
                    n_reuse: int = 1, return_scores: bool = False, workspace=None,
                    causal_window: bool = False) -> CompressResult:
    """Allocate outputs with torch and run chunkkv_compress_layers on the current stream."""
    k0 = k[0]
    q0 = next(x for x in q_win if x is not None)
    p, keep = params_for(q0, k0, cu_seqlens, Hkv=Hkv, w=w, c=c, L_max=L_max, causal_window=causal_window)
    assert p.Hq == Hq
    n_cap, c_max = chunkkv_out_capacity(p)
    n_layers = len(k)
    groups = -(-n_layers // n_reuse)
    B = len(cu_seqlens) - 1
    dev = k0.device
    d = k0.shape[2]
    k_out = [torch.empty(B, Hkv, n_cap, d, dtype=k0.dtype, device=dev) for _ in range(n_layers)]
    v_out = [torch.empty(B, Hkv, n_cap, d, dtype=k0.dtype, device=dev) for _ in range(n_layers)]
    indices = torch.empty(groups, B, Hkv, max(n_cap, 1), dtype=torch.int32, device=dev)
    counts = torch.empty(groups, B, Hkv, dtype=torch.int32, device=dev)
    scores = torch.empty(groups, B, Hkv, max(c_max, 1), dtype=torch.float32, device=dev) \
        if return_scores else None
    if workspace is None:
        ws_bytes = chunkkv_workspace_size(p, n_layers, n_reuse)
        workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    chunkkv_compress_layers(p, n_reuse, q_win, k, v, k_out, v_out, indices, counts, scores, workspace)
    del keep
    return CompressResult(k_out, v_out, indices, counts, scores, workspace)


def compress_tail(q_win, k, v, cu_seqlens, n_prev, *, Hq: int, Hkv: int, w: int, c: int, L_tail: int,
                  n_reuse: int = 1, return_scores: bool = False, workspace=None) -> CompressResult:
    """Allocate outputs with torch and run chunkkv_compress_tail on the current stream.  q_win, k, v are
    tensors (one layer) or lists of per-layer tensors (q_win None for reuse layers)."""
    if torch.is_tensor(k):
        q_win, k, v = [q_win], [k], [v]
    k0 = k[0]
    q0 = next(x for x in q_win if x is not None)
    p, keep = params_for(q0, k0, cu_seqlens, Hkv=Hkv, w=w, c=c, L_max=L_tail)
    assert p.Hq == Hq
    n_layers = len(k)
    n_cap, c_max, ws_bytes = chunkkv_tail_sizes(p, n_prev, n_layers, n_reuse)
    groups = -(-n_layers // n_reuse)
    B = len(cu_seqlens) - 1
    dev, d = k0.device, k0.shape[2]
    k_out = [torch.empty(B, Hkv, n_cap, d, dtype=k0.dtype, device=dev) for _ in range(n_layers)]
    v_out = [torch.empty(B, Hkv, n_cap, d, dtype=k0.dtype, device=dev) for _ in range(n_layers)]
    indices = torch.empty(groups, B, Hkv, max(n_cap, 1), dtype=torch.int32, device=dev)
    counts = torch.empty(groups, B, Hkv, dtype=torch.int32, device=dev)
    scores = torch.empty(groups, B, Hkv, max(c_max, 1), dtype=torch.float32, device=dev) if return_scores else None
    if workspace is None:
        workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    chunkkv_compress_tail(p, n_prev, n_reuse, q_win, k, v, k_out, v_out, indices, counts, scores, workspace)
    del keep
    return CompressResult(k_out, v_out, indices, counts, scores, workspace)


__all__ = [
    "ChunkKVError", "CompressResult", "Params", "MAX_GATHER_LAYERS", "PHASES", "PHASE_EVENTS",
    "chunkkv_compress_layers", "chunkkv_compress_tail", "chunkkv_tail_sizes", "compress_tail", "chunkkv_gather", "chunkkv_launch_count", "chunkkv_layer_overlap",
    "chunkkv_out_capacity", "chunkkv_probe_ex2", "chunkkv_score", "chunkkv_score_noalloc", "chunkkv_score_path",
    "chunkkv_select", "chunkkv_selftest_wait_timeout", "chunkkv_set_phase_events", "chunkkv_status_check",
    "chunkkv_workspace_size", "compress_layers", "make_params", "params_for",
]
