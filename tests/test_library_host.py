"""libchunkkv.so on the host: it loads, exports the header's symbols, and checks arguments.

Nothing here launches a kernel: every call below either computes sizes or is
rejected by the host-side argument checks before any CUDA call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "chunkkv.h")
LIBPATH = os.path.join(ROOT, "chunk_level_kv_gb300", "libchunkkv.so")


@pytest.fixture(scope="module")
def ckv():
    if not os.path.exists(LIBPATH):
        import __graft_entry__
        __graft_entry__.build()
    import chunk_level_kv_gb300 as m
    return m


def test_exports_every_declared_function(ckv):
    text = open(HEADER).read()
    names = set(re.findall(r"^\s*(?:const\s+char\*|chunkkv_status|int32_t|uint64_t)\s+(chunkkv_\w+)\s*\(", text,
                           flags=re.M))
    assert {"chunkkv_score", "chunkkv_select", "chunkkv_gather", "chunkkv_compress_layers",
            "chunkkv_workspace_size", "chunkkv_out_capacity", "chunkkv_status_check"} <= names
    lib = ctypes.CDLL(LIBPATH)
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_launch_counter_only_counts_launches(ckv):
    n0 = ckv.chunkkv_launch_count()
    assert isinstance(n0, int) and n0 >= 0
    p, keep = _p(ckv)
    ckv.chunkkv_workspace_size(p, 4, 2)            # host-side sizing launches nothing
    ckv.chunkkv_out_capacity(p)
    assert ckv.chunkkv_launch_count() == n0


def test_phase_events_argument_checks(ckv):
    from chunk_level_kv_gb300._lib import LIB
    arr = (ctypes.c_void_p * 7)()                      # NULL handles
    assert LIB.chunkkv_set_phase_events(arr, 7) == 1
    assert LIB.chunkkv_set_phase_events(arr, 3) == 1
    assert LIB.chunkkv_set_phase_events(None, 0) == 0


def test_selftest_argument_checks(ckv):
    from chunk_level_kv_gb300._lib import LIB
    assert LIB.chunkkv_selftest_wait_timeout(None, 256, None) == 1
    assert LIB.chunkkv_selftest_wait_timeout(ctypes.c_void_p(16), 128, None) == 1     # too small: no launch


def test_status_strings(ckv):
    from chunk_level_kv_gb300._lib import LIB
    for code in range(6):
        assert LIB.chunkkv_status_string(code)
    assert LIB.chunkkv_status_string(0) == b"ok"


def _p(ckv, **kw):
    import torch
    args = dict(cu_seqlens=[0, 512], Hq=4, Hkv=2, d=64, w=8, c=10, L_max=128, dtype=torch.float32)
    args.update(kw)
    return ckv.make_params(**args)


@pytest.mark.parametrize("T,w,c,L_max,n_cap,C", [
    (32768, 32, 10, 6553, 6582, 3277),          # LLaMA-3-8B 32K, 20 % budget
    (131072, 64, 10, 13107, 13164, 13108),      # Qwen2-7B 128K, 10 % budget
    (8192, 32, 10, 819, 842, 820),              # LLaMA-3-8B single layer, 10 %
    (512, 8, 10, 128, 128, 52),                 # tiny
    (20, 30, 7, 7, 20, 3),                      # window longer than the prompt
    (100, 5, 10, 0, 5, 10),                     # no chunk budget: recent window only
    (0, 5, 10, 50, 0, 0),                       # empty sequence
])
def test_out_capacity(ckv, T, w, c, L_max, n_cap, C):
    import torch
    p, keep = _p(ckv, cu_seqlens=[0, T], w=w, c=c, L_max=L_max, d=128, Hq=32, Hkv=8,
                 dtype=torch.bfloat16)
    assert ckv.chunkkv_out_capacity(p) == (n_cap, C)


def test_workspace_size_grows_with_window(ckv):
    import torch
    small, k1 = _p(ckv, cu_seqlens=[0, 4096], w=8, d=128, Hq=8, Hkv=8, dtype=torch.bfloat16)
    big, k2 = _p(ckv, cu_seqlens=[0, 4096], w=64, d=128, Hq=8, Hkv=8, dtype=torch.bfloat16)
    assert 0 < ckv.chunkkv_workspace_size(small) < ckv.chunkkv_workspace_size(big)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=3, Hkv=2), 1),                      # Hq not a multiple of Hkv
    (dict(c=0), 1),
    (dict(w=-1), 1),
    (dict(L_max=-5), 1),
    (dict(d=6), 1),                              # 24-byte fp32 rows are not 16-byte multiples
    (dict(d=512), 2),                            # beyond the head-dimension limit
    (dict(cu_seqlens=[0, 10, 5]), 1),            # decreasing offsets
    (dict(cu_seqlens=[3, 10]), 1),               # offsets must start at 0
    (dict(cu_seqlens=[0] * 1100), 2),            # batch beyond CHUNKKV_MAX_BATCH
    (dict(w=2048, Hq=8, Hkv=2), 2),              # w * G beyond the window-row limit
    (dict(kv_strides=(64 * 2 + 1, 64)), 1),      # token stride breaks 16-byte rows
])
def test_invalid_params_rejected(ckv, kw, code):
    p, keep = _p(ckv, **kw)
    from chunk_level_kv_gb300._lib import LIB
    n = ctypes.c_size_t()
    assert LIB.chunkkv_workspace_size(ctypes.byref(p), 1, 1, ctypes.byref(n)) == code


def test_null_and_misaligned_pointers_rejected_before_launch(ckv):
    from chunk_level_kv_gb300._lib import LIB
    p, keep = _p(ckv)
    P = ctypes.byref(p)
    ws_bytes = ckv.chunkkv_workspace_size(p)
    # null inputs, a misaligned pointer, a workspace that is too small: no launch happens
    assert LIB.chunkkv_score(P, None, None, None, None, 0, None) == 1
    assert LIB.chunkkv_score(P, 0x1001, 0x2000, 0x3000, 0x4000, ws_bytes, None) == 1
    assert LIB.chunkkv_score(P, 0x1000, 0x2000, 0x3000, 0x4000, 16, None) == 3
    assert LIB.chunkkv_select(P, None, None, None, None) == 1
    arr = (ctypes.c_void_p * 1)(0x1000)
    assert LIB.chunkkv_gather(P, 0, 0x1000, 0x2000, arr, arr, arr, arr, None) == 1   # zero layers
    assert LIB.chunkkv_gather(P, 65, 0x1000, 0x2000, arr, arr, arr, arr, None) == 1  # too many
    bad = (ctypes.c_void_p * 1)(0x1008)
    assert LIB.chunkkv_gather(P, 1, 0x1000, 0x2000, bad, arr, arr, arr, None) == 1
    assert LIB.chunkkv_compress_layers(P, 1, 0, arr, arr, arr, arr, arr, 0x1000, 0x2000, None,
                                       0x3000, ws_bytes, None) == 1                  # n_reuse 0
    assert LIB.chunkkv_status_check(None, None, None) == 1


def test_empty_batch_is_a_no_op(ckv):
    from chunk_level_kv_gb300._lib import LIB
    p, keep = _p(ckv, cu_seqlens=[0])
    assert ckv.chunkkv_out_capacity(p) == (0, 0)
    arr = (ctypes.c_void_p * 1)(0)
    assert LIB.chunkkv_compress_layers(ctypes.byref(p), 1, 1, arr, arr, arr, arr, arr, None, None, None,
                                       None, 0, None) == 0


def _plan(seqlens, Hq, Hkv, w, c, n_layers, n_reuse, d=128, slots=304, item_tiles=2):
    """The library's workspace plan replayed for the tensor-core path (bf16, d = 128): the unit
    length (chunks per unit) that minimises waves x (tiles per item + a fixed item cost of two
    tiles) over 304 CTA slots, ties to longer units, and the workspace bytes that follow."""
    from math import gcd
    align = lambda x: (x + 255) // 256 * 256
    G = Hq // Hkv
    wG = w * G
    Cs = [-(-T // c) for T in seqlens]
    MT = -(-wG // 128)
    base = 80 // gcd(80, c)                      # chunks in lcm(80, c) keys
    base_tiles = base * c // 80
    per_unit_items = Hkv * MT
    best = cpu = None
    for m in range(1, 65):
        cc = base * m
        items = sum(-(-C // cc) for C in Cs) * per_unit_items
        if items == 0:
            break
        cost = -(-items // slots) * (m * base_tiles + item_tiles)
        if best is None or cost <= best:
            best, cpu = cost, cc
        if items <= per_unit_items:
            break
    units = sum(-(-C // cpu) for C in Cs) * Hkv
    groups = -(-n_layers // n_reuse)
    B = len(seqlens)
    slot = align(units * 2 * wG * 4) + align(units * cpu * wG * 2) + align(B * Hkv * wG * 4)
    qpack = align(B * Hkv * MT * 128 * d * 2)
    scores = align(B * Hkv * max(Cs) * 4)
    return 256 + groups * (slot + qpack + scores), cpu


@pytest.mark.parametrize("shape", ["llama_32k", "qwen_128k", "mistral_c3", "mistral_c10", "mistral_c30"])
def test_planner_unit_length(ckv, shape):
    # The workspace size follows the planner's unit length: it must match the replayed plan, and
    # for the ragged 16-prompt batch the fixed item cost must keep units several tiles long (with
    # a cost of tiles alone the planner picked one-tile units there)
    import torch
    from synthetic import configs
    mistral = configs.mistral_ragged().seqlens
    case = {"llama_32k": ((32768,), 32, 8, 32, 10, 32, 2), "qwen_128k": ((131072,), 28, 4, 64, 10, 28, 2),
            "mistral_c3": (mistral, 32, 8, 32, 3, 32, 2), "mistral_c10": (mistral, 32, 8, 32, 10, 32, 2),
            "mistral_c30": (mistral, 32, 8, 32, 30, 32, 2)}[shape]
    seqlens, Hq, Hkv, w, c, n_layers, n_reuse = case
    cu = [0]
    for T in seqlens:
        cu.append(cu[-1] + T)
    p, keep = _p(ckv, cu_seqlens=cu, Hq=Hq, Hkv=Hkv, d=128, w=w, c=c, L_max=256, dtype=torch.bfloat16)
    want, cpu = _plan(seqlens, Hq, Hkv, w, c, n_layers, n_reuse)
    assert ckv.chunkkv_workspace_size(p, n_layers, n_reuse) == want
    if shape.startswith("mistral"):
        assert cpu * c >= 4 * 80, f"units of {cpu * c} keys"


def test_rescale_inputs_cross_the_threshold(ckv):
    # The GPU test of the scoring kernel's rescale relies on two facts checked here on the CPU: the
    # library plans 240-key work items for one 8192-token LLaMA-shaped layer (so the planted key at
    # offset 150 of every item lies in its second tile), and with bf16 inputs that key stands more
    # than 23 bits above the first tile's maximum for the rows along u, and far below for the others.
    import math
    import torch
    from synthetic import configs
    from test_gpu_parity_limits import _rescale_inputs
    wl = configs.llama_layer()
    p, keep = _p(ckv, cu_seqlens=[0, wl.T_total], Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                 L_max=wl.L_max, dtype=torch.bfloat16)
    want, cpu = _plan((wl.T_total,), wl.Hq, wl.Hkv, wl.w, wl.c, 1, 1)
    assert ckv.chunkkv_workspace_size(p, 1, 1) == want and cpu * wl.c == 240
    q, k, _, pos = _rescale_inputs(wl.T_total, wl.Hq, wl.Hkv, wl.w, wl.d, 240, 150)
    q, k = q.to(torch.bfloat16).double(), k.to(torch.bfloat16).double()
    G = wl.Hq // wl.Hkv
    for h in range(wl.Hkv):
        rows = torch.cat([q[0, :, h * G + g, :] for g in range(G)], 0)                 # (member, window row)
        s = rows @ k[:, h, :].T / math.sqrt(wl.d) * (1 / math.log(2))                # base-2 logits
        for u0 in range(0, wl.T_total - 240, 240):
            lift = s[:, u0 + 150] - s[:, u0:u0 + 80].max(dim=1).values
            assert lift[0::2].min() > 23 and lift[1::2].max() < -23


def test_tail_pass_sizes_and_argument_checks(ckv):
    # the incremental pass sizes its outputs from the new tails, its workspace from prefix + tail
    from chunk_level_kv_gb300._lib import LIB
    p, keep = _p(ckv, cu_seqlens=[0, 500, 1300], c=10, w=8, L_max=50)
    n_cap, c_max, ws = ckv.chunkkv_tail_sizes(p, [300, 0])
    assert (n_cap, c_max) == (58, 80)                  # tails of 200 and 800 tokens; k = 5
    assert ws >= ckv.chunkkv_workspace_size(p) > 0
    assert ckv.chunkkv_tail_sizes(p, [500, 800])[:2] == (0, 0)      # nothing new: nothing to append
    P = ctypes.byref(p)
    n_cap_, c_, w_ = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    out = (ctypes.byref(n_cap_), ctypes.byref(c_), ctypes.byref(w_))

    def sizes(n_prev, n_layers=1, n_reuse=1):
        arr = (ctypes.c_int32 * 2)(*n_prev) if n_prev is not None else None
        return LIB.chunkkv_tail_sizes(P, arr, n_layers, n_reuse, *out)
    assert sizes([501, 0]) == 1                        # a prefix longer than its cache
    assert sizes([-1, 0]) == 1
    assert sizes(None) == 1
    assert sizes([300, 0], 0, 1) == 1 and sizes([300, 0], 4, 0) == 1      # no layers, no reuse depth
    assert sizes([300, 0], 4, 2) == 0 and w_.value > ws                    # two scoring layers: two scratch slots
    pc, keep_c = _p(ckv, cu_seqlens=[0, 500, 1300], causal_window=True)
    assert LIB.chunkkv_tail_sizes(ctypes.byref(pc), (ctypes.c_int32 * 2)(0, 0), 1, 1, *out) == 2
    pb, keep_b = _p(ckv, cu_seqlens=list(range(0, 600)))   # 599 caches: the paired table would exceed the batch limit
    assert LIB.chunkkv_tail_sizes(ctypes.byref(pb), (ctypes.c_int32 * 599)(), 1, 1, *out) == 2
    # null or misaligned pointers and a short workspace are rejected before any launch
    n_prev = (ctypes.c_int32 * 2)(300, 0)
    arr = lambda x: (ctypes.c_void_p * 1)(x)
    assert LIB.chunkkv_compress_tail(P, n_prev, 1, 1, None, None, None, None, None, None, None, None, None, 0,
                                     None) == 1
    assert LIB.chunkkv_compress_tail(P, n_prev, 1, 1, arr(0x1000), arr(0x2008), arr(0x3000), arr(0x4000),
                                     arr(0x5000), 0x6000, 0x7000, None, 0x8000, ws, None) == 1
    assert LIB.chunkkv_compress_tail(P, n_prev, 1, 1, arr(0x1000), arr(0x2000), arr(0x3000), arr(0x4000),
                                     arr(0x5000), 0x6000, 0x7000, None, 0x8000, 16, None) == 3
