"""chunkkv_score_noalloc: the scoring entry point for callers that cannot allocate.

Callers that run inside a memory pool or an allocator callback, or under a
device-memory budget fixed at start-up, cannot call cudaMalloc and may have no
workspace to lend.  chunkkv_score_noalloc keeps its scratch in a fixed device
array inside the library instead.  These tests call it through the C-ABI twice
in a row (the second call runs over scratch the first one left behind) and
hold every call to the CPU oracle and to chunkkv_score, which uses a caller
workspace, within the chunk-score tolerance used everywhere else
(abs 1e-5 + rel 1e-3).  The cases cover a ragged two-sequence bf16 batch, the
tiny fp32 layer, and the causal window, where rows see no key of some units.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import ATOL, RTOL, check_scores, f64
from synthetic import configs, generator as gen

pytestmark = pytest.mark.gpu


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return bool(np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)))


def _oracle_scores(wl, q, k, causal):
    qf, cu = f64(q), wl.cu_seqlens
    out = []
    for b in range(wl.B):
        kb = f64(k[cu[b]:cu[b + 1]])
        T = cu[b + 1] - cu[b]
        row = []
        for h in range(wl.Hkv):
            rows = oracle.group_window_rows(qf[b], h, wl.G)
            lim = oracle.window_limits(rows.shape[0], T, wl.w) if causal else None
            row.append(oracle.chunk_scores(oracle.key_scores(rows, kb[:, h], lim), wl.c))
        out.append(row)
    return out


@pytest.mark.parametrize("case", ["ragged_bf16", "tiny_f32", "causal_ragged_bf16"])
def test_noalloc_matches_the_oracle_and_workspace_scoring_twice_in_a_row(case):
    import chunk_level_kv_gb300 as ckv
    dev = torch.device("cuda:0")
    causal = case.startswith("causal")
    if case == "tiny_f32":
        wl = configs.tiny()
    else:
        # the second sequence is shorter than the causal window's reach into a unit: some rows of its
        # last unit see no key there
        wl = configs.llama_layer().with_params(seqlens=(8192, 1500) if not causal else (3001, 20), B=2,
                                               name=f"noalloc_{case}")
    q, k, v, _ = gen.make_all_layers(wl, dev)
    p, keep = ckv.params_for(q[0], k[0], wl.cu_seqlens, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max,
                             causal_window=causal)
    n_cap, C_max = ckv.chunkkv_out_capacity(p)
    ws = torch.zeros(ckv.chunkkv_workspace_size(p), dtype=torch.uint8, device=dev)
    want = torch.zeros(wl.B, wl.Hkv, C_max, device=dev)
    ckv.chunkkv_score(p, q[0], k[0], want, ws)
    ref = _oracle_scores(wl, q[0], k[0], causal)
    for call in range(2):
        got = torch.full((wl.B, wl.Hkv, C_max), float("nan"), device=dev)
        ckv.chunkkv_score_noalloc(p, q[0], k[0], got)
        torch.cuda.synchronize()
        g = got.cpu().numpy()
        for b in range(wl.B):
            C = -(-wl.seqlens[b] // wl.c)
            for h in range(wl.Hkv):
                check_scores(g[b, h, :C], ref[b][h], f"{wl.name} call {call} seq {b} head {h}")
            assert _close(got[b, :, :C], want[b, :, :C]), wl.name


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import chunk_level_kv_gb300 as ckv
    dev = torch.device("cuda:0")
    # 128K tokens with 448 window rows needs ~94 MB of scratch, far beyond the fixed array
    wl = configs.qwen_128k()
    p, keep = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                              L_max=wl.L_max, dtype=torch.bfloat16)
    buf = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ckv.ChunkKVError) as e:
        ckv.chunkkv_score_noalloc(p, buf, buf, buf)
    assert e.value.code == 3          # CHUNKKV_ERR_WORKSPACE_TOO_SMALL, nothing launched
    torch.cuda.synchronize()
