"""CUDA library vs CPU oracle on seeded inputs (needs a GB300; calls go through the C-ABI)."""
import itertools
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from parity import check_gather, check_indices, check_scores, f64
from synthetic import configs, generator as gen
from synthetic.generator import NeedleSpec

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def ckv():
    import chunk_level_kv_gb300 as m     # fails loudly if the library was not built
    return m


_POOL = ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1)))


def oracle_group_scores(wl, q, k, heads, seqs, causal=False):
    """Oracle chunk scores {(b, h): A} of one scoring layer (q [B, w, Hq, d], k [T_total, Hkv, d]) for the
    given sequences and heads; the heads of one sequence run in parallel threads (numpy releases the
    interpreter lock inside its array loops and BLAS)."""
    qf = f64(q)
    cu = wl.cu_seqlens
    out = {}
    for b in seqs:
        T = cu[b + 1] - cu[b]
        kb = f64(k[cu[b]:cu[b + 1]])

        def one(h, b=b, T=T, kb=kb):
            rows = oracle.group_window_rows(qf[b], h, wl.G)
            lim = oracle.window_limits(rows.shape[0], T, wl.w) if causal else None
            return oracle.chunk_scores(oracle.key_scores(rows, kb[:, h], lim), wl.c)

        for h, A in zip(heads, _POOL.map(one, heads)):
            out[(b, h)] = A
        del kb
    return out


def run_and_check(ckv, wl, layers_to_check=None, heads=None, seqs=None, qs=None, ks=None, vs=None,
                  spans=None, causal=False, oracle_cache=None):
    """Compress all layers on the GPU; compare scoring groups / heads / sequences with the oracle.

    oracle_cache: optional dict {(group, b, h): A} of oracle chunk scores to reuse (they depend on the
    inputs, c and the causal option only, not on L_max); filled with what this call computes."""
    if ks is None:
        qs, ks, vs, spans = gen.make_all_layers(wl, DEV)
    out = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c,
                              L_max=wl.L_max, n_reuse=wl.n_reuse, return_scores=True, causal_window=causal)
    assert ckv.chunkkv_status_check(out.workspace) == 0
    cu = wl.cu_seqlens
    groups = range(-(-wl.n_layers // wl.n_reuse)) if layers_to_check is None else layers_to_check
    heads = list(range(wl.Hkv)) if heads is None else list(heads)
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    scores = out.chunk_scores.cpu().numpy()
    idx = out.indices.cpu().numpy()
    cnt = out.counts.cpu().numpy()
    verdicts = []
    for g in groups:
        layer = g * wl.n_reuse
        if oracle_cache is not None and all((g, b, h) in oracle_cache for b in seqs for h in heads):
            ref = {(b, h): oracle_cache[(g, b, h)] for b in seqs for h in heads}
        else:
            ref = oracle_group_scores(wl, qs[layer], ks[layer], heads, seqs, causal)
            if oracle_cache is not None:
                oracle_cache.update({(g, b, h): A for (b, h), A in ref.items()})
        for b in seqs:
            T = cu[b + 1] - cu[b]
            for h in heads:
                A = ref[(b, h)]
                what = f"{wl.name} group {g} seq {b} head {h}"
                check_scores(scores[g, b, h], A, what)
                n = int(cnt[g, b, h])
                verdicts.append(check_indices(idx[g, b, h, :n], A, T, wl.c, wl.w, wl.L_max, what))
                for layer2 in range(layer, min(layer + wl.n_reuse, wl.n_layers)):
                    src = ks[layer2][cu[b]:cu[b + 1], h]
                    check_gather(out.k_out[layer2][b, h, :n], src, idx[g, b, h, :n], what + " K'")
                    check_gather(out.v_out[layer2][b, h, :n], vs[layer2][cu[b]:cu[b + 1], h],
                                 idx[g, b, h, :n], what + " V'")
    return out, verdicts


def test_tiny_fp32_exact(ckv):
    wl = configs.tiny()
    out, verdicts = run_and_check(ckv, wl)
    assert verdicts == ["exact", "exact"]
    # the planted chunk wins in both heads
    spans = gen.needle_spans(wl)[0][0]
    (s, e), = spans
    sc = out.chunk_scores[0, 0].cpu().numpy()
    assert all(int(np.argmax(sc[h, :52])) == s // wl.c for h in range(2))


@pytest.mark.parametrize("T,c,w,Hq,Hkv,L_max", [
    (3001, 10, 32, 32, 8, 300),      # several tiles, ragged last chunk and unit
    (2999, 3, 16, 8, 8, 256),        # c = 3, G = 1
    (4500, 30, 64, 28, 4, 900),      # c = 30, G = 7, window rows 448
    (1777, 1, 8, 4, 2, 100),         # token-level selection (c = 1)
    (640, 7, 5, 6, 2, 70),           # odd chunk, odd window
    (5000, 10, 48, 40, 8, 500),      # window rows 240: two M tiles in one CTA, the second partly padding
    (2500, 5, 40, 32, 4, 300),       # window rows 320: three M tiles, the last CTA's second tile all padding
    (3333, 16, 64, 16, 2, 512),      # window rows 512: four full M tiles, c = 16
    (2345, 15, 32, 32, 8, 450),      # c = 15 (the notes' ablation): chunk size read at run time
    (1999, 2, 32, 28, 4, 200),       # c = 2, window rows 224: a chunk end in every column pair
    (4100, 100, 16, 16, 4, 1000),    # c = 100: chunks spanning tiles, a whole-tile unit of 400 keys
    (3000, 1, 32, 28, 4, 256),       # token-level selection on 224 window rows (two M tiles)
    (3001, 1, 64, 28, 4, 700),       # token-level, two passes on 448 window rows (last M tile half padding)
    (2600, 1, 32, 32, 8, 400),       # token-level, two passes on 128 window rows
    (2100, 1, 24, 28, 4, 300),       # token-level, two passes on packed window rows (w = 24), 168 rows
])
def test_bf16_shapes(ckv, T, c, w, Hq, Hkv, L_max):
    wl = configs.llama_layer().with_params(seqlens=(T,), c=c, w=w, Hq=Hq, Hkv=Hkv, L_max=L_max,
                                           name=f"bf16_T{T}_c{c}_w{w}_G{Hq // Hkv}")
    p, keep = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                              L_max=wl.L_max, dtype=torch.bfloat16)
    assert ckv.chunkkv_score_path(p) == 1          # every chunk size up to 4096 on the tensor cores
    run_and_check(ckv, wl)


@pytest.mark.parametrize("c", [1, 7, 15])
def test_tensor_core_chunk_sizes_on_a_ragged_batch(ckv, c):
    # token-level chunks and chunk sizes read at run time, over ragged sequences (empty, shorter than
    # the window, shorter than one tile, several units) and two reuse groups, with the causal window too
    wl = configs.mistral_ragged().with_params(seqlens=(1000, 0, 20, 2500, 7, 333), B=6, n_layers=3,
                                              L_max=256, c=c, name=f"ragged_tc_c{c}")
    run_and_check(ckv, wl)
    run_and_check(ckv, wl.with_params(name=f"ragged_tc_c{c}_causal"), causal=True)


def test_ragged_batch_with_degenerate_sequences(ckv):
    # empty sequence, shorter than the window, shorter than one chunk, budget above T
    wl = configs.mistral_ragged().with_params(seqlens=(1000, 0, 20, 2500, 7, 333), B=6, n_layers=3,
                                              L_max=256, name="ragged6")
    run_and_check(ckv, wl)


@pytest.mark.parametrize("kw", [
    dict(L_max=100000),              # every chunk kept: K' = K
    dict(L_max=5),                   # L_max < c: only the recent window
    dict(w=0),                       # no window: scores all zero, ties to the lowest chunks
    dict(c=5000),                    # one chunk longer than the prompt
])
def test_degenerate_parameters(ckv, kw):
    wl = configs.llama_layer().with_params(seqlens=(1234,), name=f"deg_{list(kw)[0]}", **kw)
    out, _ = run_and_check(ckv, wl)
    if kw.get("L_max") == 100000:
        n = int(out.counts[0, 0, 0])
        assert n == 1234 and torch.equal(out.indices[0, 0, 0, :n].cpu(), torch.arange(1234, dtype=torch.int32))


def test_maximum_batch_ragged(ckv):
    # CHUNKKV_MAX_BATCH sequences of 0..400 tokens (empty, shorter than the window, several units)
    rng = np.random.default_rng(2024)
    seqlens = tuple(int(x) for x in rng.integers(0, 401, size=1024))
    seqlens = (0,) + seqlens[1:511] + (7,) + seqlens[512:]
    wl = configs.mistral_ragged().with_params(seqlens=seqlens, B=1024, Hq=8, Hkv=2, w=16, L_max=64,
                                              n_layers=2, n_reuse=2, needles=NeedleSpec(kind="none"),
                                              name="max_batch_1024")
    run_and_check(ckv, wl, seqs=[0, 1, 2, 511, 700, 1023])


def test_maximum_window_rows(ckv):
    # w*G = 4096 window rows per KV head (the library's limit): 32 M tiles on the tensor-core path
    wl = configs.llama_layer().with_params(seqlens=(1500,), Hq=32, Hkv=1, w=128, L_max=300, name="wG4096")
    p, keep = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                              L_max=wl.L_max, dtype=torch.bfloat16)
    assert ckv.chunkkv_score_path(p) == 1
    run_and_check(ckv, wl)


@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (256, "bf16"), (256, "f32")])
def test_other_head_dims_portable_path(ckv, d, dtype):
    wl = configs.llama_layer().with_params(seqlens=(900,), d=d, dtype=dtype, Hq=8, Hkv=2, w=8, L_max=100,
                                           name=f"d{d}_{dtype}")
    run_and_check(ckv, wl)


@pytest.mark.parametrize("Hq,Hkv,w", [(32, 8, 32), (28, 4, 64)])
def test_layer_reuse_groups(ckv, Hq, Hkv, w):
    # one scoring launch covers the three reuse groups (one and two M tiles per CTA)
    wl = configs.llama_model().with_params(seqlens=(2048,), n_layers=5, n_reuse=2, L_max=409, Hq=Hq, Hkv=Hkv,
                                           w=w, name=f"reuse5_G{Hq // Hkv}_w{w}")
    out, _ = run_and_check(ckv, wl)
    assert out.indices.shape[0] == 3


@pytest.mark.parametrize("B,w,Hq,launches", [(1, 32, 32, 5), (1, 48, 40, 6), (5, 32, 32, 3), (12, 32, 32, 5)])
def test_one_launch_per_phase(ckv, B, w, Hq, launches):
    # score (all reuse groups), log-sum-exp, finalize, select, gather (all layers).  A packing launch
    # comes first only when the scoring kernel cannot read the window rows from Q_w through a tensor
    # map (w does not divide 128).  With 5 sequences x 8 KV heads x 3 reuse groups = 120 heads (one
    # wave of one CTA per SM, 79 % of 152 SMs) one kernel takes log-sum-exp, finalisation and
    # selection; with 12 sequences (288 heads, two waves) the separate kernels run again.
    wl = configs.llama_model().with_params(seqlens=(3000,) * B, B=B, n_layers=6, n_reuse=2, L_max=600, w=w,
                                           Hq=Hq, name=f"phases_B{B}_w{w}")
    qs, ks, vs, _ = gen.make_all_layers(wl, DEV)
    ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max,
                        n_reuse=wl.n_reuse)
    torch.cuda.synchronize()
    n0 = ckv.chunkkv_launch_count()
    out = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max,
                              n_reuse=wl.n_reuse)
    assert ckv.chunkkv_launch_count() - n0 == launches
    assert ckv.chunkkv_status_check(out.workspace) == 0


def test_head_kernel_on_a_ragged_batch(ckv):
    # 5 ragged sequences (one empty, two shorter than the window, one several units long) x 8 KV heads
    # x 3 reuse groups = 120 heads, one wave: log-sum-exp, finalisation and selection run as one kernel
    # per head (three launches per call); checked against the oracle like every other path
    seqlens = (3000, 77, 5, 4096, 0)
    wl = configs.mistral_ragged().with_params(seqlens=seqlens, B=len(seqlens), n_layers=6, n_reuse=2, L_max=600,
                                              needles=NeedleSpec(kind="none"), name="head_ragged5")
    n0 = ckv.chunkkv_launch_count()
    out, _ = run_and_check(ckv, wl)
    assert ckv.chunkkv_launch_count() - n0 == 3                    # score, head_kernel, gather
    assert not out.counts[:, 4].any()                              # the empty sequence keeps nothing


def test_phase_events_mark_every_phase(ckv):
    wl = configs.llama_model().with_params(seqlens=(3000,), n_layers=4, n_reuse=2, L_max=600, name="phase_events")
    qs, ks, vs, _ = gen.make_all_layers(wl, DEV)
    kw = dict(Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max, n_reuse=wl.n_reuse)
    ref = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, **kw)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(ckv.PHASES) + 1)]
    ckv.chunkkv_set_phase_events(evs)
    try:
        out = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, **kw)
    finally:
        ckv.chunkkv_set_phase_events(None)
    torch.cuda.synchronize()
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(ckv.PHASES))]
    assert all(t >= 0 for t in times) and times[1] > 0 and times[-1] > 0
    assert torch.equal(out.indices, ref.indices) and torch.equal(out.counts, ref.counts)
    assert all(torch.equal(a, b) for a, b in zip(out.k_out, ref.k_out))


@pytest.mark.parametrize("n_layers,n_reuse,seqlens", [(6, 2, (2500, 0, 4100)), (64, 1, (700, 333))])
def test_claimed_items_counter_returns_to_zero(ckv, n_layers, n_reuse, seqlens):
    # The tensor-core scoring CTAs claim their work items from a counter in the workspace header
    # (int32 words 4 and 5: next item, finished CTAs), which the launch's last CTA sets back to zero.
    # Calls that share a workspace then see every item: repeated calls give identical outputs, and so
    # does the second scoring launch of a call with more than 32 reuse groups (64 layers, N_reuse 1).
    wl = configs.llama_model().with_params(seqlens=seqlens, B=len(seqlens), n_layers=n_layers, n_reuse=n_reuse, L_max=300,
                                           name=f"claim_counter_{n_layers}L")
    qs, ks, vs, spans = gen.make_all_layers(wl, DEV)
    p, _ = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                           L_max=wl.L_max, dtype=torch.bfloat16)
    assert ckv.chunkkv_score_path(p) == 1
    first, _ = run_and_check(ckv, wl, qs=qs, ks=ks, vs=vs, spans=spans,
                             layers_to_check=None if n_layers < 10 else [0, 31, 32, 63])
    header = lambda out: out.workspace[:32].view(torch.int32).cpu()
    assert header(first)[4] == 0 and header(first)[5] == 0
    kw = dict(Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max, n_reuse=wl.n_reuse, return_scores=True)
    cu = wl.cu_seqlens
    n_chunks = [-(-(cu[b + 1] - cu[b]) // wl.c) for b in range(wl.B)]   # entries past them are not written
    for _ in range(3):
        again = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, workspace=first.workspace, **kw)
        assert ckv.chunkkv_status_check(again.workspace) == 0
        assert header(again)[4] == 0 and header(again)[5] == 0
        assert torch.equal(again.counts, first.counts)
        for b, C in enumerate(n_chunks):
            assert torch.equal(again.chunk_scores[:, b, :, :C], first.chunk_scores[:, b, :, :C])
            for grp in range(first.counts.shape[0]):
                for h in range(wl.Hkv):
                    n = int(first.counts[grp, b, h])
                    assert torch.equal(again.indices[grp, b, h, :n], first.indices[grp, b, h, :n])
                    for layer in range(grp * wl.n_reuse, min((grp + 1) * wl.n_reuse, wl.n_layers)):
                        assert torch.equal(again.k_out[layer][b, h, :n], first.k_out[layer][b, h, :n])
                        assert torch.equal(again.v_out[layer][b, h, :n], first.v_out[layer][b, h, :n])


def test_bounded_wait_gives_up_and_reports(ckv):
    import ctypes
    from chunk_level_kv_gb300._lib import LIB
    from chunk_level_kv_gb300.api import _stream
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    pattern = torch.arange(64, dtype=torch.uint8, device=DEV) * 3 + 7
    ws[128:192] = pattern                                 # what the self test copies asynchronously
    ckv.chunkkv_selftest_wait_timeout(ws)
    code = ctypes.c_int32()
    st = LIB.chunkkv_status_check(ctypes.c_void_p(ws.data_ptr()), _stream(ws.device), ctypes.byref(code))
    assert st == 5 and code.value == 0x1FF                 # CHUNKKV_ERR_TIMEOUT, the self-test site
    # after giving up, the kernel waited for its own copy to land before it returned (the teardown
    # drain of the scoring kernel): the copied bytes are what it wrote back
    assert torch.equal(ws[64:128], pattern)
    assert ckv.chunkkv_status_check(ws) == 0              # the word was cleared ...
    wl = configs.tiny()                                   # ... and the context still computes
    out, verdicts = run_and_check(ckv, wl)
    assert verdicts == ["exact", "exact"]


@pytest.mark.parametrize("case", ["llama6", "ragged3"])
def test_layer_overlap_counts(ckv, case):
    # adjacent-layer overlap of the kept lists of independently scored layers (n_reuse = 1),
    # bit-exact against the oracle's set counts on the GPU's own lists
    if case == "llama6":
        wl = configs.llama_model().with_params(seqlens=(3000,), n_layers=6, n_reuse=1, L_max=600, name="overlap6")
    else:
        wl = configs.mistral_ragged().with_params(seqlens=(1000, 0, 20, 2500, 7, 333), B=6, n_layers=3,
                                                  n_reuse=1, L_max=256, name="overlap_ragged")
    qs, ks, vs, _ = gen.make_all_layers(wl, DEV)
    out = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max,
                              n_reuse=1)
    p, keep = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                              L_max=wl.L_max, dtype=ks[0].dtype)
    inter, uni = ckv.chunkkv_layer_overlap(p, out.indices, out.counts)
    idx, cnt = out.indices.cpu().numpy(), out.counts.cpu().numpy()
    inter, uni = inter.cpu().numpy(), uni.cpu().numpy()
    jac = []
    for l in range(wl.n_layers - 1):
        for b in range(wl.B):
            for h in range(wl.Hkv):
                want = oracle.layer_overlap(idx[l, b, h, :cnt[l, b, h]], idx[l + 1, b, h, :cnt[l + 1, b, h]])
                assert (int(inter[l, b, h]), int(uni[l, b, h])) == want, (l, b, h)
                if want[1]:
                    jac.append(want[0] / want[1])
    if case == "llama6":
        # 16 of 20 needle spans survive from layer to layer: selections overlap well above chance
        assert np.mean(jac) > 0.2


def test_layer_overlap_on_given_lists(ckv):
    # identical, disjoint and partly overlapping lists, and positions outside [0, T) ignored
    T, n_cap = 100, 8
    p, keep = ckv.make_params(cu_seqlens=[0, T], Hq=2, Hkv=2, d=64, w=4, c=2, L_max=4, dtype=torch.float32)
    lists = np.full((3, 1, 2, n_cap), -1, dtype=np.int32)
    cnt = np.zeros((3, 1, 2), dtype=np.int32)
    lists[0, 0, 0, :4], cnt[0, 0, 0] = [1, 5, 9, 97], 4
    lists[1, 0, 0, :4], cnt[1, 0, 0] = [1, 5, 9, 97], 4
    lists[2, 0, 0, :3], cnt[2, 0, 0] = [2, 5, 98], 3
    lists[0, 0, 1, :2], cnt[0, 0, 1] = [0, 1], 2
    lists[1, 0, 1, :3], cnt[1, 0, 1] = [2, 3, 150], 3          # 150 >= T: ignored by the probe
    lists[2, 0, 1, :0], cnt[2, 0, 1] = [], 0
    n_cap_lib, _ = ckv.chunkkv_out_capacity(p)
    buf = np.full((3, 1, 2, n_cap_lib), -1, dtype=np.int32)
    buf[..., :n_cap] = lists
    inter, uni = ckv.chunkkv_layer_overlap(p, torch.from_numpy(buf).to(DEV), torch.from_numpy(cnt).to(DEV))
    assert inter.cpu().tolist() == [[[4, 0]], [[1, 0]]]
    assert uni.cpu().tolist() == [[[4, 5]], [[6, 3]]]


@pytest.mark.parametrize("case", ["tiny_f32", "bf16_G4", "bf16_G7_c30", "ragged_short"])
def test_causal_window(ckv, case):
    # chunkkv_params.causal_window = 1: window query q sees keys up to T - w + q (reading R10)
    if case == "tiny_f32":
        wl = configs.tiny()
    elif case == "bf16_G4":
        wl = configs.llama_layer().with_params(seqlens=(3001,), L_max=300, name="causal_G4")
    elif case == "bf16_G7_c30":
        wl = configs.llama_layer().with_params(seqlens=(4500,), c=30, w=64, Hq=28, Hkv=4, L_max=900,
                                               name="causal_G7")
    else:
        wl = configs.mistral_ragged().with_params(seqlens=(1000, 0, 20, 2500, 7, 333), B=6, n_layers=3,
                                                  L_max=256, name="causal_ragged")
    out, _ = run_and_check(ckv, wl, causal=True)
    # the option changes the scores of the chunks inside the window
    plain, _ = run_and_check(ckv, wl, causal=False)
    assert not torch.equal(out.chunk_scores, plain.chunk_scores)


def test_hybrid_chunk_then_token_level(ckv):
    # §5.7 hybrid policy: chunk-level selection (c = 10) in the lower half of the layers and
    # token-level selection (c = 1) in the upper half, as two calls over the two halves
    wl = configs.llama_model().with_params(seqlens=(2500,), n_layers=4, n_reuse=1, L_max=500, name="hybrid")
    qs, ks, vs, spans = gen.make_all_layers(wl, DEV)
    lower = wl.with_params(n_layers=2, name="hybrid_lower_c10")
    upper = wl.with_params(n_layers=2, c=1, name="hybrid_upper_c1")
    out_lo, _ = run_and_check(ckv, lower, qs=qs[:2], ks=ks[:2], vs=vs[:2], spans=spans[:2])
    out_hi, _ = run_and_check(ckv, upper, qs=qs[2:], ks=ks[2:], vs=vs[2:], spans=spans[2:])
    assert out_lo.indices.shape[-1] >= 500 and out_hi.indices.shape[-1] >= 500


def test_decode_time_recompression(ckv):
    # Decode-time compression (reading R11): the score-based paradigm of Kara §2 Eqs. (2)-(3)
    # compresses again once the cache reaches its threshold.  Here the cache of each (sequence,
    # KV head) is its compressed prompt followed by the tokens decoded since, and Algorithm 1 runs
    # over it with the latest w queries as the window.  Heads keep different counts after the
    # first pass, so the second pass treats every head's cache as a sequence of its own (one KV
    # head, its G query heads).
    wl = configs.llama_layer().with_params(seqlens=(3001,), L_max=600, name="decode_prefill")
    out1, _ = run_and_check(ckv, wl)
    n1 = [int(x) for x in out1.counts[0, 0].cpu()]
    tail = 347                                   # tokens decoded since the first pass
    assert all(n + tail > wl.L_max + wl.w for n in n1)
    wl2 = wl.with_params(seqlens=tuple(n + tail for n in n1), B=wl.Hkv, Hq=wl.G, Hkv=1, seed=wl.seed + 500,
                         needles=NeedleSpec(kind="none"), name="decode_recompress")
    q2 = gen.gen_q_window(wl2, 0, DEV)
    k2 = gen.gen_kv_raw(wl2, 0, gen.TENSOR_K, DEV)
    v2 = gen.gen_kv_raw(wl2, 0, gen.TENSOR_V, DEV)
    cu2 = wl2.cu_seqlens
    for h, n in enumerate(n1):                   # the compressed prompt, then the decoded tokens
        k2[cu2[h]:cu2[h] + n, 0] = out1.k_out[0][0, h, :n]
        v2[cu2[h]:cu2[h] + n, 0] = out1.v_out[0][0, h, :n]
    out2, _ = run_and_check(ckv, wl2, qs=[q2], ks=[k2], vs=[v2], spans=[None])
    # the second pass keeps the newest w tokens of every cache
    for h, n in enumerate(n1):
        cnt = int(out2.counts[0, h, 0])
        got = out2.indices[0, h, 0, :cnt].cpu().numpy()
        T2 = n + tail
        assert (got[-wl.w:] == np.arange(T2 - wl.w, T2)).all()


def test_select_is_bit_exact_on_given_scores(ckv):
    # both sides decide on the same fp32 scores: the selection must match exactly (ties included)
    rng = np.random.default_rng(0)
    seqlens = [1000, 57, 0, 4096, 333]
    cu = [0] + list(itertools.accumulate(seqlens))
    c, w, L_max, Hkv = 10, 16, 200, 3
    p, keep = ckv.make_params(cu_seqlens=cu, Hq=Hkv, Hkv=Hkv, d=64, w=w, c=c, L_max=L_max,
                              dtype=torch.bfloat16)
    n_cap, C_max = ckv.chunkkv_out_capacity(p)
    scores = rng.integers(0, 6, size=(len(seqlens), Hkv, C_max)).astype(np.float32) * 0.125
    scores[1] = -scores[1]                    # negative scores and -0.0 order correctly too
    dev_scores = torch.from_numpy(scores).to(DEV)
    indices = torch.full((len(seqlens), Hkv, n_cap), -1, dtype=torch.int32, device=DEV)
    counts = torch.zeros(len(seqlens), Hkv, dtype=torch.int32, device=DEV)
    ckv.chunkkv_select(p, dev_scores, indices, counts)
    torch.cuda.synchronize()
    for b, T in enumerate(seqlens):
        C = -(-T // c)
        for h in range(Hkv):
            A = scores[b, h, :C].astype(np.float64)
            want = oracle.kept_indices(oracle.top_chunks(A, oracle.n_select(T, c, L_max)), T, c, w)
            n = int(counts[b, h])
            assert n == len(want)
            assert np.array_equal(indices[b, h, :n].cpu().numpy(), want)


def test_gather_is_bit_exact(ckv):
    rng = np.random.default_rng(1)
    seqlens = [300, 1, 77]
    cu = [0] + list(itertools.accumulate(seqlens))
    Hkv, d = 2, 128
    p, keep = ckv.make_params(cu_seqlens=cu, Hq=Hkv, Hkv=Hkv, d=d, w=4, c=10, L_max=64,
                              dtype=torch.bfloat16)
    n_cap, _ = ckv.chunkkv_out_capacity(p)
    k = [torch.randn(cu[-1], Hkv, d, device=DEV).to(torch.bfloat16) for _ in range(3)]
    v = [torch.randn(cu[-1], Hkv, d, device=DEV).to(torch.bfloat16) for _ in range(3)]
    counts = torch.tensor([[min(n_cap, T), min(n_cap, T) // 2] for T in seqlens], dtype=torch.int32)
    idx = torch.zeros(len(seqlens), Hkv, n_cap, dtype=torch.int32)
    for b, T in enumerate(seqlens):
        for h in range(Hkv):
            n = int(counts[b, h])
            idx[b, h, :n] = torch.from_numpy(np.sort(rng.choice(T, size=n, replace=False))).int()
    ko = [torch.zeros(len(seqlens), Hkv, n_cap, d, dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    vo = [torch.zeros_like(x) for x in ko]
    ckv.chunkkv_gather(p, idx.to(DEV), counts.to(DEV), k, v, ko, vo)
    torch.cuda.synchronize()
    for layer in range(3):
        for b in range(len(seqlens)):
            for h in range(Hkv):
                n = int(counts[b, h])
                check_gather(ko[layer][b, h, :n], k[layer][cu[b]:cu[b + 1], h], idx[b, h, :n].numpy())
                check_gather(vo[layer][b, h, :n], v[layer][cu[b]:cu[b + 1], h], idx[b, h, :n].numpy())
                assert not ko[layer][b, h, n:].any()          # rows beyond the count are untouched


def test_gather_operands_in_pinned_host_memory(ckv):
    # K, V read from and K', V' written to pinned host memory by the gather kernel itself (the GPU
    # addresses it across the host link): bit-exact, rows beyond the count untouched
    rng = np.random.default_rng(2)
    seqlens = [500, 3, 129]
    cu = [0] + list(itertools.accumulate(seqlens))
    Hkv, d = 4, 128
    p, keep = ckv.make_params(cu_seqlens=cu, Hq=Hkv, Hkv=Hkv, d=d, w=8, c=10, L_max=100,
                              dtype=torch.bfloat16)
    n_cap, _ = ckv.chunkkv_out_capacity(p)
    k = [torch.randn(cu[-1], Hkv, d).to(torch.bfloat16).pin_memory() for _ in range(2)]
    v = [torch.randn(cu[-1], Hkv, d).to(torch.bfloat16).pin_memory() for _ in range(2)]
    counts = torch.tensor([[min(n_cap, T) - (h % 2) * min(n_cap, T) // 3 for h in range(Hkv)] for T in seqlens],
                          dtype=torch.int32)
    idx = torch.zeros(len(seqlens), Hkv, n_cap, dtype=torch.int32)
    for b, T in enumerate(seqlens):
        for h in range(Hkv):
            n = int(counts[b, h])
            idx[b, h, :n] = torch.from_numpy(np.sort(rng.choice(T, size=n, replace=False))).int()
    ko = [torch.zeros(len(seqlens), Hkv, n_cap, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    vo = [torch.zeros_like(x).pin_memory() for x in ko]
    ckv.chunkkv_gather(p, idx.to(DEV), counts.to(DEV), k, v, ko, vo)
    torch.cuda.synchronize()
    for layer in range(2):
        for b in range(len(seqlens)):
            for h in range(Hkv):
                n = int(counts[b, h])
                check_gather(ko[layer][b, h, :n], k[layer][cu[b]:cu[b + 1], h], idx[b, h, :n].numpy())
                check_gather(vo[layer][b, h, :n], v[layer][cu[b]:cu[b + 1], h], idx[b, h, :n].numpy())
                assert not ko[layer][b, h, n:].any() and not vo[layer][b, h, n:].any()


def test_compress_with_host_resident_kv(ckv):
    # the scoring layers' keys in device memory (the tensor-core kernel reads them through TMA), the
    # other layers' K and every V in pinned host memory, K' and V' written to pinned host memory:
    # identical to the all-device call.  A scoring layer's keys in host memory are rejected before
    # anything is launched.
    wl = configs.llama_model().with_params(seqlens=(3000, 1234), B=2, n_layers=4, n_reuse=2, L_max=600,
                                           name="host_kv")
    qs, ks, vs, _ = gen.make_all_layers(wl, DEV)
    ref = ckv.compress_layers(qs, ks, vs, wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, w=wl.w, c=wl.c,
                              L_max=wl.L_max, n_reuse=wl.n_reuse)
    p, keep = ckv.params_for(next(q for q in qs if q is not None), ks[0], wl.cu_seqlens, Hkv=wl.Hkv, w=wl.w,
                             c=wl.c, L_max=wl.L_max)
    assert ckv.chunkkv_score_path(p) == 1
    hk = [x.cpu().pin_memory() for x in ks]
    hv = [x.cpu().pin_memory() for x in vs]
    kmix = [ks[layer] if layer % wl.n_reuse == 0 else hk[layer] for layer in range(wl.n_layers)]
    hko = [torch.zeros(x.shape, dtype=x.dtype).pin_memory() for x in ref.k_out]
    hvo = [torch.zeros(x.shape, dtype=x.dtype).pin_memory() for x in ref.v_out]
    idx, cnt = torch.empty_like(ref.indices), torch.empty_like(ref.counts)
    ws = torch.zeros(ckv.chunkkv_workspace_size(p, wl.n_layers, wl.n_reuse), dtype=torch.uint8, device=DEV)
    ckv.chunkkv_compress_layers(p, wl.n_reuse, qs, kmix, hv, hko, hvo, idx, cnt, None, ws)
    torch.cuda.synchronize()
    assert torch.equal(cnt, ref.counts)
    counts = cnt.cpu()
    for layer in range(wl.n_layers):
        grp = layer // wl.n_reuse
        for b in range(wl.B):
            for h in range(wl.Hkv):
                n = int(counts[grp, b, h])
                assert torch.equal(idx[grp, b, h, :n], ref.indices[grp, b, h, :n])
                for got, want in ((hko, ref.k_out), (hvo, ref.v_out)):
                    assert torch.equal(got[layer][b, h, :n].view(torch.int16),
                                       want[layer][b, h, :n].cpu().view(torch.int16))
                    assert not got[layer][b, h, n:].any()
    assert ckv.chunkkv_status_check(ws) == 0
    kbad = [hk[0]] + list(ks[1:])
    with pytest.raises(ckv.ChunkKVError) as e:
        ckv.chunkkv_compress_layers(p, wl.n_reuse, qs, kbad, hv, hko, hvo, idx, cnt, None, ws)
    assert e.value.code == 1                  # CHUNKKV_ERR_INVALID_ARG, nothing launched


@pytest.mark.parametrize("c", [10, 1])
def test_score_entry_point_alone(ckv, c):
    # c = 1 takes the two passes over the keys (row lse, then per-key sums) inside chunkkv_score too
    wl = configs.llama_layer().with_params(seqlens=(5000, 3000), B=2, c=c, name=f"score_only_c{c}")
    q, k, v, _ = gen.make_all_layers(wl, DEV)
    p, keep = ckv.params_for(q[0], k[0], wl.cu_seqlens, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max)
    n_cap, C_max = ckv.chunkkv_out_capacity(p)
    ws = torch.zeros(ckv.chunkkv_workspace_size(p), dtype=torch.uint8, device=DEV)
    scores = torch.zeros(2, wl.Hkv, C_max, device=DEV)
    ckv.chunkkv_score(p, q[0], k[0], scores, ws)
    assert ckv.chunkkv_status_check(ws) == 0
    qf = f64(q[0])
    cu = wl.cu_seqlens
    for b in range(2):
        kb = f64(k[0][cu[b]:cu[b + 1]])
        for h in (0, 5):
            A = oracle.chunk_scores(oracle.key_scores(oracle.group_window_rows(qf[b], h, wl.G), kb[:, h]), wl.c)
            check_scores(scores[b, h].cpu().numpy(), A, f"seq {b} head {h}")


# ------------------------------------------------------------------ full-size workloads

def test_full_llama_layer_8k(ckv):
    _, verdicts = run_and_check(ckv, configs.llama_layer())
    assert len(verdicts) == 8


def test_full_llama_model_32k(ckv):
    # all 32 layers run exactly as the benchmark runs them; every reuse group, every head is compared
    # with the oracle, and every layer's gather is checked bit-exactly
    wl = configs.llama_model()
    _, verdicts = run_and_check(ckv, wl)
    assert len(verdicts) == 16 * 8


def test_full_qwen_128k(ckv):
    # every one of the 14 reuse groups x 4 KV heads (13108 chunk scores and 13164 kept indices each)
    wl = configs.qwen_128k()
    _, verdicts = run_and_check(ckv, wl)
    assert len(verdicts) == 14 * 4


@pytest.mark.parametrize("c,L_max", configs.MISTRAL_SWEEP)
def test_full_mistral_ragged_sweep(ckv, c, L_max, mistral_inputs):
    # every sweep point in full: 16 reuse groups x 16 ragged sequences x 8 KV heads; the oracle's
    # chunk scores depend on c only, so the three budgets of a chunk size share them
    wl, qs, ks, vs, spans, cache = mistral_inputs
    wl = wl.with_params(c=c, L_max=L_max, name=f"mistral_c{c}_L{L_max}")
    _, verdicts = run_and_check(ckv, wl, qs=qs, ks=ks, vs=vs, spans=spans,
                                oracle_cache=cache.setdefault(c, {}))
    assert len(verdicts) == 16 * 16 * 8


@pytest.fixture(scope="module")
def mistral_inputs():
    wl = configs.mistral_ragged()
    qs, ks, vs, spans = gen.make_all_layers(wl, DEV)
    return wl, qs, ks, vs, spans, {}


def test_tensor_core_path_is_selected_for_bf16_d128(ckv):
    # the shapes of the LLaMA / Mistral / Qwen workloads run the tcgen05 kernel
    for wl in (configs.llama_layer(), configs.llama_model(), configs.qwen_128k(),
               configs.mistral_ragged(c=3), configs.mistral_ragged(c=30),
               configs.llama_layer().with_params(c=1), configs.llama_layer().with_params(c=15)):
        p, keep = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                                  L_max=wl.L_max, dtype=torch.bfloat16)
        assert ckv.chunkkv_score_path(p) == 1, wl.name
    p, keep = ckv.make_params(cu_seqlens=[0, 512], Hq=4, Hkv=2, d=64, w=8, c=10, L_max=128, dtype=torch.float32)
    assert ckv.chunkkv_score_path(p) == 0
