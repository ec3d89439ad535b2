"""Incremental compression during decoding (reading R12) through the C-ABI, against the CPU oracle.

A cache of one (sequence, KV head) holds the positions kept by earlier passes followed by the
tokens decoded since.  chunkkv_compress_tail re-scores only the new tail: every window row's
softmax runs over all keys of the cache (Kara §2 Eq. (1)), the tail is chunked from its first
token and ChunkKV §4.1 Algorithm 1 steps 2-6 select from it; with several layers, the layers that
do not score gather with their group's list (§4.2 Algorithm 2).  The oracle is
oracle.compress_tail_head; the comparison rules are tests/parity.py's (scores within 1e-5 + 1e-3
relative, indices exact unless the oracle's cut is a near-tie, gathered rows bit-exact).
"""
import pytest
import torch

import oracle
from parity import check_gather, check_indices, check_scores, f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def ckv():
    import chunk_level_kv_gb300 as m     # fails loudly if the library was not built
    return m


def _caches(pairs, Hkv, G, d, w, dtype, seed, needle_len=0):
    """Seeded caches [(n_prev, n_new)]: q [B, w, Hkv*G, d], k, v [sum T, Hkv, d]; with needle_len, a
    run of tail keys in each cache is set along its heads' mean window query (found if selection works)."""
    g = torch.Generator().manual_seed(seed)
    B = len(pairs)
    cu = [0]
    for n_prev, n_new in pairs:
        cu.append(cu[-1] + n_prev + n_new)
    q = torch.randn(B, w, Hkv * G, d, generator=g)
    scale = torch.empty(Hkv, d).uniform_(0.5, 2.0, generator=g)
    k = torch.randn(cu[-1], Hkv, d, generator=g) * scale
    v = torch.randn(cu[-1], Hkv, d, generator=g)
    if needle_len:
        for b, (n_prev, n_new) in enumerate(pairs):
            if n_new < needle_len + w + 1:
                continue
            s = n_prev + int(torch.randint(0, n_new - needle_len - w, (1,), generator=g))
            for h in range(Hkv):
                qm = q[b, :, h * G:(h + 1) * G].reshape(-1, d).mean(0)
                k[cu[b] + s: cu[b] + s + needle_len, h] = 3 * d ** 0.5 * qm / qm.norm()
    return cu, q.to(dtype).to(DEV), k.to(dtype).to(DEV), v.to(dtype).to(DEV)


def _check_pass(out, cu, pairs, q, k, v, G, c, w, L, what):
    scores = out.chunk_scores[0].cpu().numpy()
    idx = out.indices[0].cpu().numpy()
    cnt = out.counts[0].cpu().numpy()
    qf, kf = f64(q), f64(k)
    for b, (n_prev, n_new) in enumerate(pairs):
        for h in range(k.shape[1]):
            rows = oracle.group_window_rows(qf[b], h, G)
            A, sel, want = oracle.compress_tail_head(rows, kf[cu[b]:cu[b + 1], h], n_prev, c, w, L)
            tag = f"{what} cache {b} head {h}"
            check_scores(scores[b, h], A, tag)
            n = int(cnt[b, h])
            got = idx[b, h, :n]
            if n_new == 0:
                assert n == 0, tag
                continue
            check_indices(got, A, n_new, c, w, L, tag)
            tail = slice(cu[b] + n_prev, cu[b + 1])
            check_gather(out.k_out[0][b, h, :n], k[tail, h], got, tag + " K'")
            check_gather(out.v_out[0][b, h, :n], v[tail, h], got, tag + " V'")


@pytest.mark.parametrize("dtype,d,c,w,G,Hkv", [
    (torch.bfloat16, 128, 10, 32, 4, 2),        # tensor-core scoring, window rows read by a tensor map
    (torch.bfloat16, 128, 3, 24, 7, 1),         # tensor-core scoring, window rows packed (w does not divide 128)
    (torch.float32, 64, 7, 8, 2, 2),            # portable scoring
])
def test_tail_pass_matches_oracle(ckv, dtype, d, c, w, G, Hkv):
    # ragged caches: no kept prefix, a tail shorter than the window, an empty tail, long tails
    pairs = [(1500, 900), (0, 1200), (733, w - 3), (2048, 0), (410, 3001), (1, 97)]
    L = 200
    cu, q, k, v = _caches(pairs, Hkv, G, d, w, dtype, seed=11, needle_len=2 * c)
    n_prev = [p for p, _ in pairs]
    out = ckv.compress_tail(q, k, v, cu, n_prev, Hq=Hkv * G, Hkv=Hkv, w=w, c=c, L_tail=L, return_scores=True)
    assert ckv.chunkkv_status_check(out.workspace) == 0
    _check_pass(out, cu, pairs, q, k, v, G, c, w, L, f"{dtype} c={c}")


def test_prefill_then_two_incremental_passes(ckv):
    # Prefill compression of a 6000-token prompt, then per-head caches that grow by decoding and are
    # compressed twice by incremental passes; each pass appends its kept tail to the cache.
    d, G, Hkv, w, c, L = 128, 4, 2, 32, 10, 400
    g = torch.Generator().manual_seed(5)
    T = 6000
    q0 = torch.randn(1, w, Hkv * G, d, generator=g).to(torch.bfloat16).to(DEV)
    k0 = torch.randn(T, Hkv, d, generator=g).to(torch.bfloat16).to(DEV)
    v0 = torch.randn(T, Hkv, d, generator=g).to(torch.bfloat16).to(DEV)
    pre = ckv.compress_layers([q0], [k0], [v0], [0, T], Hq=Hkv * G, Hkv=Hkv, w=w, c=c, L_max=600)
    kept = [int(x) for x in pre.counts[0, 0].cpu()]
    cache_k = [pre.k_out[0][0, h, :kept[h]].clone() for h in range(Hkv)]
    cache_v = [pre.v_out[0][0, h, :kept[h]].clone() for h in range(Hkv)]
    for step, n_new in enumerate((1111, 530)):
        n_prev = [x.shape[0] for x in cache_k]
        # every head's cache is a sequence of its own (one KV head, its G query heads)
        new_k = [torch.randn(n_new, d, generator=g).to(torch.bfloat16).to(DEV) for _ in range(Hkv)]
        new_v = [torch.randn(n_new, d, generator=g).to(torch.bfloat16).to(DEV) for _ in range(Hkv)]
        k = torch.cat([torch.cat([cache_k[h], new_k[h]]) for h in range(Hkv)]).unsqueeze(1)
        v = torch.cat([torch.cat([cache_v[h], new_v[h]]) for h in range(Hkv)]).unsqueeze(1)
        cu = [0]
        for h in range(Hkv):
            cu.append(cu[-1] + n_prev[h] + n_new)
        qw = torch.randn(Hkv, w, G, d, generator=g).to(torch.bfloat16).to(DEV)
        out = ckv.compress_tail(qw, k, v, cu, n_prev, Hq=G, Hkv=1, w=w, c=c, L_tail=L, return_scores=True)
        assert ckv.chunkkv_status_check(out.workspace) == 0
        pairs = [(n_prev[h], n_new) for h in range(Hkv)]
        _check_pass(out, cu, pairs, qw, k, v, G, c, w, L, f"pass {step}")
        for h in range(Hkv):                         # append what the pass kept
            n = int(out.counts[0, h, 0])
            assert 0 < n <= L // c * c + w
            cache_k[h] = torch.cat([cache_k[h], out.k_out[0][h, 0, :n]])
            cache_v[h] = torch.cat([cache_v[h], out.v_out[0][h, 0, :n]])
    assert all(x.shape[0] > kept[h] for h, x in enumerate(cache_k))


def test_tail_pass_over_layers_with_index_reuse(ckv):
    # ChunkKV §4.2 Algorithm 2 during decoding: layers 0 and 2 re-score their new tails, layers 1 and 3
    # gather with the index lists of layers 0 and 2 (every layer's cache has the same lengths)
    pairs = [(700, 900), (0, 640), (1200, 75)]
    d, G, Hkv, w, c, L, n_layers, n_reuse = 128, 4, 2, 32, 10, 150, 4, 2
    qs, ks, vs = [], [], []
    for layer in range(n_layers):
        cu, q, k, v = _caches(pairs, Hkv, G, d, w, torch.bfloat16, seed=20 + layer, needle_len=2 * c)
        qs.append(q if layer % n_reuse == 0 else None)
        ks.append(k)
        vs.append(v)
    n_prev = [p for p, _ in pairs]
    out = ckv.compress_tail(qs, ks, vs, cu, n_prev, Hq=Hkv * G, Hkv=Hkv, w=w, c=c, L_tail=L, n_reuse=n_reuse,
                            return_scores=True)
    assert ckv.chunkkv_status_check(out.workspace) == 0
    scores = out.chunk_scores.cpu().numpy()
    idx = out.indices.cpu().numpy()
    cnt = out.counts.cpu().numpy()
    for grp in range(n_layers // n_reuse):
        src = oracle.scoring_layer(grp * n_reuse, n_reuse)
        qf, kf = f64(qs[src]), f64(ks[src])
        for b, (n_p, n_new) in enumerate(pairs):
            for h in range(Hkv):
                A, _, _ = oracle.compress_tail_head(oracle.group_window_rows(qf[b], h, G), kf[cu[b]:cu[b + 1], h],
                                                    n_p, c, w, L)
                tag = f"group {grp} cache {b} head {h}"
                check_scores(scores[grp, b, h], A, tag)
                n = int(cnt[grp, b, h])
                got = idx[grp, b, h, :n]
                check_indices(got, A, n_new, c, w, L, tag)
                tail = slice(cu[b] + n_p, cu[b + 1])
                for layer in range(grp * n_reuse, (grp + 1) * n_reuse):
                    check_gather(out.k_out[layer][b, h, :n], ks[layer][tail, h], got, f"{tag} layer {layer} K'")
                    check_gather(out.v_out[layer][b, h, :n], vs[layer][tail, h], got, f"{tag} layer {layer} V'")


def test_tail_pass_records_phase_events(ckv):
    # the phase events of chunkkv_set_phase_events mark the incremental pass's phases too, and a recorded
    # pass computes what an unrecorded one does
    pairs = [(700, 900), (0, 640)]
    d, G, Hkv, w, c, L = 128, 4, 2, 32, 10, 150
    cu, q, k, v = _caches(pairs, Hkv, G, d, w, torch.bfloat16, seed=31, needle_len=2 * c)
    n_prev = [p for p, _ in pairs]
    kw = dict(Hq=Hkv * G, Hkv=Hkv, w=w, c=c, L_tail=L, return_scores=True)
    ref = ckv.compress_tail(q, k, v, cu, n_prev, **kw)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(ckv.PHASES) + 1)]
    ckv.chunkkv_set_phase_events(evs)
    try:
        out = ckv.compress_tail(q, k, v, cu, n_prev, **kw)
    finally:
        ckv.chunkkv_set_phase_events(None)
    torch.cuda.synchronize()
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(ckv.PHASES))]
    assert all(t >= 0 for t in times) and times[1] > 0 and times[-1] > 0       # scoring and gather ran
    assert torch.equal(out.counts, ref.counts)
    for b, (n_p, n_new) in enumerate(pairs):
        C = -(-n_new // c)                                  # chunk scores past the tail's are not written
        assert torch.equal(out.chunk_scores[0, b, :, :C], ref.chunk_scores[0, b, :, :C])
        for h in range(Hkv):
            n = int(ref.counts[0, b, h])
            assert torch.equal(out.indices[0, b, h, :n], ref.indices[0, b, h, :n])
            assert torch.equal(out.k_out[0][b, h, :n], ref.k_out[0][b, h, :n])


def test_tail_pass_replays_from_a_cuda_graph(ckv):
    # every step of the pass is a stream-ordered launch, so a decode loop can capture it once and replay
    # it; the replayed pass (its claim counter reset by each launch) computes what the eager one does
    pairs = [(700, 900), (0, 640), (1200, 75)]
    d, G, Hkv, w, c, L = 128, 4, 2, 32, 10, 150
    cu, q, k, v = _caches(pairs, Hkv, G, d, w, torch.bfloat16, seed=41, needle_len=2 * c)
    n_prev = [p for p, _ in pairs]
    kw = dict(Hq=Hkv * G, Hkv=Hkv, w=w, c=c, L_tail=L, return_scores=True)
    ref = ckv.compress_tail(q, k, v, cu, n_prev, **kw)
    out = ckv.compress_tail(q, k, v, cu, n_prev, **kw)              # warm-up; outputs and workspace reused
    p, keep = ckv.params_for(q, k, cu, Hkv=Hkv, w=w, c=c, L_max=L)
    for x in (out.indices, out.counts, out.chunk_scores, *out.k_out, *out.v_out):
        x.fill_(-1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ckv.chunkkv_compress_tail(p, n_prev, 1, [q], [k], [v], out.k_out, out.v_out, out.indices, out.counts,
                                  out.chunk_scores, out.workspace)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert ckv.chunkkv_status_check(out.workspace) == 0
    assert torch.equal(out.counts, ref.counts)
    for b, (n_p, n_new) in enumerate(pairs):
        C = -(-n_new // c)
        assert torch.equal(out.chunk_scores[0, b, :, :C], ref.chunk_scores[0, b, :, :C])
        for h in range(Hkv):
            n = int(ref.counts[0, b, h])
            assert torch.equal(out.indices[0, b, h, :n], ref.indices[0, b, h, :n])
            assert torch.equal(out.k_out[0][b, h, :n], ref.k_out[0][b, h, :n])
            assert torch.equal(out.v_out[0][b, h, :n], ref.v_out[0][b, h, :n])
    del keep
