"""Pins of the CPU oracle to facts fixed outside of it.

Each test ties the oracle to something it could not get right by accident:
hand-derived closed forms (tests/golden), a high-precision brute force written
in a different form, invariants of the softmax, exhaustive subset search for
the top-k, a textbook per-token top-k for c = 1, and the structure of
Algorithm 2.  Citations: "ChunkKV ... (NeurIPS'25) notes" §4.1 Algorithm 1,
§4.2 Algorithm 2; "Kara" §2 Eq. (1).
"""
import heapq
import itertools
import json
import math
import os

import mpmath
import numpy as np
import pytest
import torch

import oracle
from synthetic import configs, generator as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _ev(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt, "log": math.log,
                                                    "exp": math.exp}))


def _load_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    q = np.array([[[_ev(x) for x in row] for row in hq] for hq in case["q_win"]])   # [w,Hq,d]
    k = np.array([[[_ev(x) for x in row] for row in tok] for tok in case["k"]])      # [T,Hkv,d]
    G = case["Hq"] // case["Hkv"]
    for h in range(case["Hkv"]):
        A, sel, idx = oracle.chunkkv_head(oracle.group_window_rows(q, h, G), k[:, h, :],
                                          case["c"], case["w"], case["L_max"])
        want = [_ev(x) for x in case["expect_scores"][h]]
        assert np.allclose(A, want, rtol=1e-13, atol=1e-14), (A, want)
        assert idx.tolist() == case["expect_indices"][h]


def _brute_scores(rows, keys, c):
    """Chunk scores at 50 digits: p_qj = 1 / sum_j' exp(s_qj' - s_qj), tokens mapped to chunks."""
    mpmath.mp.dps = 50
    R, d = rows.shape
    T = keys.shape[0]
    inv = 1 / mpmath.sqrt(d)
    bins = {}
    for q in range(R):
        s = [mpmath.fsum(mpmath.mpf(float(rows[q, e])) * mpmath.mpf(float(keys[j, e]))
                         for e in range(d)) * inv for j in range(T)]
        for j in range(T):
            pj = 1 / mpmath.fsum(mpmath.e ** (s[i] - s[j]) for i in range(T))
            bins[j // c] = bins.get(j // c, mpmath.mpf(0)) + pj
    return [float(bins[i]) for i in range(len(bins))]


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_high_precision(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 13))
    d = int(rng.integers(1, 5))
    R = int(rng.integers(1, 5))
    c = int(rng.integers(1, 5))
    rows = rng.normal(size=(R, d)) * 2
    keys = rng.normal(size=(T, d)) * 2
    A = oracle.chunk_scores(oracle.key_scores(rows, keys), c)
    assert np.allclose(A, _brute_scores(rows, keys, c), rtol=1e-12, atol=1e-14)


def _rand_case(seed, T=97, d=16, w=5, G=3, Hkv=2, c=7):
    rng = np.random.default_rng(100 + seed)
    q = rng.normal(size=(w, G * Hkv, d))
    k = rng.normal(size=(T, Hkv, d)) * 1.5
    return q, k, G, c


@pytest.mark.parametrize("seed", range(4))
def test_scores_sum_to_window_times_group(seed):
    # every softmax row sums to one, so the chunk scores of a KV head add up to w * G
    q, k, G, c = _rand_case(seed)
    w = q.shape[0]
    for h in range(k.shape[1]):
        A = oracle.chunk_scores(oracle.key_scores(oracle.group_window_rows(q, h, G), k[:, h]), c)
        assert abs(A.sum() - w * G) < 1e-11


def test_zero_keys_give_uniform_mass():
    # K = 0: every logit is 0, p = 1/T, so A_i = w G |chunk_i| / T (last chunk short)
    T, c, w, G, d = 53, 10, 4, 2, 8
    q = np.random.default_rng(1).normal(size=(w, G, d))
    A = oracle.chunk_scores(oracle.key_scores(oracle.group_window_rows(q, 0, G), np.zeros((T, d))), c)
    sizes = [10, 10, 10, 10, 10, 3]
    assert np.allclose(A, [w * G * s / T for s in sizes], rtol=1e-14)


@pytest.mark.parametrize("seed", range(3))
def test_shift_of_all_keys_leaves_scores_unchanged(seed):
    # adding one vector u to every key adds <q,u>/sqrt(d) to a whole softmax row
    q, k, G, c = _rand_case(seed)
    u = np.random.default_rng(seed).normal(size=k.shape[2])
    rows = oracle.group_window_rows(q, 1, G)
    a0 = oracle.key_scores(rows, k[:, 1])
    a1 = oracle.key_scores(rows, k[:, 1] + u)
    assert np.allclose(a0, a1, rtol=1e-10, atol=1e-13)
    # ...while scaling the keys does change them (the normalisation is per query row)
    assert not np.allclose(a0, oracle.key_scores(rows, 2 * k[:, 1]), rtol=1e-3)


def test_single_query_is_textbook_softmax():
    # G = 1, w = 1, c = 1: the chunk scores are one softmax row of q.k / sqrt(d)
    rng = np.random.default_rng(5)
    q = rng.normal(size=(1, 1, 8))
    k = rng.normal(size=(20, 8))
    s = torch.tensor(k @ q[0, 0] / math.sqrt(8))
    want = torch.softmax(s, dim=0).numpy()
    A = oracle.chunk_scores(oracle.key_scores(oracle.group_window_rows(q, 0, 1), k), 1)
    assert np.allclose(A, want, rtol=1e-12)


def test_top_chunks_brute_force_subsets():
    rng = np.random.default_rng(7)
    for trial in range(60):
        C = int(rng.integers(1, 11))
        k = int(rng.integers(0, C + 1))
        A = rng.integers(0, 4, size=C).astype(np.float64)   # integers: exact sums, many ties
        best, best_set = None, None
        for comb in itertools.combinations(range(C), k):     # lexicographic order
            s = sum(A[i] for i in comb)
            if best is None or s > best:
                best, best_set = s, list(comb)
        assert oracle.top_chunks(A, k) == best_set, (A, k)


def test_all_equal_scores_keep_lowest_chunks():
    assert oracle.top_chunks(np.full(9, 0.25), 4) == [0, 1, 2, 3]


def test_chunk_size_one_is_per_token_topk():
    # c = 1: selection is a plain top-L_max over per-token mass (ties to the lower token)
    q, k, G, _ = _rand_case(3, T=64)
    rows = oracle.group_window_rows(q, 0, G)
    a = oracle.key_scores(rows, k[:, 0])
    L_max, w = 11, 5
    A, sel, idx = oracle.chunkkv_head(rows, k[:, 0], 1, w, L_max)
    want = sorted(heapq.nlargest(L_max, range(64), key=lambda j: (a[j], -j)))
    assert sel == want
    assert idx.tolist() == sorted(set(want) | set(range(64 - w, 64)))


@pytest.mark.parametrize("T,c,w,L_max", [(97, 7, 5, 30), (97, 7, 0, 30), (20, 7, 30, 7),
                                         (64, 8, 8, 16), (10, 3, 2, 0), (1, 4, 1, 4)])
def test_kept_indices_characterised(T, c, w, L_max):
    q, k, G, _ = _rand_case(1, T=T)
    rows = oracle.group_window_rows(q, 0, G)
    A, sel, idx = oracle.chunkkv_head(rows, k[:, 0], c, w, L_max)
    C = -(-T // c)
    assert len(sel) == min(L_max // c, C) and len(set(sel)) == len(sel)
    idx = idx.tolist()
    assert all(b > a for a, b in zip(idx, idx[1:])) and all(0 <= j < T for j in idx)
    recent = set(range(max(0, T - w), T))
    for j in range(T):       # j kept  <=>  its chunk was selected or it is recent
        assert (j in idx) == ((j // c) in sel or j in recent)


def test_budget_at_least_prompt_keeps_everything():
    q, k, G, c = _rand_case(2, T=45)
    rows = oracle.group_window_rows(q, 0, G)
    A, sel, idx = oracle.chunkkv_head(rows, k[:, 0], c, 3, 45)
    assert idx.tolist() == list(range(45))
    assert np.array_equal(oracle.gather(k[:, 0], idx), k[:, 0])


def test_planted_chunk_is_selected_tiny():
    wl = configs.tiny()
    q, k, v, spans = gen.make_all_layers(wl, "cpu")
    (s, e), = spans[0][0]
    res = oracle.compress_layers([q[0].numpy()], [k[0].numpy()], [v[0].numpy()], wl.cu_seqlens,
                                 wl.Hq, wl.Hkv, wl.w, wl.c, wl.L_max, wl.n_reuse)
    for h in range(wl.Hkv):
        assert s // wl.c in res["chunks"][0][0][h]
        A = res["scores"][0][0][h]
        assert int(np.argmax(A)) == s // wl.c


def test_needle_spans_are_found_llama_layer():
    # every needle span at least one chunk long contains a selected chunk, in every KV head
    wl = configs.llama_layer()
    q, k, v, spans = gen.make_all_layers(wl, "cpu")
    qf = q[0].float().numpy()
    kf = k[0].float().numpy()
    G = wl.G
    for h in range(wl.Hkv):
        A, sel, idx = oracle.chunkkv_head(oracle.group_window_rows(qf[0], h, G), kf[:, h],
                                          wl.c, wl.w, wl.L_max)
        sel = set(sel)
        for (s, e) in spans[0][0]:
            full = [i for i in range(-(-s // wl.c), e // wl.c) if (i + 1) * wl.c <= e]
            if full:
                assert sel & set(full), (h, s, e)


@pytest.mark.parametrize("name", ["llama_model", "qwen_128k", "mistral_ragged"])
def test_needle_spans_are_found_full_size(name):
    # the same on the first layer of the 32K and 128K models and of the 16-sequence ragged batch:
    # in every sequence and KV head, every needle span at least one chunk long contains a selected
    # chunk (the heads run in parallel threads: numpy releases the interpreter lock in its loops)
    from concurrent.futures import ThreadPoolExecutor
    wl = getattr(configs, name)()
    spans = gen.needle_spans(wl)
    q, k, v = gen.make_layer(wl, 0, "cpu", spans=spans[0])
    qf = q.float().numpy()
    cu = wl.cu_seqlens
    n_checked = 0
    with ThreadPoolExecutor(max_workers=8) as ex:
        for b in range(wl.B):
            kf = k[cu[b]:cu[b + 1]].float().numpy()
            T = cu[b + 1] - cu[b]
            assert oracle.n_select(T, wl.c, wl.L_max) >= len(spans[0][b])
            sels = ex.map(lambda h: set(oracle.chunkkv_head(oracle.group_window_rows(qf[b], h, wl.G), kf[:, h],
                                                             wl.c, wl.w, wl.L_max)[1]), range(wl.Hkv))
            for h, sel in enumerate(sels):
                for (s, e) in spans[0][b]:
                    full = [i for i in range(-(-s // wl.c), e // wl.c) if (i + 1) * wl.c <= e]
                    if full:
                        assert sel & set(full), (name, b, h, s, e)
                        n_checked += 1
    assert n_checked >= wl.B * wl.Hkv * 5


def _layers(n_layers, T=40, Hkv=2, G=2, w=4, d=8, seed=0):
    rng = np.random.default_rng(seed)
    qs = [rng.normal(size=(1, w, Hkv * G, d)) for _ in range(n_layers)]
    ks = [rng.normal(size=(T, Hkv, d)) for _ in range(n_layers)]
    vs = [rng.normal(size=(T, Hkv, d)) for _ in range(n_layers)]
    return qs, ks, vs


def test_reuse_layers_share_indices_and_gather_their_own_kv():
    qs, ks, vs = _layers(5)
    r = oracle.compress_layers(qs, ks, vs, [0, 40], 4, 2, 4, 5, 15, n_reuse=2)
    assert sorted(r["indices"]) == [0, 1, 2]                  # layers 0, 2, 4 score
    for layer in range(5):
        g = layer // 2
        for h in range(2):
            idx = r["indices"][g][0][h]
            assert np.array_equal(r["k_out"][layer][0][h], ks[layer][idx, h])
            assert np.array_equal(r["v_out"][layer][0][h], vs[layer][idx, h])


def test_reuse_depth_changes_only_the_reusing_layers():
    qs, ks, vs = _layers(4, seed=3)
    r1 = oracle.compress_layers(qs, ks, vs, [0, 40], 4, 2, 4, 5, 15, n_reuse=1)
    r2 = oracle.compress_layers(qs, ks, vs, [0, 40], 4, 2, 4, 5, 15, n_reuse=2)
    for layer in (0, 2):                                       # scoring layers agree
        for h in range(2):
            assert np.array_equal(r1["indices"][layer][0][h], r2["indices"][layer // 2][0][h])
    # with N_reuse = 1 layer 1 selects from its own scores; they differ from layer 0 here
    assert any(not np.array_equal(r1["indices"][1][0][h], r1["indices"][0][0][h]) for h in range(2))


def test_ragged_batch_is_per_sequence():
    rng = np.random.default_rng(11)
    T = [30, 0, 17]
    cu = [0, 30, 30, 47]
    q = rng.normal(size=(3, 4, 4, 8))
    k = rng.normal(size=(47, 2, 8))
    v = rng.normal(size=(47, 2, 8))
    r = oracle.compress_layers([q], [k], [v], cu, 4, 2, 4, 5, 10, 1)
    for b in range(3):
        for h in range(2):
            A, sel, idx = oracle.chunkkv_head(oracle.group_window_rows(q[b], h, 2),
                                              k[cu[b]:cu[b + 1], h], 5, 4, 10)
            assert np.array_equal(r["indices"][0][b][h], idx)
    assert r["indices"][0][1][0].size == 0


# ---------------------------------------------------------------- adjacent-layer overlap (reading R9)

def _merge_counts(a, b):
    """Two-pointer merge over sorted, duplicate-free arrays: (|A ∩ B|, |A ∪ B|), a formulation
    independent of the oracle's set arithmetic."""
    i = j = inter = union = 0
    while i < len(a) or j < len(b):
        if j == len(b) or (i < len(a) and a[i] < b[j]):
            i += 1
        elif i == len(a) or b[j] < a[i]:
            j += 1
        else:
            inter += 1
            i += 1
            j += 1
        union += 1
    return inter, union


def test_layer_overlap_closed_forms():
    a = np.arange(100, 200)
    assert oracle.layer_overlap(a, a) == (100, 100) and oracle.layer_jaccard(a, a) == 1.0
    assert oracle.layer_overlap(a, a + 100) == (0, 200) and oracle.layer_jaccard(a, a + 100) == 0.0
    assert oracle.layer_overlap(a, a[10:30]) == (20, 100)                       # nested
    assert oracle.layer_overlap(np.arange(0, 10), np.arange(5, 15)) == (5, 15)
    assert oracle.layer_jaccard([], []) == 1.0 and oracle.layer_overlap([], [3]) == (0, 1)
    # a fractional value: |A ∩ B| = 5 over |A ∪ B| = 15 (not the Dice ratio 2·5 / 20)
    assert oracle.layer_jaccard(np.arange(0, 10), np.arange(5, 15)) == pytest.approx(1 / 3, rel=1e-15)
    assert oracle.layer_jaccard(a, a[10:30]) == pytest.approx(0.2, rel=1e-15)


def test_layer_overlap_against_merge_counts():
    rng = np.random.default_rng(17)
    for _ in range(200):
        T = int(rng.integers(1, 400))
        a = np.sort(rng.choice(T, size=int(rng.integers(0, T + 1)), replace=False))
        b = np.sort(rng.choice(T, size=int(rng.integers(0, T + 1)), replace=False))
        assert oracle.layer_overlap(a, b) == _merge_counts(a, b)
        assert oracle.layer_overlap(a, b) == oracle.layer_overlap(b, a)


def test_window_only_budget_gives_identical_lists():
    # L_max < c keeps only the recent window in every layer, so adjacent layers overlap fully
    rng = np.random.default_rng(3)
    T, w, c, d = 300, 16, 10, 8
    rows = rng.standard_normal((w, d))
    i1 = oracle.chunkkv_head(rows, rng.standard_normal((T, d)), c, w, 5)[2]
    i2 = oracle.chunkkv_head(rows, rng.standard_normal((T, d)), c, w, 5)[2]
    assert oracle.layer_jaccard(i1, i2) == 1.0 and len(i1) == w


# ---------------------------------------------------------------- causal window option (reading R10)

def test_causal_window_of_one_row_is_unmasked():
    # the single window query sits at T - 1 and sees every key
    rng = np.random.default_rng(21)
    rows, keys = rng.standard_normal((3, 8)), rng.standard_normal((57, 8))      # G = 3 rows of one window position
    lim = oracle.window_limits(3, 57, 1)
    assert np.array_equal(lim, [56, 56, 56])
    assert np.allclose(oracle.key_scores(rows, keys, lim), oracle.key_scores(rows, keys), rtol=0, atol=1e-15)


def test_causal_window_zero_keys_closed_form():
    # K = 0: window query q sees T - w + q + 1 keys with equal probability
    T, w, G, d = 23, 5, 2, 4
    rows = np.random.default_rng(1).standard_normal((G * w, d))
    a = oracle.key_scores(rows, np.zeros((T, d)), oracle.window_limits(G * w, T, w))
    want = np.zeros(T)
    for q in range(w):
        n = T - w + q + 1
        want[:n] += G / n
    assert np.allclose(a, want, rtol=0, atol=1e-14)
    assert math.isclose(a.sum(), G * w, rel_tol=1e-14)


def test_causal_window_brute_force_50_digits():
    rng = np.random.default_rng(8)
    T, w, d = 9, 4, 3
    rows, keys = rng.standard_normal((w, d)), rng.standard_normal((T, d))
    lim = oracle.window_limits(w, T, w)
    got = oracle.key_scores(rows, keys, lim)
    mpmath.mp.dps = 50
    want = [mpmath.mpf(0)] * T
    for r in range(w):
        s = [sum(mpmath.mpf(float(rows[r, e])) * mpmath.mpf(float(keys[j, e])) for e in range(d)) / mpmath.sqrt(d)
             for j in range(T)]
        for j in range(int(lim[r]) + 1):
            want[j] += 1 / sum(mpmath.e ** (s[i] - s[j]) for i in range(int(lim[r]) + 1))
    assert np.allclose(got, [float(x) for x in want], rtol=1e-13, atol=1e-15)


def test_causal_window_group_rows_brute_force_50_digits():
    # G = 2 query heads share the KV head: the row of (member g, window row q) sits at T - w + q
    # whatever g is, so each member's rows see the same growing key prefixes
    rng = np.random.default_rng(12)
    T, w, G, Hkv, d, h = 8, 3, 2, 2, 3, 1
    q_win = rng.standard_normal((w, G * Hkv, d))
    keys = rng.standard_normal((T, d))
    rows = oracle.group_window_rows(q_win, h, G)
    got = oracle.key_scores(rows, keys, oracle.window_limits(G * w, T, w))
    mpmath.mp.dps = 50
    want = [mpmath.mpf(0)] * T
    for g in range(G):
        for qi in range(w):
            x = q_win[qi, h * G + g]
            last = T - w + qi
            s = [sum(mpmath.mpf(float(x[e])) * mpmath.mpf(float(keys[j, e])) for e in range(d)) / mpmath.sqrt(d)
                 for j in range(last + 1)]
            for j in range(last + 1):
                want[j] += 1 / sum(mpmath.e ** (s[i] - s[j]) for i in range(last + 1))
    assert np.allclose(got, [float(x) for x in want], rtol=1e-13, atol=1e-15)


def test_causal_window_rows_before_the_sequence_add_nothing():
    # T < w: window queries at negative positions see no key
    rng = np.random.default_rng(4)
    T, w, d = 3, 5, 4
    rows, keys = rng.standard_normal((w, d)), rng.standard_normal((T, d))
    lim = oracle.window_limits(w, T, w)                       # -2, -1, 0, 1, 2
    a = oracle.key_scores(rows, keys, lim)
    assert math.isclose(a.sum(), 3.0, rel_tol=1e-14)          # only the three rows at 0, 1, 2 count
    assert np.allclose(a, oracle.key_scores(rows[2:], keys, lim[2:]), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- decoding: incremental pass (reading R12)

def test_tail_pass_with_no_kept_prefix_is_algorithm_1():
    # n_prev = 0: the whole cache is new, and the pass is ChunkKV §4.1 Algorithm 1 on it
    q, k, G, c = _rand_case(4, T=83)
    rows = oracle.group_window_rows(q, 1, G)
    A, sel, idx = oracle.compress_tail_head(rows, k[:, 1], 0, c, 5, 30)
    A0, sel0, idx0 = oracle.chunkkv_head(rows, k[:, 1], c, 5, 30)
    assert np.array_equal(A, A0) and sel == sel0 and idx.tolist() == idx0.tolist()


def test_tail_pass_zero_keys_closed_form():
    # K = 0: p = 1 / (n_prev + n_new) for every key of the cache, so a tail chunk scores
    # w G |chunk| / (n_prev + n_new), chunks counted from the tail's first token (last one short)
    n_prev, n_new, c, w, G, d = 41, 23, 5, 3, 2, 4
    q = np.random.default_rng(2).normal(size=(w, G, d))
    A, sel, idx = oracle.compress_tail_head(oracle.group_window_rows(q, 0, G), np.zeros((n_prev + n_new, d)),
                                            n_prev, c, w, 10)
    assert np.allclose(A, [w * G * s / (n_prev + n_new) for s in (5, 5, 5, 5, 3)], rtol=1e-14)
    # all full tail chunks tie: the two lowest are kept, then the last w tokens of the tail
    assert sel == [0, 1]
    assert idx.tolist() == list(range(n_prev, n_prev + 10)) + list(range(n_prev + n_new - w, n_prev + n_new))


@pytest.mark.parametrize("seed", range(4))
def test_tail_pass_brute_force_50_digits(seed):
    # every window row normalised over the whole cache, tail tokens binned from the tail's start
    rng = np.random.default_rng(30 + seed)
    n_prev, n_new = int(rng.integers(0, 9)), int(rng.integers(1, 9))
    d, R, c = int(rng.integers(1, 4)), int(rng.integers(1, 4)), int(rng.integers(1, 4))
    rows, keys = rng.normal(size=(R, d)) * 2, rng.normal(size=(n_prev + n_new, d)) * 2
    A, _, _ = oracle.compress_tail_head(rows, keys, n_prev, c, 1, c)
    mpmath.mp.dps = 50
    T = n_prev + n_new
    want = [mpmath.mpf(0)] * (-(-n_new // c))
    for r in range(R):
        s = [sum(mpmath.mpf(float(rows[r, e])) * mpmath.mpf(float(keys[j, e])) for e in range(d)) / mpmath.sqrt(d)
             for j in range(T)]
        for j in range(n_prev, T):
            want[(j - n_prev) // c] += 1 / sum(mpmath.e ** (s[i] - s[j]) for i in range(T))
    assert np.allclose(A, [float(x) for x in want], rtol=1e-12, atol=1e-15)


def test_tail_pass_normalises_over_the_whole_cache():
    # Hand-built: row 0 attends mostly to a kept key (logit 10/sqrt 2), row 1 does not.  Over the
    # whole cache, tail token y (favoured by row 1) outscores x (favoured by row 0):
    #   row 0: Z = e^7.07 + e^1.41 + 2  -> p(x) = 0.0035, p(y) = 0.0008
    #   row 1: Z = 3 + e^0.85           -> p(x) = 0.187,  p(y) = 0.438
    # so A(y) = 0.44 > A(x) = 0.19; normalised over the tail alone, x would win (0.90 vs 0.70).
    rows = np.array([[2.0, 0.0], [0.0, 2.0]])
    keys = np.array([[5.0, 0.0],      # kept by an earlier pass
                     [1.0, 0.0],      # x
                     [0.0, 0.6],      # y
                     [0.0, 0.0]])     # the most recent token (forced in by w = 1)
    A, sel, idx = oracle.compress_tail_head(rows, keys, 1, 1, 1, 1)
    z0 = math.exp(10 / math.sqrt(2)) + math.exp(2 / math.sqrt(2)) + 2
    z1 = 3 + math.exp(1.2 / math.sqrt(2))
    want = [math.exp(2 / math.sqrt(2)) / z0 + 1 / z1, 1 / z0 + math.exp(1.2 / math.sqrt(2)) / z1, 1 / z0 + 1 / z1]
    assert np.allclose(A, want, rtol=1e-13)
    assert sel == [1] and idx.tolist() == [2, 3]


@pytest.mark.parametrize("n_prev,n_new,c,w,L", [(30, 47, 7, 5, 20), (0, 10, 3, 2, 0), (12, 3, 4, 6, 8),
                                               (5, 64, 8, 8, 100)])
def test_tail_pass_kept_positions_characterised(n_prev, n_new, c, w, L):
    q, k, G, _ = _rand_case(5, T=n_prev + n_new)
    rows = oracle.group_window_rows(q, 0, G)
    A, sel, idx = oracle.compress_tail_head(rows, k[:, 0], n_prev, c, w, L)
    C = -(-n_new // c)
    assert len(A) == C and len(sel) == min(L // c, C)
    idx = idx.tolist()
    assert all(b > a for a, b in zip(idx, idx[1:])) and all(n_prev <= j < n_prev + n_new for j in idx)
    for t in range(n_new):   # tail token t appended  <=>  its tail chunk was selected or it is recent
        assert ((n_prev + t) in idx) == ((t // c) in sel or t >= n_new - w)
