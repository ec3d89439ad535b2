"""The oracle's pins catch plausible mistakes: each mutant below plants one in the oracle (on the CPU)
and at least one pin of tests/test_oracle_pins.py must then fail.

A mutant replaces one oracle function, in the package and in the module that defines it, so the
oracle's own calls (chunkkv_head, compress_layers) see it too.  The mistakes are the kinds a
restatement of ChunkKV §4.1 Algorithm 1 and §4.2 Algorithm 2 (with the probabilities of Kara §2
Eq. (1)) could plausibly contain: a dropped or wrong scale, a softmax over the wrong axis, a sum
read as a mean, the GQA group dropped or mis-indexed, the short last chunk lost, an off-by-one in
the budget, the tie rule or the recent window, the wrong layer reused, a causal limit off by one, and, for the incremental pass during decoding,
the softmax over the tail alone, the tail chunked on the cache's grid, or tail-local positions.
"""
import importlib.util
import math
import os

import numpy as np
import pytest

import oracle
import oracle.chunkkv_oracle as O

ORIG = {name: getattr(O, name) for name in oracle.__all__}


def _load_pins():
    path = os.path.join(os.path.dirname(__file__), "test_oracle_pins.py")
    spec = importlib.util.spec_from_file_location("_oracle_pins_for_mutants", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pin_calls(mod):
    """(name, thunk) for every pin test and every parameter set it runs with."""
    calls = []
    for name, fn in sorted(vars(mod).items()):
        if not (name.startswith("test_") and callable(fn)):
            continue
        if name.endswith("_full_size"):
            continue               # the full-size needle pins repeat the 8K one at 10-30x the cost
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn))
            continue
        assert len(marks) == 1, name
        argnames, values = marks[0].args[0], marks[0].args[1]
        names = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for i, val in enumerate(values):
            args = val if len(names) > 1 else (val,)
            calls.append((f"{name}[{i}]", lambda fn=fn, kw=dict(zip(names, args)): fn(**kw)))
    return calls


PINS = _pin_calls(_load_pins())


def _failing_pins(monkeypatch, name, fn):
    with monkeypatch.context() as m:
        if name is not None:
            m.setattr(O, name, fn)
            m.setattr(oracle, name, fn)
        failed = []
        for pin, call in PINS:
            try:
                call()
            except Exception as e:          # an assertion, or a crash the pin's checks lead to
                failed.append((pin, type(e).__name__))
        return failed


# ---------------------------------------------------------------- the mutants

def ks_scale_by_d(rows, keys, limits=None):            # 1/d instead of 1/sqrt(d)
    return ORIG["key_scores"](np.asarray(rows) / math.sqrt(keys.shape[1]), keys, limits)


def ks_unscaled(rows, keys, limits=None):              # the 1/sqrt(d) dropped
    return ORIG["key_scores"](np.asarray(rows) * math.sqrt(keys.shape[1]), keys, limits)


def ks_softmax_over_rows(rows, keys, limits=None):     # normalised over the window, not the keys
    T, d = keys.shape
    if T == 0 or rows.shape[0] == 0:
        return np.zeros(T)
    s = np.asarray(rows, np.float64) @ np.asarray(keys, np.float64).T / math.sqrt(d)
    p = np.exp(s - s.max(axis=0, keepdims=True))
    return (p / p.sum(axis=0, keepdims=True)).sum(axis=0)


def ks_mean_over_rows(rows, keys, limits=None):        # a mean over the window rows, not a sum
    return ORIG["key_scores"](rows, keys, limits) / max(rows.shape[0], 1)


def ks_raw_logits(rows, keys, limits=None):            # step 1 read as the plain product, no softmax
    T, d = keys.shape
    if T == 0 or rows.shape[0] == 0:
        return np.zeros(T)
    return (np.asarray(rows, np.float64) @ np.asarray(keys, np.float64).T / math.sqrt(d)).sum(axis=0)


def ks_limits_ignored(rows, keys, limits=None):       # the causal option never applied
    return ORIG["key_scores"](rows, keys, None)


def rows_first_member_only(q, h, G):                   # the GQA sum dropped
    return ORIG["group_window_rows"](q, h, G)[: q.shape[0]]


def rows_interleaved_group(q, h, G):                   # query head g * Hkv + h instead of h * G + g
    Hkv = q.shape[1] // G
    return np.concatenate([q[:, g * Hkv + h, :] for g in range(G)], axis=0).astype(np.float64)


def chunks_tail_dropped(a, c):                         # C = floor(T / c)
    return ORIG["chunk_scores"](a[: (len(a) // c) * c], c)


def chunks_mean(a, c):                                 # chunk score normalised by its length
    s = ORIG["chunk_scores"](a, c)
    sizes = np.minimum(c, len(a) - np.arange(len(s)) * c)
    return s / sizes


def chunks_from_end(a, c):                             # chunks aligned to the last token, short one first
    T = len(a)
    return ORIG["chunk_scores"](a[::-1], c)[::-1].copy() if T else np.zeros(0)


def nsel_ceil(T, c, L_max):                            # k = ceil(L_max / c)
    return min(-(-L_max // c), -(-T // c))


def top_ties_high(A, k):                               # ties to the higher chunk index
    order = sorted(range(len(A)), key=lambda i: (-float(A[i]), -i))
    return sorted(order[:k])


def top_smallest(A, k):                                # the k lowest scores
    order = sorted(range(len(A)), key=lambda i: (float(A[i]), i))
    return sorted(order[:k])


def top_in_score_order(A, k):                          # best first, not ascending chunk ids
    return sorted(range(len(A)), key=lambda i: (-float(A[i]), i))[:k]


def kept_window_short(chunks, T, c, w):                # w - 1 recent tokens
    return ORIG["kept_indices"](chunks, T, c, max(w - 1, 0))


def kept_no_window(chunks, T, c, w):                   # the recent window not forced in
    return ORIG["kept_indices"](chunks, T, c, 0)


def kept_chunk_offset(chunks, T, c, w):                # chunk i taken as tokens i*c+1 .. i*c+c
    keep = set(range(max(0, T - w), T))
    for i in chunks:
        keep.update(j for j in range(i * c + 1, i * c + c + 1) if j < T)
    return np.array(sorted(keep), dtype=np.int64)


def layer_group_index(layer, n_reuse):                 # floor(l / N) instead of floor(l / N) * N
    return layer // n_reuse


def layer_next_scoring(layer, n_reuse):                # a reuse layer takes the next scoring layer
    return -(-layer // n_reuse) * n_reuse


def limits_off_by_one(n_rows, T, w):                   # query q sees keys < T - w + q only
    return ORIG["window_limits"](n_rows, T, w) - 1


def limits_row_order(n_rows, T, w):                    # rows taken as (window row, group member)
    G = max(n_rows // max(w, 1), 1)
    return T - w + np.arange(n_rows) // G


def overlap_sum_of_sizes(a, b):                        # |A| + |B| for the union
    inter, _ = ORIG["layer_overlap"](a, b)
    return inter, len(np.asarray(a).ravel()) + len(np.asarray(b).ravel())


def jaccard_dice(a, b):                                # 2|A ∩ B| / (|A| + |B|)
    inter, union = ORIG["layer_overlap"](a, b)
    return 1.0 if union == 0 else 2 * inter / (union + inter)


def gather_prefix(x, idx):                             # the first len(idx) rows, not rows idx
    return x[: len(idx)]


def tail_normalised_over_tail(rows, keys, n_prev):    # the softmax over the new tail only
    return ORIG["key_scores"](rows, keys[n_prev:])


def tail_chunks_from_cache_start(rows, keys, n_prev, c, w, L_tail):   # tail chunks on the cache's chunk grid
    a = ORIG["key_scores"](rows, keys)
    first = n_prev // c
    A = ORIG["chunk_scores"](a, c)[first:]
    n_new = keys.shape[0] - n_prev
    sel = ORIG["top_chunks"](A, ORIG["n_select"](n_new, c, L_tail))
    keep = set()
    for i in sel:
        keep.update(range((first + i) * c, min((first + i) * c + c, keys.shape[0])))
    keep.update(range(max(n_prev, keys.shape[0] - w), keys.shape[0]))
    return A, sel, np.array(sorted(keep), dtype=np.int64)


def tail_positions_not_offset(rows, keys, n_prev, c, w, L_tail):       # tail-local positions returned
    A, sel, idx = ORIG["compress_tail_head"](rows, keys, n_prev, c, w, L_tail)
    return A, sel, idx - n_prev


MUTANTS = {
    "key_scores": [ks_scale_by_d, ks_unscaled, ks_softmax_over_rows, ks_mean_over_rows, ks_raw_logits,
                   ks_limits_ignored],
    "group_window_rows": [rows_first_member_only, rows_interleaved_group],
    "chunk_scores": [chunks_tail_dropped, chunks_mean, chunks_from_end],
    "n_select": [nsel_ceil],
    "top_chunks": [top_ties_high, top_smallest, top_in_score_order],
    "kept_indices": [kept_window_short, kept_no_window, kept_chunk_offset],
    "scoring_layer": [layer_group_index, layer_next_scoring],
    "window_limits": [limits_off_by_one, limits_row_order],
    "layer_overlap": [overlap_sum_of_sizes],
    "layer_jaccard": [jaccard_dice],
    "gather": [gather_prefix],
    "tail_key_scores": [tail_normalised_over_tail],
    "compress_tail_head": [tail_chunks_from_cache_start, tail_positions_not_offset],
}
CASES = [(name, fn) for name, fns in MUTANTS.items() for fn in fns]


def test_pins_pass_on_the_oracle_itself(monkeypatch):
    assert len(PINS) >= 40
    assert _failing_pins(monkeypatch, None, None) == []


@pytest.mark.parametrize("name,fn", CASES, ids=[f"{n}:{f.__name__}" for n, f in CASES])
def test_a_planted_mistake_fails_a_pin(monkeypatch, name, fn):
    failed = _failing_pins(monkeypatch, name, fn)
    assert failed, f"no pin catches {fn.__name__} planted in {name}"
    assert getattr(O, name) is ORIG[name] and getattr(oracle, name) is ORIG[name]
