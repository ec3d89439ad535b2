"""CPU oracle for ChunkKV chunk-level KV-cache compression (TEST INFRASTRUCTURE ONLY).

This module is the plain, slow, fp64 statement of what the CUDA library must
compute.  It exists to check that library: only the test suite, the smoke
check of __graft_entry__ and the CPU-baseline / reference arm of bench.py may
import it.  The library never calls it and has no fallback to it.

Sources (cited per function below):
  * "ChunkKV: Semantic-Preserving KV Cache Compression for Efficient
    Long-Context LLM Inference" (NeurIPS'25 reading notes), §4.1
    Algorithm 1 (chunk-level compression) and §4.2 Algorithm 2 (layer-wise
    index reuse).
  * "Kara: ... sliding-window KV cache compression", §2 Preliminaries,
    Eq. (1): attention probabilities are softmax(Q K^T / sqrt(d)) per query row.

Readings where the notes are silent or loose (each is a choice of the plainest
form the rest supports):
  R1  Algorithm 1 step 1 prints the raw product Q_w K^T; the scores used here
      are the attention probabilities of Eq. (1): softmax over all T keys of
      each window-query row of Q_w K^T / sqrt(d).  No causal mask inside the
      window.
  R2  GQA: the scores of one KV head are summed over the window queries of
      every query head in its group; query head hq belongs to KV head
      hq // (Hq / Hkv).
  R3  Chunks are contiguous from token 0; the last one may be short and its
      score is a plain sum (no length normalisation).
  R4  k = floor(L_max / c), capped at the chunk count C; top-k order is
      score descending, ties to the lower chunk index.
  R5  The top-k runs over all C chunks, including those that overlap the recent
      window; the kept index list is the sorted set union of the selected
      chunks' tokens and the last w tokens (no duplicates).
  R6  Selection is independent per (sequence, layer, KV head); a reuse layer
      reuses the index list of the same (sequence, KV head).
  R9  The adjacent-layer similarity behind Algorithm 2 (§4.2, "observation":
      the indices ChunkKV selects are highly similar from one layer to the next,
      by Jaccard similarity) is taken over the kept index sets I_l of layers
      scored independently (N_reuse = 1), per (sequence, KV head):
      J = |I_l ∩ I_{l+1}| / |I_l ∪ I_{l+1}|.
  R10 Optional causal window (an option beside reading R1's unmasked window):
      window query q (0 <= q < w) sits at sequence position T - w + q and sees
      only keys j <= T - w + q; a query whose position is negative (T < w) sees
      no key and adds nothing.
  R12 Incremental compression during decoding (the notes keep the compressed
      cache through decoding, §5.6; Kara §2 Eqs. (2)-(3) compress again when
      the cache reaches its threshold).  A cache of one (sequence, KV head)
      holds n_prev positions kept by earlier passes followed by n_new tokens
      decoded since.  A pass re-scores only the new tail: the window rows
      attend to every key of the cache (the softmax of Eq. (1) runs over all
      n_prev + n_new keys), the tail is cut into chunks from its first token,
      Algorithm 1 steps 2-6 run on the tail alone (k = floor(L / c) of its
      chunks plus its last w tokens, L being the pass's budget for the tail),
      and the kept tail positions are appended to the n_prev kept ones, which
      stay as they are.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------- Algorithm 1

def group_window_rows(q_win_seq: np.ndarray, h: int, G: int) -> np.ndarray:
    """Window-query rows of KV head h: every query head of its group, every window row.

    q_win_seq: [w, Hq, d] (the last w query rows of one sequence).
    Returns [G * w, d] in fp64, ordered by (group member g, window row q).
    Reading R2 (GQA grouping hq -> hq // G).
    """
    rows = [q_win_seq[:, h * G + g, :] for g in range(G)]
    return np.concatenate(rows, axis=0).astype(np.float64)


def key_scores(rows: np.ndarray, keys: np.ndarray, limits=None) -> np.ndarray:
    """Per-key attention mass a_j = sum over window rows of softmax_j(rows . keys^T / sqrt(d)).

    ChunkKV §4.1 Algorithm 1 step 1 (window attention A, w x T_k) with the
    probabilities of Kara §2 Eq. (1) (reading R1).  rows [R, d], keys [T, d].
    limits: None, or per row the last key index the row may see (reading R10):
    the softmax of row r runs over keys 0..limits[r] only, and a row with a
    negative limit adds nothing.
    """
    T, d = keys.shape
    if T == 0:
        return np.zeros(0)
    if rows.shape[0] == 0:
        return np.zeros(T)
    logits = (rows.astype(np.float64) @ keys.astype(np.float64).T) / math.sqrt(d)   # [R, T]
    if limits is None:
        logits -= logits.max(axis=1, keepdims=True)
        p = np.exp(logits)
        p /= p.sum(axis=1, keepdims=True)                                            # each row sums to 1
        return p.sum(axis=0)
    a = np.zeros(T)
    for r, lim in enumerate(limits):
        n = min(int(lim), T - 1) + 1                                                 # keys 0 .. lim
        if n <= 0:
            continue
        x = logits[r, :n] - logits[r, :n].max()
        p = np.exp(x)
        a[:n] += p / p.sum()
    return a


def chunk_scores(a: np.ndarray, c: int) -> np.ndarray:
    """A_i = sum of a_j over the tokens of chunk i; C = ceil(T / c) chunks.

    ChunkKV §4.1 Algorithm 1 steps 2-3 (reading R3: the last chunk may hold
    fewer than c tokens and is not normalised).
    """
    T = a.shape[0]
    C = -(-T // c)
    out = np.zeros(C)
    for i in range(C):
        out[i] = a[i * c: min(i * c + c, T)].sum()
    return out


def n_select(T: int, c: int, L_max: int) -> int:
    """k = floor(L_max / c), capped at C (ChunkKV §4.1 Algorithm 1 step 4; reading R4)."""
    C = -(-T // c)
    return min(L_max // c, C)


def top_chunks(A: np.ndarray, k: int) -> list:
    """Indices of the k chunks with the largest score, ties to the lower index, ascending.

    ChunkKV §4.1 Algorithm 1 step 4 (TopK over chunk scores; reading R4).
    """
    order = sorted(range(len(A)), key=lambda i: (-float(A[i]), i))
    return sorted(order[:k])


def kept_indices(chunks: list, T: int, c: int, w: int) -> np.ndarray:
    """Sorted union of the selected chunks' tokens and the last w tokens.

    ChunkKV §4.1 Algorithm 1 steps 5-6 (recent window forced in, index list
    built for index_select; reading R5).
    """
    keep = set()
    for i in chunks:
        keep.update(range(i * c, min(i * c + c, T)))
    keep.update(range(max(0, T - w), T))
    return np.array(sorted(keep), dtype=np.int64)


def window_limits(n_rows: int, T: int, w: int) -> np.ndarray:
    """Last visible key of each window row under the causal window (reading R10): rows are ordered
    (group member g, window row q) as group_window_rows returns them; row q sits at T - w + q."""
    q = np.arange(n_rows) % max(w, 1)
    return T - w + q


def chunkkv_head(rows: np.ndarray, keys: np.ndarray, c: int, w: int, L_max: int, causal: bool = False):
    """Algorithm 1 for one (sequence, KV head): returns (A, selected chunks, kept indices)."""
    T = keys.shape[0]
    limits = window_limits(rows.shape[0], T, w) if causal else None
    A = chunk_scores(key_scores(rows, keys, limits), c)
    sel = top_chunks(A, n_select(T, c, L_max))
    return A, sel, kept_indices(sel, T, c, w)


def gather(x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """K' = index_select(K, indices) (ChunkKV §4.1 Algorithm 1 step 6)."""
    return x[idx]


# ---------------------------------------------------------------- decoding (reading R12)

def tail_key_scores(rows: np.ndarray, keys: np.ndarray, n_prev: int) -> np.ndarray:
    """a_j of the tail keys j >= n_prev of a cache, each window row's softmax running over all of
    the cache's keys (Kara §2 Eq. (1) over the whole cache; reading R12)."""
    return key_scores(rows, keys)[n_prev:]


def compress_tail_head(rows: np.ndarray, keys: np.ndarray, n_prev: int, c: int, w: int, L_tail: int):
    """One incremental pass over the cache of one (sequence, KV head) (reading R12): the tail
    [n_prev, T) is chunked from its first token and Algorithm 1 steps 2-6 (ChunkKV §4.1) select
    from it with budget L_tail.  Returns (A over the tail's chunks, selected tail chunks, the
    appended cache positions n_prev + i, ascending)."""
    n_new = keys.shape[0] - n_prev
    A = chunk_scores(tail_key_scores(rows, keys, n_prev), c)
    sel = top_chunks(A, n_select(n_new, c, L_tail))
    return A, sel, n_prev + kept_indices(sel, n_new, c, w)


# ---------------------------------------------------------------- Algorithm 2

def scoring_layer(layer: int, n_reuse: int) -> int:
    """Layer whose index list layer l uses: floor(l / N_reuse) * N_reuse (ChunkKV §4.2 Algorithm 2)."""
    return (layer // n_reuse) * n_reuse


def compress_layers(q_win, k, v, cu_seqlens, Hq: int, Hkv: int, w: int, c: int, L_max: int,
                    n_reuse: int, want_kv: bool = True, causal: bool = False):
    """ChunkKV with layer-wise index reuse over all layers of a batch of sequences.

    q_win[l]: [B, w, Hq, d] (read for layers with l mod N_reuse == 0 only);
    k[l], v[l]: [T_total, Hkv, d] with sequence b at rows cu_seqlens[b]..cu_seqlens[b+1].
    ChunkKV §4.2 Algorithm 2: layers with l mod N_reuse == 0 run Algorithm 1,
    the others gather with the indices of layer floor(l / N_reuse) * N_reuse.

    Returns a dict with, per scoring layer index g (group):
      scores[g][b][h]  fp64 chunk scores A,   chunks[g][b][h] selected chunk ids,
      indices[g][b][h] kept token positions (sequence-local, ascending),
    and, when want_kv, k_out[l][b][h] / v_out[l][b][h] (rows of K, V in input dtype).
    """
    n_layers = len(k)
    G = Hq // Hkv
    B = len(cu_seqlens) - 1
    res = {"scores": {}, "chunks": {}, "indices": {}, "k_out": {}, "v_out": {}}
    for layer in range(n_layers):
        src = scoring_layer(layer, n_reuse)
        if layer == src:
            sc, ch, ix = [], [], []
            for b in range(B):
                t0, t1 = cu_seqlens[b], cu_seqlens[b + 1]
                qb = np.asarray(q_win[layer][b])
                row_s, row_c, row_i = [], [], []
                for h in range(Hkv):
                    A, sel, idx = chunkkv_head(group_window_rows(qb, h, G),
                                               np.asarray(k[layer][t0:t1, h, :]), c, w, L_max, causal)
                    row_s.append(A)
                    row_c.append(sel)
                    row_i.append(idx)
                sc.append(row_s)
                ch.append(row_c)
                ix.append(row_i)
            g = src // n_reuse
            res["scores"][g], res["chunks"][g], res["indices"][g] = sc, ch, ix
        if want_kv:
            idx = res["indices"][src // n_reuse]
            ko, vo = [], []
            for b in range(B):
                t0, t1 = cu_seqlens[b], cu_seqlens[b + 1]
                ko.append([gather(np.asarray(k[layer][t0:t1, h, :]), idx[b][h]) for h in range(Hkv)])
                vo.append([gather(np.asarray(v[layer][t0:t1, h, :]), idx[b][h]) for h in range(Hkv)])
            res["k_out"][layer], res["v_out"][layer] = ko, vo
    return res


# ---------------------------------------------------------------- §4.2 observation (reading R9)

def layer_overlap(idx_a: np.ndarray, idx_b: np.ndarray) -> tuple:
    """(|A ∩ B|, |A ∪ B|) of two kept index sets: the counts behind the adjacent-layer Jaccard
    similarity that motivates Algorithm 2 (ChunkKV §4.2, observation; reading R9)."""
    a = set(int(x) for x in np.asarray(idx_a).ravel())
    b = set(int(x) for x in np.asarray(idx_b).ravel())
    return len(a & b), len(a | b)


def layer_jaccard(idx_a: np.ndarray, idx_b: np.ndarray) -> float:
    """|A ∩ B| / |A ∪ B| (1.0 for two empty sets)."""
    inter, union = layer_overlap(idx_a, idx_b)
    return 1.0 if union == 0 else inter / union

