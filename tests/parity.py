"""Comparison rules between the CUDA library and the CPU oracle.

Chunk scores: |gpu - oracle| <= 1e-5 + 1e-3 |oracle|.
Kept indices: identical to the oracle's, except when the oracle's k-th and
(k+1)-th largest chunk scores differ by less than that tolerance; then the list
of any selection of exactly k chunks that is the top-k of some scores each
within that tolerance of the oracle's is accepted (the GPU selects exactly on
its own scores, which check_scores holds to that tolerance); chunks inside the
recent window leave no trace in the list, so the check asks that such a
selection exists.
K', V': bit-exact rows of K, V at the GPU's indices.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL, RTOL = 1e-5, 1e-3


def f64(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def check_scores(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    got = np.asarray(got[: len(want)], dtype=np.float64)
    bad = ~(np.abs(got - want) <= ATOL + RTOL * np.abs(want))      # NaN fails too
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} chunk scores off, first at {i}: "
                             f"gpu {got[i]!r} oracle {want[i]!r}")


def check_indices(got_idx: np.ndarray, A: np.ndarray, T: int, c: int, w: int, L_max: int,
                  what: str = "") -> str:
    """Returns 'exact' or 'near-tie' (accepted); raises on a mismatch.

    A list other than the oracle's passes only at a near-tie, when the oracle's k-th and (k+1)-th
    largest chunk scores differ by less than the chunk-score tolerance, and only when it is the list
    of a selection S of exactly k chunks that is the top-k of some scores each within that tolerance
    of the oracle's: min over S of (A_i + tol_i) >= max over the other chunks of (A_j - tol_j).
    Chunks inside the recent window leave no trace in the list; the best of them (largest A) fill
    the slots the list leaves, which is the choice that makes the condition easiest to meet.
    """
    got = [int(x) for x in got_idx]
    k = oracle.n_select(T, c, L_max)
    sel = oracle.top_chunks(A, k)
    want = oracle.kept_indices(sel, T, c, w).tolist()
    if got == want:
        return "exact"
    C = len(A)
    if not (0 < k < C):
        raise AssertionError(f"{what}: index list differs (k={k}, C={C}, no tie possible)")
    srt = np.sort(A)[::-1]
    a_k, a_k1 = srt[k - 1], srt[k]
    if a_k - a_k1 >= ATOL + RTOL * abs(a_k):
        raise AssertionError(f"{what}: index list differs from the oracle and the cut is clear "
                             f"({a_k!r} vs {a_k1!r}); first difference "
                             f"{next((i for i, (x, y) in enumerate(zip(got, want)) if x != y), None)}")
    R = max(0, T - w)
    chosen = sorted({j // c for j in got if j < R})
    hidden = sorted((i for i in range(C) if i * c >= R), key=lambda i: -A[i])
    fill = k - len(chosen)
    if fill < 0 or fill > len(hidden) or got != oracle.kept_indices(chosen, T, c, w).tolist():
        raise AssertionError(f"{what}: index list is not the list of any {k} chunks; first difference "
                             f"{next((i for i, (x, y) in enumerate(zip(got, want)) if x != y), None)}")
    S = set(chosen) | set(hidden[:fill])
    tol = ATOL + RTOL * np.abs(A)
    low = min(A[i] + tol[i] for i in S)
    high = max(A[j] - tol[j] for j in range(C) if j not in S)
    if low < high:
        raise AssertionError(f"{what}: selection differs from the oracle's beyond the score tolerance "
                             f"(weakest kept {low!r} < strongest dropped {high!r})")
    return "near-tie"


def check_gather(k_out_rows: torch.Tensor, k_src: torch.Tensor, idx: np.ndarray, what: str = "") -> None:
    ref = k_src[torch.as_tensor(np.asarray(idx, dtype=np.int64), device=k_src.device)]
    if not torch.equal(k_out_rows, ref):
        bad = (k_out_rows != ref).any(dim=-1).nonzero()
        raise AssertionError(f"{what}: gathered rows differ from K[indices] at rows {bad[:5].tolist()}")
