"""Comparison rules between the CUDA library and the CPU oracle.

Chunk scores: |gpu - oracle| <= 1e-5 + 1e-3 |oracle|.
Kept indices: identical to the oracle's, except when the oracle's k-th and
(k+1)-th largest chunk scores are closer than that tolerance; then any
selection of exactly k chunks that holds every chunk clearly above the cut and
only chunks not clearly below it is accepted, and the index list must be
exactly the one that selection defines (chunks inside the recent window leave
no trace in the list, so the check asks that such a selection exists).
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
    """Returns 'exact' or 'near-tie' (accepted); raises on a mismatch."""
    got = [int(x) for x in got_idx]
    k = oracle.n_select(T, c, L_max)
    sel = oracle.top_chunks(A, k)
    want = oracle.kept_indices(sel, T, c, w).tolist()
    if got == want:
        return "exact"
    C = len(A)
    srt = np.sort(A)[::-1]
    if not (0 < k < C):
        raise AssertionError(f"{what}: index list differs (k={k}, C={C}, no tie possible)")
    a_k, a_k1 = srt[k - 1], srt[k]
    tol = ATOL + RTOL * abs(a_k)
    if a_k - a_k1 >= tol:
        raise AssertionError(f"{what}: index list differs from the oracle and the cut is clear "
                             f"({a_k!r} vs {a_k1!r}); first difference "
                             f"{next((i for i, (x, y) in enumerate(zip(got, want)) if x != y), None)}")
    R = max(0, T - w)
    visible = {i for i in range(C) if i * c < R}
    chosen = sorted({j // c for j in got if j < R})
    must = {i for i in range(C) if A[i] > a_k + tol}
    allowed = {i for i in range(C) if A[i] >= a_k1 - tol}
    # the selection is chosen plus k - |chosen| chunks inside the window, which the list cannot
    # show: it exists when the window holds every clear winner it must and enough allowed chunks
    ok = (must & visible) <= set(chosen) <= allowed \
        and len(must - visible) <= k - len(chosen) <= len(allowed - visible) \
        and got == oracle.kept_indices(chosen, T, c, w).tolist()
    if not ok:
        raise AssertionError(f"{what}: near-tie at the cut but the selection is not a valid one")
    return "near-tie"


def check_gather(k_out_rows: torch.Tensor, k_src: torch.Tensor, idx: np.ndarray, what: str = "") -> None:
    ref = k_src[torch.as_tensor(np.asarray(idx, dtype=np.int64), device=k_src.device)]
    if not torch.equal(k_out_rows, ref):
        bad = (k_out_rows != ref).any(dim=-1).nonzero()
        raise AssertionError(f"{what}: gathered rows differ from K[indices] at rows {bad[:5].tolist()}")
