"""The comparison rules of tests/parity.py reject planted errors (CPU only, no library).

The GPU parity tests pass only as long as these rules do: each case below hands a rule an output
that the library could plausibly produce when wrong and checks that it raises, and hands it the
legitimate outputs (exact, or a different choice at a near-tie cut) and checks that it accepts them.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import ATOL, RTOL, check_gather, check_indices, check_scores


def _kept(sel, T, c, w):
    return oracle.kept_indices(sorted(sel), T, c, w)


def test_scores_within_and_outside_the_tolerance():
    want = np.array([0.0, 1e-6, 0.5, 3.0, 250.0])
    check_scores(want * (1 + 0.9 * RTOL), want)
    check_scores(want + 0.9 * ATOL, want)
    for i in range(len(want)):
        bad = want.copy()
        bad[i] += ATOL + RTOL * abs(want[i]) * 1.2 + 1e-9
        with pytest.raises(AssertionError):
            check_scores(bad, want)
    with pytest.raises(AssertionError):
        check_scores(np.full(5, np.nan), want)


# T = 60, c = 5: 12 chunks; w = 7: the window covers tokens 53..59, so R = 53 and chunks 0..10 start
# before it (chunk 10 straddles); L_max = 20: k = 4.
T, C_, W, L_MAX = 60, 5, 7, 20
K = oracle.n_select(T, C_, L_MAX)


def _scores(cut_gap):
    """Chunk scores whose 4th and 5th largest (chunks 6 and 2) differ by cut_gap."""
    A = np.linspace(1.0, 2.0, 12)[::-1].copy() * 0.1      # descending, clearly apart
    A[[1, 4, 9]] = [5.0, 4.0, 3.0]                          # three clear winners
    A[6] = 2.0
    A[2] = 2.0 - cut_gap
    return A


def test_exact_lists_pass_and_a_clear_cut_is_exact():
    A = _scores(0.5)
    sel = oracle.top_chunks(A, K)
    assert sel == [1, 4, 6, 9]
    assert check_indices(_kept(sel, T, C_, W), A, T, C_, W, L_MAX) == "exact"
    for wrong in ([1, 4, 2, 9], [1, 4, 9], [1, 4, 6, 9, 2]):
        with pytest.raises(AssertionError):
            check_indices(_kept(wrong, T, C_, W), A, T, C_, W, L_MAX)


def test_near_tie_accepts_either_chunk_at_the_cut():
    A = _scores(0.2 * (ATOL + RTOL * 2.0))
    assert check_indices(_kept([1, 4, 6, 9], T, C_, W), A, T, C_, W, L_MAX) == "exact"
    assert check_indices(_kept([1, 2, 4, 9], T, C_, W), A, T, C_, W, L_MAX) == "near-tie"


def test_near_tie_rejects_planted_errors():
    A = _scores(0.2 * (ATOL + RTOL * 2.0))
    cases = {
        "a clear winner dropped": _kept([2, 4, 6, 9], T, C_, W),
        "a chunk clearly below the cut": _kept([0, 1, 4, 9], T, C_, W),
        "one chunk too few": _kept([1, 4, 9], T, C_, W),
        "one chunk too many": _kept([1, 2, 4, 6, 9], T, C_, W),
        "the window one token short": _kept([1, 2, 4, 9], T, C_, W - 1),
        "a token of a kept chunk missing": np.delete(_kept([1, 2, 4, 9], T, C_, W), 3),
        "a duplicate token": np.sort(np.append(_kept([1, 2, 4, 9], T, C_, W), 11)),
        "descending order": _kept([1, 2, 4, 9], T, C_, W)[::-1].copy(),
    }
    for what, got in cases.items():
        with pytest.raises(AssertionError):
            check_indices(got, A, T, C_, W, L_MAX, what)


def test_near_tie_with_a_window_chunk_in_the_selection():
    # chunk 11 (tokens 55..59) lies inside the window: the kept list cannot show whether it was
    # selected, so a list that holds only k - 1 chunks before the window passes when chunk 11 may
    # fill the last slot, and fails when it cannot
    A = _scores(0.5)
    A[11] = 2.0 - 0.2 * (ATOL + RTOL * 2.0)                 # ties with chunk 6 at the cut
    short = _kept([1, 4, 9], T, C_, W)
    assert check_indices(short, A, T, C_, W, L_MAX) == "near-tie"
    A[11] = 0.01                                            # now clearly below the cut
    A[2] = 2.0 - 0.2 * (ATOL + RTOL * 2.0)                  # the near tie is chunk 2 vs chunk 6
    with pytest.raises(AssertionError):
        check_indices(short, A, T, C_, W, L_MAX, "k - 1 chunks and no window chunk to fill the slot")


def test_no_tie_possible_when_everything_or_nothing_is_kept():
    A = np.full(12, 0.25)
    all_kept = np.arange(T)
    assert check_indices(all_kept, A, T, C_, W, 1000) == "exact"
    with pytest.raises(AssertionError):
        check_indices(all_kept[1:], A, T, C_, W, 1000)
    assert check_indices(np.arange(T - W, T), A, T, C_, W, 3) == "exact"
    with pytest.raises(AssertionError):
        check_indices(np.arange(T - W + 1, T), A, T, C_, W, 3)


def test_gather_rows_must_match_bit_for_bit():
    k = torch.arange(60 * 8, dtype=torch.float32).reshape(60, 8).to(torch.bfloat16)
    idx = np.array([0, 5, 6, 7, 59])
    rows = k[torch.as_tensor(idx)].clone()
    check_gather(rows, k, idx)
    bad = rows.clone()
    bad[2, 3] = bad[2, 3] + 1
    with pytest.raises(AssertionError):
        check_gather(bad, k, idx)
    with pytest.raises(AssertionError):
        check_gather(k[torch.as_tensor(idx[:-1] + 1)], k, idx[:-1])      # rows one token off


def test_near_tie_rule_against_brute_force():
    # On small cases every subset of chunks gives a candidate list.  The rule must accept the
    # oracle's list and, when the oracle's k-th and (k+1)-th scores differ by less than the
    # tolerance, exactly the lists of the k-chunk selections that scores within the tolerance can
    # produce.  Built here by construction: raise the selection's scores by their tolerance and
    # lower the others by theirs; the selection is reachable iff it is then the oracle's top-k.
    import itertools
    rng = np.random.default_rng(31)
    n_near = 0
    for trial in range(60):
        c = int(rng.integers(1, 4))
        C = int(rng.integers(2, 8))
        T = C * c - int(rng.integers(0, c))                   # ragged last chunk when c > 1
        w = int(rng.integers(0, 2 * c + 1))
        L_max = int(rng.integers(c, C * c))
        k = oracle.n_select(T, c, L_max)
        # scores on a coarse grid with offsets inside and outside the tolerance
        A = rng.integers(0, 3, size=C) + rng.choice([0.0, 3e-4, 4e-3], size=C)
        tol = ATOL + RTOL * np.abs(A)
        srt = np.sort(A)[::-1]
        near = 0 < k < C and srt[k - 1] - srt[k] < ATOL + RTOL * abs(srt[k - 1])
        valid = {tuple(_kept(oracle.top_chunks(A, k), T, c, w).tolist())}
        for Sv in itertools.combinations(range(C), k) if near else ():
            up = np.array([A[i] + tol[i] if i in Sv else A[i] - tol[i] for i in range(C)])
            if oracle.top_chunks(up, k) == list(Sv):
                valid.add(tuple(_kept(list(Sv), T, c, w).tolist()))
        for r in range(C + 1):
            for S in itertools.combinations(range(C), r):
                got = _kept(list(S), T, c, w)
                try:
                    verdict = check_indices(got, A, T, c, w, L_max)
                except AssertionError:
                    verdict = None
                assert (verdict is not None) == (tuple(got.tolist()) in valid), (A, k, S, T, c, w)
                n_near += verdict == "near-tie"
    assert n_near > 20                          # the cases reach the near-tie branch often
