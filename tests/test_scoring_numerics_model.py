"""The single-pass scoring scheme's error budget, replayed in numpy float32 against the oracle (CPU only).

The tensor-core path scores a work item (one unit of keys, one KV head) per row in one pass:
  - the row's reference R is the largest base-2 logit of the item's first 80-key tile, plus a shift
    of 86 so that every term 2^(t - R) is at most 2^-86 and the 16-bit code of a bin is the rounded
    upper half of its fp32 pattern;
  - the terms are summed per chunk in fp32 and each chunk's sum is stored as a 16-bit code; the row
    sum l of the item is kept in fp32;
  - when l outgrows (1 - 2^-10) 2^-63 after a tile, the row moves R to that tile's maximum (+86),
    multiplies the codes it already wrote (decoded, rescaled, encoded again), l and the running chunk
    sum by 2^(R_old - R_new), and redoes the tile;
  - afterwards a row's base-2 log-sum-exp merges the (R, l) pairs of all its items, and a chunk
    scores sum over rows of bin * 2^(R - lse).
This model states those steps in numpy float32 (exp2 exact to float32 rounding, where the kernel uses
ex2.approx) and checks, on inputs chosen to stress them, that the chunk scores stay within the parity
tolerance of the oracle (abs 1e-5 + rel 1e-3).  It tests the scheme, not the CUDA code.
"""
import math

import numpy as np
import pytest

import oracle
from parity import ATOL, RTOL

SHIFT = 86
BIG = np.float32((1 - 2.0 ** -10) * 2.0 ** -63)
TILE = 80


def enc(v):
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) >> 13).astype(np.uint32)


def dec(code):
    return (np.asarray(code, np.uint64) << 13).astype(np.uint32).view(np.float32)


def model_chunk_scores(rows, keys, c, unit_keys, rescale_codes=True):
    """Chunk scores of one KV head by the single-pass scheme (rows [R, d], keys [T, d], fp64 inputs).

    unit_keys: keys per work item, a multiple of lcm(80, c) as the planner makes them (items hold
    whole tiles and whole chunks).  rescale_codes=False plants a fault: a rescale leaves the codes
    already written as they were.
    """
    T, d = keys.shape
    assert unit_keys % (TILE * c // math.gcd(TILE, c)) == 0
    n_rows = rows.shape[0]
    alpha = np.float32(1.0 / math.log(2) / math.sqrt(d))
    s_all = (rows.astype(np.float32) @ keys.astype(np.float32).T).astype(np.float32)      # fp32 MMA
    C = -(-T // c)
    items = []                                         # (first chunk, R [rows], l [rows], codes [chunks, rows])
    for k0 in range(0, T, unit_keys):
        nk = min(unit_keys, T - k0)
        n_ch = -(-nk // c)
        codes = np.zeros((n_ch, n_rows), np.uint32)
        s = s_all[:, k0:k0 + nk]
        R = (s[:, :min(TILE, nk)].max(axis=1) * alpha + np.float32(SHIFT)).astype(np.float32)
        l = np.zeros(n_rows, np.float32)
        carry = np.zeros(n_rows, np.float32)
        for t0 in range(0, nk, TILE):
            cols = range(t0, min(t0 + TILE, nk))
            for attempt in range(2):
                l_t, carry_t, writes = l.copy(), carry.copy(), {}
                for j in cols:
                    e = np.exp2((s[:, j] * alpha - R).astype(np.float32)).astype(np.float32)
                    carry_t = (carry_t + e).astype(np.float32)
                    if (j + 1) % c == 0 or j + 1 == nk:              # a chunk ends here
                        writes[j // c] = carry_t.copy()
                        l_t = (l_t + carry_t).astype(np.float32)
                        carry_t = np.zeros(n_rows, np.float32)
                over = ~(l_t <= BIG)
                if attempt == 1 or not over.any():
                    break
                tm = (s[:, cols.start:cols.stop].max(axis=1) * alpha + np.float32(SHIFT)).astype(np.float32)
                R2 = np.where(over, np.maximum(R, tm), R).astype(np.float32)
                f = np.exp2((R - R2).astype(np.float32)).astype(np.float32)
                done = t0 // c                                   # chunks completed before this tile
                if rescale_codes:
                    codes[:done] = np.where(over[None, :], enc(dec(codes[:done]) * f[None, :]), codes[:done])
                l = (l * f).astype(np.float32)
                carry = (carry * f).astype(np.float32)
                R = R2
            assert not over.any() or attempt == 1
            for ch, v in writes.items():
                codes[ch] = enc(v)
            l, carry = l_t, carry_t
        items.append((k0 // c, R, l, codes))
    # base-2 log-sum-exp of every row over its items
    M = np.full(n_rows, -np.inf, np.float32)
    S = np.zeros(n_rows, np.float32)
    for _, R, l, _ in items:
        Mn = np.maximum(M, R)
        S = (S * np.exp2(M - Mn) + l * np.exp2(R - Mn)).astype(np.float32)
        M = Mn
    lse = (M + np.log2(S)).astype(np.float32)
    A = np.zeros(C)
    for ch0, R, l, codes in items:
        wgt = np.exp2((R - lse).astype(np.float32)).astype(np.float32)
        A[ch0:ch0 + codes.shape[0]] = (dec(codes) * wgt[None, :]).astype(np.float64).sum(axis=1)
    return A


def _oracle(rows, keys, c):
    return oracle.chunk_scores(oracle.key_scores(rows, keys), c)


def _bf16(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def _check(rows, keys, c, unit_keys, **kw):
    rows, keys = _bf16(rows), _bf16(keys)
    got = model_chunk_scores(rows, keys, c, unit_keys, **kw)
    want = _oracle(rows, keys, c)
    err = np.abs(got - want) / (ATOL + RTOL * np.abs(want))
    assert err.max() <= 1.0, f"worst error {err.max():.3f} of the tolerance at chunk {int(err.argmax())}"
    return err.max()


def test_model_matches_the_oracle_on_plain_random_inputs():
    rng = np.random.default_rng(1)
    worst = _check(rng.standard_normal((128, 128)), rng.standard_normal((2000, 128)), 10, 240)
    assert worst < 0.5


def _ramp_case(seed=3):
    # rows sharing a component along v and keys whose logits climb along v key by key (about 15 bits
    # a tile for most rows), so that most rows outgrow their first-tile reference in every item
    rng = np.random.default_rng(seed)
    d = 128
    v = rng.standard_normal(d)
    v /= np.linalg.norm(v)
    rows = rng.standard_normal((64, d)) + 3.0 * v[None, :]
    keys = rng.standard_normal((1001, d)) + 0.5 * np.arange(1001)[:, None] * v[None, :]
    return rows, keys


def test_model_with_a_climbing_maximum_and_short_chunks():
    # c = 3 with a ragged last chunk and a ragged last item; the planted fault shows the rescale is hit
    rows, keys = _ramp_case()
    _check(rows, keys, 3, 240)
    with pytest.raises(AssertionError):
        _check(rows, keys, 3, 240, rescale_codes=False)


def test_model_with_flat_and_peaked_rows():
    rng = np.random.default_rng(4)
    d = 128
    keys = np.zeros((777, d))                           # every logit 0: uniform mass, no rescale
    _check(rng.standard_normal((32, d)), keys, 7, 560)
    keys = 0.1 * rng.standard_normal((777, d))
    keys[500] = 60.0 * np.ones(d) / math.sqrt(d)       # one key far above all others, in a later tile
    rows = np.ones((32, d)) + 0.1 * rng.standard_normal((32, d))
    _check(rows, keys, 7, 560)


def _rescale_case(seed=2, n=128, T=2400):
    rng = np.random.default_rng(seed)
    d = 128
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    sign = np.where(np.arange(n) % 2 == 0, 1.0, -1.0)
    rows = rng.standard_normal((n, d)) + 10.0 * sign[:, None] * u[None, :]
    keys = 0.3 * rng.standard_normal((T, d))
    keys[150::240] = 34.0 * u
    return rows, keys


def test_model_rescales_rows_that_outgrow_their_first_tile():
    # half the rows along a direction u meet a key about 30 natural-log units above their first tile
    # in the second tile of every item; the other half point against u
    rows, keys = _rescale_case()
    _check(rows, keys, 10, 240)


def test_a_rescale_that_forgets_the_written_codes_breaks_the_tolerance():
    # the same inputs with the planted fault: the check must fail, so the inputs do reach the rescale
    rows, keys = _rescale_case()
    with pytest.raises(AssertionError):
        _check(rows, keys, 10, 240, rescale_codes=False)


# ---------------------------------------------------------------- token-level chunks: two passes
def model_two_pass_token_scores(rows, keys, unit_keys, drop_lse_of_later_items=False):
    """Per-token scores (c = 1) of one KV head by the two-pass scheme of the tensor-core path.

    Pass 1 forms each work item's (R, l) per row exactly as the single pass does (R = first-tile
    maximum + 86, l summed in fp32, a row whose l outgrows the bound moves R to that tile's maximum and
    rescales l), but writes no bins; the rows' base-2 log-sum-exps merge the pairs of all items.  Pass 2
    recomputes the logits and forms 2^(t - lse) in fp32, sums them per key over each warp's 32 rows,
    then over the warps in order.  drop_lse_of_later_items plants a fault: the normaliser of a row is
    that of its first item only.
    """
    T, d = keys.shape
    n_rows = rows.shape[0]
    alpha = np.float32(1.0 / math.log(2) / math.sqrt(d))
    s_all = (rows.astype(np.float32) @ keys.astype(np.float32).T).astype(np.float32)
    pairs = []
    for k0 in range(0, T, unit_keys):
        nk = min(unit_keys, T - k0)
        s = s_all[:, k0:k0 + nk]
        R = (s[:, :min(TILE, nk)].max(axis=1) * alpha + np.float32(SHIFT)).astype(np.float32)
        l = np.zeros(n_rows, np.float32)
        for t0 in range(0, nk, TILE):
            blk = s[:, t0:min(t0 + TILE, nk)]
            l_t = (l + np.exp2((blk * alpha - R[:, None]).astype(np.float32)).astype(np.float32).sum(axis=1,
                                                                                                 dtype=np.float32))
            over = ~(l_t <= BIG)
            if over.any():
                tm = (blk.max(axis=1) * alpha + np.float32(SHIFT)).astype(np.float32)
                R2 = np.where(over, np.maximum(R, tm), R).astype(np.float32)
                l = (l * np.exp2((R - R2).astype(np.float32))).astype(np.float32)
                R = R2
                l_t = (l + np.exp2((blk * alpha - R[:, None]).astype(np.float32)).astype(np.float32).sum(
                    axis=1, dtype=np.float32))
            l = l_t.astype(np.float32)
        pairs.append((R, l))
    if drop_lse_of_later_items:
        pairs = pairs[:1]
    M = np.full(n_rows, -np.inf, np.float32)
    S = np.zeros(n_rows, np.float32)
    for R, l in pairs:
        Mn = np.maximum(M, R)
        S = (S * np.exp2(M - Mn) + l * np.exp2(R - Mn)).astype(np.float32)
        M = Mn
    lse = (M + np.log2(S)).astype(np.float32)
    p = np.exp2((s_all * alpha - lse[:, None]).astype(np.float32)).astype(np.float32)
    A = np.zeros(T, np.float32)
    for r0 in range(0, n_rows, 32):                     # warp partial sums, then the warps in order
        A = (A + p[r0:r0 + 32].sum(axis=0, dtype=np.float32)).astype(np.float32)
    return A.astype(np.float64)


def _check_two_pass(rows, keys, unit_keys, **kw):
    rows, keys = _bf16(rows), _bf16(keys)
    got = model_two_pass_token_scores(rows, keys, unit_keys, **kw)
    want = _oracle(rows, keys, 1)
    err = np.abs(got - want) / (ATOL + RTOL * np.abs(want))
    assert err.max() <= 1.0, f"worst error {err.max():.3f} of the tolerance at key {int(err.argmax())}"
    return err.max()


def test_two_pass_token_level_model_matches_the_oracle():
    rng = np.random.default_rng(7)
    worst = _check_two_pass(rng.standard_normal((128, 128)), rng.standard_normal((1500, 128)), 240)
    assert worst < 0.05                                 # fp32 sums: far inside the tolerance
    rows, keys = _rescale_case()                        # rows whose maximum climbs past the first tile's
    _check_two_pass(rows, keys, 240)
    rows, keys = _ramp_case()
    _check_two_pass(rows, keys, 160)


def test_two_pass_needs_the_normaliser_over_every_item():
    # planted fault: a row's lse from its first item alone scores every key too high
    rows, keys = _rescale_case()
    with pytest.raises(AssertionError):
        _check_two_pass(rows, keys, 240, drop_lse_of_later_items=True)
