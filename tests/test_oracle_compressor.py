"""Pins for the oracle's THD compressor core (miles PR 2038 report,
compressor.py _forward_thd grouping and _overlap_transform_thd; the pooling
after the transform is a reading, see the oracle's comment).

What pins it, apart from the oracle itself:
* slot placement, phrased from the token's side: boosting the score of one
  packed element (row t, column c) makes exactly one output element take
  that element's kv value -- the compressed row that contains t (or, for a
  first-half column with overlap, the next compressed row of the same
  sequence) at dimension c mod head_dim -- and leaves every other output
  bit-identical; rows in a sequence's tail (len % ratio) and first-half
  columns of a sequence's last group feed nothing;
* the pooling equals scipy.special.softmax over the slots on sequences of
  exactly one group (whose slots are its rows);
* closed forms with zero scores: a first group pools the mean of its own r
  rows, a later group (with overlap) the mean of 2r consecutive rows;
* invariances: a per-column constant added to every ape slot changes
  nothing; sequences are isolated; ratio 1 without overlap is the identity.
"""

import numpy as np
import pytest
from scipy import special

import oracle

LENGTHS = [11, 3, 9, 4]    # tails of 3, 3, 1, 0 rows; the length-3 sequence has no group
R, HD = 4, 3


def cu_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def token_target(t, c, lengths, r, hd, overlap):
    """(compressed row, dimension) fed by packed element (t, c), or None,
    derived from the token's position in its sequence."""
    cu = cu_of(lengths)
    b = int(np.searchsorted(cu, t, side="right") - 1)
    pos = t - cu[b]
    groups = lengths[b] // r
    first_row = sum(L // r for L in lengths[:b])
    own = pos // r
    if own >= groups:
        return None  # the tail: no compressed row
    if not overlap:
        return first_row + own, c
    if c >= hd:
        return first_row + own, c - hd
    nxt = own + 1  # the first half is pulled by the next group of the sequence
    return (first_row + nxt, c) if nxt < groups else None


@pytest.mark.parametrize("overlap", [True, False])
def test_slot_placement_from_the_token_side(overlap):
    rng = np.random.default_rng(0)
    cu = cu_of(LENGTHS)
    T = int(cu[-1])
    wd = 2 * HD if overlap else HD
    kv = rng.standard_normal((T, wd))
    base_score = np.zeros((T, wd))
    ape = rng.standard_normal((R, wd)) * 0.1
    base = oracle.compress_thd(kv, base_score, ape, cu, R, HD, overlap)
    fed = 0
    for t in range(T):
        for c in range(wd):
            score = base_score.copy()
            score[t, c] = 80.0
            out = oracle.compress_thd(kv, score, ape, cu, R, HD, overlap)
            target = token_target(t, c, LENGTHS, R, HD, overlap)
            changed = np.argwhere(out != base)
            if target is None:
                assert len(changed) == 0, (t, c)
                continue
            fed += 1
            assert [tuple(x) for x in changed] == [target], (t, c, changed, target)
            assert out[target] == pytest.approx(kv[t, c], abs=1e-20 + 1e-12 * abs(kv[t, c]))
    n_groups = sum(L // R for L in LENGTHS)
    slots = 2 * R if overlap else R
    # every slot of every group is fed once, except the missing predecessors
    firsts = sum(1 for L in LENGTHS if L // R > 0)
    assert fed == n_groups * slots * HD - (firsts * R * HD if overlap else 0)


@pytest.mark.parametrize("overlap", [True, False])
def test_pooling_is_library_softmax_on_single_groups(overlap):
    rng = np.random.default_rng(1)
    lengths = [R, R, R]  # one group per sequence: its slots are its own rows
    cu = cu_of(lengths)
    T = int(cu[-1])
    wd = 2 * HD if overlap else HD
    kv = rng.standard_normal((T, wd))
    score = rng.standard_normal((T, wd)) * 3
    ape = rng.standard_normal((R, wd))
    out = oracle.compress_thd(kv, score, ape, cu, R, HD, overlap)
    for b in range(3):
        rows = slice(int(cu[b]), int(cu[b + 1]))
        cols = slice(HD, 2 * HD) if overlap else slice(0, HD)
        p = special.softmax(score[rows, cols] + ape[:, cols], axis=0)
        np.testing.assert_allclose(out[b], (p * kv[rows, cols]).sum(0), rtol=1e-13, atol=1e-15)


def test_zero_scores_closed_form():
    lengths = [13, 2, 8]
    cu = cu_of(lengths)
    T = int(cu[-1])
    kv = np.repeat(np.arange(T, dtype=float)[:, None], 2 * HD, axis=1)  # every column = row index
    out = oracle.compress_thd(kv, np.zeros((T, 2 * HD)), None, cu, R, HD, True)
    g = 0
    for b, L in enumerate(lengths):
        for j in range(L // R):
            start = cu[b] + j * R
            want = start + (R - 1) / 2 if j == 0 else start - R + (2 * R - 1) / 2
            np.testing.assert_allclose(out[g], want, rtol=0, atol=1e-12)
            g += 1
    assert g == out.shape[0]


def test_invariances():
    rng = np.random.default_rng(2)
    cu = cu_of(LENGTHS)
    T = int(cu[-1])
    kv = rng.standard_normal((T, 2 * HD))
    score = rng.standard_normal((T, 2 * HD))
    ape = rng.standard_normal((R, 2 * HD))
    base = oracle.compress_thd(kv, score, ape, cu, R, HD, True)
    # a per-column constant on every slot: the two halves meet in one
    # softmax per dimension, so shift both halves of dimension e alike
    shift = rng.standard_normal(HD)
    ape2 = ape + np.concatenate([shift, shift])[None, :]
    np.testing.assert_allclose(oracle.compress_thd(kv, score, ape2, cu, R, HD, True), base,
                               rtol=1e-12, atol=1e-14)
    # isolation: rows of the last sequence change, the others' outputs do not
    kv2, score2 = kv.copy(), score.copy()
    kv2[cu[3]:] += 5.0
    score2[cu[3]:] -= 2.0
    out2 = oracle.compress_thd(kv2, score2, ape, cu, R, HD, True)
    n_before = sum(L // R for L in LENGTHS[:3])
    assert np.array_equal(out2[:n_before], base[:n_before])
    assert not np.allclose(out2[n_before:], base[n_before:])
    # ratio 1 without overlap is the identity
    np.testing.assert_allclose(oracle.compress_thd(kv[:, :HD], score[:, :HD], None, cu, 1, HD,
                                                   False), kv[:, :HD], rtol=0, atol=0)
