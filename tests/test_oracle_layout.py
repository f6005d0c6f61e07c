"""Pins for the oracle's integer steps: compressed cu_seqlens and window rows.

Checked against worked values derived by hand from the pages (golden file),
against brute-force enumeration, and against invariants.
"""

import os

import numpy as np
import pytest

import oracle
from oracle import dense_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_pack_layout.txt")


def load_golden():
    cu = cuc = None
    win, vis = {}, {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            vals = [int(v) for v in vals]
            if tag == "cu":
                cu = vals
            elif tag == "cu_cmp":
                cuc = vals
            elif tag == "win":
                win[vals[0]] = vals[1:]
            elif tag == "vis":
                vis[vals[0]] = vals[1:]
    return cu, cuc, win, vis


def brute_compress(lengths, r):
    """Count complete groups of r rows per segment by walking the segment."""
    out = [0]
    for L in lengths:
        groups, start = 0, 0
        while start + r <= L:
            groups += 1
            start += r
        out.append(out[-1] + groups)
    return out


def brute_window(lengths, W):
    """Row lists by set membership: same segment, not after t, fewer than W back."""
    seg = []
    for b, L in enumerate(lengths):
        seg += [b] * L
    T = len(seg)
    rows = []
    for t in range(T):
        members = sorted(s for s in range(T) if seg[s] == seg[t] and s <= t and t - s < W)
        rows.append(members + [-1] * (W - len(members)))
    return np.array(rows, dtype=np.int32).reshape(T, W)


def test_golden_tiny_pack():
    cu, cuc, win, _ = load_golden()
    assert oracle.compress_cu_seqlens(cu, 4).tolist() == cuc
    idx = oracle.window_idx(cu, 256, 15)
    assert idx.shape == (256, 16)
    for t, row in win.items():
        assert idx[t].tolist() == row, t


def test_compress_edge_segments():
    # zero-length, shorter than r, exactly r, r+1, multiples
    lengths = [0, 1, 3, 4, 5, 7, 8, 0, 9, 128, 127, 129]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    for r in (1, 2, 4, 128):
        assert oracle.compress_cu_seqlens(cu, r).tolist() == brute_compress(lengths, r)


@pytest.mark.parametrize("seed", range(6))
def test_compress_random(seed):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(0, 300, size=rng.integers(1, 20)).tolist()
    cu = np.concatenate([[0], np.cumsum(lengths)])
    for r in (3, 4, 128):
        got = oracle.compress_cu_seqlens(cu, r)
        assert got.tolist() == brute_compress(lengths, r)
        # the dense oracle's grouping (written separately) must agree
        cseg, first, last = dense_ref.compressed_layout(lengths, r)
        assert len(cseg) == got[-1]
        assert np.all(last - first == r - 1)


@pytest.mark.parametrize("W", [1, 2, 16, 128])
def test_window_brute_force(W):
    rng = np.random.default_rng(W)
    lengths = [1, 3, 4, 5] + rng.integers(1, 200, size=5).tolist()
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T = int(cu[-1])
    got = oracle.window_idx(cu, T, W - 1)
    np.testing.assert_array_equal(got, brute_window(lengths, W))
    # invariant: the number of valid rows is min(W, pos + 1)
    seg = dense_ref.segment_ids(lengths)
    pos = np.arange(T) - cu[seg]
    np.testing.assert_array_equal((got >= 0).sum(1), np.minimum(W, pos + 1))
    # and it matches the dense window mask
    np.testing.assert_array_equal((got >= 0).sum(1), dense_ref.window_mask(lengths, W).sum(1))


def test_window_rejects_bad_cu():
    with pytest.raises(ValueError):
        oracle.window_idx([0, 5, 3], 3, 4)  # decreasing
    with pytest.raises(ValueError):
        oracle.window_idx([1, 5], 4, 4)  # does not start at 0


def test_visible_blocks_golden():
    """The dense visibility rule reproduces the hand-derived block ranges."""
    cu, cuc, _, vis = load_golden()
    lengths = np.diff(cu).tolist()
    mask = dense_ref.visible_mask(lengths, 4)
    for t, (count, first, last) in vis.items():
        rows = np.nonzero(mask[t])[0]
        assert len(rows) == count, t
        if count:
            assert rows[0] == first and rows[-1] == last, t


def test_window_rows_of_listed_tokens_match_the_whole_table():
    rng = np.random.default_rng(3)
    cu = np.concatenate([[0], np.cumsum(rng.integers(1, 300, size=9))]).astype(np.int32)
    T = int(cu[-1])
    toks = rng.integers(0, T, size=50).astype(np.int32)
    for W in (1, 16, 128):
        whole = oracle.window_idx(cu, T, W - 1)
        np.testing.assert_array_equal(oracle.window_idx(cu, T, W - 1, toks), whole[toks])
