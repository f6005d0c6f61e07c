"""Pins for the oracle's lightning-indexer score and top-k.

Hand-computed values, special cases that need no scoring, exact ties, the
independent dense oracle and selection invariants.
"""

import numpy as np
import pytest
import torch

import oracle
from csa_inputs import packs
from oracle import dense_ref


def run_topk(q, k, w, lengths, r, K, tokens=None):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cuc = oracle.compress_cu_seqlens(cu, r)
    T = int(cu[-1])
    qr = q if tokens is None else q[tokens]
    wr = w if tokens is None else w[tokens]
    return oracle.indexer_topk(qr, k, wr, T, cu, cuc, r, K, tokens=tokens), cuc


def test_hand_computed_scores():
    # One segment of 8 rows, r=4: blocks 0 and 1. Two heads, dim 2.
    T, Hi, Di = 8, 2, 2
    q = np.zeros((T, Hi, Di))
    w = np.zeros((T, Hi))
    q[7] = [[1, 0], [0, 1]]
    w[7] = [1.0, -1.0]
    q[3] = [[0.5, 0.5], [1, 1]]
    w[3] = [2.0, 0.25]
    k = np.array([[2.0, 3.0], [-1.0, 2.0]])
    (idx, val, kth, nxt, nvis), _ = run_topk(q, k, w, [8], 4, 2)
    # token 7: block0 = 1*relu(2) + (-1)*relu(3) = -1 ; block1 = 1*relu(-1) + (-1)*relu(2) = -2
    assert idx[7].tolist() == [0, 1]
    assert val[7].tolist() == [-1.0, -2.0]
    assert nvis[7] == 2
    # token 3 sees block 0 only: 2*relu(2.5) + 0.25*relu(5) = 6.25
    assert idx[3].tolist() == [0, -1]
    assert val[3][0] == 6.25 and val[3][1] == -np.inf
    assert nvis[3] == 1 and np.isnan(kth[3]) and np.isnan(nxt[3])
    # tokens 0..2 see nothing
    assert (idx[:3] == -1).all()
    # top-1 of token 7 keeps the higher score, and reports the k-th/k+1-th
    (idx1, val1, kth1, nxt1, _), _ = run_topk(q, k, w, [8], 4, 1)
    assert idx1[7].tolist() == [0] and val1[7].tolist() == [-1.0]
    assert kth1[7] == -1.0 and nxt1[7] == -2.0


def test_exact_ties_go_to_lower_index():
    lengths = [37, 64]
    T, Hi, Di, r, K = sum(lengths), 4, 8, 4, 5
    q = np.zeros((T, Hi, Di))  # every score is exactly 0
    rng = np.random.default_rng(0)
    k = rng.standard_normal((T // r, Di))
    w = rng.random((T, Hi))
    (idx, val, _, _, nvis), cuc = run_topk(q, k[: 9 + 16], w, lengths, r, K)
    for t in range(T):
        b = 0 if t < 37 else 1
        pos = t - (0 if b == 0 else 37)
        n = (pos + 1) // r
        expect = [cuc[b] + j for j in range(min(K, n))]
        assert idx[t].tolist() == expect + [-1] * (K - len(expect)), t
        assert nvis[t] == n


def test_topk_covering_all_visible_needs_no_scores():
    spec = packs.pack_spec("tiny")
    lengths = list(spec.lengths)
    rng = np.random.default_rng(1)
    T = sum(lengths)
    q, w = rng.standard_normal((T, 4, 64)), rng.standard_normal((T, 4))
    k = rng.standard_normal((63, 64))
    (idx, _, _, _, _), _ = run_topk(q, k, w, lengths, 4, 32)  # 32 >= max visible (29)
    vis = dense_ref.visible_mask(lengths, 4)
    for t in range(T):
        expect = np.nonzero(vis[t])[0].tolist()
        assert idx[t].tolist() == expect + [-1] * (32 - len(expect))


@pytest.mark.parametrize("K", [1, 3, 8])
def test_against_dense_oracle_tiny_pack(K):
    spec = packs.pack_spec("tiny")
    layer = spec.layers[0]
    t = packs.draw_pack(spec)[0]
    lengths = list(spec.lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    tc = int(oracle.compress_cu_seqlens(cu, 4)[-1])
    q = t["q_idx"].double().numpy()
    k = t["k_idx"][:tc].double().numpy()
    w = t["w"].double().numpy()
    (idx, val, kth, nxt, _), _ = run_topk(q, k, w, lengths, layer.cmp_ratio, K)
    scores = dense_ref.indexer_scores(q, k, w)
    vis = dense_ref.visible_mask(lengths, layer.cmp_ratio)
    np.testing.assert_array_equal(idx, dense_ref.topk_dense(scores, vis, K))
    sel = idx >= 0
    rows = np.nonzero(sel)
    np.testing.assert_allclose(val[sel], scores[rows[0], idx[sel]], rtol=1e-12, atol=1e-12)


def test_selection_invariants_random_pack():
    rng = np.random.default_rng(7)
    lengths = [1, 3, 250, 5, 130, 77]
    T, Hi, Di, r, K = sum(lengths), 8, 16, 4, 10
    q = rng.standard_normal((T, Hi, Di))
    w = rng.standard_normal((T, Hi))
    k = rng.standard_normal((T // r, Di))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    tc = int(oracle.compress_cu_seqlens(cu, r)[-1])
    (idx, val, kth, nxt, nvis), cuc = run_topk(q, k[:tc], w, lengths, r, K)
    scores = dense_ref.indexer_scores(q, k[:tc], w)
    vis = dense_ref.visible_mask(lengths, r)
    for t in range(T):
        sel = [j for j in idx[t] if j >= 0]
        assert len(sel) == min(K, vis[t].sum())
        assert sel == sorted(sel) and len(set(sel)) == len(sel)
        assert all(vis[t, j] for j in sel)
        rest = [j for j in np.nonzero(vis[t])[0] if j not in sel]
        if sel and rest:
            # the two computations round differently, so compare within 1e-12
            assert min(scores[t, sel]) >= max(scores[t, rest]) - 1e-12
            assert kth[t] == pytest.approx(min(scores[t, sel]), rel=1e-12, abs=1e-12)
            assert nxt[t] == pytest.approx(max(scores[t, rest]), rel=1e-12, abs=1e-12)


def test_token_list_matches_full_run():
    rng = np.random.default_rng(3)
    lengths = [90, 41]
    T, Hi, Di, r, K = 131, 4, 16, 4, 6
    q = rng.standard_normal((T, Hi, Di))
    w = rng.standard_normal((T, Hi))
    k = rng.standard_normal((32, Di))
    (idx, val, *_), _ = run_topk(q, k, w, lengths, r, K)
    toks = np.array([130, 0, 89, 90, 45])
    (idx2, val2, *_), _ = run_topk(q, k, w, lengths, r, K, tokens=toks)
    np.testing.assert_array_equal(idx2, idx[toks])
    np.testing.assert_array_equal(val2, val[toks])


def test_bf16_inputs_widen_exactly():
    x = torch.randn(4, 4, 8).bfloat16()
    assert np.array_equal(x.double().numpy(), x.float().double().numpy())
