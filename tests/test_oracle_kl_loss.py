"""Pins for the oracle's indexer KL-loss gradient (the hyper-parallel RFC,
section 3, sparse_lightning_indexer_kl_loss_grad: the indexer's backward
with a KL loss against the main attention's distribution).

What pins it, apart from the oracle itself:
* the per-token loss equals scipy.stats.entropy(p, softmax(I)) (a library
  KL divergence, which also L1-normalises p), with the scores I taken from
  the independent dense NumPy restatement and the entry set S from its
  visibility mask;
* every gradient element equals the central finite difference of
  grad_scale * sum(loss) in the input it belongs to;
* closed forms: p proportional to softmax(I) gives zero loss and zero
  gradients; w = 0 makes softmax(I) uniform, so the loss is log|S| - H(p),
  d_q and d_k vanish and d_w is the uniform-minus-target weighting of the
  ReLU'd dot products; a single entry gives zero loss;
* invariances: the order of a token's entries (with their targets), the
  scale of a token's targets, and computing tokens one at a time.
"""

import numpy as np
import pytest
from scipy import special, stats

import oracle
from oracle import dense_ref

LENGTHS = [13, 3, 22, 9]   # the length-3 segment has no compressed row
R, HI, DI, TOPK = 4, 3, 8, 6
GRAD_SCALE = 0.37


def cu_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def make_case(seed, topk=TOPK, w_zero=False):
    rng = np.random.default_rng(seed)
    cu = cu_of(LENGTHS)
    cuc = oracle.compress_cu_seqlens(cu, R)
    T, tc = int(cu[-1]), int(cuc[-1])
    vis = dense_ref.visible_mask(LENGTHS, R)
    idx = -np.ones((T, topk), dtype=np.int32)
    a = rng.uniform(0.05, 1.0, size=(T, topk)) * 0.8
    for t in range(T):
        cand = np.flatnonzero(vis[t])
        rng.shuffle(cand)
        m = min(topk - 1, len(cand))
        idx[t, :m] = cand[:m]
    # entries the rule must skip: a block of the token's segment that is not
    # complete yet, a row out of range, a row of another segment
    seg1_first = int(cu[2])                 # third segment, first token
    idx[seg1_first, -1] = int(cuc[2]) + 1   # not visible yet
    idx[seg1_first + 9, -1] = tc + 3        # out of range
    idx[int(cu[3]) + 8, -1] = int(cuc[0])   # first segment's block, other segment
    # a token whose listed entries all carry zero mass
    zero_tok = int(cu[2]) + 20
    a[zero_tok, :] = 0.0
    q = rng.standard_normal((T, HI, DI))
    k = rng.standard_normal((tc, DI))
    w = np.zeros((T, HI)) if w_zero else rng.standard_normal((T, HI))
    return dict(cu=cu, cuc=cuc, T=T, tc=tc, idx=idx, a=a, q=q, k=k, w=w, vis=vis,
                zero_tok=zero_tok)


def run(c, q=None, k=None, w=None, a=None, idx=None, tokens=None, scale=GRAD_SCALE):
    sel = slice(None) if tokens is None else np.asarray(tokens)
    return oracle.indexer_kl_loss_grad((c["q"] if q is None else q)[sel], c["k"] if k is None else k,
                                       (c["w"] if w is None else w)[sel],
                                       (c["idx"] if idx is None else idx)[sel],
                                       (c["a"] if a is None else a)[sel], c["T"], c["cu"],
                                       c["cuc"], R, scale, tokens=tokens)


def entry_set(c, t):
    """Entries of token t that name a visible row, from the dense mask."""
    return [s for s, j in enumerate(c["idx"][t]) if 0 <= j < c["tc"] and c["vis"][t, j]]


def test_loss_is_library_kl_of_dense_scores():
    c = make_case(1)
    res = run(c)
    scores = dense_ref.indexer_scores(c["q"], c["k"], c["w"])
    n_checked = 0
    for t in range(c["T"]):
        S = entry_set(c, t)
        if not S or c["a"][t, S].sum() == 0:
            assert res["loss"][t] == 0.0
            continue
        I = scores[t, c["idx"][t, S]]
        want = stats.entropy(c["a"][t, S], special.softmax(I))
        assert res["loss"][t] == pytest.approx(want, rel=1e-10, abs=1e-12), t
        n_checked += 1
    assert n_checked > 20
    # the skipped entries really were in the lists
    assert (c["idx"] >= c["tc"]).any() and res["loss"][c["zero_tok"]] == 0.0


def _fd(c, name, pos, eps=1e-6):
    def total(x):
        return GRAD_SCALE * run(c, **{name: x})["loss"].sum()
    x = c[name].copy()
    x[pos] += eps
    up = total(x)
    x[pos] -= 2 * eps
    down = total(x)
    return (up - down) / (2 * eps)


@pytest.mark.parametrize("seed", [2, 3])
def test_gradients_match_finite_differences(seed):
    c = make_case(seed)
    # no dot product sits on the ReLU's kink
    dots = np.einsum("thd,jd->thj", c["q"], c["k"])
    assert np.abs(dots).min() > 1e-4
    res = run(c)
    rng = np.random.default_rng(seed)
    for name, grad in (("q", res["d_q"]), ("w", res["d_w"]), ("k", res["d_k"])):
        flat = np.argwhere(np.ones(grad.shape, bool))
        picks = flat[rng.choice(len(flat), size=min(60, len(flat)), replace=False)]
        # include the largest-magnitude elements too
        big = np.unravel_index(np.argsort(np.abs(grad), axis=None)[-10:], grad.shape)
        picks = list(map(tuple, picks)) + list(zip(*big))
        for pos in picks:
            want = _fd(c, name, tuple(int(i) for i in pos))
            assert grad[pos] == pytest.approx(want, rel=1e-5, abs=1e-7), (name, pos)
    assert np.abs(res["d_q"]).max() > 1e-3 and np.abs(res["d_k"]).max() > 1e-3


def test_target_equal_to_indexer_softmax_gives_zero():
    c = make_case(4)
    scores = dense_ref.indexer_scores(c["q"], c["k"], c["w"])
    a = np.zeros_like(c["a"])
    for t in range(c["T"]):
        S = entry_set(c, t)
        if S:
            # any positive multiple: the target is L1-normalised over S
            a[t, S] = 2.5 * special.softmax(scores[t, c["idx"][t, S]])
    res = run(c, a=a)
    assert np.abs(res["loss"]).max() < 1e-12
    for g in ("d_q", "d_w", "d_k"):
        assert np.abs(res[g]).max() < 1e-12, g


def test_zero_weights_uniform_closed_form():
    c = make_case(5, w_zero=True)
    res = run(c)
    dots = np.einsum("thd,jd->thj", c["q"], c["k"])
    assert np.abs(res["d_q"]).max() == 0.0 and np.abs(res["d_k"]).max() == 0.0
    for t in range(c["T"]):
        S = entry_set(c, t)
        if not S or c["a"][t, S].sum() == 0:
            continue
        p = c["a"][t, S] / c["a"][t, S].sum()
        n = len(S)
        assert res["loss"][t] == pytest.approx(np.log(n) - stats.entropy(p), abs=1e-12)
        rows = c["idx"][t, S]
        want = GRAD_SCALE * ((1.0 / n - p)[None, :] * np.maximum(dots[t][:, rows], 0)).sum(1)
        np.testing.assert_allclose(res["d_w"][t], want, rtol=1e-12, atol=1e-14)


def test_single_entry_is_zero():
    c = make_case(6, topk=1)
    res = run(c)
    assert np.abs(res["loss"]).max() < 1e-15
    assert np.abs(res["d_q"]).max() < 1e-15 and np.abs(res["d_k"]).max() < 1e-15


def test_invariances():
    c = make_case(7)
    base = run(c)
    rng = np.random.default_rng(7)
    perm = np.stack([rng.permutation(TOPK) for _ in range(c["T"])])
    idx_p = np.take_along_axis(c["idx"], perm, axis=1)
    a_p = np.take_along_axis(c["a"], perm, axis=1)
    # scale each token's targets by its own factor: L1 normalisation undoes it
    a_p = a_p * rng.uniform(0.1, 10.0, size=(c["T"], 1))
    res = run(c, a=a_p, idx=idx_p)
    for key in ("loss", "d_q", "d_w", "d_k"):
        np.testing.assert_allclose(res[key], base[key], rtol=1e-11, atol=1e-13, err_msg=key)
    # token by token: per-token outputs unchanged, and d_k is their sum
    dk = np.zeros_like(base["d_k"])
    for t in range(c["T"]):
        one = run(c, tokens=[t])
        np.testing.assert_allclose(one["d_q"][0], base["d_q"][t], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(one["d_w"][0], base["d_w"][t], rtol=1e-12, atol=1e-15)
        assert one["loss"][0] == pytest.approx(base["loss"][t], rel=1e-12, abs=1e-15)
        dk += one["d_k"]
    np.testing.assert_allclose(dk, base["d_k"], rtol=1e-11, atol=1e-13)
    # gradients are linear in grad_scale, the loss is not scaled
    res2 = run(c, scale=2 * GRAD_SCALE)
    np.testing.assert_allclose(res2["d_q"], 2 * base["d_q"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(res2["loss"], base["loss"], rtol=1e-12, atol=1e-15)


def test_score_gradient_output():
    """g = dL/dI per entry: it sums to zero over a token's entries (softmax
    minus a normalised target), vanishes on skipped entries, and gives back
    the finite-difference-pinned d_w through sum_s g_s relu(q . k)."""
    c = make_case(8)
    res = run(c)
    g = res["g"]
    dots = np.einsum("thd,jd->thj", c["q"], c["k"])
    for t in range(c["T"]):
        S = entry_set(c, t)
        skipped = [s for s in range(TOPK) if s not in S]
        assert (g[t, skipped] == 0).all()
        if not S:
            continue
        assert abs(g[t].sum()) < 1e-12
        rows = c["idx"][t, S]
        want = (g[t, S][None, :] * np.maximum(dots[t][:, rows], 0)).sum(1)
        np.testing.assert_allclose(res["d_w"][t], want, rtol=1e-12, atol=1e-14)
    assert np.abs(g).max() > 0.01
