"""Pins for the oracle's backward of the shared-KV MLA attention with sinks.

The gradients are checked against central finite differences of
sum(dout * out) computed with the oracle's own forward (which the forward
pins tie to the pages), element by element, in both compressed modes (top-k
list, every visible block) and with and without sinks. The head-averaged
attention distributions are checked against the independent dense NumPy
oracle's weights and against the identity that a token's weights over its
keys and the sink sum to one.
"""

import numpy as np
import pytest

import oracle
from oracle import dense_ref


def cu_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


LENGTHS = [9, 11, 6]
H, D, R, WIN_LEFT, SCALE = 3, 8, 4, 4, 0.37


def make_case(seed, with_sinks, topk):
    rng = np.random.default_rng(seed)
    cu = cu_of(LENGTHS)
    cuc = oracle.compress_cu_seqlens(cu, R)
    T, tc = int(cu[-1]), int(cuc[-1])
    c = dict(cu=cu, cuc=cuc, T=T, tc=tc,
             q=rng.standard_normal((T, H, D)), okv=rng.standard_normal((T, D)),
             ckv=rng.standard_normal((tc, D)), g=rng.standard_normal((T, H, D)),
             sinks=rng.standard_normal(H) if with_sinks else None, idx=None)
    if topk:
        # per token: up to `topk` distinct visible blocks in a random order,
        # then -1; one token also lists a block that is not visible yet
        vis = dense_ref.visible_mask(LENGTHS, R)
        idx = -np.ones((T, topk), dtype=np.int32)
        for t in range(T):
            cand = np.flatnonzero(vis[t])
            rng.shuffle(cand)
            idx[t, : min(topk, len(cand))] = cand[:topk]
        late = int(cu[1]) + 1  # second segment, before its first block is complete
        idx[late, -1] = int(cuc[1]) + 1
        c["idx"] = idx
    return c


def loss(c, q=None, okv=None, ckv=None, sinks="c"):
    out, _ = oracle.sparse_mla_fwd(c["q"] if q is None else q, c["okv"] if okv is None else okv,
                                   c["ckv"] if ckv is None else ckv, c["idx"], c["cu"], c["cuc"],
                                   c["T"], c["sinks"] if isinstance(sinks, str) else sinks,
                                   SCALE, R, WIN_LEFT)
    return float(np.sum(out * c["g"]))


def fd(c, name, eps=1e-5):
    base = c[name]
    grad = np.zeros_like(base)
    flat = grad.reshape(-1)
    for i in range(base.size):
        p = base.copy().reshape(-1)
        p[i] += eps
        lp = loss(c, **{name: p.reshape(base.shape)})
        p[i] -= 2 * eps
        lm = loss(c, **{name: p.reshape(base.shape)})
        flat[i] = (lp - lm) / (2 * eps)
    return grad


def bwd(c):
    return oracle.sparse_mla_bwd(c["q"], c["g"], c["okv"], c["ckv"], c["idx"], c["cu"], c["cuc"],
                                 c["sinks"], SCALE, R, WIN_LEFT)


@pytest.mark.parametrize("topk", [0, 2])
@pytest.mark.parametrize("with_sinks", [True, False])
def test_gradients_match_finite_differences(topk, with_sinks):
    c = make_case(11 + topk + with_sinks, with_sinks, topk)
    res = bwd(c)
    pairs = [("q", "d_q"), ("okv", "d_ori_kv"), ("ckv", "d_cmp_kv")]
    if with_sinks:
        pairs.append(("sinks", "d_sinks"))
    for name, key in pairs:
        ref = fd(c, name)
        got = res[key]
        scale = max(1.0, float(np.abs(ref).max()))
        assert np.abs(got - ref).max() <= 1e-6 * scale, (name, np.abs(got - ref).max())
        assert np.abs(ref).max() > 1e-3, f"{name}: gradient vanished, the check proves nothing"
    if not with_sinks:
        assert res["d_sinks"] is None


def test_distributions_match_dense_weights_and_sum_to_one():
    c = make_case(5, True, 2)
    res = bwd(c)
    T, tc, W = c["T"], c["tc"], WIN_LEFT + 1
    selected = np.zeros((T, tc), dtype=bool)
    vis = dense_ref.visible_mask(LENGTHS, R)
    for t in range(T):
        for j in c["idx"][t]:
            if 0 <= j < tc and vis[t, j]:
                selected[t, j] = True
    _, lse, p = dense_ref.attention_dense(c["q"], c["okv"], c["ckv"], LENGTHS, W, R, selected,
                                          c["sinks"], SCALE, return_probs=True)
    pm = p.mean(axis=1)  # [T, T + Tc + 1], head average
    for t in range(T):
        start = max(t - W + 1, int(c["cu"][np.searchsorted(c["cu"], t, side="right") - 1]))
        for i in range(W):
            want = pm[t, start + i] if start + i <= t else 0.0
            assert abs(res["ori_l1"][t, i] - want) < 1e-12
        for s, j in enumerate(c["idx"][t]):
            want = pm[t, T + j] if (0 <= j < tc and vis[t, j]) else 0.0
            assert abs(res["cmp_l1"][t, s] - want) < 1e-12
    sink_mean = np.exp(c["sinks"][None, :] - lse).mean(axis=1)
    total = res["ori_l1"].sum(axis=1) + res["cmp_l1"].sum(axis=1) + sink_mean
    assert np.abs(total - 1.0).max() < 1e-12
