"""Pins for the oracle's shared-KV MLA sparse attention with sinks.

The C oracle is checked against: the independent dense NumPy oracle, a
library softmax-attention routine (sink of -inf), a closed form for the
single-key case, the normalisation identity, and invariances (segment
isolation, head independence, key-order independence, window and causal
boundaries).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from csa_inputs import packs
from oracle import dense_ref


def cu_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def small_case(seed, lengths, H=4, D=32, r=4, with_sinks=True):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    cu = cu_of(lengths)
    cuc = oracle.compress_cu_seqlens(cu, r)
    tc = int(cuc[-1])
    q = rng.standard_normal((T, H, D))
    okv = rng.standard_normal((T, D))
    ckv = rng.standard_normal((tc, D))
    sinks = rng.standard_normal(H) if with_sinks else None
    return dict(q=q, okv=okv, ckv=ckv, sinks=sinks, cu=cu, cuc=cuc, T=T, r=r)


def run(c, W, idx=None, tokens=None, sinks="default", scale=None, q=None, okv=None, ckv=None):
    qq = c["q"] if q is None else q
    if tokens is not None:
        qq = qq[tokens]
        if idx is not None:
            idx = idx[tokens]
    sk = c["sinks"] if isinstance(sinks, str) else sinks
    D = c["q"].shape[2]
    return oracle.sparse_mla_fwd(
        qq, c["okv"] if okv is None else okv, c["ckv"] if ckv is None else ckv, idx, c["cu"],
        c["cuc"], c["T"], sk, 1.0 / math.sqrt(D) if scale is None else scale, c["r"], W - 1,
        tokens=tokens)


def test_matches_dense_oracle_all_visible():
    lengths = [1, 3, 37, 60, 19]
    c = small_case(0, lengths)
    W = 16
    out, lse = run(c, W)  # compressor-only: every visible block
    sel = dense_ref.visible_mask(lengths, c["r"])
    out_d, lse_d = dense_ref.attention_dense(c["q"], c["okv"], c["ckv"], lengths, W, c["r"], sel,
                                             c["sinks"], 1.0 / math.sqrt(32))
    np.testing.assert_allclose(out, out_d, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_d, rtol=1e-11, atol=1e-12)


def test_matches_dense_oracle_tiny_pack_with_topk():
    spec = packs.pack_spec("tiny")
    t = packs.draw_pack(spec)[0]
    lengths = list(spec.lengths)
    cu = cu_of(lengths)
    cuc = oracle.compress_cu_seqlens(cu, 4)
    tc = int(cuc[-1])
    K, W = 8, 16
    idx, *_ = oracle.indexer_topk(t["q_idx"], t["k_idx"][:tc], t["w"], 256, cu, cuc, 4, K)
    q = t["q"].double().numpy()
    okv = t["ori_kv"].double().numpy()
    ckv = t["cmp_kv"][:tc].double().numpy()
    sinks = t["sinks"].double().numpy()
    out, lse = oracle.sparse_mla_fwd(q, okv, ckv, idx, cu, cuc, 256, sinks, spec.scale, 4, W - 1)
    sel = np.zeros((256, tc), dtype=bool)
    for tt in range(256):
        for j in idx[tt]:
            if j >= 0:
                sel[tt, j] = True
    out_d, lse_d = dense_ref.attention_dense(q, okv, ckv, lengths, W, 4, sel, sinks, spec.scale)
    np.testing.assert_allclose(out, out_d, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_d, rtol=1e-11, atol=1e-12)
    # with topk covering every visible block the indexer choice drops out
    idx_all, *_ = oracle.indexer_topk(t["q_idx"], t["k_idx"][:tc], t["w"], 256, cu, cuc, 4, 29)
    out_a, _ = oracle.sparse_mla_fwd(q, okv, ckv, idx_all, cu, cuc, 256, sinks, spec.scale, 4, W - 1)
    out_h, _ = oracle.sparse_mla_fwd(q, okv, ckv, None, cu, cuc, 256, sinks, spec.scale, 4, W - 1)
    np.testing.assert_array_equal(out_a, out_h)


@pytest.mark.parametrize("sink", [None, -np.inf])
def test_no_sink_is_library_softmax_attention(sink):
    lengths = [23, 50]
    c = small_case(1, lengths, H=3, D=16)
    W = 8
    sinks = None if sink is None else np.full(3, sink)
    out, lse = run(c, W, sinks=sinks)
    mask = np.concatenate([dense_ref.window_mask(lengths, W),
                           dense_ref.visible_mask(lengths, c["r"])], axis=1)
    kv = torch.from_numpy(np.concatenate([c["okv"], c["ckv"]], axis=0))
    q = torch.from_numpy(c["q"]).transpose(0, 1)  # [H, T, D]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, kv[None].expand(3, -1, -1), kv[None].expand(3, -1, -1),
        attn_mask=torch.from_numpy(mask)[None].expand(3, -1, -1), scale=1.0 / 4.0)
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)
    logits = (q @ kv.T * 0.25).masked_fill(~torch.from_numpy(mask)[None], -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(logits, -1).T.numpy(), rtol=1e-12)


def test_single_key_closed_form():
    # the first token of a segment sees only its own row (no compressed block is complete)
    lengths = [5, 9, 6]
    c = small_case(2, lengths, H=4, D=16)
    for scale in (0.25, 0.7):
        out, lse = run(c, 16, scale=scale)
        for t in (0, 5, 14):
            v = c["okv"][t]
            for h in range(4):
                l = scale * float(c["q"][t, h] @ v)
                s = c["sinks"][h]  # the sink logit is not scaled
                np.testing.assert_allclose(out[t, h], v / (1.0 + math.exp(s - l)), rtol=1e-13)
                assert lse[t, h] == pytest.approx(math.log(math.exp(l) + math.exp(s)), rel=1e-13)


def test_probability_identity_with_one_hot_rows():
    # with distinct one-hot value rows, out[d] is the probability of the key placed at d,
    # so sum_d out + exp(sink - lse) = 1
    lengths = [40, 24]
    T, D, r = 64, 128, 4
    c = small_case(3, lengths, H=2, D=D, r=r)
    okv = np.eye(D)[:T]
    ckv = np.eye(D)[T:T + c["ckv"].shape[0]]
    out, lse = run(c, 16, okv=okv, ckv=ckv)
    total = out.sum(axis=2) + np.exp(c["sinks"][None, :] - lse)
    np.testing.assert_allclose(total, 1.0, rtol=0, atol=1e-13)
    assert (out >= 0).all()


def test_segment_isolation():
    lengths = [30, 45, 21]
    c = small_case(4, lengths)
    out, lse = run(c, 16)
    c2 = dict(c)
    rng = np.random.default_rng(99)
    q2, okv2, ckv2 = c["q"].copy(), c["okv"].copy(), c["ckv"].copy()
    q2[:30] = rng.standard_normal(q2[:30].shape)
    okv2[75:] = rng.standard_normal(okv2[75:].shape)
    ckv2[:7] = rng.standard_normal(ckv2[:7].shape)  # segment 0 blocks
    ckv2[18:] = rng.standard_normal(ckv2[18:].shape)  # segment 2 blocks
    out2, lse2 = run(c2, 16, q=q2, okv=okv2, ckv=ckv2)
    np.testing.assert_array_equal(out2[30:75], out[30:75])
    np.testing.assert_array_equal(lse2[30:75], lse[30:75])
    assert not np.allclose(out2[:30], out[:30])


def test_head_independence():
    lengths = [33, 17]
    c = small_case(5, lengths, H=5)
    out, lse = run(c, 8)
    perm = np.array([3, 0, 4, 1, 2])
    out_p, lse_p = run(c, 8, q=c["q"][:, perm], sinks=c["sinks"][perm])
    np.testing.assert_array_equal(out_p, out[:, perm])
    np.testing.assert_array_equal(lse_p, lse[:, perm])


def test_index_order_and_invalid_entries():
    lengths = [64, 40]
    c = small_case(6, lengths)
    T = c["T"]
    rng = np.random.default_rng(6)
    vis = dense_ref.visible_mask(lengths, c["r"])
    K = 6
    idx = -np.ones((T, K), dtype=np.int32)
    for t in range(T):
        cand = np.nonzero(vis[t])[0]
        pick = rng.choice(cand, size=min(4, len(cand)), replace=False) if len(cand) else []
        idx[t, : len(pick)] = np.sort(pick)
    out, lse = run(c, 16, idx=idx)
    shuffled = idx.copy()
    for t in range(T):
        rng.shuffle(shuffled[t])
    out_s, lse_s = run(c, 16, idx=shuffled)
    np.testing.assert_allclose(out_s, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_s, lse, rtol=1e-13)
    # entries out of range or not visible are skipped like -1
    bad = idx.copy()
    tc = c["ckv"].shape[0]
    for t in range(T):
        invis = np.nonzero(~vis[t])[0]
        bad[t, 4] = tc + 5
        bad[t, 5] = invis[0] if len(invis) else -7
    out_b, lse_b = run(c, 16, idx=bad)
    np.testing.assert_array_equal(out_b, out)
    np.testing.assert_array_equal(lse_b, lse)


def test_window_and_causal_boundaries():
    lengths = [70]
    c = small_case(7, lengths, r=4)
    W, t = 16, 50
    out, _ = run(c, W)
    rng = np.random.default_rng(1)
    # row t-W is outside the window: no effect; row t-W+1 is inside: effect
    okv = c["okv"].copy()
    okv[t - W] = rng.standard_normal(okv.shape[1])
    assert np.array_equal(run(c, W, okv=okv)[0][t], out[t])
    okv = c["okv"].copy()
    okv[t - W + 1] = rng.standard_normal(okv.shape[1])
    assert not np.allclose(run(c, W, okv=okv)[0][t], out[t])
    # block 12 pools rows 48..51: complete at token 51, not at token 50
    ckv = c["ckv"].copy()
    ckv[12] = rng.standard_normal(ckv.shape[1])
    out2, _ = run(c, W, ckv=ckv)
    assert np.array_equal(out2[50], out[50])
    assert not np.allclose(out2[51], out[51])


def test_token_list_matches_full_run():
    c = small_case(8, [50, 50])
    out, lse = run(c, 16)
    toks = np.array([99, 0, 50, 13])
    out2, lse2 = run(c, 16, tokens=toks)
    np.testing.assert_array_equal(out2, out[toks])
    np.testing.assert_array_equal(lse2, lse[toks])
