"""Dense brute-force restatement of the CSA forward path (NumPy, fp64).

TEST INFRASTRUCTURE ONLY, tiny packs only. It is written independently of
``csa_oracle.c`` and pins it: instead of per-token key lists it builds the
full boolean mask over every (token, key) pair of the pack, with the
visibility rules phrased from the other side (which rows a block pools,
which rows lie inside a window), then runs ordinary dense masked softmax
with an extra sink column.

Sources, as for the C oracle: miles PR 2038 report (THD helpers, compressor
grouping, tail rule), hyper-parallel RFC sections 1-2 (lightning_indexer and
sparse_flash_mla schemas), Megatron-LM PR 7 (verl) environment note
(head_dim = d_v = 512, shared K/V row).
"""

from __future__ import annotations

import numpy as np


def segment_ids(lengths):
    return np.repeat(np.arange(len(lengths)), np.asarray(lengths, dtype=np.int64))


def compressed_layout(lengths, r):
    """Per compressed row: its segment and the packed rows it pools.

    A segment of length L pools its leading full groups of r rows, one group
    per compressed row; the trailing L % r rows form no group."""
    lengths = np.asarray(lengths, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    seg, first, last = [], [], []
    for b, (s, L) in enumerate(zip(starts, lengths)):
        for g in range(L // r):
            seg.append(b)
            first.append(s + g * r)
            last.append(s + g * r + r - 1)
    return (np.asarray(seg, dtype=np.int64), np.asarray(first, dtype=np.int64),
            np.asarray(last, dtype=np.int64))


def window_mask(lengths, W):
    """[T, T] bool: packed row s is in token t's window."""
    seg = segment_ids(lengths)
    t = np.arange(len(seg))[:, None]
    s = np.arange(len(seg))[None, :]
    return (seg[:, None] == seg[None, :]) & (s <= t) & (t - s < W)


def visible_mask(lengths, r):
    """[T, Tc] bool: compressed row j is complete and in token t's segment."""
    seg = segment_ids(lengths)
    cseg, _, last = compressed_layout(lengths, r)
    t = np.arange(len(seg))[:, None]
    return (seg[:, None] == cseg[None, :]) & (last[None, :] <= t)


def indexer_scores(q_idx, k_idx, w):
    """[T, Tc] = sum_h w[t,h] * relu(q_idx[t,h] . k_idx[j]) for every pair."""
    dots = np.einsum("thd,jd->thj", q_idx, k_idx)
    return np.einsum("th,thj->tj", w, np.maximum(dots, 0.0))


def topk_dense(scores, visible, k):
    """Per token: k best visible blocks (ties to the lower index), ascending, -1 pad."""
    T, Tc = scores.shape
    out = -np.ones((T, k), dtype=np.int64)
    for t in range(T):
        cand = [(-scores[t, j], j) for j in range(Tc) if visible[t, j]]
        cand.sort()
        chosen = sorted(j for _, j in cand[:k])
        out[t, : len(chosen)] = chosen
    return out


def attention_dense(q, ori_kv, cmp_kv, lengths, W, r, selected, sinks, scale, return_probs=False):
    """Dense masked attention with a sink column.

    ``selected`` is a [T, Tc] bool mask of the compressed rows each token
    attends (may be None when there are no compressed rows). With
    ``return_probs`` the attention weights come back too, [T, H, T + Tc + 1]:
    original rows, then compressed rows, then the sink column."""
    T, H, D = q.shape
    kv = ori_kv if cmp_kv is None else np.concatenate([ori_kv, cmp_kv], axis=0)
    mask = window_mask(lengths, W)
    if cmp_kv is not None:
        mask = np.concatenate([mask, selected], axis=1)
    logits = scale * np.einsum("thd,kd->thk", q, kv)
    logits = np.where(mask[:, None, :], logits, -np.inf)
    sink_col = np.broadcast_to((np.full(H, -np.inf) if sinks is None else sinks)[None, :, None],
                               (T, H, 1))
    full = np.concatenate([logits, sink_col], axis=2)
    mx = full.max(axis=2, keepdims=True)
    e = np.exp(full - mx)
    z = e.sum(axis=2, keepdims=True)
    p = e / z
    out = np.einsum("thk,kd->thd", p[:, :, :-1], kv)
    lse = (mx + np.log(z))[:, :, 0]
    if return_probs:
        return out, lse, p
    return out, lse
