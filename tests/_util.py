"""Shared helpers for the GPU parity tests: seeded packs, oracle calls on the
same bits, and the comparison rules.

Comparison rules
* integer outputs (compressed cu_seqlens, window rows): bit-exact;
* top-k rows: identical, except where the oracle's topk-th and (topk+1)-th
  scores are within 1e-3 relative of each other; then every row in the
  symmetric difference must score within that band of the boundary;
* attention output (bf16): max |gpu - oracle| <= 2e-2 and mean <= 2e-3;
  LSE (fp32): max |gpu - oracle| <= 1e-3. Where a top-k row differed by a
  near-tie, the oracle attention is fed the GPU's indices for that token.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from csa_inputs import packs

# Lines for the terminal summary (tests/conftest.py): per-layer errors at full size.
REPORT = []

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3
TIE_REL = 1e-3
VAL_RTOL, VAL_ATOL = 1e-4, 2e-3


def cu_of(lengths):
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def custom_spec(lengths, heads=8, win_left=15, layers=None, seed=11, w_uniform=False):
    if layers is None:
        layers = (packs.LayerSpec(cmp_ratio=4, indexer=True, topk=16, index_heads=8,
                                  index_dim=64),)
    return packs.PackSpec("custom", tuple(int(x) for x in lengths), heads=heads, dim=512,
                          win_left=win_left, layers=tuple(layers), seed=seed, w_uniform=w_uniform)


class LayerCase:
    """One layer of a pack: CPU tensors (with cmp rows trimmed to the pack's
    compressed count from the oracle) and their CUDA copies."""

    def __init__(self, spec, layer, tensors, device="cuda"):
        self.spec, self.layer = spec, layer
        self.cu = cu_of(spec.lengths)
        self.cuc = oracle.compress_cu_seqlens(self.cu, layer.cmp_ratio)
        self.T, self.Tc = int(self.cu[-1]), int(self.cuc[-1])
        self.t = dict(tensors)
        self.t["cmp_kv"] = self.t["cmp_kv"][: self.Tc].contiguous()
        if layer.indexer:
            self.t["k_idx"] = self.t["k_idx"][: self.Tc].contiguous()
        self.device = device
        self.d = {k: v.to(device) for k, v in self.t.items()} if device else None
        self.cu_d = torch.from_numpy(self.cu).to(device) if device else None


def layer_cases(spec, device="cuda"):
    return [LayerCase(spec, layer, tens, device)
            for layer, tens in zip(spec.layers, packs.draw_pack(spec))]


def sample_tokens(lengths, r, n_random=16, seed=0, cap=64):
    """Boundary tokens of every segment (first, first with a complete block,
    last) plus random ones, capped."""
    cu = cu_of(lengths)
    picks = []
    for b in range(len(lengths)):
        s, e = int(cu[b]), int(cu[b + 1])
        if e > s:
            picks += [s, min(e - 1, s + r - 1), e - 1, min(e - 1, s + 130)]
    rng = np.random.default_rng(seed)
    picks += rng.integers(0, int(cu[-1]), size=n_random).tolist()
    picks = sorted(set(picks))
    if len(picks) > cap:
        keep = rng.choice(len(picks), size=cap, replace=False)
        picks = sorted(picks[i] for i in keep)
    return np.asarray(picks, dtype=np.int32)


def oracle_topk(case, tokens=None):
    t = case.t
    qi = t["q_idx"] if tokens is None else t["q_idx"][torch.from_numpy(tokens).long()]
    w = t["w"] if tokens is None else t["w"][torch.from_numpy(tokens).long()]
    return oracle.indexer_topk(qi, t["k_idx"], w, case.T, case.cu, case.cuc,
                               case.layer.cmp_ratio, case.layer.topk, tokens=tokens)


def oracle_all_scores(case, token):
    """Every visible row's oracle score for one token (topk = n_vis)."""
    tok = np.asarray([token], dtype=np.int32)
    _, _, _, _, nvis = oracle_topk(case, tok)
    n = int(nvis[0])
    if n == 0:
        return {}
    t = case.t
    idx, val, *_ = oracle.indexer_topk(t["q_idx"][token:token + 1], t["k_idx"],
                                       t["w"][token:token + 1], case.T, case.cu, case.cuc,
                                       case.layer.cmp_ratio, n, tokens=tok)
    return {int(j): float(v) for j, v in zip(idx[0], val[0]) if j >= 0}


def check_topk(case, gpu_idx, ref, tokens=None, gpu_val=None):
    """Apply the top-k rule; returns the list of rows that differed by a
    near-tie (allowed)."""
    idx, val, kth, nxt, nvis = ref
    tok = np.arange(gpu_idx.shape[0]) if tokens is None else tokens
    allowed = []
    for i, t in enumerate(tok):
        g, r = gpu_idx[i], idx[i]
        if np.array_equal(g, r):
            continue
        a, b = kth[i], nxt[i]
        band = TIE_REL * max(abs(a), abs(b))
        assert not (math.isnan(a) or math.isnan(b)), f"token {t}: set differs without a k+1-th"
        assert abs(a - b) < band, f"token {t}: set differs but kth={a} next={b}"
        scores = oracle_all_scores(case, int(t))
        diff = set(g[g >= 0].tolist()) ^ set(r[r >= 0].tolist())
        for j in diff:
            assert j in scores, f"token {t}: row {j} not visible"
            assert abs(scores[j] - a) <= band, f"token {t}: row {j} far from the boundary"
        gs = g[g >= 0]
        assert len(gs) == len(r[r >= 0]) and np.all(np.diff(gs) > 0)
        allowed.append(i)
    if gpu_val is not None:
        same = [i for i in range(len(tok)) if i not in allowed]
        np.testing.assert_allclose(gpu_val[same], val[same], rtol=VAL_RTOL, atol=VAL_ATOL)
    return allowed


def check_attention(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = out_gpu.float().cpu().double().numpy() if torch.is_tensor(out_gpu) else out_gpu
    err = np.abs(o - out_ref)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert err.max() <= OUT_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    if lse_gpu is not None:
        l = lse_gpu.cpu().double().numpy() if torch.is_tensor(lse_gpu) else lse_gpu
        lerr = np.abs(l - lse_ref)
        assert lerr.max() <= LSE_MAX_ABS, f"{what}: lse max abs err {lerr.max():.3e}"
    return float(err.max()), float(err.mean())


def oracle_attention(case, idx_rows, tokens=None):
    """Oracle attention for the listed tokens (idx_rows per listed token, or
    None for compressor-only layers)."""
    t = case.t
    q = t["q"] if tokens is None else t["q"][torch.from_numpy(tokens).long()]
    return oracle.sparse_mla_fwd(q, t["ori_kv"], t["cmp_kv"], idx_rows, case.cu, case.cuc,
                                 case.T, t["sinks"], case.spec.scale, case.layer.cmp_ratio,
                                 case.spec.win_left, tokens=tokens)


def indices_for_oracle(case, gpu_idx_np, tokens=None):
    """Oracle top-k rows, replaced by the GPU's rows where they differ by a
    near-tie (the attention is then compared with the GPU's rows)."""
    ref = oracle_topk(case, tokens)
    sel = gpu_idx_np if tokens is None else gpu_idx_np[tokens]
    allowed = check_topk(case, sel, ref, tokens=tokens)
    rows = ref[0].copy()
    for i in allowed:
        rows[i] = sel[i]
    return rows
