"""GPU parity of the indexer KL-loss gradient (csa_indexer_kl_loss_grad)
against the oracle's fp64 version, element by element, on ragged packs that
span several 32-row chunks, with lists from the oracle's top-k (including
-1 padding and entries the rule must skip), targets from the oracle's
attention backward or seeded draws, and at the mixed 32k pack's full size on
sampled tokens plus an identity over every token.

Tolerances: the kernel works in fp32 from bf16 inputs; each gradient is held
to 1e-2 of its largest magnitude in max-abs and 1e-3 in mean-abs, the
per-token loss to 1e-4 relative + 1e-3 absolute. One decision is not fixed
by the inputs at fp32: the ReLU's derivative where a dot product lies within
fp32 rounding of zero. Where the fp64 dot of a listed (token, head, row) is
below 1e-3 in magnitude, the elements it feeds may differ by up to that
entry's contribution (the oracle's dL/dI for the entry times the other
factors, with a 1 % margin), and that allowance is added to their bound. A separate case uses quarter-integer
inputs, whose dot products are exact in fp32, so no decision is ambiguous.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import cu_of, layer_cases, oracle_topk, sample_tokens

pytestmark = pytest.mark.gpu

GRAD_MAX, GRAD_MEAN = 1e-2, 1e-3
LOSS_RTOL, LOSS_ATOL = 1e-4, 1e-3
AMBIG = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def run_gpu_raw(q, k, w, idx, l1, cu, r, grad_scale):
    """CPU tensors / arrays in; CUDA tensors out."""
    dev = "cuda"
    cu_d = torch.from_numpy(np.asarray(cu, dtype=np.int32)).to(dev)
    cuc = csa.csa_compress_cu_seqlens(cu_d, r)
    res = csa.csa_indexer_kl_loss_grad(
        q.to(dev), None if k is None or k.shape[0] == 0 else k.to(dev), w.to(dev),
        torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(dev),
        torch.from_numpy(np.ascontiguousarray(l1, dtype=np.float32)).to(dev), cu_d, cuc, r,
        grad_scale)
    torch.cuda.synchronize()
    return res


def run_gpu(q, k, w, idx, l1, cu, r, grad_scale):
    """CPU tensors / arrays in; numpy dict (fp64) out."""
    res = run_gpu_raw(q, k, w, idx, l1, cu, r, grad_scale)
    return {key: (None if v is None else v.double().cpu().numpy()) for key, v in res.items()}


def allowances(q, k, w, idx, g, tokens=None, want_dk=True):
    """Per-element allowance for ReLU decisions within fp32 rounding of zero.

    ``g`` is the oracle's dL/dI per entry of the listed tokens; a flipped
    decision on entry (t, h, s) moves d_q[t,h,:] by g_s w[t,h] k[j_s,:] and
    d_k[j_s,:] by g_s w[t,h] q[t,h,:] (1 % margin for g's own fp32 error)."""
    if tokens is not None:
        sel = torch.from_numpy(np.asarray(tokens)).long()
        q, w, idx = q[sel], w[sel], idx[np.asarray(tokens)]
    qs = q.double()
    kk = k.double()
    ws = w.double()
    rows = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int64))
    ok = (rows >= 0) & (rows < kk.shape[0])
    kr = kk[torch.where(ok, rows, 0)]                        # [n, topk, Di]
    dots = torch.bmm(qs, kr.transpose(1, 2))                # [n, Hi, topk]
    amb = (dots.abs() < AMBIG) & ok[:, None, :]
    gg = torch.from_numpy(np.asarray(g, dtype=np.float64))
    coef = torch.where(amb, 1.01 * gg.abs()[:, None, :] * ws.abs()[:, :, None], 0.0)
    allow_dq = torch.bmm(coef, kr.abs()).numpy()            # [n, Hi, Di]
    allow_dk = None
    if want_dk:
        acc = torch.zeros(kk.shape, dtype=torch.float64)
        n_i, h_i, s_i = torch.nonzero(amb, as_tuple=True)
        if len(n_i):
            acc.index_add_(0, rows[n_i, s_i], coef[n_i, h_i, s_i][:, None] * qs[n_i, h_i].abs())
        allow_dk = acc.numpy()
    return allow_dq, allow_dk, int(amb.sum())


def check_grad(got, ref, allow, what):
    assert np.isfinite(got).all(), f"{what}: non-finite"
    scale = float(np.abs(ref).max())
    err = np.abs(got - ref)
    bound = GRAD_MAX * scale + (0 if allow is None else allow)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of bound, worst "
                           f"{float((err - bound).max()):.3e} over, scale {scale:.3e}")
    extra = 0.0 if allow is None else float(np.mean(allow))
    assert err.mean() <= GRAD_MEAN * scale + extra, f"{what}: mean err {err.mean():.3e}"


def check_loss(got, ref, what="loss"):
    np.testing.assert_allclose(got, ref, rtol=LOSS_RTOL, atol=LOSS_ATOL, err_msg=what)


def compare_full(q, k, w, idx, l1, cu, cuc, r, grad_scale):
    T = int(cu[-1])
    got = run_gpu(q, k, w, idx, l1, cu, r, grad_scale)
    ref = oracle.indexer_kl_loss_grad(q, k, w, idx, l1, T, cu, cuc, r, grad_scale)
    allow_dq, allow_dk, n_amb = allowances(q, k, w, idx, ref["g"])
    check_loss(got["loss"], ref["loss"])
    check_grad(got["d_w"], ref["d_w"], None, "d_w")
    check_grad(got["d_q"], ref["d_q"], allow_dq, "d_q")
    check_grad(got["d_k"], ref["d_k"], allow_dk, "d_k")
    return got, ref, n_amb


def plant_skipped_entries(idx, cu, cuc, tc):
    """Entries the rule must skip, written over the last slot of a few tokens:
    out of range, a block of the own segment not complete yet, another
    segment's block."""
    idx = idx.copy()
    nb = len(cu) - 1
    long_b = int(np.argmax(np.diff(cu)))
    s = int(cu[long_b])
    idx[s + 5, -1] = tc + 5
    if cuc[long_b + 1] - cuc[long_b] > 3:
        idx[s + 6, -1] = int(cuc[long_b]) + 3          # complete only at local position 15
    other = (long_b + 1) % nb
    if cuc[other + 1] > cuc[other]:
        idx[s + 40, -1] = int(cuc[other])
    return idx


def test_tiny_pack_attention_targets():
    """Lists from the oracle's top-k, targets from the oracle's attention
    backward for those lists (the distribution the pages feed this call)."""
    spec = packs.pack_spec("tiny")
    case = layer_cases(spec, device=None)[0]
    t = case.t
    idx = oracle_topk(case)[0]
    bwd = oracle.sparse_mla_bwd(t["q"], torch.zeros_like(t["q"]), t["ori_kv"], t["cmp_kv"], idx,
                                case.cu, case.cuc, t["sinks"], spec.scale, 4, spec.win_left)
    l1 = bwd["cmp_l1"].astype(np.float32)
    assert (l1 > 0).any()
    compare_full(t["q_idx"], t["k_idx"], t["w"], idx, l1, case.cu, case.cuc, 4, 1.0 / case.T)


@pytest.mark.parametrize("hi,di,k,w_scale", [(64, 128, 64, 1.0), (16, 64, 150, 1.0),
                                             (33, 128, 8, 1e-3)])
def test_medium_pack(hi, di, k, w_scale):
    lengths = [1, 3, 700, 5, 260, 333, 2]
    cu = cu_of(lengths)
    cuc = oracle.compress_cu_seqlens(cu, 4)
    T, tc = int(cu[-1]), int(cuc[-1])
    tens = packs.draw_indexer_tensors(T, T // 4, hi, di, seed=hi + di + k)
    q, kk, w = tens["q_idx"], tens["k_idx"][:tc].contiguous(), tens["w"] * w_scale
    idx = oracle.indexer_topk(q, kk, w, T, cu, cuc, 4, k)[0]
    idx = plant_skipped_entries(idx, cu, cuc, tc)
    l1 = packs.draw_uniform((T, k), seed=7 + k).numpy()
    l1[l1 < 0.1] = 0.0
    l1[int(cu[2]) + 100, :] = 0.0  # a token whose entries carry no mass
    got, ref, _ = compare_full(q, kk, w, idx, l1, cu, cuc, 4, 1.0 / T)
    assert got["loss"][int(cu[2]) + 100] == 0.0
    assert np.abs(got["d_q"][int(cu[2]) + 100]).max() == 0.0
    assert (got["loss"][: int(cu[2]) + 3] == 0.0).all()  # no complete block yet


def test_exact_dots_long_lists():
    """Quarter-integer q and k: every dot product is exact in fp32, so every
    ReLU decision matches the oracle's. Lists of 300 entries (two compaction
    passes, ten chunks) drawn from the whole segment's compressed rows, with
    rows not yet complete, duplicates and -1."""
    lengths = [600, 450]
    cu = cu_of(lengths)
    cuc = oracle.compress_cu_seqlens(cu, 4)
    T, tc = int(cu[-1]), int(cuc[-1])
    hi, di, k = 16, 128, 300
    gen = torch.Generator().manual_seed(31)
    q = (torch.randint(-8, 9, (T, hi, di), generator=gen).float() / 4).to(torch.bfloat16)
    kk = (torch.randint(-8, 9, (tc, di), generator=gen).float() / 4).to(torch.bfloat16)
    w = torch.randn(T, hi, generator=gen) * 0.01
    rng = np.random.default_rng(31)
    idx = np.empty((T, k), dtype=np.int32)
    for b in range(len(lengths)):
        rows = rng.integers(int(cuc[b]), int(cuc[b + 1]), size=(lengths[b], k))
        idx[int(cu[b]):int(cu[b + 1])] = rows
    idx[rng.random((T, k)) < 0.05] = -1
    l1 = packs.draw_uniform((T, k), seed=32).numpy()
    got, ref, n_amb = compare_full(q, kk, w, idx, l1, cu, cuc, 4, 0.5)
    # with exact dots only exact zeros are flagged, and they agree anyway
    assert np.abs(got["d_q"] - ref["d_q"]).max() <= GRAD_MAX * np.abs(ref["d_q"]).max()


def test_no_compressed_rows():
    lengths = [1, 3, 2, 3]
    cu = cu_of(lengths)
    T = int(cu[-1])
    tens = packs.draw_indexer_tensors(T, 0, 4, 64, seed=3)
    idx = np.full((T, 8), -1, dtype=np.int32)
    l1 = np.ones((T, 8), dtype=np.float32)
    got = run_gpu(tens["q_idx"], None, tens["w"], idx, l1, cu, 4, 1.0)
    assert got["d_k"] is None
    assert (got["loss"] == 0).all() and (got["d_q"] == 0).all() and (got["d_w"] == 0).all()


def test_full_size_mixed32k_sampled():
    """The mixed 32k pack's r=4 layer at full size (64 heads x 128, lists of
    512): sampled tokens against the oracle, and over every token the
    identity <d_k, k> = <d_q, q> = <w, d_w> (the ReLU is positively
    homogeneous, so each side equals sum_t sum_s g_s I_s)."""
    spec = packs.pack_spec("mixed32k")
    lengths = spec.lengths
    cu = cu_of(lengths)
    cuc = oracle.compress_cu_seqlens(cu, 4)
    T, tc = int(cu[-1]), int(cuc[-1])
    K = 512
    tens = packs.draw_indexer_tensors(T, T // 4, 64, 128, seed=55)
    q, kk, w = tens["q_idx"], tens["k_idx"][:tc].contiguous(), tens["w"]
    # lists shaped like the indexer's: every visible block while they fit,
    # else a sorted random 512 of them; -1 padding
    rng = np.random.default_rng(55)
    idx = np.full((T, K), -1, dtype=np.int32)
    for b in range(len(lengths)):
        s, e, c0 = int(cu[b]), int(cu[b + 1]), int(cuc[b])
        for t in range(s, e):
            nvis = (t - s + 1) // 4
            if nvis <= K:
                idx[t, :nvis] = c0 + np.arange(nvis)
            else:
                idx[t] = c0 + np.sort(rng.choice(nvis, size=K, replace=False))
    l1 = packs.draw_uniform((T, K), seed=56).numpy()
    gs = 1.0 / T
    res = run_gpu_raw(q, kk, w, idx, l1, cu, 4, gs)
    toks = sample_tokens(lengths, 4, n_random=24, cap=48)
    sel = torch.from_numpy(toks).long()
    ref = oracle.indexer_kl_loss_grad(q[sel], kk, w[sel], idx[toks], l1[toks], T, cu, cuc, 4,
                                      gs, tokens=toks, want_dk=False)
    allow_dq, _, _ = allowances(q, kk, w, idx, ref["g"], tokens=toks, want_dk=False)
    dev_sel = sel.cuda()
    check_loss(res["loss"][dev_sel].double().cpu().numpy(), ref["loss"])
    check_grad(res["d_w"][dev_sel].double().cpu().numpy(), ref["d_w"], None, "d_w")
    check_grad(res["d_q"][dev_sel].double().cpu().numpy(), ref["d_q"], allow_dq, "d_q")
    # the identity over every token, in fp64 on the device
    wd = w.cuda().double() * res["d_w"].double()
    lhs_w = float(wd.sum())
    scale = float(wd.abs().sum())
    lhs_q = float((q.cuda().double() * res["d_q"].double()).sum())
    lhs_k = float((kk.cuda().double() * res["d_k"].double()).sum())
    assert scale > 0
    assert abs(lhs_q - lhs_w) <= 1e-4 * scale, (lhs_q, lhs_w, scale)
    assert abs(lhs_k - lhs_w) <= 1e-4 * scale, (lhs_k, lhs_w, scale)
