"""GPU parity of the sparse MLA backward (csa_sparse_mla_bwd) against the
oracle's fp64 backward, element by element, on packs that span several key
tiles and head groups, with ragged segments, in the three modes (top-k list,
every visible block, window only), with and without sinks.

Tolerances: the kernel works in fp32 from bf16 inputs; the forward's bf16
output enters only through Dv = dout . out, whose rounding (2^-9 relative per
element) is small against dout . k (of order sqrt(D) |dout| |k|), so the
gradients carry about 1e-3 relative error. Each gradient is held to 1e-2 of
its largest magnitude in max-abs and 1e-3 in mean-abs. d_sinks has only H
entries, each a sum over every token of P_sink * Dv whose terms all carry
that rounding (about 2e-3 relative where a token has few keys and a heavy
sink), so it is held to the max-abs bound alone. The head-averaged
distributions (probabilities in [0, 1]) are held to 1e-4 absolute.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import custom_spec, layer_cases

pytestmark = pytest.mark.gpu

GRAD_MAX, GRAD_MEAN, DIST_ABS = 1e-2, 1e-3, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def run_case(lengths, heads, win_left, mode, with_sinks, topk=8, seed=0):
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=topk, index_heads=4, index_dim=64)
    case = layer_cases(custom_spec(lengths, heads=heads, win_left=win_left, layers=(layer,),
                                   seed=seed))[0]
    d, t = case.d, case.t
    gen = torch.Generator().manual_seed(1000 + seed)
    dout_cpu = torch.randn(t["q"].shape, generator=gen).to(torch.bfloat16)
    dout = dout_cpu.cuda()
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, 4)
    ckv = None if mode == "window" else d["cmp_kv"]
    idx = None
    if mode == "topk":
        idx, _ = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc, 4, topk)
    sinks = d["sinks"] if with_sinks else None
    out, lse = csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], ckv, idx, case.cu_d, case.cu_d, cuc,
                                      sinks, case.spec.scale, 4, win_left,
                                      return_softmax_lse=True)
    got = csa.csa_sparse_mla_bwd(d["q"], dout, out, lse, d["ori_kv"], ckv, idx, case.cu_d,
                                 case.cu_d, cuc, sinks, case.spec.scale, 4, win_left)
    torch.cuda.synchronize()
    ref = oracle.sparse_mla_bwd(t["q"], dout_cpu, t["ori_kv"],
                                None if mode == "window" else t["cmp_kv"],
                                None if idx is None else idx.cpu().numpy(), case.cu, case.cuc,
                                t["sinks"] if with_sinks else None, case.spec.scale, 4, win_left)
    return got, ref


def check_grad(got, ref, what, mean=True):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite"
    scale = float(np.abs(ref).max())
    err = np.abs(g - ref)
    assert err.max() <= GRAD_MAX * scale, f"{what}: max err {err.max():.3e} vs scale {scale:.3e}"
    if mean:
        assert err.mean() <= GRAD_MEAN * scale, f"{what}: mean err {err.mean():.3e}"


def check_all(got, ref, mode, with_sinks):
    check_grad(got["d_q"], ref["d_q"], "d_q")
    check_grad(got["d_ori_kv"], ref["d_ori_kv"], "d_ori_kv")
    if mode != "window":
        check_grad(got["d_cmp_kv"], ref["d_cmp_kv"], "d_cmp_kv")
    if with_sinks:
        check_grad(got["d_sinks"], ref["d_sinks"], "d_sinks", mean=False)
    else:
        assert got["d_sinks"] is None
    e = np.abs(got["ori_l1"].double().cpu().numpy() - ref["ori_l1"]).max()
    assert e <= DIST_ABS, f"ori_l1 err {e:.3e}"
    if mode == "topk":
        e = np.abs(got["cmp_l1"].double().cpu().numpy() - ref["cmp_l1"]).max()
        assert e <= DIST_ABS, f"cmp_l1 err {e:.3e}"


LENGTHS = [1, 3, 70, 5, 150, 41, 2]


@pytest.mark.parametrize("mode", ["topk", "all_visible", "window"])
@pytest.mark.parametrize("with_sinks", [True, False])
def test_bwd_modes(mode, with_sinks):
    got, ref = run_case(LENGTHS, heads=8, win_left=15, mode=mode, with_sinks=with_sinks,
                        seed=3 if with_sinks else 4)
    check_all(got, ref, mode, with_sinks)


@pytest.mark.parametrize("heads,win_left,topk", [(64, 127, 64), (40, 40, 300), (4, 0, 5)])
def test_bwd_shapes(heads, win_left, topk):
    """Two head groups (64), a partial second group (40), a lone head group of
    4 with a one-row window; windows and top-k lists over several key tiles."""
    got, ref = run_case([1, 3, 520, 5, 333, 150, 4], heads=heads, win_left=win_left,
                        mode="topk", with_sinks=True, topk=topk, seed=heads)
    check_all(got, ref, "topk", True)


def test_bwd_distributions_sum_to_one():
    """Per token, the distributions over the listed keys plus the mean sink
    weight add up to one (a property, checked on the GPU's own numbers)."""
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=16, index_heads=4, index_dim=64)
    case = layer_cases(custom_spec([300, 90], heads=16, win_left=31, layers=(layer,), seed=9))[0]
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, 4)
    idx, _ = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc, 4, 16)
    out, lse = csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], d["cmp_kv"], idx, case.cu_d, case.cu_d,
                                      cuc, d["sinks"], case.spec.scale, 4, 31,
                                      return_softmax_lse=True)
    dout = torch.randn_like(d["q"].float()).to(torch.bfloat16)
    got = csa.csa_sparse_mla_bwd(d["q"], dout, out, lse, d["ori_kv"], d["cmp_kv"], idx, case.cu_d,
                                 case.cu_d, cuc, d["sinks"], case.spec.scale, 4, 31)
    sink_mean = torch.exp(d["sinks"][None, :] - lse).mean(dim=1)
    total = got["ori_l1"].sum(dim=1) + got["cmp_l1"].sum(dim=1) + sink_mean
    assert torch.allclose(total, torch.ones_like(total), atol=1e-4)
