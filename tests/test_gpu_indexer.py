"""GPU parity of the lightning-indexer score + top-k against the oracle."""

import numpy as np
import pytest
import torch

import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import (LayerCase, check_topk, custom_spec, layer_cases, oracle_topk,
                         sample_tokens)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def run_gpu(case, topk=None, return_value=True):
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, case.layer.cmp_ratio)
    idx, val = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc,
                                    case.layer.cmp_ratio, topk or case.layer.topk,
                                    return_value=return_value)
    return idx.cpu().numpy(), (val.cpu().numpy() if val is not None else None)


def test_tiny_pack_full():
    case = layer_cases(packs.pack_spec("tiny"))[0]
    idx, val = run_gpu(case)
    ref = oracle_topk(case)
    check_topk(case, idx, ref, gpu_val=val)


@pytest.mark.parametrize("hi,di,k", [(64, 128, 64), (8, 64, 16), (4, 64, 1), (64, 64, 300),
                                     (12, 128, 8), (33, 64, 40)])
def test_medium_pack_full(hi, di, k):
    lengths = [1, 3, 700, 5, 1100, 260, 4, 9]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=k, index_heads=hi, index_dim=di)
    spec = custom_spec(lengths, heads=4, layers=(layer,), seed=hi + di + k)
    case = layer_cases(spec)[0]
    idx, val = run_gpu(case)
    ref = oracle_topk(case)
    check_topk(case, idx, ref, gpu_val=val)


def test_topk_covers_visible_and_index_only():
    lengths = [77, 130, 2]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=40, index_heads=16, index_dim=128)
    case = layer_cases(custom_spec(lengths, layers=(layer,)))[0]
    idx, _ = run_gpu(case, return_value=False)
    ref = oracle_topk(case)
    np.testing.assert_array_equal(idx, ref[0])


def test_exact_ties_lowest_rows_win():
    lengths = [300, 41]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=20, index_heads=4, index_dim=64)
    case = layer_cases(custom_spec(lengths, layers=(layer,)))[0]
    case.t["q_idx"].zero_()
    case.d["q_idx"].zero_()
    idx, val = run_gpu(case)
    ref = oracle_topk(case)
    np.testing.assert_array_equal(idx, ref[0])
    assert (val[idx >= 0] == 0).all()


def test_no_compressed_rows():
    lengths = [1, 3, 2, 3]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=8, index_heads=4, index_dim=64)
    spec = custom_spec(lengths, layers=(layer,))
    tens = packs.draw_pack(spec)[0]
    case = LayerCase(spec, layer, tens)
    assert case.Tc == 0
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, 4)
    idx, val = csa.csa_indexer_topk(d["q_idx"], None, d["w"], case.cu_d, cuc, 4, 8,
                                    return_value=True)
    assert (idx.cpu() == -1).all() and torch.isinf(val.cpu()).all()


@pytest.mark.parametrize("name", ["prefill4k", "long16k", "mixed32k"])
def test_full_size_sampled(name):
    spec = packs.pack_spec(name)
    case = layer_cases(spec)[0]
    idx, val = run_gpu(case)
    toks = sample_tokens(spec.lengths, case.layer.cmp_ratio, n_random=24, cap=48)
    if name == "long16k":
        toks = np.unique(np.concatenate([toks, [16383, 16382, 8191, 2047, 2048, 4095]])).astype(
            np.int32)
    ref = oracle_topk(case, toks)
    check_topk(case, idx[toks], ref, tokens=toks, gpu_val=val[toks])


@pytest.mark.parametrize("entry", ["workspace", "noalloc"])
@pytest.mark.parametrize("return_value", [True, False])
def test_spill_path_against_oracle(entry, return_value):
    """One 24,576-token sequence at ratio 4 (6,144 compressed rows): its late
    tokens see more rows than the kernel keeps in shared memory, so their
    scores go through the global scratch (the caller's workspace, or the
    library's own array for the no-allocation entry point)."""
    T, K = 24576, 512
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=K, index_heads=64, index_dim=128)
    case = layer_cases(custom_spec([T], heads=4, layers=(layer,), seed=97))[0]
    assert case.Tc == T // 4
    # more rows than shared memory keeps: the ordinary entry point wants a workspace
    assert csa.csa_indexer_topk_workspace_size(T, case.Tc, 64, 128, K) > 0
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, 4)
    call = csa.csa_indexer_topk if entry == "workspace" else csa.csa_indexer_topk_noalloc
    idx, val = call(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc, 4, K,
                    return_value=return_value)
    torch.cuda.synchronize()
    assert csa.csa_device_error()[0] == 0
    rng = np.random.default_rng(5)
    late = rng.integers(5120 * 4 - 1, T, size=40)  # positions that see > 5120 rows
    toks = np.unique(np.concatenate([late, [T - 1, 20478, 20479, 20480, 2051, 7, 0]]))
    toks = toks.astype(np.int32)
    ref = oracle_topk(case, toks)
    gi = idx.cpu().numpy()[toks]
    gv = val.cpu().numpy()[toks] if return_value else None
    check_topk(case, gi, ref, tokens=toks, gpu_val=gv)
    # every scored late token keeps K distinct rows of its own sequence, ascending
    assert (gi[toks >= 20480] >= 0).all()


@pytest.mark.parametrize("scores", ["shared", "workspace"])
def test_one_warp_selection(scores):
    """The one-warp selection (taken for tokens with more visible rows than
    the two-warp selection's bound) on ordinary inputs, with the bound
    lowered to 256 rows: rows in shared memory (a ragged pack) and rows in
    the workspace (a 24,576-token sequence). Outputs equal those of the
    two-warp selection, and agree with the oracle."""
    if scores == "shared":
        layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=64, index_heads=16, index_dim=64)
        case = layer_cases(custom_spec([1, 3, 700, 5, 2600, 333, 2], heads=1, layers=(layer,),
                                       seed=113))[0]
        toks = None
    else:
        layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=512, index_heads=64,
                                index_dim=128)
        case = layer_cases(custom_spec([24576], heads=1, layers=(layer,), seed=97))[0]
        rng = np.random.default_rng(8)
        toks = np.unique(np.concatenate([rng.integers(20480, 24576, size=24),
                                         [24575, 2051, 1100]])).astype(np.int32)
    d, K = case.d, case.layer.topk
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, 4)
    ref_idx, ref_val = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc, 4, K,
                                            return_value=True)
    try:
        csa.csa_set_pair_select_rows(256)
        idx, val = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc, 4, K,
                                        return_value=True)
        torch.cuda.synchronize()
    finally:
        csa.csa_set_pair_select_rows(0)
    assert csa.csa_device_error()[0] == 0
    assert torch.equal(idx, ref_idx) and torch.equal(val, ref_val)
    ref = oracle_topk(case, toks)
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    if toks is not None:
        gi, gv = gi[toks], gv[toks]
    check_topk(case, gi, ref, tokens=toks, gpu_val=gv)
