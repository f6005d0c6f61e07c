"""GPU parity of the shared-KV MLA sparse attention with sinks against the
oracle: full comparisons on packs that span several key tiles and ragged
segments, sampled comparisons at full size, and invariances."""

import numpy as np
import pytest
import torch

import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import (check_attention, custom_spec, indices_for_oracle, layer_cases,
                         oracle_attention, sample_tokens)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def gpu_attention(case, idx_dev, sinks="default", cmp=True, q=None, okv=None, ckv=None):
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, case.layer.cmp_ratio)
    sk = d["sinks"] if isinstance(sinks, str) else sinks
    out, lse = csa.csa_sparse_mla_fwd(
        d["q"] if q is None else q, d["ori_kv"] if okv is None else okv,
        (d["cmp_kv"] if ckv is None else ckv) if cmp else None, idx_dev, case.cu_d, case.cu_d,
        cuc, sk, case.spec.scale, case.layer.cmp_ratio, case.spec.win_left,
        return_softmax_lse=True)
    return out, lse


def gpu_topk(case):
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, case.layer.cmp_ratio)
    idx, _ = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc,
                                  case.layer.cmp_ratio, case.layer.topk)
    return idx


def test_tiny_pack_full():
    case = layer_cases(packs.pack_spec("tiny"))[0]
    idx = gpu_topk(case)
    out, lse = gpu_attention(case, idx)
    rows = indices_for_oracle(case, idx.cpu().numpy())
    ref_out, ref_lse = oracle_attention(case, rows)
    check_attention(out, lse, ref_out, ref_lse, "tiny")


@pytest.mark.parametrize("heads,win_left,k", [(64, 127, 64), (16, 127, 300), (12, 40, 8),
                                              (4, 0, 5)])
def test_medium_pack_indexer(heads, win_left, k):
    lengths = [1, 3, 520, 5, 333, 150, 4]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=k, index_heads=8, index_dim=64)
    spec = custom_spec(lengths, heads=heads, win_left=win_left, layers=(layer,),
                       seed=heads + k)
    case = layer_cases(spec)[0]
    idx = gpu_topk(case)
    out, lse = gpu_attention(case, idx)
    rows = indices_for_oracle(case, idx.cpu().numpy())
    ref_out, ref_lse = oracle_attention(case, rows)
    check_attention(out, lse, ref_out, ref_lse, f"H={heads}")


@pytest.mark.parametrize("r", [128, 4])
def test_medium_pack_compressor_only(r):
    lengths = [700, 300, 129, 127, 1, 260]
    layer = packs.LayerSpec(cmp_ratio=r, indexer=False)
    case = layer_cases(custom_spec(lengths, heads=16, win_left=127, layers=(layer,)))[0]
    out, lse = gpu_attention(case, None)
    ref_out, ref_lse = oracle_attention(case, None)
    check_attention(out, lse, ref_out, ref_lse, f"hca r={r}")


def test_window_only_and_no_sinks():
    lengths = [200, 57]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=False)
    case = layer_cases(custom_spec(lengths, heads=8, win_left=63, layers=(layer,)))[0]
    out, lse = gpu_attention(case, None, cmp=False)
    import oracle
    ref_out, ref_lse = oracle.sparse_mla_fwd(case.t["q"], case.t["ori_kv"], None, None, case.cu,
                                             case.cuc, case.T, case.t["sinks"], case.spec.scale,
                                             4, 63)
    check_attention(out, lse, ref_out, ref_lse, "window only")
    # sinks NULL == sinks of -inf, bit for bit
    o1, l1 = gpu_attention(case, None, sinks=None)
    o2, l2 = gpu_attention(case, None, sinks=torch.full_like(case.d["sinks"], -float("inf")))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_out, ref_lse = oracle.sparse_mla_fwd(case.t["q"], case.t["ori_kv"], case.t["cmp_kv"],
                                             None, case.cu, case.cuc, case.T, None,
                                             case.spec.scale, 4, 63)
    check_attention(o1, l1, ref_out, ref_lse, "no sinks")


def test_invalid_indices_are_skipped():
    lengths = [90, 200]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=12, index_heads=4, index_dim=64)
    case = layer_cases(custom_spec(lengths, heads=8, layers=(layer,)))[0]
    idx = gpu_topk(case)
    bad = idx.clone()
    bad[:, -1] = case.Tc + 3          # out of range
    bad[:, -2] = -5                   # negative
    bad[100:, -3] = 0                 # row of another sequence
    out, lse = gpu_attention(case, bad)
    ref_out, ref_lse = oracle_attention(case, bad.cpu().numpy())
    check_attention(out, lse, ref_out, ref_lse, "invalid indices")


def test_segment_isolation_bit_exact():
    lengths = [150, 260, 90]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=32, index_heads=8, index_dim=64)
    case = layer_cases(custom_spec(lengths, heads=16, layers=(layer,)))[0]
    idx = gpu_topk(case)
    out, lse = gpu_attention(case, idx)
    q2, okv2, ckv2 = case.d["q"].clone(), case.d["ori_kv"].clone(), case.d["cmp_kv"].clone()
    g = torch.Generator(device="cuda").manual_seed(3)
    q2[:150] = torch.randn(q2[:150].shape, generator=g, device="cuda").bfloat16()
    okv2[410:] = torch.randn(okv2[410:].shape, generator=g, device="cuda").bfloat16()
    ckv2[:37] = torch.randn(ckv2[:37].shape, generator=g, device="cuda").bfloat16()
    out2, lse2 = gpu_attention(case, idx, q=q2, okv=okv2, ckv=ckv2)
    assert torch.equal(out2[150:410], out[150:410])
    assert torch.equal(lse2[150:410], lse[150:410])


def test_index_order_permutation():
    lengths = [400]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=64, index_heads=8, index_dim=64)
    case = layer_cases(custom_spec(lengths, heads=16, layers=(layer,)))[0]
    idx = gpu_topk(case)
    out, lse = gpu_attention(case, idx)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(0)).cuda()
    out2, lse2 = gpu_attention(case, idx[:, perm].contiguous())
    assert (out2.float() - out.float()).abs().max().item() <= 1e-2
    assert (lse2 - lse).abs().max().item() <= 1e-4


@pytest.mark.parametrize("name", ["prefill4k", "long16k", "hca32k", "mixed32k"])
def test_full_size_sampled(name):
    spec = packs.pack_spec(name)
    for li, case in enumerate(layer_cases(spec)):
        toks = sample_tokens(spec.lengths, case.layer.cmp_ratio, n_random=16, cap=40, seed=li)
        if case.layer.indexer:
            idx = gpu_topk(case)
            out, lse = gpu_attention(case, idx)
            rows = indices_for_oracle(case, idx.cpu().numpy(), toks)
        else:
            out, lse = gpu_attention(case, None)
            rows = None
        ref_out, ref_lse = oracle_attention(case, rows, toks)
        tk = torch.from_numpy(toks).long().cuda()
        check_attention(out[tk], lse[tk], ref_out, ref_lse, f"{name} layer {li}")
        del case
        torch.cuda.empty_cache()


@pytest.mark.parametrize("win_left", [300, 1023])
def test_wide_window(win_left):
    """Windows wider than one key tile (several window tiles per token, no ring)."""
    lengths = [1200, 5, 300]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=64, index_heads=8, index_dim=64)
    case = layer_cases(custom_spec(lengths, heads=16, win_left=win_left, layers=(layer,),
                                   seed=win_left))[0]
    idx = gpu_topk(case)
    toks = sample_tokens(lengths, 4, n_random=24, cap=48, seed=5)
    out, lse = gpu_attention(case, idx)
    rows = indices_for_oracle(case, idx.cpu().numpy(), toks)
    ref_out, ref_lse = oracle_attention(case, rows, toks)
    check_attention(out[toks], lse[toks], ref_out, ref_lse, f"window {win_left + 1}")


def test_many_short_sequences():
    """More sequences than the kernels keep offsets for on chip; many CTAs
    start and end mid-sequence; hundreds of tokens see one or two keys, so
    their outputs are single V rows (|out| up to ~4) and any rounding of the
    largest weight shows directly."""
    rng = np.random.default_rng(7)
    lengths = [int(x) for x in rng.integers(1, 40, size=700)]
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=6, index_heads=4, index_dim=64)
    case = layer_cases(custom_spec(lengths, heads=8, win_left=15, layers=(layer,), seed=3))[0]
    idx = gpu_topk(case)
    rows = indices_for_oracle(case, idx.cpu().numpy())
    out, lse = gpu_attention(case, idx)
    ref_out, ref_lse = oracle_attention(case, rows)
    check_attention(out, lse, ref_out, ref_lse, "700 sequences")


def test_no_compress_ratio_one():
    """NO_COMPRESS: the compressor gives no rows and the ratio is 1; the
    attention is the window alone (with sinks)."""
    import oracle
    lengths = [300, 1, 129, 57]
    layer = packs.LayerSpec(cmp_ratio=1, indexer=False)
    case = layer_cases(custom_spec(lengths, heads=16, win_left=127, layers=(layer,)))[0]
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, 1)
    np.testing.assert_array_equal(cuc.cpu().numpy(), case.cu)  # ratio 1: every token a row
    d = case.d
    out, lse = csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], None, None, case.cu_d, case.cu_d, cuc,
                                      d["sinks"], case.spec.scale, 1, 127,
                                      return_softmax_lse=True)
    ref_out, ref_lse = oracle.sparse_mla_fwd(case.t["q"], case.t["ori_kv"], None, None, case.cu,
                                             case.cu, case.T, case.t["sinks"], case.spec.scale,
                                             1, 127)
    check_attention(out, lse, ref_out, ref_lse, "ratio 1, window only")
    # compressed rows at ratio 1 are not an accepted request
    with pytest.raises(csa.CsaError) as e:
        csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], d["ori_kv"], None, case.cu_d, case.cu_d, cuc,
                               d["sinks"], case.spec.scale, 1, 127)
    assert e.value.code == 3  # CSA_ERR_UNSUPPORTED
