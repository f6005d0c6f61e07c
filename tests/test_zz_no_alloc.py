"""csa_indexer_topk_noalloc against csa_indexer_topk.

The no-allocation entry point is for callers that cannot allocate device
memory themselves -- for instance a plugin that a host framework hands only
its input and output buffers, or a runtime held to a memory budget fixed at
start-up -- and so cannot provide the workspace the ordinary entry point
takes. It uses the library's own fixed-size scratch array instead.

The pack here is one sequence long enough that its late tokens see more
compressed rows than the kernel keeps in shared memory, so their scores go
through the scratch. Two calls in a row must both give what the ordinary
entry point gives with a workspace from the caller, and sampled tokens of
both must follow the fp64 oracle's top-k rule. This file is named to be
collected last.
"""

import ctypes as C
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import sparse_attention_csa_gb300 as csa
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import VAL_ATOL, VAL_RTOL, check_topk, oracle_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()


def test_noalloc_matches_workspace_entry_point():
    T, r, Hi, Di, K = 170_000, 4, 4, 64, 16  # 42,500 compressed rows in one sequence
    g = torch.Generator(device="cuda").manual_seed(1234)
    q = torch.randn((T, Hi, Di), generator=g, device="cuda").bfloat16()
    k = torch.randn((T // r, Di), generator=g, device="cuda").bfloat16()
    w = torch.rand((T, Hi), generator=g, device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    cuc = csa.csa_compress_cu_seqlens(cu, r)
    assert cuc.cpu().tolist() == [0, T // r]
    # the ordinary entry point needs a caller workspace for this pack
    assert csa.csa_indexer_topk_workspace_size(T, T // r, Hi, Di, K) > 0
    ref_idx, ref_val = csa.csa_indexer_topk(q, k, w, cu, cuc, r, K, return_value=True)
    ref_idx, ref_val = ref_idx.cpu(), ref_val.cpu().numpy()
    for _ in range(2):
        idx, val = csa.csa_indexer_topk_noalloc(q, k, w, cu, cuc, r, K, return_value=True)
        assert torch.equal(idx.cpu(), ref_idx)
        np.testing.assert_allclose(val.cpu().numpy(), ref_val, rtol=VAL_RTOL, atol=VAL_ATOL)
    assert csa.csa_device_error()[0] == 0
    # the last token sees every row and keeps the 16 best of 42,500
    assert (ref_idx[-1] >= 0).all() and ref_idx[-1].unique().numel() == K
    # and both agree with the fp64 oracle on sampled tokens, late ones included
    case = SimpleNamespace(
        t={"q_idx": q.cpu(), "k_idx": k.cpu(), "w": w.cpu()}, T=T, cu=np.array([0, T], np.int32),
        cuc=np.array([0, T // r], np.int32),
        layer=SimpleNamespace(cmp_ratio=r, topk=K))
    rng = np.random.default_rng(11)
    toks = np.unique(np.concatenate([rng.integers(5120 * r, T, size=32), [T - 1, 3, 100]]))
    toks = toks.astype(np.int32)
    ref = oracle_topk(case, toks)
    check_topk(case, idx.cpu().numpy()[toks], ref, tokens=toks, gpu_val=val.cpu().numpy()[toks])


def test_noalloc_rejects_more_rows_than_the_scratch_holds():
    L = csa.lib()
    p = C.c_void_p(0x1000)  # never dereferenced: the size check comes first
    for rows in ((1 << 21) + 1, (1 << 23) + 1):  # one CTA slot holds 4 x rows floats
        rc = L.csa_indexer_topk_noalloc(p, p, p, 1 << 24, rows, 4, 64, p, p, 1, 4, 8, p,
                                        None, None)
        assert rc == 4  # CSA_ERR_WORKSPACE
