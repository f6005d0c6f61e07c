"""GPU parity of the THD compressor core (csa_compress_thd) against the
oracle, on every output element: a ragged pack with sequences shorter than
one group, the mixed 32k pack at full size for both ratios (4 and 128,
head_dim 512, overlap), the no-overlap 128-wide variant (the indexer's keys)
and a pack with no compressed row.

Tolerance: the kernel accumulates the softmax online in fp32 from fp32
inputs; against the fp64 oracle each output may differ by 2e-5 absolute
plus 1e-5 relative (outputs are convex combinations of N(0,1) values)."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import cu_of

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-5, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def run_case(lengths, r, hd, overlap, with_ape, seed):
    cu = cu_of(lengths)
    T = int(cu[-1])
    wd = 2 * hd if overlap else hd
    kv = packs.draw_normal((T, wd), seed)
    score = packs.draw_normal((T, wd), seed + 1)
    ape = packs.draw_normal((r, wd), seed + 2) if with_ape else None
    cu_d = torch.from_numpy(cu).cuda()
    cuc = csa.csa_compress_cu_seqlens(cu_d, r)
    tc = int(cuc[-1].item())
    out = csa.csa_compress_thd(kv.cuda(), score.cuda(), None if ape is None else ape.cuda(), cu_d,
                               cuc, tc, r, hd, overlap)
    got = out.double().cpu().numpy()
    ref = oracle.compress_thd(kv, score, ape, cu, r, hd, overlap)
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=RTOL, atol=ATOL)
    return got


def test_ragged_pack():
    run_case([1, 3, 700, 5, 260, 333, 2], 4, 512, True, True, seed=10)


@pytest.mark.parametrize("r", [4, 128])
def test_mixed32k_full_size(r):
    run_case(packs.pack_spec("mixed32k").lengths, r, 512, True, True, seed=20 + r)


def test_no_overlap_index_keys():
    run_case([1, 3, 700, 5, 260, 333, 2], 4, 128, False, False, seed=30)


def test_no_compressed_rows():
    lengths = [1, 3, 2]
    cu_d = torch.from_numpy(cu_of(lengths)).cuda()
    cuc = csa.csa_compress_cu_seqlens(cu_d, 4)
    assert int(cuc[-1].item()) == 0
    kv = torch.zeros((6, 1024), device="cuda")
    out = csa.csa_compress_thd(kv, kv, None, cu_d, cuc, 0, 4, 512, True)
    assert out.shape == (0, 512)
