"""GPU parity of the THD compressor core (csa_compress_thd) against the
oracle, on every output element: a ragged pack with sequences shorter than
one group, the mixed 32k pack at full size for both ratios (4 and 128,
head_dim 512, overlap), the no-overlap 128-wide variant (the indexer's keys),
ratios 1 to 128 and widths 64 to 1024 (every thread-row split of the slots),
the per-dimension path (odd widths, unaligned arrays) and a pack with no
compressed row.

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


def on_device(x, misalign):
    """x on the GPU; with misalign, at an address 4 bytes past a 16-byte
    boundary (the kernel's per-dimension path)."""
    if not misalign:
        return x.cuda()
    buf = torch.empty(x.numel() + 1, dtype=x.dtype, device="cuda")
    view = buf[1:].view(x.shape)
    view.copy_(x)
    return view


def run_case(lengths, r, hd, overlap, with_ape, seed, misalign=False):
    cu = cu_of(lengths)
    T = int(cu[-1])
    wd = 2 * hd if overlap else hd
    kv = packs.draw_normal((T, wd), seed)
    score = packs.draw_normal((T, wd), seed + 1)
    ape = packs.draw_normal((r, wd), seed + 2) if with_ape else None
    cu_d = torch.from_numpy(cu).cuda()
    cuc = csa.csa_compress_cu_seqlens(cu_d, r)
    tc = int(cuc[-1].item())
    out = csa.csa_compress_thd(on_device(kv, misalign), on_device(score, False),
                               None if ape is None else ape.cuda(), cu_d, cuc, tc, r, hd, overlap)
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


@pytest.mark.parametrize("r,hd,overlap", [(1, 512, True), (2, 64, False), (3, 512, True),
                                           (8, 512, True), (64, 512, True), (16, 1024, True),
                                           (8, 128, False), (16, 96, False), (128, 128, False)])
def test_ratios_and_widths(r, hd, overlap):
    """Ratios from 1 to 128 and widths from 64 to 1024: the thread-row split
    of the slots (1 to 8 rows, rows holding no slot), two dimension blocks per
    row, and the 32-thread blocks of narrow rows."""
    run_case([1, 3, 700, 5, 260, 333, 2, 1500], r, hd, overlap, True, seed=40 + r)


@pytest.mark.parametrize("hd,misalign", [(130, False), (512, True)])
def test_per_dimension_path(hd, misalign):
    """Widths that are not a multiple of 4, and arrays not 16-byte aligned,
    take the one-dimension-per-thread kernel."""
    run_case([1, 3, 700, 5, 260, 333, 2], 4, hd, True, True, seed=50 + hd, misalign=misalign)


def test_no_compressed_rows():
    lengths = [1, 3, 2]
    cu_d = torch.from_numpy(cu_of(lengths)).cuda()
    cuc = csa.csa_compress_cu_seqlens(cu_d, 4)
    assert int(cuc[-1].item()) == 0
    kv = torch.zeros((6, 1024), device="cuda")
    out = csa.csa_compress_thd(kv, kv, None, cu_d, cuc, 0, 4, 512, True)
    assert out.shape == (0, 512)
