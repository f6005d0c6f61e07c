"""GPU parity of the integer steps: compressed cu_seqlens and window rows,
bit-exact against the oracle (tiny pack, random packs, edge segments)."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_csa_gb300 as csa
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import cu_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


EDGE = [0, 1, 3, 4, 5, 0, 7, 8, 127, 128, 129, 255, 256, 257, 2]


@pytest.mark.parametrize("r", [1, 2, 3, 4, 128])
def test_compress_edge_and_random(r):
    rng = np.random.default_rng(r)
    for lengths in (EDGE, rng.integers(0, 600, size=40).tolist(), [100, 37, 119], [16384]):
        cu = cu_of(lengths)
        got = csa.csa_compress_cu_seqlens(dev(cu), r).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.compress_cu_seqlens(cu, r))


def test_compress_many_segments_and_empty():
    rng = np.random.default_rng(5)
    lengths = rng.integers(0, 50, size=5000).tolist()  # several scan chunks of 1024
    cu = cu_of(lengths)
    got = csa.csa_compress_cu_seqlens(dev(cu), 4).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.compress_cu_seqlens(cu, 4))
    got0 = csa.csa_compress_cu_seqlens(dev([0]), 4).cpu().numpy()
    assert got0.tolist() == [0]


@pytest.mark.parametrize("W", [1, 2, 16, 127, 128, 129])
def test_window_random_and_edges(W):
    rng = np.random.default_rng(W)
    for lengths in (EDGE, rng.integers(1, 400, size=12).tolist(), [100, 37, 119]):
        cu = cu_of(lengths)
        T = int(cu[-1])
        got = csa.csa_window_idx(dev(cu), T, W - 1).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.window_idx(cu, T, W - 1))


def test_window_full_size_pack():
    from csa_inputs import packs
    for name in ("mixed32k", "long16k"):
        spec = packs.pack_spec(name)
        cu = cu_of(spec.lengths)
        got = csa.csa_window_idx(dev(cu), spec.total_tokens, 127).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.window_idx(cu, spec.total_tokens, 127))


def test_window_unaligned_output_and_empty():
    cu = cu_of([9, 30])
    buf = torch.full((39 * 16 + 1,), 7, dtype=torch.int32, device="cuda")
    out = buf[1:].view(39, 16)  # 4-byte aligned, not 16-byte aligned
    assert not out.is_contiguous() or out.data_ptr() % 16 != 0
    csa.csa_window_idx(dev(cu), 39, 15, out=out)
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.window_idx(cu, 39, 15))
    assert buf[0].item() == 7
    empty = torch.empty((0, 16), dtype=torch.int32, device="cuda")
    csa.csa_window_idx(dev([0]), 0, 15, out=empty)


def test_inconsistent_cu_sets_device_error():
    # cu_seqlens covers 10 rows but 16 tokens are requested: rows 10..15 get -1
    cu = dev([0, 4, 10])
    out = csa.csa_window_idx(cu, 16, 3).cpu().numpy()
    assert (out[10:] == -1).all()
    np.testing.assert_array_equal(out[:10], oracle.window_idx([0, 4, 10], 10, 3))
    st, word = csa.csa_device_error()
    assert st == 6 and word != 0
    assert csa.csa_device_error()[0] == 0  # cleared
