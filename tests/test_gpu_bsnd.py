"""GPU parity of the BSND entry points (csa_sparse_mla_fwd_bsnd,
csa_indexer_topk_bsnd) against the oracle. Each batch's valid rows are
compared with the oracle run on that batch alone as one THD sequence, where
batch-local rows are the oracle's own rows; rows past seqused are
unspecified and not compared. Same tolerances as the THD tests."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import check_attention, check_topk

pytestmark = pytest.mark.gpu

B, S, H, D, R = 3, 200, 8, 512, 4
SC = S // R
HI, DI, TOPK, WIN_LEFT = 8, 64, 16, 31
SCALE = 1.0 / np.sqrt(D)


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


def draw(seed):
    gen = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    t = {"q": torch.randn(B, S, H, D, generator=gen).to(bf),
         "ori_kv": torch.randn(B, S, D, generator=gen).to(bf),
         "cmp_kv": torch.randn(B, SC, D, generator=gen).to(bf),
         "q_idx": torch.randn(B, S, HI, DI, generator=gen).to(bf),
         "k_idx": torch.randn(B, SC, DI, generator=gen).to(bf),
         "w": torch.randn(B, S, HI, generator=gen),
         "sinks": torch.randn(H, generator=gen)}
    return t


class OneBatch:
    """Batch b's valid rows as a one-sequence THD case (for check_topk)."""

    def __init__(self, t, b, used):
        nc = used // R
        self.T, self.cu = used, np.array([0, used], dtype=np.int32)
        self.cuc = np.array([0, nc], dtype=np.int32)
        self.t = {"q_idx": t["q_idx"][b, :used].contiguous(),
                  "k_idx": t["k_idx"][b, :nc].contiguous(), "w": t["w"][b, :used].contiguous(),
                  "q": t["q"][b, :used].contiguous(), "ori_kv": t["ori_kv"][b, :used].contiguous(),
                  "cmp_kv": t["cmp_kv"][b, :nc].contiguous(), "sinks": t["sinks"]}
        self.layer = packs.LayerSpec(cmp_ratio=R, indexer=True, topk=TOPK, index_heads=HI,
                                     index_dim=DI)

    def oracle_topk(self):
        c = self.t
        return oracle.indexer_topk(c["q_idx"], c["k_idx"], c["w"], self.T, self.cu, self.cuc, R,
                                   TOPK)


def lists_from_oracle(t, used):
    """Batch-local top-k lists from the oracle, -1 on padding rows."""
    idx = -np.ones((B, S, TOPK), dtype=np.int32)
    for b in range(B):
        ob = OneBatch(t, b, int(used[b]))
        idx[b, : ob.T] = ob.oracle_topk()[0]
    return idx


@pytest.mark.parametrize("seqused", [None, (200, 57, 131)])
def test_indexer_bsnd(seqused):
    t = draw(1)
    used = np.full(B, S) if seqused is None else np.asarray(seqused)
    su = None if seqused is None else torch.tensor(seqused, dtype=torch.int32, device="cuda")
    idx, val = csa.csa_indexer_topk_bsnd(t["q_idx"].cuda(), t["k_idx"].cuda(), t["w"].cuda(), su,
                                         R, TOPK, return_value=True)
    idx, val = idx.cpu().numpy(), val.cpu().numpy()
    for b in range(B):
        ob = OneBatch(t, b, int(used[b]))
        check_topk(ob, idx[b, : ob.T], ob.oracle_topk(), gpu_val=val[b, : ob.T])


@pytest.mark.parametrize("mode", ["topk", "all", "window"])
@pytest.mark.parametrize("seqused", [None, (200, 57, 131)])
def test_sparse_mla_bsnd(mode, seqused):
    t = draw(2)
    used = np.full(B, S) if seqused is None else np.asarray(seqused)
    su = None if seqused is None else torch.tensor(seqused, dtype=torch.int32, device="cuda")
    idx = lists_from_oracle(t, used) if mode == "topk" else None
    if idx is not None:
        idx[0, 150, -1] = SC + 3       # out of range: skipped
        idx[2, 100, -1] = SC - 1       # not complete at row 100: skipped
    ckv = None if mode == "window" else t["cmp_kv"].cuda()
    out, lse = csa.csa_sparse_mla_fwd_bsnd(
        t["q"].cuda(), t["ori_kv"].cuda(), ckv,
        None if idx is None else torch.from_numpy(idx).cuda(), su, t["sinks"].cuda(), SCALE, R,
        WIN_LEFT, return_softmax_lse=True)
    out, lse = out.cpu(), lse.cpu()
    for b in range(B):
        ob = OneBatch(t, b, int(used[b]))
        c = ob.t
        ref_out, ref_lse = oracle.sparse_mla_fwd(
            c["q"], c["ori_kv"], None if mode == "window" else c["cmp_kv"],
            None if idx is None else idx[b, : ob.T], ob.cu, ob.cuc, ob.T, c["sinks"], SCALE, R,
            WIN_LEFT)
        check_attention(out[b, : ob.T], lse[b, : ob.T], ref_out, ref_lse, f"batch {b} {mode}")


def test_seqused_out_of_range_is_reported():
    t = draw(3)
    su = torch.tensor([S + 5, 10, -1], dtype=torch.int32, device="cuda")
    out, _ = csa.csa_sparse_mla_fwd_bsnd(t["q"].cuda(), t["ori_kv"].cuda(), None, None, su,
                                         t["sinks"].cuda(), SCALE, R, WIN_LEFT)
    st, word = csa.csa_device_error()
    assert st == 6 and (word >> 16) & 0xFF == 7  # a device check, from the BSND offsets
    assert csa.csa_device_error()[0] == 0        # read once, cleared
    # the clamped batch (all S rows valid) still matches the oracle
    ob = OneBatch(t, 0, S)
    c = ob.t
    ref_out, _ = oracle.sparse_mla_fwd(c["q"], c["ori_kv"], None, None, ob.cu, ob.cuc, S,
                                       c["sinks"], SCALE, R, WIN_LEFT)
    check_attention(out[0].cpu(), None, ref_out, None, "clamped batch")
