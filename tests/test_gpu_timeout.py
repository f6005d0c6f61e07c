"""The bounded-wait timeout path of the indexer and sparse-attention kernels.

With a pipeline-wait limit of a fraction of a microsecond (csa_set_wait_limit_ns),
waits of both kernels give up: each launch must still end, report
CSA_ERR_TIMEOUT (kind 2 in the device error word, with the kernel's id), and
leave the context usable, so that the next launches at the default limit are
clean and match the oracle. No GPU fault, trap or endless wait is involved:
the kernels' own bounded waits run out."""

import numpy as np
import pytest
import torch

import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import check_attention, indices_for_oracle, layer_cases, oracle_attention

pytestmark = pytest.mark.gpu

CSA_ERR_TIMEOUT = 7
KERNEL_INDEXER, KERNEL_MLA = 3, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    csa.csa_set_wait_limit_ns(0)
    assert csa.csa_device_error()[0] == 0


def run(case):
    d = case.d
    cuc = csa.csa_compress_cu_seqlens(case.cu_d, case.layer.cmp_ratio)
    idx, _ = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc,
                                  case.layer.cmp_ratio, case.layer.topk, return_value=True)
    st_idx = csa.csa_device_error()
    out, lse = csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], d["cmp_kv"], idx, case.cu_d, case.cu_d,
                                      cuc, d["sinks"], case.spec.scale, case.layer.cmp_ratio,
                                      case.spec.win_left, return_softmax_lse=True)
    st_mla = csa.csa_device_error()
    return idx, out, lse, st_idx, st_mla


def test_short_wait_limit_times_out_and_next_launch_is_clean():
    case = layer_cases(packs.pack_spec("prefill4k"))[0]
    assert csa.csa_device_error()[0] == 0
    try:
        csa.csa_set_wait_limit_ns(200)
        for _ in range(2):
            _, _, _, (st_i, w_i), (st_m, w_m) = run(case)
            assert st_i == CSA_ERR_TIMEOUT and (w_i >> 24) == 2 and ((w_i >> 16) & 0xFF) == KERNEL_INDEXER
            assert st_m == CSA_ERR_TIMEOUT and (w_m >> 24) == 2 and ((w_m >> 16) & 0xFF) == KERNEL_MLA
    finally:
        csa.csa_set_wait_limit_ns(0)
    idx, out, lse, (st_i, _), (st_m, _) = run(case)
    assert st_i == 0 and st_m == 0
    toks = np.arange(0, case.T, 97, dtype=np.int32)
    rows = indices_for_oracle(case, idx.cpu().numpy(), toks)
    ref_out, ref_lse = oracle_attention(case, rows, toks)
    tk = torch.from_numpy(toks).long().cuda()
    check_attention(out[tk], lse[tk], ref_out, ref_lse, "after timeouts")
