"""Every token of the full-size packs against the fp64 oracle.

For each layer of prefill4k, long16k, hca32k and mixed32k (both layers), the
GPU runs the layer as the product path does (indexer without values, then the
sparse attention), and the oracle recomputes every token in chunks:
* top-k rows: bit-exact, except where the oracle's k-th and (k+1)-th scores
  are within the near-tie band (tests/_util.check_topk); the values path
  (every token scored) is checked too, with its values;
* attention: max |out - oracle| <= 2e-2 and mean <= 2e-3 over the whole
  output of the layer, LSE max <= 1e-3; where a top-k row differed by a
  near-tie the oracle is fed the GPU's rows for that token.
The per-layer errors are printed in the run's parity report.
"""

import numpy as np
import pytest
import torch

import sparse_attention_csa_gb300 as csa
from csa_inputs import packs
from sparse_attention_csa_gb300 import build as csa_build
from tests._util import (LSE_MAX_ABS, OUT_MAX_ABS, OUT_MEAN_ABS, REPORT, check_topk, layer_cases,
                         oracle_attention, oracle_topk)

pytestmark = pytest.mark.gpu

CHUNK = 2048  # tokens per oracle call


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa_build.build()
    yield
    assert csa.csa_device_error()[0] == 0


@pytest.mark.parametrize("name", ["prefill4k", "long16k", "hca32k", "mixed32k"])
def test_every_token(name):
    spec = packs.pack_spec(name)
    for li, case in enumerate(layer_cases(spec)):
        d, layer, T = case.d, case.layer, case.T
        cuc = csa.csa_compress_cu_seqlens(case.cu_d, layer.cmp_ratio)
        idx_np = val_idx = val_np = None
        idx = None
        if layer.indexer:
            idx, _ = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc,
                                          layer.cmp_ratio, layer.topk)
            vi, vv = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], case.cu_d, cuc,
                                          layer.cmp_ratio, layer.topk, return_value=True)
            idx_np, val_idx, val_np = idx.cpu().numpy(), vi.cpu().numpy(), vv.cpu().numpy()
            del vi, vv
        out, lse = csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], d["cmp_kv"], idx, case.cu_d,
                                          case.cu_d, cuc, d["sinks"], spec.scale, layer.cmp_ratio,
                                          spec.win_left, return_softmax_lse=True)
        torch.cuda.synchronize()
        assert csa.csa_device_error()[0] == 0
        lse_np = lse.cpu().double().numpy()
        mx = lmx = 0.0
        tot, cnt, ties = 0.0, 0, 0
        for t0 in range(0, T, CHUNK):
            t1 = min(T, t0 + CHUNK)
            toks = np.arange(t0, t1, dtype=np.int32)
            rows = None
            if layer.indexer:
                ref = oracle_topk(case, toks)
                allowed = check_topk(case, idx_np[t0:t1], ref, tokens=toks)
                check_topk(case, val_idx[t0:t1], ref, tokens=toks, gpu_val=val_np[t0:t1])
                rows = ref[0].copy()
                for i in allowed:
                    rows[i] = idx_np[t0 + i]
                ties += len(allowed)
            ref_out, ref_lse = oracle_attention(case, rows, toks)
            o = out[t0:t1].float().cpu().double().numpy()
            assert np.isfinite(o).all(), f"{name} layer {li}: non-finite output"
            err = np.abs(o - ref_out)
            mx = max(mx, float(err.max()))
            tot += float(err.sum())
            cnt += err.size
            lmx = max(lmx, float(np.abs(lse_np[t0:t1] - ref_lse).max()))
        mean = tot / cnt
        REPORT.append(f"{name} layer {li} (r={layer.cmp_ratio}), all {T} tokens: out max|err| "
                      f"{mx:.3e} mean {mean:.3e}, lse max|err| {lmx:.3e}"
                      + (f", near-tie top-k rows {ties}" if layer.indexer else ""))
        assert mx <= OUT_MAX_ABS, f"{name} layer {li}: max abs err {mx:.3e}"
        assert mean <= OUT_MEAN_ABS, f"{name} layer {li}: mean abs err {mean:.3e}"
        assert lmx <= LSE_MAX_ABS, f"{name} layer {li}: lse max abs err {lmx:.3e}"
        del out, lse, idx, case
        torch.cuda.empty_cache()
