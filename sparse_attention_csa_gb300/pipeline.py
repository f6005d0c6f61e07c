"""One CSA / HCA attention layer forward, chaining the four C-ABI calls.

Order of the path (miles PR 2038 report, the attention forward excerpt:
compressed cu_seqlens, then the indexer, then sparse attention over the window
rows plus the selected compressed rows):

1. ``csa_compress_cu_seqlens``  compressed cu_seqlens of the pack;
2. ``csa_window_idx``           the window rows (returned for the caller; the
                                attention kernel derives the band itself);
3. ``csa_indexer_topk``         top-k compressed rows (INDEXER layers only);
4. ``csa_sparse_mla_fwd``       attention with sinks (COMPRESSOR_ONLY layers
                                attend every visible compressed row).

Everything runs on the current CUDA stream (the window rows optionally on a
side stream, joined before returning); nothing synchronises.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (csa_compress_cu_seqlens, csa_indexer_topk, csa_indexer_topk_workspace_size,
               csa_sparse_mla_fwd, csa_window_idx)


@dataclass
class LayerOutputs:
    out: torch.Tensor                 # [T, H, 512] bf16
    lse: torch.Tensor | None          # [T, H] fp32
    topk_idx: torch.Tensor | None     # [T, topk] int32 (INDEXER layers)
    window_idx: torch.Tensor | None   # [T, W] int32
    cu_seqlens_cmp: torch.Tensor      # [batch+1] int32


def allocate_outputs(T, H, D, W, topk, batch, device, with_window=True, with_lse=True):
    """Preallocated outputs for repeated calls (benchmarks, CUDA graphs)."""
    return LayerOutputs(
        out=torch.empty((T, H, D), dtype=torch.bfloat16, device=device),
        lse=torch.empty((T, H), dtype=torch.float32, device=device) if with_lse else None,
        topk_idx=torch.empty((T, topk), dtype=torch.int32, device=device) if topk else None,
        window_idx=torch.empty((T, W), dtype=torch.int32, device=device) if with_window else None,
        cu_seqlens_cmp=torch.empty((batch + 1,), dtype=torch.int32, device=device),
    )


def csa_layer_forward(q, ori_kv, cmp_kv, cu_seqlens, sinks, softmax_scale: float, cmp_ratio: int,
                      ori_win_left: int, q_idx=None, k_idx=None, w=None, topk: int = 0,
                      return_softmax_lse: bool = True, with_window: bool = True,
                      outputs: LayerOutputs | None = None, workspace=None,
                      window_stream=None) -> LayerOutputs:
    """Forward of one layer. ``q_idx``/``k_idx``/``w``/``topk`` given -> INDEXER
    layer (CSA); omitted -> COMPRESSOR_ONLY layer (HCA, every visible block).
    ``cmp_kv`` must hold exactly the pack's compressed row count.
    ``window_stream`` (a CUDA stream): the window rows, which nothing else of
    the layer reads, are computed there, beside the indexer, and the current
    stream waits for them before returning."""
    T, H, D = q.shape
    batch = cu_seqlens.numel() - 1
    indexer = q_idx is not None
    if outputs is None:
        outputs = allocate_outputs(T, H, D, ori_win_left + 1, topk if indexer else 0, batch,
                                   q.device, with_window, return_softmax_lse)
    csa_compress_cu_seqlens(cu_seqlens, cmp_ratio, out=outputs.cu_seqlens_cmp)
    main = torch.cuda.current_stream()
    win_done = None
    if with_window:
        if window_stream is None:
            csa_window_idx(cu_seqlens, T, ori_win_left, 0, out=outputs.window_idx)
        else:
            window_stream.wait_stream(main)
            csa_window_idx(cu_seqlens, T, ori_win_left, 0, out=outputs.window_idx,
                           stream=window_stream)
            win_done = torch.cuda.Event()
            win_done.record(window_stream)
    idx = None
    if indexer:
        if workspace is None:
            need = csa_indexer_topk_workspace_size(T, k_idx.shape[0], q_idx.shape[1],
                                                   q_idx.shape[2], topk)
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
        idx, _ = csa_indexer_topk(q_idx, k_idx, w, cu_seqlens, outputs.cu_seqlens_cmp, cmp_ratio,
                                  topk, workspace=workspace, out=outputs.topk_idx)
    csa_sparse_mla_fwd(q, ori_kv, cmp_kv, idx, cu_seqlens, cu_seqlens, outputs.cu_seqlens_cmp,
                       sinks, softmax_scale, cmp_ratio, ori_win_left, 0, return_softmax_lse,
                       out=outputs.out, lse=outputs.lse)
    if win_done is not None:
        main.wait_event(win_done)
    return outputs
