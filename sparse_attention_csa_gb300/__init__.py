"""GB300 (sm_103a) forward path of DeepSeek-V4 Compressed Sparse Attention
(THD, and BSND batches), the backward of its sparse MLA attention and the
indexer's KL-loss gradient.

Thin Python binding of the C ABI declared in ``include/csa.h`` (same call
names). It only marshals arguments: every step of the path runs in the CUDA
kernels of ``libcsa_gb300.so``; there is no CPU or PyTorch fallback, and a
call fails loudly when the library has not been built.

PyTorch supplies device memory and the current CUDA stream. All tensors are
CUDA tensors in THD layout, contiguous, with the dtypes ``include/csa.h``
states (bf16 activations, fp32 weights/sinks/outputs, int32 indices).
"""

from __future__ import annotations

import ctypes as C
import os

import torch

__all__ = [
    "CsaError", "lib", "library_path", "csa_status_string", "csa_compress_cu_seqlens",
    "csa_window_idx", "csa_indexer_topk_workspace_size", "csa_indexer_topk",
    "csa_sparse_mla_fwd", "csa_sparse_mla_bwd", "csa_device_error", "csa_indexer_topk_noalloc",
    "csa_indexer_kl_loss_grad", "csa_bsnd_mla_workspace_size", "csa_sparse_mla_fwd_bsnd",
    "csa_bsnd_indexer_workspace_size", "csa_indexer_topk_bsnd", "csa_compress_thd",
    "csa_set_wait_limit_ns", "csa_set_pair_select_rows", "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_build", "libcsa_gb300.so")

# Every entry point include/csa.h declares.
EXPORTED_SYMBOLS = (
    "csa_status_string", "csa_compress_cu_seqlens", "csa_window_idx",
    "csa_indexer_topk_workspace_size", "csa_indexer_topk", "csa_sparse_mla_fwd",
    "csa_sparse_mla_bwd", "csa_device_error", "csa_indexer_topk_noalloc",
    "csa_indexer_kl_loss_grad", "csa_bsnd_mla_workspace_size", "csa_sparse_mla_fwd_bsnd",
    "csa_bsnd_indexer_workspace_size", "csa_indexer_topk_bsnd", "csa_compress_thd",
    "csa_set_wait_limit_ns", "csa_set_pair_select_rows",
)

_STATUS = {0: "CSA_OK", 1: "CSA_ERR_NULL", 2: "CSA_ERR_SHAPE", 3: "CSA_ERR_UNSUPPORTED",
           4: "CSA_ERR_WORKSPACE", 5: "CSA_ERR_CUDA", 6: "CSA_ERR_DEVICE_CHECK",
           7: "CSA_ERR_TIMEOUT"}


class CsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {csa_status_string(code)}")


_lib = None
_vp, _i32, _sz, _f32 = C.c_void_p, C.c_int32, C.c_size_t, C.c_float


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = C.CDLL(library_path)
        L.csa_status_string.restype = C.c_char_p
        L.csa_status_string.argtypes = [C.c_int]
        L.csa_compress_cu_seqlens.argtypes = [_vp, _i32, _i32, _vp, _vp]
        L.csa_window_idx.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp]
        L.csa_indexer_topk_workspace_size.restype = _sz
        L.csa_indexer_topk_workspace_size.argtypes = [_i32] * 5
        L.csa_indexer_topk.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _i32, _i32,
                                       _i32, _vp, _vp, _vp, _sz, _vp]
        L.csa_sparse_mla_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                         _i32, _i32, _vp, _f32, _i32, _i32, _i32, _vp, _vp, _i32,
                                         _vp]
        L.csa_sparse_mla_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                         _i32, _i32, _i32, _i32, _i32, _vp, _f32, _i32, _i32,
                                         _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.csa_device_error.argtypes = [_vp, C.POINTER(_i32)]
        L.csa_indexer_topk_noalloc.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp,
                                               _i32, _i32, _i32, _vp, _vp, _vp]
        L.csa_indexer_kl_loss_grad.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                               _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _vp,
                                               _vp, _vp]
        L.csa_bsnd_mla_workspace_size.restype = _sz
        L.csa_bsnd_mla_workspace_size.argtypes = [_i32] * 3
        L.csa_sparse_mla_fwd_bsnd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                              _i32, _i32, _vp, _f32, _i32, _i32, _i32, _vp, _vp,
                                              _i32, _vp, _sz, _vp]
        L.csa_bsnd_indexer_workspace_size.restype = _sz
        L.csa_bsnd_indexer_workspace_size.argtypes = [_i32] * 6
        L.csa_indexer_topk_bsnd.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                            _i32, _i32, _vp, _vp, _vp, _sz, _vp]
        L.csa_compress_thd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                       _i32, _vp, _vp]
        L.csa_set_wait_limit_ns.argtypes = [C.c_uint64]
        L.csa_set_pair_select_rows.argtypes = [_i32]
        for name in ("csa_compress_cu_seqlens", "csa_window_idx", "csa_indexer_topk",
                     "csa_sparse_mla_fwd", "csa_sparse_mla_bwd", "csa_device_error",
                     "csa_indexer_topk_noalloc", "csa_indexer_kl_loss_grad",
                     "csa_sparse_mla_fwd_bsnd", "csa_indexer_topk_bsnd", "csa_compress_thd",
                     "csa_set_wait_limit_ns", "csa_set_pair_select_rows"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def csa_status_string(code: int) -> str:
    try:
        return lib().csa_status_string(int(code)).decode()
    except RuntimeError:
        return _STATUS.get(int(code), "unknown")


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name, dtype, ndim=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _check(rc, where):
    if rc != 0:
        raise CsaError(rc, where)


def csa_compress_cu_seqlens(cu_seqlens, cmp_ratio: int, out=None, stream=None):
    """cu_seqlens_cmp[b+1] = cu_seqlens_cmp[b] + floor(len_b / cmp_ratio)."""
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if out is None:
        out = torch.empty_like(cu_seqlens)
    _need(out, "out", torch.int32, 1)
    _check(lib().csa_compress_cu_seqlens(_ptr(cu_seqlens), cu_seqlens.numel() - 1, int(cmp_ratio),
                                         _ptr(out), _stream(stream)), "csa_compress_cu_seqlens")
    return out


def csa_window_idx(cu_seqlens, total_tokens: int, ori_win_left: int, ori_win_right: int = 0,
                   out=None, stream=None):
    """[T, ori_win_left+1] int32 window rows (stream-absolute, -1 padded)."""
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if out is None:
        out = torch.empty((total_tokens, ori_win_left + 1), dtype=torch.int32,
                          device=cu_seqlens.device)
    _need(out, "out", torch.int32, 2)
    _check(lib().csa_window_idx(_ptr(cu_seqlens), cu_seqlens.numel() - 1, int(total_tokens),
                                int(ori_win_left), int(ori_win_right), _ptr(out), _stream(stream)),
           "csa_window_idx")
    return out


def csa_indexer_topk_workspace_size(total_tokens, total_cmp, index_heads, index_dim, topk) -> int:
    return int(lib().csa_indexer_topk_workspace_size(int(total_tokens), int(total_cmp),
                                                     int(index_heads), int(index_dim), int(topk)))


def csa_indexer_topk(q, k, w, cu_seqlens_q, cu_seqlens_cmp_kv, cmp_ratio: int, topk: int,
                     return_value: bool = False, workspace=None, out=None, out_val=None,
                     stream=None):
    """Top-k compressed rows per token by lightning-indexer score.

    Returns ``(topk_idx [T, topk] int32, topk_val [T, topk] fp32 or None)``."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_cmp_kv, "cu_seqlens_cmp_kv", torch.int32, 1)
    T, Hi, Di = q.shape
    Tc = 0 if k is None else k.shape[0]
    if out is None:
        out = torch.empty((T, topk), dtype=torch.int32, device=q.device)
    if return_value and out_val is None:
        out_val = torch.empty((T, topk), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.int32, 2)
    _need(out_val, "out_val", torch.float32, 2)
    need = csa_indexer_topk_workspace_size(T, Tc, Hi, Di, topk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().csa_indexer_topk(
        _ptr(q), _ptr(k) if Tc else None, _ptr(w), T, Tc, Hi, Di, _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_cmp_kv), cu_seqlens_q.numel() - 1, int(cmp_ratio), int(topk), _ptr(out),
        _ptr(out_val) if return_value else None, _ptr(workspace), ws_bytes, _stream(stream)),
        "csa_indexer_topk")
    return out, (out_val if return_value else None)


def csa_indexer_topk_noalloc(q, k, w, cu_seqlens_q, cu_seqlens_cmp_kv, cmp_ratio: int,
                             topk: int, return_value: bool = False, out=None, out_val=None,
                             stream=None):
    """Same result as :func:`csa_indexer_topk`, for callers that cannot
    allocate device memory: no workspace, the library's own fixed 32 MiB
    scratch array instead (shared by every call; order calls on one stream)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_cmp_kv, "cu_seqlens_cmp_kv", torch.int32, 1)
    T, Hi, Di = q.shape
    Tc = 0 if k is None else k.shape[0]
    if out is None:
        out = torch.empty((T, topk), dtype=torch.int32, device=q.device)
    if return_value and out_val is None:
        out_val = torch.empty((T, topk), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.int32, 2)
    _need(out_val, "out_val", torch.float32, 2)
    _check(lib().csa_indexer_topk_noalloc(
        _ptr(q), _ptr(k) if Tc else None, _ptr(w), T, Tc, Hi, Di, _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_cmp_kv), cu_seqlens_q.numel() - 1, int(cmp_ratio), int(topk), _ptr(out),
        _ptr(out_val) if return_value else None, _stream(stream)), "csa_indexer_topk_noalloc")
    return out, (out_val if return_value else None)


def csa_sparse_mla_fwd(q, ori_kv, cmp_kv, cmp_sparse_indices, cu_seqlens_q, cu_seqlens_ori_kv,
                       cu_seqlens_cmp_kv, sinks, softmax_scale: float, cmp_ratio: int,
                       ori_win_left: int, ori_win_right: int = 0,
                       return_softmax_lse: bool = False, out=None, lse=None, stream=None):
    """Shared-KV MLA sparse attention with sinks.

    ``cmp_sparse_indices`` None attends every visible compressed row (HCA);
    ``cmp_kv`` None attends the window only. Returns ``(out, lse or None)``."""
    _need(q, "q", torch.bfloat16, 3)
    _need(ori_kv, "ori_kv", torch.bfloat16, 2)
    _need(cmp_kv, "cmp_kv", torch.bfloat16, 2)
    _need(cmp_sparse_indices, "cmp_sparse_indices", torch.int32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_ori_kv, "cu_seqlens_ori_kv", torch.int32, 1)
    _need(cu_seqlens_cmp_kv, "cu_seqlens_cmp_kv", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    T, H, D = q.shape
    Tc = 0 if cmp_kv is None else cmp_kv.shape[0]
    topk = 0 if cmp_sparse_indices is None else cmp_sparse_indices.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if return_softmax_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    _check(lib().csa_sparse_mla_fwd(
        _ptr(q), _ptr(ori_kv), _ptr(cmp_kv) if Tc else None, _ptr(cmp_sparse_indices),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_ori_kv), _ptr(cu_seqlens_cmp_kv),
        cu_seqlens_q.numel() - 1, T, Tc, H, D, topk, _ptr(sinks), float(softmax_scale),
        int(cmp_ratio), int(ori_win_left), int(ori_win_right), _ptr(out),
        _ptr(lse) if return_softmax_lse else None, 1 if return_softmax_lse else 0,
        _stream(stream)), "csa_sparse_mla_fwd")
    return out, (lse if return_softmax_lse else None)


def csa_sparse_mla_bwd(q, dout, out, lse, ori_kv, cmp_kv, cmp_sparse_indices, cu_seqlens_q,
                       cu_seqlens_ori_kv, cu_seqlens_cmp_kv, sinks, softmax_scale: float,
                       cmp_ratio: int, ori_win_left: int, ori_win_right: int = 0,
                       want_l1: bool = True, stream=None):
    """Backward of ``csa_sparse_mla_fwd`` from its ``out`` and ``lse``.

    Returns a dict of fp32 tensors: d_q [T,H,D], d_ori_kv [T,D], d_cmp_kv
    [Tc,D] (None without compressed rows), d_sinks [H] (None without sinks),
    ori_l1 [T, ori_win_left+1] and cmp_l1 [T, topk] (None without a top-k
    list, or both None when ``want_l1`` is false)."""
    for t, n, dt, nd in ((q, "q", torch.bfloat16, 3), (dout, "dout", torch.bfloat16, 3),
                         (out, "out", torch.bfloat16, 3), (lse, "lse", torch.float32, 2),
                         (ori_kv, "ori_kv", torch.bfloat16, 2), (cmp_kv, "cmp_kv", torch.bfloat16, 2),
                         (cmp_sparse_indices, "cmp_sparse_indices", torch.int32, 2),
                         (cu_seqlens_q, "cu_seqlens_q", torch.int32, 1),
                         (cu_seqlens_ori_kv, "cu_seqlens_ori_kv", torch.int32, 1),
                         (cu_seqlens_cmp_kv, "cu_seqlens_cmp_kv", torch.int32, 1),
                         (sinks, "sinks", torch.float32, 1)):
        _need(t, n, dt, nd)
    T, H, D = q.shape
    Tc = 0 if cmp_kv is None else cmp_kv.shape[0]
    topk = 0 if cmp_sparse_indices is None else cmp_sparse_indices.shape[1]
    f32 = dict(dtype=torch.float32, device=q.device)
    res = {
        "d_q": torch.empty((T, H, D), **f32),
        "d_ori_kv": torch.empty((T, D), **f32),
        "d_cmp_kv": torch.empty((Tc, D), **f32) if Tc else None,
        "d_sinks": torch.empty((H,), **f32) if sinks is not None else None,
        "ori_l1": torch.empty((T, ori_win_left + 1), **f32) if want_l1 else None,
        "cmp_l1": (torch.empty((T, topk), **f32)
                   if want_l1 and Tc and cmp_sparse_indices is not None else None),
    }
    _check(lib().csa_sparse_mla_bwd(
        _ptr(q), _ptr(dout), _ptr(out), _ptr(lse), _ptr(ori_kv), _ptr(cmp_kv) if Tc else None,
        _ptr(cmp_sparse_indices), _ptr(cu_seqlens_q), _ptr(cu_seqlens_ori_kv),
        _ptr(cu_seqlens_cmp_kv), cu_seqlens_q.numel() - 1, T, Tc, H, D, topk, _ptr(sinks),
        float(softmax_scale), int(cmp_ratio), int(ori_win_left), int(ori_win_right),
        _ptr(res["d_q"]), _ptr(res["d_ori_kv"]), _ptr(res["d_cmp_kv"]), _ptr(res["d_sinks"]),
        _ptr(res["ori_l1"]), _ptr(res["cmp_l1"]), _stream(stream)), "csa_sparse_mla_bwd")
    return res


def csa_indexer_kl_loss_grad(q, k, w, sparse_indices, attn_softmax_l1_norm, cu_seqlens_q,
                             cu_seqlens_cmp_kv, cmp_ratio: int, grad_scale: float = 1.0,
                             want_loss: bool = True, stream=None):
    """Indexer KL loss against the attention distribution, and its gradients.

    Returns a dict of fp32 tensors: d_q [T,Hi,Di], d_k [Tc,Di] (None when
    Tc == 0), d_w [T,Hi] and loss [T] (the unscaled KL per token; None unless
    ``want_loss``). The gradients are those of ``grad_scale * loss.sum()``."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(sparse_indices, "sparse_indices", torch.int32, 2)
    _need(attn_softmax_l1_norm, "attn_softmax_l1_norm", torch.float32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_cmp_kv, "cu_seqlens_cmp_kv", torch.int32, 1)
    T, Hi, Di = q.shape
    Tc = 0 if k is None else k.shape[0]
    topk = sparse_indices.shape[1]
    if tuple(attn_softmax_l1_norm.shape) != (T, topk) or sparse_indices.shape[0] != T:
        raise ValueError("sparse_indices and attn_softmax_l1_norm must both be [T, topk]")
    f32 = dict(dtype=torch.float32, device=q.device)
    res = {"d_q": torch.empty((T, Hi, Di), **f32),
           "d_k": torch.empty((Tc, Di), **f32) if Tc else None,
           "d_w": torch.empty((T, Hi), **f32),
           "loss": torch.empty((T,), **f32) if want_loss else None}
    _check(lib().csa_indexer_kl_loss_grad(
        _ptr(q), _ptr(k) if Tc else None, _ptr(w), _ptr(sparse_indices),
        _ptr(attn_softmax_l1_norm), T, Tc, Hi, Di, _ptr(cu_seqlens_q), _ptr(cu_seqlens_cmp_kv),
        cu_seqlens_q.numel() - 1, int(cmp_ratio), int(topk), float(grad_scale), _ptr(res["d_q"]),
        _ptr(res["d_k"]), _ptr(res["d_w"]), _ptr(res["loss"]), _stream(stream)),
        "csa_indexer_kl_loss_grad")
    return res


def _workspace(need, device, workspace):
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    size = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return workspace, size


def csa_sparse_mla_fwd_bsnd(q, ori_kv, cmp_kv, cmp_sparse_indices, seqused, sinks,
                            softmax_scale: float, cmp_ratio: int, ori_win_left: int,
                            ori_win_right: int = 0, return_softmax_lse: bool = False,
                            workspace=None, out=None, lse=None, stream=None):
    """Sparse MLA forward in BSND layout: q [B,S,H,D], ori_kv [B,S,D], cmp_kv
    [B,Sc,D] or None, cmp_sparse_indices [B,S,topk] batch-local or None,
    seqused [B] int32 or None. Returns ``(out [B,S,H,D], lse [B,S,H] or None)``;
    rows past seqused are unspecified."""
    _need(q, "q", torch.bfloat16, 4)
    _need(ori_kv, "ori_kv", torch.bfloat16, 3)
    _need(cmp_kv, "cmp_kv", torch.bfloat16, 3)
    _need(cmp_sparse_indices, "cmp_sparse_indices", torch.int32, 3)
    _need(seqused, "seqused", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    B, S, H, D = q.shape
    Sc = 0 if cmp_kv is None else cmp_kv.shape[1]
    topk = 0 if cmp_sparse_indices is None else cmp_sparse_indices.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if return_softmax_lse and lse is None:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    list_used = topk if Sc else 0
    need = int(lib().csa_bsnd_mla_workspace_size(B, S, list_used))
    workspace, ws_bytes = _workspace(need, q.device, workspace)
    _check(lib().csa_sparse_mla_fwd_bsnd(
        _ptr(q), _ptr(ori_kv), _ptr(cmp_kv) if Sc else None, _ptr(cmp_sparse_indices),
        _ptr(seqused), B, S, Sc, H, D, topk, _ptr(sinks), float(softmax_scale), int(cmp_ratio),
        int(ori_win_left), int(ori_win_right), _ptr(out),
        _ptr(lse) if return_softmax_lse else None, 1 if return_softmax_lse else 0,
        _ptr(workspace), ws_bytes, _stream(stream)), "csa_sparse_mla_fwd_bsnd")
    return out, (lse if return_softmax_lse else None)


def csa_indexer_topk_bsnd(q, k, w, seqused, cmp_ratio: int, topk: int,
                          return_value: bool = False, workspace=None, out=None, out_val=None,
                          stream=None):
    """Lightning-indexer top-k in BSND layout: q [B,S,Hi,Di], k [B,Sc,Di],
    w [B,S,Hi], seqused [B] int32 or None. Returns ``(topk_idx [B,S,topk]
    batch-local rows, topk_val or None)``; rows past seqused are unspecified."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 3)
    _need(w, "w", torch.float32, 3)
    _need(seqused, "seqused", torch.int32, 1)
    B, S, Hi, Di = q.shape
    Sc = 0 if k is None else k.shape[1]
    if out is None:
        out = torch.empty((B, S, topk), dtype=torch.int32, device=q.device)
    if return_value and out_val is None:
        out_val = torch.empty((B, S, topk), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.int32, 3)
    _need(out_val, "out_val", torch.float32, 3)
    need = int(lib().csa_bsnd_indexer_workspace_size(B, S, Sc, Hi, Di, int(topk)))
    workspace, ws_bytes = _workspace(need, q.device, workspace)
    _check(lib().csa_indexer_topk_bsnd(
        _ptr(q), _ptr(k) if Sc else None, _ptr(w), _ptr(seqused), B, S, Sc, Hi, Di,
        int(cmp_ratio), int(topk), _ptr(out), _ptr(out_val) if return_value else None,
        _ptr(workspace), ws_bytes, _stream(stream)), "csa_indexer_topk_bsnd")
    return out, (out_val if return_value else None)


def csa_compress_thd(kv, score, ape, cu_seqlens, cu_seqlens_cmp, total_cmp: int,
                     cmp_ratio: int, head_dim: int, overlap: bool = True, out=None, stream=None):
    """Compressed rows [total_cmp, head_dim] fp32 from the projections kv and
    score [T, Wd] fp32 (Wd = 2 head_dim with overlap) and ape [cmp_ratio, Wd]
    or None: per-sequence groups, overlap transform, softmax pooling over
    the slots. ``total_cmp`` is cu_seqlens_cmp's last entry (a host int)."""
    _need(kv, "kv", torch.float32, 2)
    _need(score, "score", torch.float32, 2)
    _need(ape, "ape", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(cu_seqlens_cmp, "cu_seqlens_cmp", torch.int32, 1)
    T, wd = kv.shape
    if tuple(score.shape) != (T, wd) or wd != (2 * head_dim if overlap else head_dim):
        raise ValueError("kv and score must both be [T, 2*head_dim] (overlap) or [T, head_dim]")
    if out is None:
        out = torch.empty((total_cmp, head_dim), dtype=torch.float32, device=kv.device)
    _need(out, "out", torch.float32, 2)
    _check(lib().csa_compress_thd(
        _ptr(kv), _ptr(score), _ptr(ape), _ptr(cu_seqlens), _ptr(cu_seqlens_cmp),
        cu_seqlens.numel() - 1, T, int(total_cmp), int(cmp_ratio), int(head_dim),
        1 if overlap else 0, _ptr(out), _stream(stream)), "csa_compress_thd")
    return out


def csa_device_error(stream=None):
    """Synchronise the stream; return (status, raw word) of the device error word."""
    detail = _i32(0)
    rc = lib().csa_device_error(_stream(stream), C.byref(detail))
    return int(rc), int(detail.value)


def csa_set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of the indexer and sparse-attention kernels' pipeline waits, in
    ns (0: the default 2 s). A wait that gives up records CSA_ERR_TIMEOUT in
    the device error word; for testing the timeout path."""
    _check(lib().csa_set_wait_limit_ns(int(limit_ns)), "csa_set_wait_limit_ns")


def csa_set_pair_select_rows(rows: int) -> None:
    """Rows above which the indexer selects a token's top-k with one warp
    instead of two (0: the default bound); for testing the one-warp path."""
    _check(lib().csa_set_pair_select_rows(int(rows)), "csa_set_pair_select_rows")
