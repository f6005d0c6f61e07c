"""fp64 CPU oracle for the CSA forward path.

TEST INFRASTRUCTURE ONLY. Importers allowed: the test suite, the smoke check
in ``__graft_entry__`` and the benchmark's CPU-baseline / reference leg.
The product (``sparse_attention_csa_gb300``) never imports this package, and
the two share no code.

``oracle/csa_oracle.c`` holds the arithmetic (plain loops, double precision,
one function per step of the path); this module only marshals NumPy arrays
into it. ``oracle/dense_ref.py`` is a second, independent NumPy restatement
(dense masked attention) used to pin the C code on tiny packs.
"""

from __future__ import annotations

import ctypes as C

import numpy as np

from .build import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build())
        i32p = C.POINTER(C.c_int32)
        f64p = C.POINTER(C.c_double)
        i32 = C.c_int32
        _lib.csa_ref_num_threads.restype = C.c_int
        _lib.csa_ref_set_num_threads.argtypes = [C.c_int]
        _lib.csa_ref_set_num_threads.restype = None
        _lib.csa_ref_compress_cu_seqlens.argtypes = [i32p, i32, i32, i32p]
        _lib.csa_ref_window_idx.argtypes = [i32p, i32, i32, i32, i32p]
        _lib.csa_ref_window_idx_tokens.argtypes = [i32p, i32, i32, i32, i32p, i32, i32p]
        _lib.csa_ref_indexer_topk.argtypes = [
            f64p, f64p, f64p, i32, i32, i32, i32, i32p, i32p, i32, i32, i32, i32p, i32,
            i32p, f64p, f64p, f64p, i32p]
        _lib.csa_ref_sparse_mla_fwd.argtypes = [
            f64p, f64p, f64p, i32p, i32p, i32p, i32, i32, i32, i32, i32, i32, f64p, C.c_double,
            i32, i32, i32p, i32, f64p, f64p]
        _lib.csa_ref_sparse_mla_bwd.argtypes = [
            f64p, f64p, f64p, f64p, i32p, i32p, i32p, i32, i32, i32, i32, i32, i32, f64p,
            C.c_double, i32, i32, f64p, f64p, f64p, f64p, f64p, f64p]
        _lib.csa_ref_indexer_kl_loss_grad.argtypes = [
            f64p, f64p, f64p, i32p, f64p, i32, i32, i32, i32, i32, i32p, i32p, i32, i32,
            C.c_double, i32p, i32, f64p, f64p, f64p, f64p, f64p]
        _lib.csa_ref_compress_thd.argtypes = [
            f64p, f64p, f64p, i32p, i32p, i32, i32, i32, i32, i32, f64p]
        for name in ("csa_ref_compress_cu_seqlens", "csa_ref_window_idx", "csa_ref_window_idx_tokens",
                     "csa_ref_indexer_topk", "csa_ref_sparse_mla_fwd", "csa_ref_sparse_mla_bwd",
                     "csa_ref_indexer_kl_loss_grad", "csa_ref_compress_thd"):
            getattr(_lib, name).restype = C.c_int
    return _lib


def _p(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(C.POINTER(ctype))


def _i32(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (bf16/fp32 widen exactly)
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (code {rc})")


def num_threads() -> int:
    return int(lib().csa_ref_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (n < 1: one per
    processor)."""
    lib().csa_ref_set_num_threads(int(n))


def compress_cu_seqlens(cu_seqlens, cmp_ratio: int) -> np.ndarray:
    cu = _i32(cu_seqlens)
    out = np.zeros_like(cu)
    _check(lib().csa_ref_compress_cu_seqlens(_p(cu, C.c_int32), len(cu) - 1, cmp_ratio,
                                             _p(out, C.c_int32)), "compress_cu_seqlens")
    return out


def window_idx(cu_seqlens, total_tokens: int, ori_win_left: int, tokens=None) -> np.ndarray:
    """Window rows of every token ([T, W]), or of the listed tokens only."""
    cu = _i32(cu_seqlens)
    if tokens is not None:
        tok = _i32(tokens)
        out = np.zeros((len(tok), ori_win_left + 1), dtype=np.int32)
        _check(lib().csa_ref_window_idx_tokens(_p(cu, C.c_int32), len(cu) - 1, total_tokens,
                                               ori_win_left, _p(tok, C.c_int32), len(tok),
                                               _p(out, C.c_int32)), "window_idx")
        return out
    out = np.zeros((total_tokens, ori_win_left + 1), dtype=np.int32)
    _check(lib().csa_ref_window_idx(_p(cu, C.c_int32), len(cu) - 1, total_tokens, ori_win_left,
                                    _p(out, C.c_int32)), "window_idx")
    return out


def indexer_topk(q_rows, k, w_rows, total_tokens: int, cu_seqlens, cu_seqlens_cmp,
                 cmp_ratio: int, topk: int, tokens=None):
    """Top-k for the listed tokens. ``q_rows``/``w_rows`` hold one row per listed
    token (all tokens when ``tokens`` is None). Returns (idx, val, kth, next, n_vis)."""
    q = _f64(q_rows)
    w = _f64(w_rows)
    kk = _f64(k)
    cu, cuc = _i32(cu_seqlens), _i32(cu_seqlens_cmp)
    tok = _i32(tokens)
    n = q.shape[0]
    hi, di = q.shape[1], q.shape[2]
    tc = 0 if kk is None else kk.shape[0]
    if kk is not None and kk.size == 0:
        kk = None
    idx = np.zeros((n, topk), dtype=np.int32)
    val = np.zeros((n, topk), dtype=np.float64)
    kth = np.zeros(n, dtype=np.float64)
    nxt = np.zeros(n, dtype=np.float64)
    nvis = np.zeros(n, dtype=np.int32)
    _check(lib().csa_ref_indexer_topk(
        _p(q, C.c_double), _p(kk, C.c_double), _p(w, C.c_double), total_tokens, tc, hi, di,
        _p(cu, C.c_int32), _p(cuc, C.c_int32), len(cu) - 1, cmp_ratio, topk,
        _p(tok, C.c_int32), n, _p(idx, C.c_int32), _p(val, C.c_double), _p(kth, C.c_double),
        _p(nxt, C.c_double), _p(nvis, C.c_int32)), "indexer_topk")
    return idx, val, kth, nxt, nvis


def sparse_mla_fwd(q_rows, ori_kv, cmp_kv, cmp_sparse_indices, cu_seqlens, cu_seqlens_cmp,
                   total_tokens: int, sinks, softmax_scale: float, cmp_ratio: int,
                   ori_win_left: int, tokens=None):
    """Attention output (fp64) and LSE for the listed tokens. ``q_rows`` and
    ``cmp_sparse_indices`` hold one row per listed token; ``cmp_sparse_indices``
    None means every visible compressed block (compressor-only mode)."""
    q = _f64(q_rows)
    okv = _f64(ori_kv)
    ckv = _f64(cmp_kv)
    if ckv is not None and ckv.size == 0:
        ckv = None
    idx = _i32(cmp_sparse_indices)
    topk = 0 if idx is None else idx.shape[1]
    cu = _i32(cu_seqlens)
    cuc = _i32(cu_seqlens_cmp)
    sk = _f64(sinks)
    tok = _i32(tokens)
    n, h, d = q.shape
    tc = 0 if ckv is None else ckv.shape[0]
    out = np.zeros((n, h, d), dtype=np.float64)
    lse = np.zeros((n, h), dtype=np.float64)
    _check(lib().csa_ref_sparse_mla_fwd(
        _p(q, C.c_double), _p(okv, C.c_double), _p(ckv, C.c_double), _p(idx, C.c_int32),
        _p(cu, C.c_int32), _p(cuc, C.c_int32), len(cu) - 1, total_tokens, tc, h, d, topk,
        _p(sk, C.c_double), float(softmax_scale), cmp_ratio, ori_win_left, _p(tok, C.c_int32), n,
        _p(out, C.c_double), _p(lse, C.c_double)), "sparse_mla_fwd")
    return out, lse


def sparse_mla_bwd(q, dout, ori_kv, cmp_kv, cmp_sparse_indices, cu_seqlens, cu_seqlens_cmp,
                   sinks, softmax_scale: float, cmp_ratio: int, ori_win_left: int):
    """Gradients of sum(dout * out) for the whole pack, in fp64, and the
    head-averaged attention distributions. Returns a dict with d_q [T,H,D],
    d_ori_kv [T,D], d_cmp_kv [Tc,D] (None without compressed rows), d_sinks
    [H] (None without sinks), ori_l1 [T,W] and cmp_l1 [T,topk] (None without
    top-k indices)."""
    qq = _f64(q)
    g = _f64(dout)
    okv = _f64(ori_kv)
    ckv = _f64(cmp_kv)
    if ckv is not None and ckv.size == 0:
        ckv = None
    idx = _i32(cmp_sparse_indices) if ckv is not None else None
    topk = 0 if idx is None else idx.shape[1]
    cu = _i32(cu_seqlens)
    cuc = _i32(cu_seqlens_cmp)
    sk = _f64(sinks)
    t, h, d = qq.shape
    tc = 0 if ckv is None else ckv.shape[0]
    w = ori_win_left + 1
    res = {
        "d_q": np.zeros((t, h, d)),
        "d_ori_kv": np.zeros((t, d)),
        "d_cmp_kv": None if ckv is None else np.zeros((tc, d)),
        "d_sinks": None if sk is None else np.zeros(h),
        "ori_l1": np.zeros((t, w)),
        "cmp_l1": None if idx is None else np.zeros((t, topk)),
    }
    _check(lib().csa_ref_sparse_mla_bwd(
        _p(qq, C.c_double), _p(g, C.c_double), _p(okv, C.c_double), _p(ckv, C.c_double),
        _p(idx, C.c_int32), _p(cu, C.c_int32), _p(cuc, C.c_int32), len(cu) - 1, t, tc, h, d,
        topk, _p(sk, C.c_double), float(softmax_scale), cmp_ratio, ori_win_left,
        _p(res["d_q"], C.c_double), _p(res["d_ori_kv"], C.c_double),
        _p(res["d_cmp_kv"], C.c_double), _p(res["d_sinks"], C.c_double),
        _p(res["ori_l1"], C.c_double), _p(res["cmp_l1"], C.c_double)), "sparse_mla_bwd")
    return res


def indexer_kl_loss_grad(q_rows, k, w_rows, sparse_indices, attn_l1, total_tokens: int,
                         cu_seqlens, cu_seqlens_cmp, cmp_ratio: int, grad_scale: float = 1.0,
                         tokens=None, want_dk: bool = True):
    """KL loss of the indexer against the attention distribution, and its
    gradients, in fp64. ``q_rows``, ``w_rows``, ``sparse_indices`` and
    ``attn_l1`` hold one row per listed token (all tokens when ``tokens`` is
    None). Returns a dict: loss [n], d_q [n,Hi,Di], d_w [n,Hi], d_k [Tc,Di]
    (the listed tokens' contributions; None unless ``want_dk``) and g [n,topk]
    (dL/dI per list entry, zero where the entry is skipped)."""
    q = _f64(q_rows)
    w = _f64(w_rows)
    kk = _f64(k)
    a = _f64(attn_l1)
    idx = _i32(sparse_indices)
    cu, cuc = _i32(cu_seqlens), _i32(cu_seqlens_cmp)
    tok = _i32(tokens)
    n, hi, di = q.shape
    topk = idx.shape[1]
    tc = 0 if kk is None else kk.shape[0]
    if kk is not None and kk.size == 0:
        kk = None
    res = {"loss": np.zeros(n), "d_q": np.zeros((n, hi, di)), "d_w": np.zeros((n, hi)),
           "d_k": np.zeros((tc, di)) if want_dk else None, "g": np.zeros((n, topk))}
    _check(lib().csa_ref_indexer_kl_loss_grad(
        _p(q, C.c_double), _p(kk, C.c_double), _p(w, C.c_double), _p(idx, C.c_int32),
        _p(a, C.c_double), total_tokens, tc, hi, di, topk, _p(cu, C.c_int32),
        _p(cuc, C.c_int32), len(cu) - 1, cmp_ratio, float(grad_scale), _p(tok, C.c_int32), n,
        _p(res["d_q"], C.c_double), _p(res["d_k"], C.c_double), _p(res["d_w"], C.c_double),
        _p(res["loss"], C.c_double), _p(res["g"], C.c_double)), "indexer_kl_loss_grad")
    return res


def compress_thd(kv, score, ape, cu_seqlens, cmp_ratio: int, head_dim: int, overlap: bool):
    """THD compressor core in fp64: grouping, ape, overlap transform and
    softmax pooling over the slots. kv/score [T, Wd] (Wd = 2 head_dim with
    overlap), ape [cmp_ratio, Wd] or None. Returns [Tc, head_dim]."""
    k = _f64(kv)
    s = _f64(score)
    a = _f64(ape)
    cu = _i32(cu_seqlens)
    cuc = compress_cu_seqlens(cu, cmp_ratio)
    out = np.zeros((int(cuc[-1]), head_dim))
    _check(lib().csa_ref_compress_thd(
        _p(k, C.c_double), _p(s, C.c_double), _p(a, C.c_double), _p(cu, C.c_int32),
        _p(cuc, C.c_int32), len(cu) - 1, int(cu[-1]), cmp_ratio, head_dim, 1 if overlap else 0,
        _p(out, C.c_double)), "compress_thd")
    return out
