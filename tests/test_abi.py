"""C-ABI checks that need no GPU: the library loads, exports every entry point
the header declares, and rejects bad host-side arguments before touching the
device. Also checks that the product never reaches into the oracle."""

import ctypes as C
import os
import re

import pytest

import sparse_attention_csa_gb300 as csa
from sparse_attention_csa_gb300 import build as csa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def L():
    csa_build.build()
    return csa.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(csa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_library_exports_nothing_undeclared(L):
    """Every csa_* symbol the shared library exports is an entry point of the
    header (no internal launcher leaks into the ABI)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    res = subprocess.run([nm, "-D", "--defined-only", csa.library_path], capture_output=True,
                         text=True, check=True)
    exported = sorted({ln.split()[-1] for ln in res.stdout.splitlines()
                       if ln.split() and ln.split()[-1].startswith("csa_")})
    assert exported == declared_symbols()


def test_status_strings(L):
    for code, name in [(0, "CSA_OK"), (1, "CSA_ERR_NULL"), (3, "CSA_ERR_UNSUPPORTED"),
                       (7, "CSA_ERR_TIMEOUT")]:
        assert csa.csa_status_string(code).startswith(name)
    assert csa.csa_status_string(99) == "unknown csa_status_t"


# Synchronous checks return before any CUDA call, so they run without a GPU.
# Dummy non-null "device pointers" are never dereferenced on these paths:
# every call below carries at least one invalid argument, so none launches.
P = C.c_void_p(0x1000)
NUL = None


def test_compress_rejects(L):
    assert L.csa_compress_cu_seqlens(NUL, 3, 4, P, NUL) == 1
    assert L.csa_compress_cu_seqlens(P, -1, 4, P, NUL) == 2
    assert L.csa_compress_cu_seqlens(P, 3, 0, P, NUL) == 3


def test_window_rejects(L):
    assert L.csa_window_idx(P, 3, 256, 15, 0, NUL, NUL) == 1
    assert L.csa_window_idx(P, 3, -5, 15, 0, P, NUL) == 2
    assert L.csa_window_idx(P, 3, 256, -1, 0, P, NUL) == 2
    assert L.csa_window_idx(P, 3, 256, 15, 1, P, NUL) == 3


def test_indexer_rejects(L):
    args = [P, P, P, 256, 63, 4, 64, P, P, 3, 4, 8, P, NUL, NUL, 0, NUL]

    def call(**kw):
        a = list(args)
        names = ["q", "k", "w", "T", "Tc", "Hi", "Di", "cu", "cuc", "batch", "r", "topk", "idx",
                 "val", "ws", "wsb", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return L.csa_indexer_topk(*a)

    assert call(q=NUL) == 1
    assert call(k=NUL) == 1
    assert call(idx=NUL) == 1
    assert call(topk=0) == 2
    assert call(T=-1) == 2
    assert call(Di=96) == 3
    assert call(Hi=65) == 3
    assert call(r=1) == 3
    need = L.csa_indexer_topk_workspace_size(4096, 10 ** 6, 64, 128, 512)
    assert need > 0
    assert call(T=4096, Tc=10 ** 6, Hi=64, Di=128, topk=512) == 4
    assert call(T=4096, Tc=10 ** 6, Hi=64, Di=128, topk=512, ws=C.c_void_p(0x1001),
                wsb=need) == 4  # misaligned


def test_mla_rejects(L):
    names = ["q", "okv", "ckv", "idx", "cuq", "cuo", "cuc", "batch", "T", "Tc", "H", "D", "topk",
             "sinks", "scale", "r", "wl", "wr", "out", "lse", "ret", "stream"]
    base = dict(q=P, okv=P, ckv=P, idx=P, cuq=P, cuo=NUL, cuc=P, batch=3, T=256, Tc=63, H=4, D=512,
                topk=8, sinks=P, scale=C.c_float(0.044), r=4, wl=15, wr=0, out=P, lse=P, ret=1,
                stream=NUL)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return L.csa_sparse_mla_fwd(*[a[n] for n in names])

    assert call(q=NUL) == 1
    assert call(out=NUL) == 1
    assert call(lse=NUL) == 1
    assert call(cuc=NUL) == 1
    assert call(H=0) == 2
    assert call(topk=0) == 2
    assert call(D=576) == 3
    assert call(H=65) == 3
    assert call(wr=1) == 3
    assert call(wl=1024) == 3
    assert call(r=1) == 3
    assert call(cuo=C.c_void_p(0x2000)) == 3  # prefix-KV cu_seqlens
    assert call(topk=1025) == 3  # beyond the per-token index list
    assert call(q=C.c_void_p(0x1002)) == 3  # 16-byte alignment


def test_mla_bwd_rejects(L):
    names = ["q", "dout", "out", "lse", "okv", "ckv", "idx", "cuq", "cuo", "cuc", "batch", "T",
             "Tc", "H", "D", "topk", "sinks", "scale", "r", "wl", "wr", "dq", "dokv", "dckv",
             "dsinks", "ol1", "cl1", "stream"]
    base = dict(q=P, dout=P, out=P, lse=P, okv=P, ckv=P, idx=P, cuq=P, cuo=NUL, cuc=P, batch=3,
                T=256, Tc=63, H=4, D=512, topk=8, sinks=P, scale=C.c_float(0.044), r=4, wl=15,
                wr=0, dq=P, dokv=P, dckv=P, dsinks=P, ol1=P, cl1=P, stream=NUL)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return L.csa_sparse_mla_bwd(*[a[n] for n in names])

    for k in ("q", "dout", "out", "lse", "okv", "cuq", "dq", "dokv", "cuc", "dckv"):
        assert call(**{k: NUL}) == 1, k
    assert call(H=0) == 2
    assert call(T=-3) == 2
    assert call(topk=0) == 2
    assert call(D=576) == 3
    assert call(H=65) == 3
    assert call(wr=1) == 3
    assert call(wl=1024) == 3
    assert call(r=1) == 3
    assert call(cuo=C.c_void_p(0x2000)) == 3  # prefix-KV cu_seqlens
    assert call(topk=1025) == 3
    assert call(dout=C.c_void_p(0x1008)) == 3  # 16-byte alignment
    assert call(dokv=C.c_void_p(0x1004)) == 3


def test_indexer_kl_rejects(L):
    names = ["q", "k", "w", "idx", "l1", "T", "Tc", "Hi", "Di", "cuq", "cuc", "batch", "r",
             "topk", "gs", "dq", "dk", "dw", "loss", "stream"]
    base = dict(q=P, k=P, w=P, idx=P, l1=P, T=256, Tc=63, Hi=4, Di=64, cuq=P, cuc=P, batch=3,
                r=4, topk=8, gs=C.c_float(1.0 / 256), dq=P, dk=P, dw=P, loss=P, stream=NUL)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return L.csa_indexer_kl_loss_grad(*[a[n] for n in names])

    for k in ("q", "k", "w", "idx", "l1", "cuq", "cuc", "dq", "dk", "dw"):
        assert call(**{k: NUL}) == 1, k
    assert call(T=-1) == 2
    assert call(Tc=-1) == 2
    assert call(topk=0) == 2
    assert call(Di=96) == 3
    assert call(Hi=0) == 3
    assert call(Hi=65) == 3
    assert call(r=1) == 3
    assert call(topk=2049) == 3
    assert call(q=C.c_void_p(0x1002)) == 3  # 16-byte alignment
    assert call(dk=C.c_void_p(0x1004)) == 3
    assert call(T=0) == 0  # nothing to do, nothing launched


def test_bsnd_rejects(L):
    names = ["q", "okv", "ckv", "idx", "su", "B", "S", "Sc", "H", "D", "topk", "sinks", "scale",
             "r", "wl", "wr", "out", "lse", "ret", "ws", "wsb", "stream"]
    need = L.csa_bsnd_mla_workspace_size(3, 200, 16)
    assert need >= 3 * 200 * 16 * 4
    assert L.csa_bsnd_mla_workspace_size(3, 200, 0) < need
    base = dict(q=P, okv=P, ckv=P, idx=P, su=NUL, B=3, S=200, Sc=50, H=8, D=512, topk=16,
                sinks=P, scale=C.c_float(0.044), r=4, wl=31, wr=0, out=P, lse=P, ret=1,
                ws=C.c_void_p(0x10000), wsb=need, stream=NUL)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return L.csa_sparse_mla_fwd_bsnd(*[a[n] for n in names])

    for k in ("q", "okv", "out", "lse"):
        assert call(**{k: NUL}) == 1, k
    assert call(B=-1) == 2
    assert call(topk=0) == 2
    assert call(B=1 << 16, S=1 << 16) == 2  # B*S beyond int32
    assert call(D=576) == 3
    assert call(H=65) == 3
    assert call(r=1) == 3
    assert call(wr=1) == 3
    assert call(q=C.c_void_p(0x1002)) == 3
    assert call(wsb=need - 1) == 4
    assert call(ws=C.c_void_p(0x10010)) == 4  # misaligned
    assert call(ws=NUL) == 4
    assert call(S=0) == 0  # nothing to do
    # indexer
    inames = ["q", "k", "w", "su", "B", "S", "Sc", "Hi", "Di", "r", "topk", "idx", "val", "ws",
              "wsb", "stream"]
    ineed = L.csa_bsnd_indexer_workspace_size(3, 200, 50, 8, 64, 16)
    assert ineed > 0
    ibase = dict(q=P, k=P, w=P, su=NUL, B=3, S=200, Sc=50, Hi=8, Di=64, r=4, topk=16, idx=P,
                 val=NUL, ws=C.c_void_p(0x10000), wsb=ineed, stream=NUL)

    def icall(**kw):
        a = dict(ibase)
        a.update(kw)
        return L.csa_indexer_topk_bsnd(*[a[n] for n in inames])

    for k in ("q", "k", "w", "idx"):
        assert icall(**{k: NUL}) == 1, k
    assert icall(topk=0) == 2
    assert icall(Sc=-1) == 2
    assert icall(Di=96) == 3
    assert icall(Hi=65) == 3
    assert icall(r=1) == 3
    assert icall(wsb=ineed - 1) == 4
    assert icall(B=0) == 0


def test_compress_thd_rejects(L):
    names = ["kv", "score", "ape", "cu", "cuc", "batch", "T", "Tc", "r", "hd", "ov", "out",
             "stream"]
    base = dict(kv=P, score=P, ape=NUL, cu=P, cuc=P, batch=3, T=256, Tc=63, r=4, hd=512, ov=1,
                out=P, stream=NUL)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return L.csa_compress_thd(*[a[n] for n in names])

    for k in ("kv", "score", "cu", "cuc", "out"):
        assert call(**{k: NUL}) == 1, k
    assert call(T=-1) == 2
    assert call(hd=0) == 2
    assert call(Tc=65) == 2  # 65 groups of 4 need more than 256 rows
    assert call(r=0) == 3
    assert call(hd=65537) == 3
    assert call(Tc=0) == 0  # nothing to pool


def test_controls(L):
    """The host-only controls: a negative selection bound is rejected; 0
    restores the defaults."""
    assert L.csa_set_pair_select_rows(-1) == 2
    assert L.csa_set_pair_select_rows(256) == 0
    assert L.csa_set_pair_select_rows(0) == 0
    assert L.csa_set_wait_limit_ns(0) == 0


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_csa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
                assert "csa_oracle" not in text and "csa_ref_" not in text, f


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(csa, "_lib", None)
    monkeypatch.setattr(csa, "library_path", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        csa.lib()
