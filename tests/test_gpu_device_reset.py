"""A device reset while the library is loaded: the next calls look the
library's device addresses (the error word) up again for the new context.

Runs in a child process that drives the C ABI through ctypes with the CUDA
runtime's own allocator (no PyTorch state to invalidate): compressed
cu_seqlens on a small pack, the device error word, cudaDeviceReset, then the
same again, checked against the oracle's offsets."""

import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle
from sparse_attention_csa_gb300 import build as csa_build

pytestmark = pytest.mark.gpu

CHILD = textwrap.dedent('''
    import ctypes as C, sys
    import numpy as np
    lib = C.CDLL(sys.argv[1])
    rt = C.CDLL("libcudart.so.13")
    vp = C.c_void_p
    rt.cudaMalloc.argtypes = [C.POINTER(vp), C.c_size_t]
    rt.cudaMemcpy.argtypes = [vp, vp, C.c_size_t, C.c_int]
    rt.cudaFree.argtypes = [vp]
    lib.csa_compress_cu_seqlens.argtypes = [vp, C.c_int32, C.c_int32, vp, vp]
    lib.csa_device_error.argtypes = [vp, C.POINTER(C.c_int32)]
    cu = np.array([int(x) for x in sys.argv[2].split(",")], dtype=np.int32)
    r = int(sys.argv[3])
    for round_ in range(2):
        d_cu, d_out = vp(), vp()
        assert rt.cudaMalloc(C.byref(d_cu), cu.nbytes) == 0
        assert rt.cudaMalloc(C.byref(d_out), cu.nbytes) == 0
        assert rt.cudaMemcpy(d_cu, cu.ctypes.data, cu.nbytes, 1) == 0
        assert lib.csa_compress_cu_seqlens(d_cu, len(cu) - 1, r, d_out, None) == 0
        word = C.c_int32(-1)
        assert lib.csa_device_error(None, C.byref(word)) == 0 and word.value == 0
        got = np.empty_like(cu)
        assert rt.cudaMemcpy(got.ctypes.data, d_out, cu.nbytes, 2) == 0
        print(",".join(str(int(x)) for x in got))
        rt.cudaFree(d_cu)
        rt.cudaFree(d_out)
        if round_ == 0:
            assert rt.cudaDeviceReset() == 0
''')


def test_calls_after_device_reset():
    lib = csa_build.build()
    lengths = [1, 3, 700, 5, 260, 333, 2]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    r = 4
    res = subprocess.run([sys.executable, "-c", CHILD, lib, ",".join(str(x) for x in cu), str(r)],
                         capture_output=True, text=True, timeout=300,
                         env=dict(os.environ))
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.strip().splitlines() if ln]
    assert len(lines) == 2
    want = oracle.compress_cu_seqlens(cu, r)
    for ln in lines:
        np.testing.assert_array_equal(np.array([int(x) for x in ln.split(",")]), want)
