"""The C-ABI library builds, loads and exports every symbol include/*.h
declares, and rejects invalid arguments on the host before anything reaches
a GPU.  CPU only: no call here launches a kernel."""
import ctypes
import glob
import os
import re

import pytest

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(tk_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_loads_and_exports_every_declared_symbol():
    lib = tk.load()
    declared = _declared_functions()
    assert "tk_attn_fwd" in declared and len(declared) >= 6
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(_lib.SIGNATURES) == declared, "Python binding and header disagree"


def test_version_and_strerror():
    lib = tk.load()
    assert lib.tk_attn_version() == (0 << 16) | 1
    for code in range(0, 12):
        assert tk.strerror(code) and tk.strerror(code) != "unknown status code"
    assert tk.strerror(999) == "unknown status code"


# Fake but well-aligned, non-overlapping addresses: validation rejects the
# arguments before any CUDA call, so they are never dereferenced.
A = 0x10000000
Bq, Bk, Bv, Bo, Bl = A, A + 0x1000000, A + 0x2000000, A + 0x3000000, A + 0x4000000


def _call(q=Bq, k=Bk, v=Bv, o=Bo, l=Bl, B=1, H=1, N=128, D=64, causal=0, scale=0.125):
    return tk.load().tk_attn_fwd(q, k, v, o, l, B, H, N, D, causal, scale, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(q=None), "TK_ERR_NULL_PTR"),
    (dict(l=None), "TK_ERR_NULL_PTR"),
    (dict(B=0), "TK_ERR_BAD_SHAPE"),
    (dict(H=-1), "TK_ERR_BAD_SHAPE"),
    (dict(N=0), "TK_ERR_BAD_SHAPE"),
    (dict(N=2**31), "TK_ERR_BAD_SHAPE"),
    (dict(B=2**20, H=2**20, N=2**20, D=128), "TK_ERR_BAD_SHAPE"),
    (dict(D=96), "TK_ERR_UNSUPPORTED_D"),
    (dict(D=256), "TK_ERR_UNSUPPORTED_D"),
    (dict(causal=2), "TK_ERR_BAD_FLAG"),
    (dict(scale=0.0), "TK_ERR_BAD_SCALE"),
    (dict(scale=-1.0), "TK_ERR_BAD_SCALE"),
    (dict(scale=float("inf")), "TK_ERR_BAD_SCALE"),
    (dict(scale=float("nan")), "TK_ERR_BAD_SCALE"),
    (dict(q=Bq + 8), "TK_ERR_MISALIGNED"),
    (dict(o=Bo + 2), "TK_ERR_MISALIGNED"),
    (dict(l=Bl + 2), "TK_ERR_MISALIGNED"),
    (dict(o=Bq + 16), "TK_ERR_ALIAS"),
    (dict(l=Bv + 64), "TK_ERR_ALIAS"),
    (dict(l=Bo + 16), "TK_ERR_ALIAS"),
])
def test_host_validation(kwargs, code):
    assert _call(**kwargs) == tk.STATUS[code]


def test_validation_order_null_before_shape():
    assert _call(q=None, N=0) == tk.STATUS["TK_ERR_NULL_PTR"]


def test_python_wrapper_rejects_bad_tensors():
    import torch
    q = torch.zeros((1, 1, 8, 64), dtype=torch.float32)
    with pytest.raises(TypeError):
        tk.fwd(q, q, q)
    qb = torch.zeros((1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        tk.fwd(qb, qb, qb)


def test_error_carries_status_name():
    e = tk.TkError(tk.STATUS["TK_ERR_BAD_SCALE"], "tk_attn_fwd")
    assert "TK_ERR_BAD_SCALE" in str(e) and e.code == 5
