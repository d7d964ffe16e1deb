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
    assert lib.tk_attn_version() == (0 << 16) | 2
    for code in range(0, 13):
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
    (dict(D=80), "TK_ERR_UNSUPPORTED_D"),
    (dict(D=192), "TK_ERR_UNSUPPORTED_D"),
    (dict(D=512), "TK_ERR_UNSUPPORTED_D"),
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


def _call_kv(q=Bq, k=Bk, v=Bv, o=Bo, l=Bl, B=1, H=1, Nq=128, Nkv=256, D=64, causal=0, scale=0.125):
    return tk.load().tk_attn_fwd_kv(q, k, v, o, l, B, H, Nq, Nkv, D, causal, scale, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(k=None), "TK_ERR_NULL_PTR"),
    (dict(Nq=0), "TK_ERR_BAD_SHAPE"),
    (dict(Nkv=0), "TK_ERR_BAD_SHAPE"),
    (dict(Nkv=2**31), "TK_ERR_BAD_SHAPE"),
    (dict(Nq=300, Nkv=200, causal=1), "TK_ERR_BAD_SHAPE"),  # a causal query would see no key
    (dict(D=48), "TK_ERR_UNSUPPORTED_D"),
    (dict(causal=3), "TK_ERR_BAD_FLAG"),
    (dict(scale=-0.5), "TK_ERR_BAD_SCALE"),
    (dict(v=Bv + 4), "TK_ERR_MISALIGNED"),
    (dict(o=Bk + 0x4000), "TK_ERR_ALIAS"),        # inside K: 256 keys x 64 x 2 B = 32 KB
    (dict(l=Bq + 0x2000), "TK_ERR_ALIAS"),        # inside Q: 128 x 64 x 2 B = 16 KB
])
def test_host_validation_kv(kwargs, code):
    assert _call_kv(**kwargs) == tk.STATUS[code]


def test_kv_validation_sizes_by_each_length():
    """K ends 32 KB after its start for Nkv = 256; an O placed just past it
    is accepted by validation (it then stops at the device-memory check,
    since the addresses are fake)."""
    rc = _call_kv(o=Bk + 256 * 64 * 2)
    assert rc != tk.STATUS["TK_ERR_ALIAS"]


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


# ---------------------------------------------------------------- backward ABI

Bdo, BdQ, BdK, BdV, Bws, Bo = (A + 0x5000000, A + 0x6000000, A + 0x7000000, A + 0x8000000,
                               A + 0x9000000, A + 0xA000000)


def _bwd(q=Bq, k=Bk, v=Bv, o=Bo, do=Bdo, l=Bl, dq=BdQ, dk=BdK, dv=BdV, ws=Bws, ws_bytes=None,
         B=1, H=1, N=128, D=64, causal=0, scale=0.125):
    lib = tk.load()
    if ws_bytes is None:
        ws_bytes = lib.tk_attn_bwd_workspace_bytes(B, H, N, D)
    return lib.tk_attn_bwd(q, k, v, o, do, l, dq, dk, dv, ws, ws_bytes, B, H, N, D, causal, scale, None)


def test_bwd_workspace_size():
    lib = tk.load()
    rows = 2 * 3 * 100
    acc = 2 * 3 * 128 * 64 * 4  # fp32 dQ accumulator over whole 128-row query tiles
    padded = 2 * 3 * 128 * 4    # Delta and -LSE*log2(e), one float per padded row each
    expect = -(-acc // 256) * 256 + 2 * (-(-padded // 256) * 256)
    assert lib.tk_attn_bwd_workspace_bytes(2, 3, 100, 64) == expect
    assert lib.tk_attn_bwd_workspace_bytes(1, 1, 0, 64) == 0
    assert lib.tk_attn_bwd_workspace_bytes(1, 1, 16, 256) == 0
    # head dims 32 and 96 run on the 64- and 128-column kernels: their accumulator is padded
    assert lib.tk_attn_bwd_workspace_bytes(1, 1, 16, 32) == lib.tk_attn_bwd_workspace_bytes(1, 1, 16, 64) > 0
    assert lib.tk_attn_bwd_workspace_bytes(1, 1, 16, 96) == lib.tk_attn_bwd_workspace_bytes(1, 1, 16, 128) > 0


@pytest.mark.parametrize("kwargs,code", [
    (dict(do=None), "TK_ERR_NULL_PTR"),
    (dict(ws=None), "TK_ERR_NULL_PTR"),
    (dict(N=0), "TK_ERR_BAD_SHAPE"),
    (dict(D=48), "TK_ERR_UNSUPPORTED_D"),
    (dict(D=256), "TK_ERR_UNSUPPORTED_D"),  # the forward takes 256; the backward does not
    (dict(causal=3), "TK_ERR_BAD_FLAG"),
    (dict(scale=-0.5), "TK_ERR_BAD_SCALE"),
    (dict(dk=BdK + 8), "TK_ERR_MISALIGNED"),
    (dict(ws=Bws + 16), "TK_ERR_WORKSPACE"),
    (dict(ws_bytes=1024), "TK_ERR_WORKSPACE"),
    (dict(dq=Bq), "TK_ERR_ALIAS"),
    (dict(dv=BdK + 256), "TK_ERR_ALIAS"),
    (dict(ws=Bdo), "TK_ERR_ALIAS"),
])
def test_bwd_host_validation(kwargs, code):
    assert _bwd(**kwargs) == tk.STATUS[code]


# ---------------------------------------------------------------- GEMM ABI

def _gemm(a=Bq, b=Bk, c=Bo, ws=None, ws_bytes=0, M=256, N=256, K=256, b_kmajor=1, stream_k=1):
    return tk.load().tk_gemm(a, b, c, ws, ws_bytes, M, N, K, b_kmajor, stream_k, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(a=None), "TK_ERR_NULL_PTR"),
    (dict(c=None), "TK_ERR_NULL_PTR"),
    (dict(M=0), "TK_ERR_BAD_SHAPE"),
    (dict(K=12), "TK_ERR_BAD_SHAPE"),     # row strides must be multiples of 16 bytes
    (dict(N=100), "TK_ERR_BAD_SHAPE"),
    (dict(K=2**31), "TK_ERR_BAD_SHAPE"),
    (dict(b_kmajor=2), "TK_ERR_BAD_FLAG"),
    (dict(stream_k=-1), "TK_ERR_BAD_FLAG"),
    (dict(b=Bk + 8), "TK_ERR_MISALIGNED"),
    (dict(c=Bq + 0x1000), "TK_ERR_ALIAS"),  # inside A (256 x 256 x 2 bytes)
])
def test_gemm_host_validation(kwargs, code):
    assert _gemm(**kwargs) == tk.STATUS[code]


def test_gemm_workspace_bytes_rejects_bad_shapes():
    lib = tk.load()
    assert lib.tk_gemm_workspace_bytes(0, 8, 8, 1) == 0
    assert lib.tk_gemm_workspace_bytes(8, 8, 12, 1) == 0
    assert lib.tk_gemm_workspace_bytes(8, 8, 8, 3) == 0


def test_gemm_uses_pairs_rejects_bad_shapes():
    """No device here: 0 for every query, valid or not, and nothing raises."""
    lib = tk.load()
    assert lib.tk_gemm_uses_pairs(0, 8, 8, 1) == 0
    assert lib.tk_gemm_uses_pairs(8, 8, 12, 1) == 0
    assert lib.tk_gemm_uses_pairs(8192, 8192, 8192, 3) == 0
    assert lib.tk_gemm_uses_pairs(8192, 8192, 8192, 1) in (0, 1)


# ---------------------------------------------------------------- Based ABI

def _based(q=Bq, k=Bk, v=Bv, o=Bo, d=Bl, B=1, H=1, N=128, Dqk=16, Dv=64, scale=0.25):
    return tk.load().tk_based_fwd(q, k, v, o, d, B, H, N, Dqk, Dv, scale, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(v=None), "TK_ERR_NULL_PTR"),
    (dict(N=0), "TK_ERR_BAD_SHAPE"),
    (dict(Dqk=32), "TK_ERR_UNSUPPORTED_D"),
    (dict(Dv=128), "TK_ERR_UNSUPPORTED_D"),
    (dict(scale=0.0), "TK_ERR_BAD_SCALE"),
    (dict(o=Bo + 8), "TK_ERR_MISALIGNED"),
    (dict(o=Bv + 1024), "TK_ERR_ALIAS"),
    (dict(d=Bo + 64), "TK_ERR_ALIAS"),
])
def test_based_host_validation(kwargs, code):
    assert _based(**kwargs) == tk.STATUS[code]


def _based_ws(q=Bq, k=Bk, v=Bv, o=Bo, d=Bl, ws=Bws, ws_bytes=1 << 20, B=1, H=1, N=128, Dqk=16, Dv=64, scale=0.25):
    return tk.load().tk_based_fwd_ws(q, k, v, o, d, ws, ws_bytes, B, H, N, Dqk, Dv, scale, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(k=None), "TK_ERR_NULL_PTR"),
    (dict(B=0), "TK_ERR_BAD_SHAPE"),
    (dict(Dqk=64), "TK_ERR_UNSUPPORTED_D"),
    (dict(scale=float("nan")), "TK_ERR_BAD_SCALE"),
    (dict(q=Bq + 2), "TK_ERR_MISALIGNED"),
    (dict(d=Bv + 256), "TK_ERR_ALIAS"),
])
def test_based_ws_host_validation(kwargs, code):
    """The segmented entry point checks its arguments like tk_based_fwd, before
    it looks at the device (the workspace checks need the device's SM count
    and are covered on the GPU)."""
    assert _based_ws(**kwargs) == tk.STATUS[code]


def test_based_workspace_bytes_without_device():
    lib = tk.load()
    assert lib.tk_based_workspace_bytes(0, 1, 128) == 0
    assert lib.tk_based_workspace_bytes(1, 1, 0) == 0


# ---------------------------------------------------------------- Hedgehog ABI

def _hh(q=Bq, k=Bk, v=Bv, wq=Bdo, wk=BdQ, o=Bo, d=Bl, B=1, H=1, N=128, Dqk=64, F=64, Dv=64):
    return tk.load().tk_hedgehog_fwd(q, k, v, wq, wk, o, d, B, H, N, Dqk, F, Dv, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(wk=None), "TK_ERR_NULL_PTR"),
    (dict(N=0), "TK_ERR_BAD_SHAPE"),
    (dict(Dqk=128), "TK_ERR_UNSUPPORTED_D"),
    (dict(F=32), "TK_ERR_UNSUPPORTED_D"),
    (dict(wq=Bdo + 8), "TK_ERR_MISALIGNED"),
    (dict(o=Bq + 4096), "TK_ERR_ALIAS"),
    (dict(d=Bdo + 64), "TK_ERR_ALIAS"),     # inside Wq
])
def test_hedgehog_host_validation(kwargs, code):
    assert _hh(**kwargs) == tk.STATUS[code]


def _hh_ws(q=Bq, k=Bk, v=Bv, wq=Bdo, wk=BdQ, o=Bo, d=Bl, ws=Bws, ws_bytes=1 << 20, B=1, H=1, N=128, Dqk=64, F=64,
           Dv=64):
    return tk.load().tk_hedgehog_fwd_ws(q, k, v, wq, wk, o, d, ws, ws_bytes, B, H, N, Dqk, F, Dv, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(wq=None), "TK_ERR_NULL_PTR"),
    (dict(H=0), "TK_ERR_BAD_SHAPE"),
    (dict(F=128), "TK_ERR_UNSUPPORTED_D"),
    (dict(wk=BdQ + 4), "TK_ERR_MISALIGNED"),
    (dict(o=Bk + 2048), "TK_ERR_ALIAS"),
])
def test_hedgehog_ws_host_validation(kwargs, code):
    assert _hh_ws(**kwargs) == tk.STATUS[code]


def test_hedgehog_workspace_bytes_without_device():
    assert tk.load().tk_hedgehog_workspace_bytes(1, 0, 128) == 0
