"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

This package is the checker, not the product (attention forward and backward,
the plain GEMM the same tile pipeline runs, and Based and Hedgehog linear
attention).  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may load
it.  It shares no code with the CUDA library and imports nothing from it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, two passes per query
row: scores and max, then weights, sum and weighted V).  This module only
compiles that file with the host C compiler and marshals numpy arrays through
ctypes.

Definition followed (the "ThunderKittens" attention forward as printed on
10100.com/article/71410160, section "writing a kernel with TK",
attn_fwd_template consumer::compute / consumer::finish, and the inner-loop
excerpt on alanwu.xyz/posts/thunderkittens):

    s_ij   = scale * <Q_i, K_j>            j in J_i  (all Nkv keys, or, if causal,
                                                     j <= i + Nkv - Nq: the Nq queries
                                                     stand at the end of the key sequence)
    LSE_i  = max_j s_ij + ln(sum_j exp(s_ij - max_j s_ij))
    O_i    = sum_j exp(s_ij - LSE_i) V_j
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtk_attn_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libtk_attn_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # -O2 without -ffast-math: IEEE fp64 semantics are kept.
        cmd = ["gcc", "-O2", "-std=gnu11", "-Wall", "-fPIC", "-shared", "-pthread",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load a compiled oracle library from ``path`` and declare its entry
    points.  ``_load`` uses it for the default build; the oracle's own
    mutation tests use it for deliberately broken copies."""
    lib = ctypes.CDLL(path)
    _declare(lib)
    return lib


def _declare(lib) -> None:
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.tkor_attn_fwd.argtypes = [P, P, P, P, P, i64, i64, i64, i64,
                                  ctypes.c_int, ctypes.c_double, ctypes.c_int]
    lib.tkor_attn_fwd.restype = ctypes.c_int
    lib.tkor_attn_fwd_rows.argtypes = [P, P, P, i64, i64, ctypes.c_int,
                                       ctypes.c_double, P, i64, P, P, ctypes.c_int]
    lib.tkor_attn_fwd_rows.restype = ctypes.c_int
    lib.tkor_attn_fwd_kv.argtypes = [P, P, P, P, P, i64, i64, i64, i64, i64,
                                     ctypes.c_int, ctypes.c_double, ctypes.c_int]
    lib.tkor_attn_fwd_kv.restype = ctypes.c_int
    lib.tkor_attn_fwd_kv_rows.argtypes = [P, P, P, i64, i64, i64, ctypes.c_int,
                                          ctypes.c_double, P, i64, P, P, ctypes.c_int]
    lib.tkor_attn_fwd_kv_rows.restype = ctypes.c_int
    lib.tkor_attn_weights.argtypes = [P, P, i64, i64, ctypes.c_int,
                                      ctypes.c_double, P]
    lib.tkor_attn_weights.restype = ctypes.c_int
    lib.tkor_attn_bwd.argtypes = [P, P, P, P, P, P, P, i64, i64, i64, i64,
                                  ctypes.c_int, ctypes.c_double, ctypes.c_int]
    lib.tkor_attn_bwd.restype = ctypes.c_int
    lib.tkor_gemm.argtypes = [P, P, P, i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.tkor_gemm.restype = ctypes.c_int
    lib.tkor_gemm_rows.argtypes = [P, P, i64, i64, i64, ctypes.c_int, P, i64, P, ctypes.c_int]
    lib.tkor_gemm_rows.restype = ctypes.c_int
    lib.tkor_based.argtypes = [P, P, P, P, P, i64, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int]
    lib.tkor_based.restype = ctypes.c_int
    lib.tkor_based_rows.argtypes = [P, P, P, i64, i64, i64, ctypes.c_double, P, i64, P, P, ctypes.c_int]
    lib.tkor_based_rows.restype = ctypes.c_int
    lib.tkor_hedgehog_rows.argtypes = [P, P, P, P, P, i64, i64, i64, i64, P, i64, P, P]
    lib.tkor_hedgehog_rows.restype = ctypes.c_int
    lib.tkor_last_threads.argtypes = []
    lib.tkor_last_threads.restype = ctypes.c_int


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _bits(a) -> np.ndarray:
    """bf16 input as a C-contiguous uint16 array of its bit patterns.

    Accepts a numpy uint16 array (already bit patterns) or a torch bfloat16
    tensor on the CPU.
    """
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(a)
    import torch  # only for the bfloat16 -> bits view
    if not isinstance(a, torch.Tensor) or a.dtype != torch.bfloat16:
        raise TypeError("expected a torch.bfloat16 tensor or uint16 bit patterns")
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def attn_fwd(q, k, v, causal: bool, scale: float, threads: int = 0, lib=None):
    """Whole problem.  q: [B,H,Nq,D], k, v: [B,H,Nkv,D] bf16 (Nq = Nkv for
    the same-length problem).  Returns (O, LSE) as float64 arrays of shapes
    [B,H,Nq,D] and [B,H,Nq]."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 4 or kb.shape != vb.shape or qb.shape[:2] + qb.shape[3:] != kb.shape[:2] + kb.shape[3:]:
        raise ValueError("q [B,H,Nq,D] and k, v [B,H,Nkv,D] must agree in B, H, D")
    B, H, Nq, D = qb.shape
    Nkv = kb.shape[2]
    O = np.empty((B, H, Nq, D), dtype=np.float64)
    L = np.empty((B, H, Nq), dtype=np.float64)
    rc = (lib or _load()).tkor_attn_fwd_kv(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(O), _ptr(L),
                                           B, H, Nq, Nkv, D, int(bool(causal)), float(scale),
                                           int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return O, L


def attn_fwd_rows(q, k, v, rows, causal: bool, scale: float, threads: int = 0):
    """Selected query rows of ONE head.  q: [Nq,D], k, v: [Nkv,D] bf16; rows:
    int indices into q.  Returns (O[len(rows),D], LSE[len(rows)]) as float64."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 2 or kb.shape != vb.shape or qb.shape[1] != kb.shape[1]:
        raise ValueError("q [Nq,D] and k, v [Nkv,D] must agree in D")
    Nq, D = qb.shape
    Nkv = kb.shape[0]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    O = np.empty((r.size, D), dtype=np.float64)
    L = np.empty((r.size,), dtype=np.float64)
    rc = _load().tkor_attn_fwd_kv_rows(_ptr(qb), _ptr(kb), _ptr(vb), Nq, Nkv, D,
                                       int(bool(causal)), float(scale), _ptr(r), r.size,
                                       _ptr(O), _ptr(L), int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return O, L


def attn_weights(q, k, causal: bool, scale: float) -> np.ndarray:
    """Attention weight matrix of ONE head (tiny N only): float64 [N,N]."""
    qb, kb = _bits(q), _bits(k)
    N, D = qb.shape
    P = np.empty((N, N), dtype=np.float64)
    rc = _load().tkor_attn_weights(_ptr(qb), _ptr(kb), N, D, int(bool(causal)),
                                   float(scale), _ptr(P))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return P


def attn_bwd(q, k, v, do, causal: bool, scale: float, threads: int = 0, lib=None):
    """Gradient of sum(O * dO) with respect to q, k, v for O = attention(q, k,
    v).  All inputs bf16 [B,H,N,D].  Returns (dQ, dK, dV) float64 arrays.

    Chain rule through the softmax, written out:  dV_j = sum_i p_ij dO_i;
    dS_ij = p_ij (<dO_i, V_j> - sum_k p_ik <dO_i, V_k>);
    dQ_i = scale sum_j dS_ij K_j;  dK_j = scale sum_i dS_ij Q_i."""
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(do)
    if qb.ndim != 4 or not (qb.shape == kb.shape == vb.shape == gb.shape):
        raise ValueError("q, k, v, do must share one [B,H,N,D] shape")
    B, H, N, D = qb.shape
    dQ = np.empty((B, H, N, D), dtype=np.float64)
    dK = np.empty((B, H, N, D), dtype=np.float64)
    dV = np.empty((B, H, N, D), dtype=np.float64)
    rc = (lib or _load()).tkor_attn_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), _ptr(dQ), _ptr(dK),
                                        _ptr(dV), B, H, N, D, int(bool(causal)), float(scale),
                                        int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return dQ, dK, dV


def gemm(a, b, b_kmajor: bool = True, rows=None, threads: int = 0, lib=None) -> np.ndarray:
    """C = a @ b.T (b_kmajor: b is [N,K]) or a @ b (b is [K,N]) in fp64 from
    the bf16 inputs; ``rows``: only those rows of C.  Returns float64
    [len(rows) or M, N]."""
    ab, bb = _bits(a), _bits(b)
    if ab.ndim != 2 or bb.ndim != 2:
        raise ValueError("a and b must be 2-D")
    M, K = ab.shape
    N, Kb = (bb.shape if b_kmajor else bb.shape[::-1])
    if Kb != K:
        raise ValueError("inner dimensions differ")
    lib = lib or _load()
    if rows is None:
        C = np.empty((M, N), dtype=np.float64)
        rc = lib.tkor_gemm(_ptr(ab), _ptr(bb), _ptr(C), M, N, K, int(bool(b_kmajor)), int(threads))
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        C = np.empty((r.size, N), dtype=np.float64)
        rc = lib.tkor_gemm_rows(_ptr(ab), _ptr(bb), M, N, K, int(bool(b_kmajor)), _ptr(r), r.size,
                                _ptr(C), int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return C


def based(q, k, v, scale: float, rows=None, threads: int = 0, lib=None):
    """Causal Based linear attention, plain quadratic form in fp64:
    w_ij = 1 + s + s^2/2 with s = scale <q_i, k_j>, j <= i;
    O_i = sum_j w_ij v_j / DEN_i, DEN_i = sum_j w_ij.
    Whole problem: q, k [B,H,N,Dqk], v [B,H,N,Dv] -> (O [B,H,N,Dv], DEN [B,H,N]).
    With ``rows``: q, k [N,Dqk], v [N,Dv] of ONE head -> (O [len,Dv], DEN [len])."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    lib = lib or _load()
    if rows is None:
        if qb.ndim != 4 or qb.shape != kb.shape or vb.shape[:3] != qb.shape[:3]:
            raise ValueError("q, k [B,H,N,Dqk] and v [B,H,N,Dv] expected")
        B, H, N, Dqk = qb.shape
        Dv = vb.shape[3]
        O = np.empty((B, H, N, Dv), dtype=np.float64)
        DEN = np.empty((B, H, N), dtype=np.float64)
        rc = lib.tkor_based(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(O), _ptr(DEN), B, H, N, Dqk, Dv,
                            float(scale), int(threads))
    else:
        if qb.ndim != 2 or qb.shape != kb.shape or vb.shape[0] != qb.shape[0]:
            raise ValueError("q, k [N,Dqk] and v [N,Dv] expected")
        N, Dqk = qb.shape
        Dv = vb.shape[1]
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        O = np.empty((r.size, Dv), dtype=np.float64)
        DEN = np.empty((r.size,), dtype=np.float64)
        rc = lib.tkor_based_rows(_ptr(qb), _ptr(kb), _ptr(vb), N, Dqk, Dv, float(scale), _ptr(r), r.size,
                                 _ptr(O), _ptr(DEN), int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return O, DEN


def hedgehog(q, k, v, wq, wk, rows=None, lib=None):
    """Causal Hedgehog linear attention, plain quadratic form in fp64, for ONE
    head: q, k [N,d], v [N,Dv], wq, wk [d,f] (bf16).  phi(x) =
    [softmax(x W), softmax(-x W)], w_ij = phi_q(q_i) . phi_k(k_j),
    O_i = sum_{j<=i} w_ij v_j / DEN_i.  Returns (O [len,Dv], DEN [len]) for
    ``rows`` (default: all rows)."""
    qb, kb, vb, wqb, wkb = _bits(q), _bits(k), _bits(v), _bits(wq), _bits(wk)
    if qb.ndim != 2 or qb.shape != kb.shape or vb.shape[0] != qb.shape[0] or wqb.shape != wkb.shape \
            or wqb.shape[0] != qb.shape[1]:
        raise ValueError("q, k [N,d], v [N,Dv], wq, wk [d,f] expected")
    N, d = qb.shape
    f = wqb.shape[1]
    Dv = vb.shape[1]
    r = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    O = np.empty((r.size, Dv), dtype=np.float64)
    DEN = np.empty((r.size,), dtype=np.float64)
    rc = (lib or _load()).tkor_hedgehog_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(wqb), _ptr(wkb), N, d, f, Dv,
                                             _ptr(r), r.size, _ptr(O), _ptr(DEN))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return O, DEN


def last_threads() -> int:
    """Threads the last oracle call actually ran on."""
    return int(_load().tkor_last_threads())
