"""ctypes binding of the C ABI in include/tk_attn.h.

Loads ``_build/libtk_attn.so`` (built in-tree by ``build.py``).  There is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

TK_OK = 0
STATUS_NAMES = {
    0: "TK_OK", 1: "TK_ERR_NULL_PTR", 2: "TK_ERR_BAD_SHAPE", 3: "TK_ERR_UNSUPPORTED_D",
    4: "TK_ERR_MISALIGNED", 5: "TK_ERR_BAD_SCALE", 6: "TK_ERR_ALIAS", 7: "TK_ERR_BAD_FLAG",
    8: "TK_ERR_UNSUPPORTED_DEVICE", 9: "TK_ERR_CUDA", 10: "TK_ERR_DEVICE_TIMEOUT",
    11: "TK_ERR_NOT_DEVICE_MEMORY", 12: "TK_ERR_WORKSPACE", 13: "TK_ERR_NOALLOC_TOO_LARGE",
}
STATUS = {v: k for k, v in STATUS_NAMES.items()}

# Every symbol the header declares, with its ctypes signature.
_P, _I64, _I, _F, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
SIGNATURES = {
    "tk_attn_fwd": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _F, _P], _I),
    "tk_attn_fwd_kv": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I, _F, _P], _I),
    "tk_attn_fwd_workspace_bytes": ([_I64, _I64, _I64, _I64, _I64, _I], ctypes.c_size_t),
    "tk_attn_fwd_ws": ([_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I64, _I64, _I64, _I64, _I64, _I, _F, _P], _I),
    "tk_attn_bwd_workspace_bytes": ([_I64, _I64, _I64, _I64], ctypes.c_size_t),
    "tk_attn_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I64, _I64, _I64, _I64,
                     _I, _F, _P], _I),
    "tk_attn_bwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _F, _P], _I),
    "tk_gemm_workspace_bytes": ([_I64, _I64, _I64, _I], ctypes.c_size_t),
    "tk_gemm_uses_pairs": ([_I64, _I64, _I64, _I], _I),
    "tk_gemm": ([_P, _P, _P, _P, ctypes.c_size_t, _I64, _I64, _I64, _I, _I, _P], _I),
    "tk_based_fwd": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _F, _P], _I),
    "tk_based_workspace_bytes": ([_I64, _I64, _I64], ctypes.c_size_t),
    "tk_based_fwd_ws": ([_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I64, _I64, _I64, _I64, _I64, _F, _P], _I),
    "tk_hedgehog_fwd": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P], _I),
    "tk_hedgehog_workspace_bytes": ([_I64, _I64, _I64], ctypes.c_size_t),
    "tk_hedgehog_fwd_ws": ([_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I64, _I64, _I64, _I64, _I64, _I64, _P],
                           _I),
    "tk_attn_device_status": ([_P, ctypes.POINTER(ctypes.c_uint32)], _I),
    "tk_attn_selftest_timeout": ([_U64, _P], _I),
    "tk_attn_strerror": ([_I], ctypes.c_char_p),
    "tk_attn_last_cuda_error": ([], _I),
    "tk_attn_version": ([], _I),
}


class TkError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, code: int, where: str, cuda_error: int = 0):
        self.code = code
        self.name = STATUS_NAMES.get(code, f"status {code}")
        msg = f"{where}: {self.name} ({strerror(code)})"
        if code == STATUS["TK_ERR_CUDA"]:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded library (built first if it is missing or stale and the
    toolkit is present)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if build_if_missing:
                try:
                    path = _build.build()
                except RuntimeError:
                    if not os.path.exists(path):
                        raise
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    try:
        return load().tk_attn_strerror(int(code)).decode()
    except Exception:  # library not loadable: still describe the code
        return STATUS_NAMES.get(code, "unknown")


def check(code: int, where: str) -> None:
    if code != TK_OK:
        raise TkError(code, where, load().tk_attn_last_cuda_error())
