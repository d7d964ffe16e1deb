"""Python entry points over the C ABI (argument marshalling only: every step
of the attention forward runs in the CUDA library)."""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
            N: int, D: int, causal: bool, scale: float, stream_handle: int) -> None:
    """tk_attn_fwd on raw device pointers; raises TkError on a non-zero status."""
    rc = _lib.load().tk_attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, D,
                                 int(bool(causal)), float(scale), stream_handle)
    _lib.check(rc, "tk_attn_fwd")


def fwd_kv_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
               Nq: int, Nkv: int, D: int, causal: bool, scale: float, stream_handle: int) -> None:
    """tk_attn_fwd_kv on raw device pointers; raises TkError on a non-zero status."""
    rc = _lib.load().tk_attn_fwd_kv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nkv, D,
                                    int(bool(causal)), float(scale), stream_handle)
    _lib.check(rc, "tk_attn_fwd_kv")


def fwd_workspace_bytes(B: int, H: int, Nq: int, Nkv: int, D: int, causal: bool) -> int:
    """Device workspace bytes tk_attn_fwd_ws needs on the current device for
    this shape (0: the last round of work units is not split)."""
    return int(_lib.load().tk_attn_fwd_workspace_bytes(B, H, Nq, Nkv, D, int(bool(causal))))


def fwd_ws_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, ws_ptr, ws_bytes: int,
               B: int, H: int, Nq: int, Nkv: int, D: int, causal: bool, scale: float,
               stream_handle: int) -> None:
    """tk_attn_fwd_ws on raw device pointers; raises TkError on a non-zero status."""
    rc = _lib.load().tk_attn_fwd_ws(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, ws_ptr, ws_bytes, B, H, Nq, Nkv, D,
                                    int(bool(causal)), float(scale), stream_handle)
    _lib.check(rc, "tk_attn_fwd_ws")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: float | None = None, out: torch.Tensor | None = None,
        lse: torch.Tensor | None = None, stream=None, workspace: torch.Tensor | None = None):
    """Fused attention forward.

    q: bf16 [B, H, Nq, D]; k, v: bf16 [B, H, Nkv, D] (Nkv = Nq usually), D
    in {32, 64, 96, 128, 256}.  Returns (O bf16 [B,H,Nq,D], LSE fp32 [B,H,Nq]) with
    O = softmax(scale QK^T [+causal]) V and LSE the natural-log row
    log-sum-exp.  Under the causal mask the queries stand at the end of the
    key sequence (query i sees keys j <= i + Nkv - Nq; needs Nkv >= Nq).
    ``scale`` defaults to 1/sqrt(D).

    CUDA inputs: the kernel is enqueued on ``stream`` (default: the current
    stream) and the call returns without synchronising.  CPU inputs (ideally
    pinned): they are copied to the current CUDA device, the kernel runs, and
    O and LSE are copied back into CPU tensors (pinned when the inputs are);
    the call then returns after the stream has finished.

    On CUDA inputs the call goes through tk_attn_fwd_ws: when the shape's last
    round of work units is split (``fwd_workspace_bytes`` > 0) it uses
    ``workspace`` (a CUDA uint8 tensor of at least that size) or allocates one
    on ``q``'s device.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{n} must be bfloat16")
        if t.dim() != 4:
            raise ValueError(f"{n} must be [B, H, N, D]")
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,D] and k, v [B,H,Nkv,D] must agree in B, H, D")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    B, H, N, D = q.shape
    Nkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)

    if q.device.type == "cpu":
        return _fwd_from_host(q, k, v, bool(causal), float(scale), stream)
    if q.device.type != "cuda":
        raise ValueError("inputs must be CUDA or CPU tensors")

    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    with torch.cuda.device(q.device):
        need = fwd_workspace_bytes(B, H, N, Nkv, D, causal)
        if need > 0 and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if need > 0 else None
        ws_bytes = workspace.numel() * workspace.element_size() if need > 0 else 0
        fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes,
                   B, H, N, Nkv, D, causal, scale, _stream_handle(stream))
    return out, lse


_side_streams = {}


def _side_stream(dev: torch.device):
    if dev.index not in _side_streams:
        _side_streams[dev.index] = torch.cuda.Stream(dev)
    return _side_streams[dev.index]


def _fwd_from_host(q, k, v, causal, scale, stream, chunk_bytes: int = 32 << 20):
    """Host tensors in and out.  With pinned inputs the heads go in chunks
    over two streams, so that one chunk's copy in, another's kernel and a
    third's copy out overlap; each chunk is one tk_attn_fwd launch over its
    heads as a [1, heads, N, D] problem."""
    dev = torch.device("cuda", torch.cuda.current_device())
    main = stream if stream is not None else torch.cuda.current_stream(dev)
    B, H, N, D = q.shape
    Nkv = k.shape[2]
    BH = B * H
    pinned = q.is_pinned() and k.is_pinned() and v.is_pinned()
    o_h = torch.empty((B, H, N, D), dtype=torch.bfloat16, pin_memory=pinned)
    l_h = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pinned)
    per_head = (N + 2 * Nkv) * D * 2
    n_chunks = max(1, min(BH, (BH * per_head) // chunk_bytes)) if pinned else 1
    qf, kf, vf = q.reshape(BH, N, D), k.reshape(BH, Nkv, D), v.reshape(BH, Nkv, D)
    of, lf = o_h.reshape(BH, N, D), l_h.reshape(BH, N)
    streams = [main, _side_stream(dev)] if n_chunks > 1 else [main]
    main_done = torch.cuda.Event()
    main_done.record(torch.cuda.current_stream(dev))
    for s in streams:
        s.wait_event(main_done)
    qd = torch.empty((BH, N, D), dtype=torch.bfloat16, device=dev)
    kd = torch.empty((BH, Nkv, D), dtype=torch.bfloat16, device=dev)
    vd = torch.empty((BH, Nkv, D), dtype=torch.bfloat16, device=dev)
    od = torch.empty((BH, N, D), dtype=torch.bfloat16, device=dev)
    ld = torch.empty((BH, N), dtype=torch.float32, device=dev)
    for c in range(n_chunks):
        h0, h1 = c * BH // n_chunks, (c + 1) * BH // n_chunks
        if h1 == h0:
            continue
        s = streams[c % len(streams)]
        with torch.cuda.stream(s):
            qd[h0:h1].copy_(qf[h0:h1], non_blocking=True)
            kd[h0:h1].copy_(kf[h0:h1], non_blocking=True)
            vd[h0:h1].copy_(vf[h0:h1], non_blocking=True)
            ptrs = (qd[h0].data_ptr(), kd[h0].data_ptr(), vd[h0].data_ptr(), od[h0].data_ptr(), ld[h0].data_ptr())
            if Nkv == N:
                fwd_raw(*ptrs, 1, h1 - h0, N, D, causal, scale, int(s.cuda_stream))
            else:
                fwd_kv_raw(*ptrs, 1, h1 - h0, N, Nkv, D, causal, scale, int(s.cuda_stream))
            of[h0:h1].copy_(od[h0:h1], non_blocking=True)
            lf[h0:h1].copy_(ld[h0:h1], non_blocking=True)
    for s in streams:
        s.synchronize()
    return o_h, l_h


def bwd_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    """Device workspace bytes tk_attn_bwd needs (0 for an unsupported shape)."""
    return int(_lib.load().tk_attn_bwd_workspace_bytes(B, H, N, D))


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        do: torch.Tensor, causal: bool = False, scale: float | None = None, workspace=None,
        stream=None):
    """Attention backward: (dQ, dK, dV), bf16 like q, for O = fwd(q, k, v)
    with its LSE and the incoming gradient dO.  CUDA tensors only; enqueued
    on ``stream`` (default: current) without synchronising.  ``workspace``
    (optional) is a CUDA uint8 tensor of at least ``bwd_workspace_bytes``;
    otherwise one is allocated with torch for the call."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.device.type != "cuda":
            raise ValueError(f"{n} must be a CUDA bf16 [B,H,N,D] tensor")
        if t.shape != q.shape:
            raise ValueError("q, k, v, o, do must have the same shape")
    B, H, N, D = q.shape
    if lse.dtype != torch.float32 or lse.shape != (B, H, N):
        raise ValueError("lse must be fp32 [B,H,N]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q, k, v, o, do, lse = (t.contiguous() for t in (q, k, v, o, do, lse))
    need = bwd_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    with torch.cuda.device(q.device):
        rc = _lib.load().tk_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                     B, H, N, D, int(bool(causal)), float(scale),
                                     _stream_handle(stream))
    _lib.check(rc, "tk_attn_bwd")
    return dq, dk, dv


def device_status(stream=None) -> tuple[int, int]:
    """(status, detail): synchronises the stream, reads and clears the device
    status word.  status is 0 or TK_ERR_DEVICE_TIMEOUT."""
    detail = ctypes.c_uint32(0)
    rc = _lib.load().tk_attn_device_status(_stream_handle(stream), ctypes.byref(detail))
    if rc not in (_lib.TK_OK, _lib.STATUS["TK_ERR_DEVICE_TIMEOUT"]):
        _lib.check(rc, "tk_attn_device_status")
    return rc, detail.value


def selftest_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue the bounded-wait self test (a wait nothing ends, given up after
    ``limit_ns``)."""
    _lib.check(_lib.load().tk_attn_selftest_timeout(int(limit_ns), _stream_handle(stream)),
               "tk_attn_selftest_timeout")


def gemm_workspace_bytes(M: int, N: int, K: int, stream_k: bool = True) -> int:
    """Device workspace bytes tk_gemm needs on the current device (0: none)."""
    return int(_lib.load().tk_gemm_workspace_bytes(M, N, K, int(bool(stream_k))))


def gemm_uses_pairs(M: int, N: int, K: int, stream_k: bool = True) -> bool:
    """Whether tk_gemm runs this shape on CTA pairs on the current device."""
    return bool(_lib.load().tk_gemm_uses_pairs(M, N, K, int(bool(stream_k))))


def gemm(a: torch.Tensor, b: torch.Tensor, b_kmajor: bool = True, stream_k: bool = True,
         out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """C = a @ b.T (b_kmajor: b is [N, K]) or a @ b (b is [K, N]); bf16 CUDA
    tensors, fp32 accumulation, bf16 result [M, N].  Enqueued on ``stream``
    (default: current) without synchronising."""
    for t, n in ((a, "a"), (b, "b")):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.device.type != "cuda":
            raise ValueError(f"{n} must be a 2-D CUDA bf16 tensor")
    M, K = a.shape
    N = b.shape[0] if b_kmajor else b.shape[1]
    if (b.shape[1] if b_kmajor else b.shape[0]) != K:
        raise ValueError("inner dimensions of a and b differ")
    a, b = a.contiguous(), b.contiguous()
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    need = gemm_workspace_bytes(M, N, K, stream_k)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    with torch.cuda.device(a.device):
        rc = _lib.load().tk_gemm(a.data_ptr(), b.data_ptr(), out.data_ptr(), ws_ptr, ws_len, M, N, K,
                                 int(bool(b_kmajor)), int(bool(stream_k)), _stream_handle(stream))
    _lib.check(rc, "tk_gemm")
    return out


def based_workspace_bytes(B: int, H: int, N: int) -> int:
    """Workspace tk_based_fwd_ws needs on the current device (0: no segments)."""
    return int(_lib.load().tk_based_workspace_bytes(B, H, N))


def based(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
          out: torch.Tensor | None = None, den: torch.Tensor | None = None, stream=None,
          workspace: torch.Tensor | None = None, segments: bool = True):
    """Causal Based linear attention.  q, k: bf16 [B,H,N,16]; v: bf16
    [B,H,N,64] (CUDA).  Returns (O bf16 [B,H,N,64], DEN fp32 [B,H,N]) with
    w_ij = 1 + s + s^2/2, s = scale <q_i,k_j>, O_i = sum_{j<=i} w_ij v_j / DEN_i.
    ``scale`` defaults to 1/sqrt(16).  With ``segments`` (the default) the
    work is balanced over the SMs (tk_based_fwd_ws; ``workspace`` is allocated
    here unless given): with fewer heads than SMs each head's sequence is
    split into segments; with more heads than SMs, not a multiple of them, the
    heads' chunks are cut into one equal run per SM.  ``segments=False`` is
    tk_based_fwd (one CTA per head).  Enqueued without synchronising."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.device.type != "cuda":
            raise ValueError(f"{n} must be a CUDA bf16 [B,H,N,D] tensor")
    if q.shape != k.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k [B,H,N,Dqk] and v [B,H,N,Dv] must agree in B, H, N")
    B, H, N, Dqk = q.shape
    Dv = v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=torch.bfloat16, device=q.device)
    if den is None:
        den = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        if not segments:
            rc = _lib.load().tk_based_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), den.data_ptr(),
                                          B, H, N, Dqk, Dv, float(scale), _stream_handle(stream))
            _lib.check(rc, "tk_based_fwd")
            return out, den
        need = based_workspace_bytes(B, H, N) if Dqk == 16 and Dv == 64 else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = _lib.load().tk_based_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), den.data_ptr(),
                                         ws_ptr, ws_bytes, B, H, N, Dqk, Dv, float(scale), _stream_handle(stream))
    _lib.check(rc, "tk_based_fwd_ws")
    return out, den


def hedgehog_workspace_bytes(B: int, H: int, N: int) -> int:
    """Workspace tk_hedgehog_fwd_ws needs on the current device (0: no segments)."""
    return int(_lib.load().tk_hedgehog_workspace_bytes(B, H, N))


def hedgehog(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, wq: torch.Tensor, wk: torch.Tensor,
             out: torch.Tensor | None = None, den: torch.Tensor | None = None, stream=None,
             workspace: torch.Tensor | None = None, segments: bool = True):
    """Causal Hedgehog linear attention.  q, k, v: bf16 [B,H,N,64]; wq, wk:
    bf16 [H,64,64] (CUDA).  phi(x) = [softmax(x W), softmax(-x W)];
    returns (O bf16 [B,H,N,64], DEN fp32 [B,H,N]).  With ``segments`` (the
    default) and fewer heads than SMs, each head's sequence is split into
    segments (tk_hedgehog_fwd_ws; ``workspace`` is allocated here unless
    given); ``segments=False`` is tk_hedgehog_fwd.  Enqueued without
    synchronising."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.device.type != "cuda":
            raise ValueError(f"{n} must be a CUDA bf16 [B,H,N,D] tensor")
    for t, n in ((wq, "wq"), (wk, "wk")):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or t.device.type != "cuda":
            raise ValueError(f"{n} must be a CUDA bf16 [H,d,f] tensor")
    if q.shape != k.shape or v.shape[:3] != q.shape[:3] or wq.shape != wk.shape or wq.shape[0] != q.shape[1]:
        raise ValueError("q, k [B,H,N,d], v [B,H,N,Dv], wq, wk [H,d,f] must agree")
    B, H, N, d = q.shape
    f, Dv = wq.shape[2], v.shape[3]
    q, k, v, wq, wk = (t.contiguous() for t in (q, k, v, wq, wk))
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=torch.bfloat16, device=q.device)
    if den is None:
        den = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        if not segments:
            rc = _lib.load().tk_hedgehog_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                                             out.data_ptr(), den.data_ptr(), B, H, N, d, f, Dv, _stream_handle(stream))
            _lib.check(rc, "tk_hedgehog_fwd")
            return out, den
        need = hedgehog_workspace_bytes(B, H, N) if (d, f, Dv) == (64, 64, 64) else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = _lib.load().tk_hedgehog_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                                            out.data_ptr(), den.data_ptr(), ws_ptr, ws_bytes, B, H, N, d, f, Dv,
                                            _stream_handle(stream))
    _lib.check(rc, "tk_hedgehog_fwd_ws")
    return out, den
