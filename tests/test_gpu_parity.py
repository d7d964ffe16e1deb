"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bar (the tolerance of the attention-forward target): O within max-abs 2e-2
and mean-abs 2e-3 of the oracle, LSE within max-abs 1e-3, over every checked
element.  The GPU rounds P to bf16 before the second contraction and O to
bf16 at the end (as the "ThunderKittens" kernel on 10100.com/article/71410160
does, section "writing a kernel with TK", consumer::compute "convert to bf16
for mma"); both roundings stay well inside the bar.

Small cases are compared in full (head dims 32, 64, 96 and 128; 32 and 96
fill half of the last 64-column box).  The five named workloads run at full size,
in the same single launch the benchmark times, and are compared on sampled
heads (and, for the longest one, sampled rows) that the oracle computes.
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import (WORKLOADS, make_qkv, sample_heads, sample_rows,
                                             workload_inputs)

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _gpu(*ts):
    return [t.cuda() for t in ts]


def _run(q, k, v, causal, scale):
    o, lse = tk.fwd(*_gpu(q, k, v), causal=causal, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    return o.cpu(), lse.cpu()


def _assert_close(o, lse, O_ref, L_ref, what):
    o = o.double().numpy()
    lse = lse.double().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    err = np.abs(o - O_ref)
    lerr = np.abs(lse - L_ref)
    assert err.max() <= O_MAX, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: O mean-abs {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"{what}: LSE max-abs {lerr.max():.3e}"


def _check_full(oracle_mod, q, k, v, causal, scale, what):
    o, lse = _run(q, k, v, causal, scale)
    O_ref, L_ref = oracle_mod.attn_fwd(q, k, v, causal, scale)
    _assert_close(o, lse, O_ref, L_ref, what)
    return o, lse


# ---------------------------------------------------------------- shape sweep

@pytest.mark.parametrize("D", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 384, 1000])
def test_shape_sweep(oracle_mod, N, D, causal):
    q, k, v = make_qkv(1, 2, N, D, 5000 + N + D)
    _check_full(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), f"N={N} D={D} causal={causal}")


def test_batched_heads_small(oracle_mod):
    q, k, v = make_qkv(3, 5, 200, 64, 77)
    _check_full(oracle_mod, q, k, v, True, 0.125, "B3 H5 N200")


# ---------------------------------------------------------------- named workloads

@pytest.mark.parametrize("idx", [1, 2])
def test_workload_full_check(oracle_mod, idx):
    w = WORKLOADS[idx]
    q, k, v = workload_inputs(w)
    _check_full(oracle_mod, q, k, v, w.causal, w.scale, w.name)


@pytest.mark.parametrize("idx", [3, 4, 5])
def test_workload_sampled(oracle_mod, idx):
    """Full-size launch; the oracle checks sampled heads (all rows, or for
    the N=16384 workload a seeded sample of rows including tile edges)."""
    w = WORKLOADS[idx]
    q, k, v = workload_inputs(w)
    o, lse = _run(q, k, v, w.causal, w.scale)
    heads = sample_heads(w, 8 if idx in (3, 4) else 2)
    for b, h in heads:
        qh, kh, vh = q[b, h], k[b, h], v[b, h]
        if w.N <= 4096:
            rows = list(range(w.N))
        else:
            rows = sample_rows(w.N, 384)
        O_ref, L_ref = oracle_mod.attn_fwd_rows(qh, kh, vh, rows, w.causal, w.scale)
        _assert_close(o[b, h, rows], lse[b, h, rows], O_ref, L_ref, f"{w.name} head ({b},{h})")


# ---------------------------------------------------------------- special cases

@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_closed_form(causal):
    """Q = 0: every allowed key weighs the same.  LSE_i = ln|J_i| and O_i is
    the mean of V over J_i (prefix mean under the causal mask)."""
    N, D = 300, 128
    _, k, v = make_qkv(1, 1, N, D, 9)
    q = torch.zeros_like(k)
    o, lse = _run(q, k, v, causal, 0.1)
    vd = v.double().numpy()[0, 0]
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    ref_o = (np.cumsum(vd, axis=0) / counts[:, None]) if causal else np.broadcast_to(vd.mean(0), (N, D))
    _assert_close(o[0, 0], lse[0, 0], ref_o, np.log(counts.astype(np.float64)), "Q=0")


def test_constant_values():
    q, k, _ = make_qkv(1, 2, 333, 64, 10)
    vrow = torch.randn((1, 2, 1, 64), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    v = vrow.expand(1, 2, 333, 64).contiguous()
    o, _ = _run(q, k, v, False, 0.125)
    err = (o.double() - vrow.double()).abs().max().item()
    assert err <= 1e-2, err


def test_causal_first_row_is_first_value():
    q, k, v = make_qkv(1, 1, 257, 128, 12)
    o, lse = _run(q, k, v, True, 1 / math.sqrt(128))
    assert torch.equal(o[0, 0, 0], v[0, 0, 0]), "row 0 sees key 0 only"
    ref = (q[0, 0, 0].double() @ k[0, 0, 0].double()).item() / math.sqrt(128)
    assert abs(lse[0, 0, 0].item() - ref) <= 1e-3


# ---------------------------------------------------------------- metamorphic / determinism

def test_deterministic_bitwise():
    q, k, v = _gpu(*make_qkv(2, 4, 1000, 128, 31))
    o1, l1 = tk.fwd(q, k, v, causal=True)
    o2, l2 = tk.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_head_swap():
    q, k, v = make_qkv(1, 3, 400, 64, 32)
    o, l = _run(q, k, v, False, 0.125)
    perm = [2, 0, 1]
    o2, l2 = _run(q[:, perm].contiguous(), k[:, perm].contiguous(), v[:, perm].contiguous(), False, 0.125)
    assert torch.equal(o2, o[:, perm]) and torch.equal(l2, l[:, perm])


def test_key_permutation_noncausal():
    q, k, v = make_qkv(1, 1, 512, 128, 33)
    o, l = _run(q, k, v, False, 0.09)
    perm = torch.randperm(512, generator=torch.Generator().manual_seed(4))
    o2, l2 = _run(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, 0.09)
    assert (o2.double() - o.double()).abs().max().item() <= 1e-2
    assert (l2.double() - l.double()).abs().max().item() <= 1e-4


def test_side_stream_and_preallocated_outputs(oracle_mod):
    q, k, v = make_qkv(2, 2, 300, 64, 34)
    qd, kd, vd = _gpu(q, k, v)
    out = torch.empty_like(qd)
    lse = torch.empty((2, 2, 300), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    tk.fwd(qd, kd, vd, causal=False, scale=0.2, out=out, lse=lse, stream=s)
    s.synchronize()
    O_ref, L_ref = oracle_mod.attn_fwd(q, k, v, False, 0.2)
    _assert_close(out.cpu(), lse.cpu(), O_ref, L_ref, "side stream")


def test_host_inputs_roundtrip(oracle_mod):
    q, k, v = make_qkv(1, 2, 150, 128, 35)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = tk.fwd(q, k, v, causal=True)
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    O_ref, L_ref = oracle_mod.attn_fwd(q, k, v, True, 1 / math.sqrt(128))
    _assert_close(o, lse, O_ref, L_ref, "host inputs")


# ---------------------------------------------------------------- errors on a GPU

def test_rejects_host_memory_and_misaligned_device_pointer():
    lib = tk.load()
    q, k, v = _gpu(*make_qkv(1, 1, 128, 64, 36))
    o = torch.empty_like(q)
    l = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    host = torch.empty_like(q.cpu())
    rc = lib.tk_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), host.data_ptr(), l.data_ptr(),
                         1, 1, 128, 64, 0, 0.125, None)
    assert rc == tk.STATUS["TK_ERR_NOT_DEVICE_MEMORY"]
    rc = lib.tk_attn_fwd(q.data_ptr() + 2, k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                         1, 1, 127, 64, 0, 0.125, None)
    assert rc == tk.STATUS["TK_ERR_MISALIGNED"]


def test_bounded_wait_reports_timeout_and_context_survives(oracle_mod):
    """A wait that nothing ends gives up after its limit: the status word
    reports the timeout, the kernel returns, and the next call still works."""
    assert tk.device_status()[0] == 0
    tk.selftest_timeout(2_000_000)  # 2 ms
    status, detail = tk.device_status()
    assert status == tk.STATUS["TK_ERR_DEVICE_TIMEOUT"]
    assert detail >> 24 == 4, hex(detail)
    assert tk.device_status()[0] == 0, "status must clear after reading"
    q, k, v = make_qkv(1, 1, 64, 64, 37)
    _check_full(oracle_mod, q, k, v, False, 0.125, "after timeout")


@pytest.mark.gpu
@pytest.mark.parametrize("causal,Nkv", [(False, 700), (True, 700), (True, 1100)])
def test_host_inputs_in_chunks_equal_device_launch(causal, Nkv):
    """Pinned host inputs go to the device in chunks of heads over two streams
    (copies overlapping kernels); each chunk is its own launch over its heads.
    Heads are independent and each launch is deterministic, so the result
    equals one launch over all heads bit for bit."""
    from tiled_attention_tk_gb300 import attention
    from tiled_attention_tk_gb300.inputs import make_qkv_rect
    B, H, Nq, D = 2, 5, 700, 128
    q, k, v = make_qkv_rect(B, H, Nq, Nkv, D, 5150 + Nkv + causal)
    o_dev, l_dev = tk.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h, l_h = attention._fwd_from_host(qh, kh, vh, causal, 1.0 / math.sqrt(D), None, chunk_bytes=600_000)
    torch.cuda.synchronize()
    assert o_h.device.type == "cpu" and o_h.is_pinned()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())
    st, detail = tk.device_status()
    assert st == 0, (st, detail)
