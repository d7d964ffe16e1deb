"""Every kernel past 2^31 elements per tensor, through the C ABI.

B4 H4112 N1024 D128 holds 2^31 + 2^23 elements per tensor (4.3 GB in bf16), so
the element offsets of the last 64 heads exceed 31 bits, and the byte offsets
of the fp32 dQ accumulator exceed 32 bits from its middle on.  Heads repeat with period 61 (head h is a
seeded head h mod 61 of one make_qkv draw): a 32-bit wrap of an element or
byte offset moves by 16384 heads, which is not a multiple of 61, so it reads
another head's data and fails the comparison.  Heads on both sides of the
2^31-element boundary, and the last head, are compared with the fp64 oracle
under the usual bars (O max-abs 2e-2, mean 2e-3, LSE 1e-3; gradients max-abs
0.02 max|G| + 1e-4, mean-abs 0.01 mean|G| + 1e-5).

The same construction covers the other kernels: Based on B8 H4100 N4096 (Q, K
and V all past 2^31 elements: 16 and 64 dims per row), Hedgehog on B2 H4100
N4096 (64 dims, its per-head projections repeating with the heads), and the
GEMM with C = 40960 x 53248 (2.18e9 elements), checked on rows beyond the
2^31-element mark; each with its own bars (Based and Hedgehog: O max-abs 2e-2,
DEN relative 1e-2; GEMM: one bf16 ulp of C plus the fp32 accumulation bound).
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

B, H, N, D = 4, 4112, 1024, 128
PERIOD = 61
HEADS = [0, 8191, 16383, 16384, B * H - 1]  # 16384 heads = 2^31 elements


def _big(block):
    """[B, H, N, D] on the GPU with head h = block[0, h mod PERIOD]."""
    idx = torch.arange(B * H, device="cuda") % PERIOD
    return torch.index_select(block[0].cuda(), 0, idx).view(B, H, N, D)


def _need_memory(gb):
    free, _ = torch.cuda.mem_get_info()
    if free < gb * (1 << 30):
        pytest.skip(f"needs {gb} GB of free device memory")


def _head(t, h):
    return t[h // H, h % H]


def test_forward_beyond_2p31_elements(oracle_mod):
    _need_memory(40)
    assert B * H * N * D > 2 ** 31
    q1, k1, v1 = make_qkv(1, PERIOD, N, D, 9700)
    q, k, v = _big(q1), _big(k1), _big(v1)
    scale = 1.0 / math.sqrt(D)
    o, lse = tk.fwd(q, k, v, causal=False, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    del q, k, v
    try:
        for h in HEADS:
            j = h % PERIOD
            sl = (slice(0, 1), slice(j, j + 1))
            O_ref, L_ref = oracle_mod.attn_fwd(q1[sl].contiguous(), k1[sl].contiguous(), v1[sl].contiguous(),
                                               False, scale)
            got_o = _head(o, h).cpu().double().numpy()
            got_l = _head(lse, h).cpu().double().numpy()
            err = np.abs(got_o - O_ref[0, 0])
            lerr = np.abs(got_l - L_ref[0, 0])
            assert np.all(np.isfinite(got_o)), f"head {h}: non-finite O"
            assert err.max() <= 2e-2 and err.mean() <= 2e-3, f"head {h}: O max {err.max():.3e} mean {err.mean():.3e}"
            assert lerr.max() <= 1e-3, f"head {h}: LSE max {lerr.max():.3e}"
    finally:
        del o, lse
        torch.cuda.empty_cache()


def test_backward_beyond_2p31_elements(oracle_mod):
    _need_memory(70)
    q1, k1, v1 = make_qkv(1, PERIOD, N, D, 9710)
    do1 = make_qkv(1, PERIOD, N, D, 9711)[0]
    q, k, v, do = _big(q1), _big(k1), _big(v1), _big(do1)
    scale = 1.0 / math.sqrt(D)
    o, lse = tk.fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = tk.bwd(q, k, v, o, lse, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    del q, k, v, do, o, lse
    try:
        for h in HEADS:
            j = h % PERIOD
            sl = (slice(0, 1), slice(j, j + 1))
            ref = oracle_mod.attn_bwd(q1[sl].contiguous(), k1[sl].contiguous(), v1[sl].contiguous(),
                                      do1[sl].contiguous(), True, scale)
            for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
                got = _head(g, h).cpu().double().numpy()
                r = r[0, 0]
                err = np.abs(got - r)
                assert np.all(np.isfinite(got)), f"head {h} {name}: non-finite"
                assert err.max() <= 0.02 * np.abs(r).max() + 1e-4, f"head {h} {name}: max err {err.max():.3e}"
                assert err.mean() <= 0.01 * np.abs(r).mean() + 1e-5, f"head {h} {name}: mean err {err.mean():.3e}"
    finally:
        del dq, dk, dv
        torch.cuda.empty_cache()


def _big_heads(block, B, H):
    """[B, H, N, d] on the GPU with head h = block[0, h mod PERIOD]."""
    idx = torch.arange(B * H, device="cuda") % PERIOD
    return torch.index_select(block[0].cuda(), 0, idx).view(B, H, *block.shape[2:])


def _linear_rows(N):
    return np.concatenate([np.arange(0, 64), np.arange(N - 192, N)])


def test_based_beyond_2p31_elements(oracle_mod):
    _need_memory(60)
    Bb, Hb, Nb = 8, 4100, 4096
    assert Bb * Hb * Nb * 16 > 2 ** 31
    g = torch.Generator().manual_seed(9720)
    q1 = torch.randn((1, PERIOD, Nb, 16), generator=g).to(torch.bfloat16)
    k1 = torch.randn((1, PERIOD, Nb, 16), generator=g).to(torch.bfloat16)
    v1 = torch.randn((1, PERIOD, Nb, 64), generator=g).to(torch.bfloat16)
    q, k, v = _big_heads(q1, Bb, Hb), _big_heads(k1, Bb, Hb), _big_heads(v1, Bb, Hb)
    o, den = tk.based(q, k, v)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    del q, k, v
    rows = _linear_rows(Nb)
    try:
        for h in [0, 8191, 8192, 32767, 32768, Bb * Hb - 1]:
            j = h % PERIOD
            O_ref, D_ref = oracle_mod.based(q1[0, j], k1[0, j], v1[0, j], 0.25, rows=rows)
            got_o = o[h // Hb, h % Hb].cpu().double().numpy()[rows]
            got_d = den[h // Hb, h % Hb].cpu().double().numpy()[rows]
            assert np.abs(got_o - O_ref).max() <= 2e-2, f"head {h}: O"
            assert (np.abs(got_d - D_ref) / np.abs(D_ref)).max() <= 1e-2, f"head {h}: DEN"
    finally:
        del o, den
        torch.cuda.empty_cache()


def test_hedgehog_beyond_2p31_elements(oracle_mod):
    _need_memory(40)
    Bh, Hh, Nh = 2, 4100, 4096
    assert Bh * Hh * Nh * 64 > 2 ** 31
    g = torch.Generator().manual_seed(9730)
    q1, k1, v1 = (torch.randn((1, PERIOD, Nh, 64), generator=g).to(torch.bfloat16) for _ in range(3))
    wq1 = (torch.randn((PERIOD, 64, 64), generator=g) * 0.2).to(torch.bfloat16)
    wk1 = (torch.randn((PERIOD, 64, 64), generator=g) * 0.2).to(torch.bfloat16)
    q, k, v = _big_heads(q1, Bh, Hh), _big_heads(k1, Bh, Hh), _big_heads(v1, Bh, Hh)
    hidx = torch.arange(Hh, device="cuda") % PERIOD
    wq = torch.index_select(wq1.cuda(), 0, hidx)
    wk = torch.index_select(wk1.cuda(), 0, hidx)
    o, den = tk.hedgehog(q, k, v, wq, wk)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    del q, k, v
    rows = _linear_rows(Nh)
    try:
        for h in [0, 8191, 8192, Bh * Hh - 1]:
            j, hh = h % PERIOD, (h % Hh) % PERIOD  # data head, projection head
            O_ref, D_ref = oracle_mod.hedgehog(q1[0, j], k1[0, j], v1[0, j], wq1[hh], wk1[hh], rows=rows)
            got_o = o[h // Hh, h % Hh].cpu().double().numpy()[rows]
            got_d = den[h // Hh, h % Hh].cpu().double().numpy()[rows]
            assert np.abs(got_o - O_ref).max() <= 2e-2, f"head {h}: O"
            assert (np.abs(got_d - D_ref) / np.abs(D_ref)).max() <= 1e-2, f"head {h}: DEN"
    finally:
        del o, den
        torch.cuda.empty_cache()


def test_gemm_beyond_2p31_elements(oracle_mod):
    _need_memory(20)
    M, N, K = 40960, 53248, 128
    assert M * N > 2 ** 31
    g = torch.Generator().manual_seed(9740)
    a = torch.randn((M, K), generator=g).to(torch.bfloat16)
    b = torch.randn((N, K), generator=g).to(torch.bfloat16)
    c = tk.gemm(a.cuda(), b.cuda(), b_kmajor=True)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    first_big = 2 ** 31 // N + 1  # rows from here on start past 2^31 elements of C
    rows = np.concatenate([np.arange(0, 16), np.arange(first_big, first_big + 16), np.arange(M - 16, M)])
    try:
        ref = oracle_mod.gemm(a, b, True, rows=rows)
        got = c[torch.from_numpy(rows).cuda()].cpu().double().numpy()
        mag = np.abs(a.double().numpy()[rows]) @ np.abs(b.double().numpy()).T
        bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * mag
        assert not bad.any(), f"{bad.sum()} elements off, first at {np.argwhere(bad)[:3]}"
    finally:
        del c
        torch.cuda.empty_cache()
