"""The forward and backward past 2^31 elements per tensor, through the C ABI.

B4 H4112 N1024 D128 holds 2^31 + 2^23 elements per tensor (4.3 GB in bf16), so
the element offsets of the last 64 heads exceed 31 bits, and the byte offsets
of the fp32 dQ accumulator exceed 32 bits from its middle on.  Heads repeat with period 61 (head h is a
seeded head h mod 61 of one make_qkv draw): a 32-bit wrap of an element or
byte offset moves by 16384 heads, which is not a multiple of 61, so it reads
another head's data and fails the comparison.  Heads on both sides of the
2^31-element boundary, and the last head, are compared with the fp64 oracle
under the usual bars (O max-abs 2e-2, mean 2e-3, LSE 1e-3; gradients max-abs
0.02 max|G| + 1e-4, mean-abs 0.01 mean|G| + 1e-5).
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
