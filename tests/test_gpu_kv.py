"""Parity of the forward with Nq queries against Nkv keys (tk_attn_fwd_kv,
through the C ABI) with the fp64 oracle.

Under the causal mask the queries stand at the end of the key sequence:
query i sees keys j <= i + Nkv - Nq (attention inference over a cache, listed
on the groovesquid.com summary of the ThunderKittens paper).  Bar: the
forward's (O max-abs 2e-2, mean-abs 2e-3; LSE max-abs 1e-3).  The offsets
Nkv - Nq cover multiples of the 128-key tile and values between them, where
a key tile is partly visible to some rows of a query tile but not others.
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import WORKLOADS, make_qkv_rect, sample_heads, sample_rows, workload_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _run(q, k, v, causal, scale):
    o, lse = tk.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def _assert_close(o, lse, O_ref, L_ref, what):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    err, lerr = np.abs(o - O_ref), np.abs(lse - L_ref)
    assert err.max() <= O_MAX, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: O mean-abs {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"{what}: LSE max-abs {lerr.max():.3e}"


@pytest.mark.parametrize("B,H,Nq,Nkv,D,causal", [
    (1, 2, 1, 1000, 128, True),     # one new query against a cache
    (1, 2, 1, 257, 64, False),
    (1, 2, 64, 1024, 128, True),    # offset a multiple of the key tile
    (1, 2, 100, 164, 64, True),     # offset 64: key tiles partly visible to a Q tile
    (1, 2, 128, 129, 128, True),
    (1, 1, 200, 333, 128, True),    # ragged queries and keys
    (2, 3, 640, 1280, 128, True),
    (1, 2, 300, 4096, 64, True),
    (1, 2, 257, 128, 64, False),    # more queries than keys (non-causal)
    (1, 2, 1000, 17, 128, False),
    (1, 2, 384, 384, 64, True),     # equal lengths through the same entry point
    (1, 2, 200, 700, 96, True),     # half-box head dims
    (2, 2, 130, 260, 32, True),
])
def test_kv_parity(oracle_mod, B, H, Nq, Nkv, D, causal):
    q, k, v = make_qkv_rect(B, H, Nq, Nkv, D, 7000 + Nq + Nkv + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = _run(q, k, v, causal, scale)
    O_ref, L_ref = oracle_mod.attn_fwd(q, k, v, causal, scale)
    _assert_close(o, lse, O_ref, L_ref, f"B{B} H{H} Nq{Nq} Nkv{Nkv} D{D} causal={causal}")


def test_equal_lengths_match_square_entry_point():
    """tk_attn_fwd_kv with Nq = Nkv is tk_attn_fwd: same kernel, bitwise."""
    q, k, v = (t.cuda() for t in make_qkv_rect(2, 2, 300, 300, 128, 7100))
    for causal in (False, True):
        o1 = torch.empty_like(q)
        l1 = torch.empty((2, 2, 300), dtype=torch.float32, device="cuda")
        o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
        sh = torch.cuda.current_stream().cuda_stream
        tk.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), l1.data_ptr(),
                   2, 2, 300, 128, causal, 0.09, sh)
        tk.fwd_kv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(),
                      2, 2, 300, 300, 128, causal, 0.09, sh)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_rejects_more_queries_than_keys():
    q, k, v = (t.cuda() for t in make_qkv_rect(1, 1, 200, 100, 64, 7200))
    with pytest.raises(tk.TkError) as e:
        tk.fwd(q, k, v, causal=True)
    assert e.value.name == "TK_ERR_BAD_SHAPE"


def test_kv_workload_sampled(oracle_mod):
    """The benchmark's cache workload (2048 queries at the end of 16384 keys,
    32 heads), in the launch the benchmark times, checked on sampled heads
    and rows."""
    w = WORKLOADS[6]
    q, k, v = workload_inputs(w)
    o, lse = _run(q, k, v, w.causal, w.scale)
    for b, h in sample_heads(w, 3):
        rows = sample_rows(w.N, 48)
        O_ref, L_ref = oracle_mod.attn_fwd_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        _assert_close(o[b, h, rows], lse[b, h, rows], O_ref, L_ref, f"{w.name} head ({b},{h})")
