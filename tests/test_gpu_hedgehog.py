"""Parity of the Hedgehog linear attention (tk_hedgehog_fwd, through the C ABI)
with the fp64 oracle's quadratic form.

The kernel runs the chunked linear form with bf16 operands (the projections'
inputs, the feature maps, the in-chunk weights and the carried state enter
the tensor-core products as bf16; accumulation and the softmaxes are fp32; O
is stored as bf16).  Bar: O within max-abs 2e-2 and mean-abs 2e-3; DEN within
relative 1e-2 (max) and 4e-3 (mean).  Each weight passes three bf16 roundings
(phi_q, phi_k, then P or the carried state), at most 3 * 2^-9 = 5.9e-3
relative; with few rows the mean is the max of a handful of them.
"""
import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk

pytestmark = pytest.mark.gpu


def _inputs(B, H, N, seed, wscale=0.2):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    wq = (torch.randn((H, 64, 64), generator=g) * wscale).to(torch.bfloat16)
    wk = (torch.randn((H, 64, 64), generator=g) * wscale).to(torch.bfloat16)
    return q, k, v, wq, wk


def _run(q, k, v, wq, wk, segments=True):
    o, den = tk.hedgehog(q.cuda(), k.cuda(), v.cuda(), wq.cuda(), wk.cuda(), segments=segments)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    return o.cpu().double().numpy(), den.cpu().double().numpy()


def _check_heads(oracle_mod, q, k, v, wq, wk, o, den, heads, rows=None, what=""):
    for b, h in heads:
        O_ref, D_ref = oracle_mod.hedgehog(q[b, h], k[b, h], v[b, h], wq[h], wk[h], rows=rows)
        oo = o[b, h] if rows is None else o[b, h, rows]
        dd = den[b, h] if rows is None else den[b, h, rows]
        assert np.all(np.isfinite(oo)) and np.all(np.isfinite(dd)), f"{what}: non-finite output"
        err = np.abs(oo - O_ref)
        rel = np.abs(dd - D_ref) / np.abs(D_ref)
        assert err.max() <= 2e-2, f"{what} ({b},{h}): O max-abs {err.max():.3e}"
        assert err.mean() <= 2e-3, f"{what} ({b},{h}): O mean-abs {err.mean():.3e}"
        assert rel.max() <= 1e-2, f"{what} ({b},{h}): DEN max-rel {rel.max():.3e}"
        assert rel.mean() <= 4e-3, f"{what} ({b},{h}): DEN mean-rel {rel.mean():.3e}"


@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 300, 1000])
def test_hedgehog_shapes(oracle_mod, N):
    q, k, v, wq, wk = _inputs(1, 2, N, 500 + N)
    o, den = _run(q, k, v, wq, wk)
    _check_heads(oracle_mod, q, k, v, wq, wk, o, den, [(0, 0), (0, 1)], what=f"N={N}")


@pytest.mark.parametrize("wscale", [0.05, 1.0])
def test_hedgehog_projection_scales_and_heads(oracle_mod, wscale):
    """Nearly uniform features (small W) and spiky ones (large W, where the
    softmax's maximum matters)."""
    q, k, v, wq, wk = _inputs(2, 3, 400, 600, wscale)
    o, den = _run(q, k, v, wq, wk)
    _check_heads(oracle_mod, q, k, v, wq, wk, o, den, [(0, 0), (1, 2)], what=f"wscale={wscale}")


def test_hedgehog_deterministic():
    q, k, v, wq, wk = _inputs(1, 4, 700, 601)
    o1, d1 = _run(q, k, v, wq, wk)
    o2, d2 = _run(q, k, v, wq, wk)
    assert np.array_equal(o1, o2) and np.array_equal(d1, d2)


def test_hedgehog_bench_workload_sampled(oracle_mod):
    """The benchmark's B8 H16 N4096 launch, sampled heads and rows."""
    q, k, v, wq, wk = _inputs(8, 16, 4096, 602)
    o, den = _run(q, k, v, wq, wk)
    rows = [0, 1, 127, 128, 2047, 2048, 4094, 4095]
    _check_heads(oracle_mod, q, k, v, wq, wk, o, den, [(0, 0), (7, 15)], rows=rows, what="B8H16N4096")


# ---------------------------------------------------------------- segmented sequences
# Fewer heads than SMs (the binding's default path, tk_hedgehog_fwd_ws): each
# head is split into segments that start from the sum of the fp32 partial
# states before them (formed by a first pass with the same feature map).

def test_hedgehog_segments_long_sequence(oracle_mod):
    """B1 H2 N20000: sampled rows across many segment boundaries and the ragged end."""
    B, H, N = 1, 2, 20000
    assert tk.hedgehog_workspace_bytes(B, H, N) > 0
    q, k, v, wq, wk = _inputs(B, H, N, 510)
    o, den = _run(q, k, v, wq, wk)
    rows = sorted({0, 1, 127, 128, 639, 640, 641, 1279, 1280, 5119, 5120, 12799, 12800, 19200, 19967, 19968,
                   19999} | {int(x) for x in np.random.default_rng(8).integers(0, N, 10)})
    _check_heads(oracle_mod, q, k, v, wq, wk, o, den, [(0, 0), (0, 1)], rows=rows, what="segmented N20000")


@pytest.mark.parametrize("N", [1000, 2049, 9000])
def test_hedgehog_segments_match_one_cta_per_head(oracle_mod, N):
    q, k, v, wq, wk = _inputs(1, 3, N, 520 + N)
    o1, d1 = _run(q, k, v, wq, wk, segments=True)
    o2, d2 = _run(q, k, v, wq, wk, segments=False)
    # the carried state enters the products as bf16: two fp32 states that differ in
    # their last bits may round to neighbouring bf16 values (2^-8 apart at most)
    assert np.abs(o1 - o2).max() <= 1e-2 and (np.abs(d1 - d2) / np.abs(d2)).max() <= 2.0 ** -8
    if N <= 2049:
        _check_heads(oracle_mod, q, k, v, wq, wk, o1, d1, [(0, 0), (0, 2)], what=f"segmented N={N}")


def test_hedgehog_segments_deterministic():
    q, k, v, wq, wk = _inputs(1, 2, 12000, 530)
    o1, d1 = _run(q, k, v, wq, wk)
    o2, d2 = _run(q, k, v, wq, wk)
    assert np.array_equal(o1, o2) and np.array_equal(d1, d2)


def test_hedgehog_workspace_checks():
    B, H, N = 1, 2, 20000
    need = tk.hedgehog_workspace_bytes(B, H, N)
    assert need > 0 and need % 256 == 0
    q, k, v, wq, wk = (t.cuda() for t in _inputs(B, H, N, 540))
    o = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device="cuda")
    den = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    lib = tk.load()

    def call(ws_ptr, ws_bytes):
        return lib.tk_hedgehog_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                                      o.data_ptr(), den.data_ptr(), ws_ptr, ws_bytes, B, H, N, 64, 64, 64, None)
    assert call(None, 0) == tk.STATUS["TK_ERR_NULL_PTR"]
    assert call(ws.data_ptr(), need - 256) == tk.STATUS["TK_ERR_WORKSPACE"]
    assert call(ws.data_ptr() + 16, need) == tk.STATUS["TK_ERR_WORKSPACE"]
    assert call(den.data_ptr(), need) == tk.STATUS["TK_ERR_ALIAS"]
    assert call(ws.data_ptr(), need) == 0
    torch.cuda.synchronize()
    assert tk.device_status()[0] == 0
