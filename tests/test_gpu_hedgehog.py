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


def _run(q, k, v, wq, wk):
    o, den = tk.hedgehog(q.cuda(), k.cuda(), v.cuda(), wq.cuda(), wk.cuda())
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
