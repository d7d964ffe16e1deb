"""Parity of the CUDA backward (through the C ABI) with the fp64 backward
oracle, on the forward outputs of the CUDA forward.

Bar, per gradient G in (dQ, dK, dV), over every element:
    max |G_gpu - G_ref|  <= 0.02 * max |G_ref|  + 1e-4
    mean|G_gpu - G_ref|  <= 0.01 * mean|G_ref| + 1e-5
sized from a CPU emulation of the kernel's roundings (bf16 P and dS, Delta
from the bf16 forward output, fp32 LSE, bf16 outputs), whose errors stay
below 0.0063 and 0.006 of those scales; the bar leaves about 3x for the fp32
summation order of the tensor cores and the dQ atomics.  The absolute floor
covers gradients that are exactly zero (a single key: dQ = dK = 0), where the
kernel leaves fp32 rounding noise of order 1e-6 (Delta from the bf16 output
against dP from the tensor core).
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def _run(q, k, v, do, causal, scale):
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, do))
    o, lse = tk.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = tk.bwd(qd, kd, vd, o, lse, gd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    return dq.cpu(), dk.cpu(), dv.cpu()


def _check(oracle_mod, q, k, v, do, causal, scale, what):
    got = _run(q, k, v, do, causal, scale)
    ref = oracle_mod.attn_bwd(q, k, v, do, causal, scale)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = g.double().numpy()
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        err = np.abs(g - r)
        assert err.max() <= 0.02 * np.abs(r).max() + 1e-4, (
            f"{what} {name}: max err {err.max():.3e} vs max|ref| {np.abs(r).max():.3e}")
        assert err.mean() <= 0.01 * np.abs(r).mean() + 1e-5, (
            f"{what} {name}: mean err {err.mean():.3e} vs mean|ref| {np.abs(r).mean():.3e}")
    return got


@pytest.mark.parametrize("D", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 300])
def test_bwd_shape_sweep(oracle_mod, N, D, causal):
    q, k, v = make_qkv(1, 2, N, D, 9000 + N + D)
    do = make_qkv(1, 2, N, D, 9500 + N)[0]
    _check(oracle_mod, q, k, v, do, causal, 1.0 / math.sqrt(D), f"N={N} D={D} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_several_tiles(oracle_mod, causal):
    q, k, v = make_qkv(2, 3, 640, 128, 9100)
    do = make_qkv(2, 3, 640, 128, 9101)[0]
    _check(oracle_mod, q, k, v, do, causal, 1.0 / math.sqrt(128), f"B2H3N640 causal={causal}")


def test_bwd_wide_logits(oracle_mod):
    q, k, v = make_qkv(1, 4, 512, 128, 9200, "wide")
    do = make_qkv(1, 4, 512, 128, 9201)[0]
    _check(oracle_mod, q, k, v, do, False, 1.0 / math.sqrt(128), "wide logits")


def test_bwd_invariants_and_determinism():
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i hold for the exact gradient;
    dK and dV are also bitwise reproducible (dQ sums atomically)."""
    q, k, v = make_qkv(1, 2, 384, 64, 9300)
    do = make_qkv(1, 2, 384, 64, 9301)[0]
    dq, dk, dv = _run(q, k, v, do, True, 0.125)
    scale_k = dk.double().abs().sum(dim=2)
    assert (dk.double().sum(dim=2).abs() <= 0.02 * scale_k + 1e-3).all()
    sv = dv.double().sum(dim=2)
    sd = do.double().sum(dim=2)
    assert (sv - sd).abs().max().item() <= 0.02 * sd.abs().max().item() + 1e-2
    dq2, dk2, dv2 = _run(q, k, v, do, True, 0.125)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert (dq.double() - dq2.double()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("D", [32, 64, 96, 128])
def test_bwd_persistent_units(oracle_mod, D):
    """Without the mask the grid is persistent: B2 H40 N1000 has 80 heads x 8
    key tiles = 640 units, about four per CTA on 152 SMs, so every CTA runs
    several units in a row (the next unit's Q and dO loading while the last
    one finishes, K and V reloaded, dK and dV reused).  The first, a middle
    and the last head against the oracle's backward; dK and dV bitwise the
    same in a second launch."""
    B, H, N = 2, 40, 1000
    q, k, v = make_qkv(B, H, N, D, 9600 + D)
    do = make_qkv(B, H, N, D, 9601 + D)[0]
    scale = 1.0 / math.sqrt(D)
    got = _run(q, k, v, do, False, scale)
    for b, h in [(0, 0), (1, 7), (1, H - 1)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle_mod.attn_bwd(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(),
                                  do[sl].contiguous(), False, scale)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            g = g[sl].double().numpy()
            err = np.abs(g - r)
            assert err.max() <= 0.02 * np.abs(r).max() + 1e-4, (D, b, h, name, err.max())
            assert err.mean() <= 0.01 * np.abs(r).mean() + 1e-5, (D, b, h, name, err.mean())
    again = _run(q, k, v, do, False, scale)
    assert torch.equal(got[1], again[1]) and torch.equal(got[2], again[2])


@pytest.mark.parametrize("idx,heads", [(4, [(0, 0), (15, 31)]), (3, [(3, 15)])])
def test_bwd_bench_workload_sampled(oracle_mod, idx, heads):
    """The benchmark's backward launches at full size (B16 H32 N1024 D128 wide
    logits; B4 H16 N4096 D128 causal), with the incoming gradient the
    benchmark draws, checked on sampled heads against the oracle's backward of
    those heads."""
    from tiled_attention_tk_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[idx]
    q, k, v = workload_inputs(w)
    do = make_qkv(w.B, w.H, w.N, w.D, 1000 * w.index + 500, "normal")[0]
    got = _run(q, k, v, do, w.causal, w.scale)
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle_mod.attn_bwd(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(),
                                  do[sl].contiguous(), w.causal, w.scale)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            g = g[sl].double().numpy()
            err = np.abs(g - r)
            assert err.max() <= 0.02 * np.abs(r).max() + 1e-4, (
                f"{w.name} head ({b},{h}) {name}: max err {err.max():.3e} vs max|ref| {np.abs(r).max():.3e}")
            assert err.mean() <= 0.01 * np.abs(r).mean() + 1e-5, (
                f"{w.name} head ({b},{h}) {name}: mean err {err.mean():.3e}")


@pytest.mark.parametrize("D", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_dq_rows_all_written_over_poisoned_buffers(oracle_mod, causal, D):
    """Every dQ row is written and the accumulator is re-zeroed per call: dQ
    and the workspace start as NaN bytes (0xFF), the workspace is used twice
    in a row, and every dQ row must come out finite and equal to the
    oracle's, over several heads, six query tiles (a ragged last one) and,
    under the causal mask, 1 to 6 key tiles adding into a query tile; at
    D = 64 (bulk reductions of staged tiles) and D = 128 (vector reductions),
    and at D = 32 and 96, which run on those kernels with their missing
    columns read as zeros (dQ, dK and dV rows are exactly D wide here)."""
    B, H, N = 2, 3, 700
    scale = 1.0 / math.sqrt(D)
    q, k, v = make_qkv(B, H, N, D, 9400 + causal + D)
    do = make_qkv(B, H, N, D, 9402 + causal + D)[0]
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, do))
    o, lse = tk.fwd(qd, kd, vd, causal=causal, scale=scale)
    ws = torch.full((tk.bwd_workspace_bytes(B, H, N, D),), 0xFF, dtype=torch.uint8, device="cuda")
    lib = tk.load()
    outs = []
    for _ in range(2):
        dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
        rc = lib.tk_attn_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), gd.data_ptr(),
                             lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                             ws.numel(), B, H, N, D, int(causal), scale, None)
        assert rc == 0, tk.strerror(rc)
        torch.cuda.synchronize()
        status, detail = tk.device_status()
        assert status == 0, f"device status {status} detail {detail:#x}"
        outs.append((dq.cpu(), dk.cpu(), dv.cpu()))
    refs = oracle_mod.attn_bwd(q, k, v, do, causal, scale)
    for got in outs:
        for name, t, ref in zip(("dQ", "dK", "dV"), got, refs):
            g = t.double().numpy()
            assert np.all(np.isfinite(g)), f"{name} rows left unwritten: {np.argwhere(~np.isfinite(g))[:4]}"
            err = np.abs(g - ref)
            assert err.max() <= 0.02 * np.abs(ref).max() + 1e-4, name
            assert err.mean() <= 0.01 * np.abs(ref).mean() + 1e-5, name
