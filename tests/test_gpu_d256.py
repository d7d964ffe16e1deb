"""Parity of the head-dim-256 forward (its own kernel: one Q tile per work
unit, two S slots in TMEM) with the fp64 oracle, through the C ABI.

Bar: the forward's (O max-abs 2e-2, mean-abs 2e-3; LSE max-abs 1e-3), over
every element.  Shapes: one key tile and ragged tails; the causal diagonal;
several heads and units per CTA (so the K/V slots, the S slots and the Q
buffer are reused across units); queries at the end of a longer key sequence;
wide logits (many rescales); bitwise determinism.
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import make_qkv, make_qkv_rect

pytestmark = pytest.mark.gpu

D = 256


def _check(oracle_mod, q, k, v, causal, scale, what):
    o, lse = tk.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    O_ref, L_ref = oracle_mod.attn_fwd(q, k, v, causal, scale)
    o = o.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite"
    err = np.abs(o - O_ref)
    assert err.max() <= 2e-2, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= 2e-3, f"{what}: O mean-abs {err.mean():.3e}"
    assert np.abs(lse - L_ref).max() <= 1e-3, f"{what}: LSE max-abs {np.abs(lse - L_ref).max():.3e}"
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 255, 384, 1000])
def test_d256_shapes(oracle_mod, N, causal):
    q, k, v = make_qkv(1, 2, N, D, 8600 + N)
    _check(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), f"N={N} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_d256_many_units(oracle_mod, causal):
    """B2 H5 N2048: 160 units of 16 key tiles over the SMs, so CTAs run
    several units back to back."""
    q, k, v = make_qkv(2, 5, 2048, D, 8700 + causal)
    _check(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), f"B2 H5 N2048 causal={causal}")


def test_d256_wide_logits(oracle_mod):
    q, k, v = make_qkv(1, 3, 700, D, 8800, "wide")
    _check(oracle_mod, q, k, v, False, 1.0 / math.sqrt(D), "wide logits")


@pytest.mark.parametrize("Nq,Nkv,causal", [(100, 300, True), (257, 1000, True), (300, 129, False)])
def test_d256_queries_against_longer_keys(oracle_mod, Nq, Nkv, causal):
    q, k, v = make_qkv_rect(1, 2, Nq, Nkv, D, 8900 + Nq)
    _check(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), f"Nq={Nq} Nkv={Nkv}")


def test_d256_causal_mirrored_pairs(oracle_mod):
    """Under the causal mask with more query-tile pairs than CTAs, the first
    heads run their Q tiles in mirrored pairs (tile n-1-i, then tile i, on one
    CTA) and the rest heaviest first.  B1 H40 N2048 (16 Q tiles, 8 pairs per
    head): 21 heads in pairs on the device's 152 SMs.  Heads on both sides of
    that boundary, and the first and last, in full against the oracle; the
    whole launch finite."""
    H, N = 40, 2048
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    hp = N // 128 // 2
    paired = max(0, (H * hp - min(H * 2 * hp, sms)) // hp)
    assert 0 < paired < H, paired
    q, k, v = make_qkv(1, H, N, D, 8100)
    scale = 1.0 / 16.0
    o, lse = tk.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    for h in sorted({0, paired - 1, paired, H - 1}):
        O_ref, L_ref = oracle_mod.attn_fwd(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], True, scale)
        err = np.abs(o[:, h:h + 1] - O_ref)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (h, err.max(), err.mean())
        assert np.abs(lse[:, h:h + 1] - L_ref).max() <= 1e-3, h


def test_d256_deterministic():
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 1500, D, 9000))
    o1, l1 = tk.fwd(q, k, v, causal=True)
    o2, l2 = tk.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
