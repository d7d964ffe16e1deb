"""Pins for the fp64 backward oracle (gradient of sum(O * dO)): checks
against facts fixed by the mathematics, not against the oracle's code.

Each check takes ``bwd(q, k, v, do, causal, scale) -> (dQ, dK, dV)`` so the
same checks run on the oracle and on copies with a planted mistake.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from tests.oracle_pins import bf, _close
from tiled_attention_tk_gb300.inputs import make_qkv


def _dout(B, H, N, D, seed):
    return make_qkv(B, H, N, D, seed)[0]


def check_bwd_against_autograd(bwd):
    """PyTorch autograd through fp64 scaled_dot_product_attention."""
    shapes = [(1, 2, 7, 4, False), (2, 1, 9, 8, True), (1, 1, 33, 64, True), (1, 1, 20, 128, False),
              (1, 3, 5, 3, True)]
    for idx, (B, H, N, D, causal) in enumerate(shapes):
        q, k, v = make_qkv(B, H, N, D, 600 + idx)
        do = _dout(B, H, N, D, 700 + idx)
        scale = 1.0 / math.sqrt(D) * (1.0 + 0.1 * idx)
        dQ, dK, dV = bwd(q, k, v, do, causal, scale)
        qd, kd, vd = (t.double().requires_grad_() for t in (q, k, v))
        o = F.scaled_dot_product_attention(qd, kd, vd, is_causal=causal, scale=scale)
        (o * do.double()).sum().backward()
        _close(dQ, qd.grad.numpy(), 1e-11, f"dQ vs autograd {B,H,N,D,causal}")
        _close(dK, kd.grad.numpy(), 1e-11, f"dK vs autograd {B,H,N,D,causal}")
        _close(dV, vd.grad.numpy(), 1e-11, f"dV vs autograd {B,H,N,D,causal}")


def check_bwd_finite_differences(bwd):
    """Central differences of f = sum(O * dO) computed with the (pinned)
    forward oracle.  Inputs are drawn from {+-1, +-1.25, +-1.5, +-1.75} and
    moved by h = 2^-7, so every perturbed value is exact in bf16; the O(h^2)
    truncation error sets the tolerance."""
    rng = np.random.default_rng(9)
    N, D, h = 4, 3, 2.0 ** -7
    vals = np.array([1.0, 1.25, 1.5, 1.75])
    for causal in (False, True):
        x = [rng.choice(vals, size=(1, 1, N, D)) * rng.choice([-1.0, 1.0], size=(1, 1, N, D))
             for _ in range(4)]
        q, k, v, do = (bf(a) for a in x)
        scale = 0.5
        dQ, dK, dV = bwd(q, k, v, do, causal, scale)
        dod = do.double().numpy()

        def f(qq, kk, vv):
            O, _ = oracle.attn_fwd(bf(qq), bf(kk), bf(vv), causal, scale)
            return float((O * dod).sum())

        for which, grad in ((0, dQ), (1, dK), (2, dV)):
            base = [a.copy() for a in x[:3]]
            for i in range(N):
                for d in range(D):
                    up = [a.copy() for a in base]
                    dn = [a.copy() for a in base]
                    up[which][0, 0, i, d] += h
                    dn[which][0, 0, i, d] -= h
                    fd = (f(*up) - f(*dn)) / (2 * h)
                    assert abs(fd - grad[0, 0, i, d]) <= 2e-3 * max(1.0, abs(fd)), (
                        f"finite difference {('dQ', 'dK', 'dV')[which]}[{i},{d}] causal={causal}: "
                        f"{fd} vs {grad[0, 0, i, d]}")


def check_bwd_closed_forms(bwd):
    """dO = 0 gives zero gradients; a single key takes weight 1, so dQ = dK = 0
    and dV = dO; value rows all equal make every dP_ij of a row equal, so the
    softmax term vanishes and dQ = dK = 0."""
    q, k, v = make_qkv(1, 2, 13, 8, 31)
    z = torch.zeros_like(q)
    for causal in (False, True):
        dQ, dK, dV = bwd(q, k, v, z, causal, 0.4)
        _close(dQ, np.zeros(dQ.shape), 0.0, "dO=0 dQ")
        _close(dK, np.zeros(dK.shape), 0.0, "dO=0 dK")
        _close(dV, np.zeros(dV.shape), 0.0, "dO=0 dV")
    q1, k1, v1 = make_qkv(1, 1, 1, 16, 32)
    do1 = _dout(1, 1, 1, 16, 33)
    dQ, dK, dV = bwd(q1, k1, v1, do1, False, 0.7)
    _close(dQ, np.zeros(dQ.shape), 1e-15, "N=1 dQ")
    _close(dK, np.zeros(dK.shape), 1e-15, "N=1 dK")
    _close(dV, do1.double().numpy(), 1e-15, "N=1 dV")
    vrow = torch.randn((1, 2, 1, 8), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    vc = vrow.expand(1, 2, 13, 8).contiguous()
    do = _dout(1, 2, 13, 8, 34)
    for causal in (False, True):
        dQ, dK, _ = bwd(q, k, vc, do, causal, 0.4)
        _close(dQ, np.zeros(dQ.shape), 1e-12, "constant V dQ")
        _close(dK, np.zeros(dK.shape), 1e-12, "constant V dK")


def check_bwd_invariants(bwd):
    """Every row's weights sum to one and the scores are unchanged by a
    common shift of the keys, so sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i
    (causal or not).  Scores depend on scale*Q only: (2Q, scale/2) leaves dK
    and dV unchanged and halves dQ."""
    q, k, v = make_qkv(2, 2, 17, 8, 41)
    do = _dout(2, 2, 17, 8, 42)
    for causal in (False, True):
        dQ, dK, dV = bwd(q, k, v, do, causal, 0.3)
        _close(dK.sum(axis=2), np.zeros((2, 2, 8)), 1e-12, "sum of dK")
        _close(dV.sum(axis=2), do.double().numpy().sum(axis=2), 1e-12, "sum of dV")
        q2 = (q.float() * 2).to(torch.bfloat16)
        dQ2, dK2, dV2 = bwd(q2, k, v, do, causal, 0.15)
        _close(dQ2, dQ / 2, 1e-12, "scale homogeneity dQ")
        _close(dK2, dK, 1e-12, "scale homogeneity dK")
        _close(dV2, dV, 1e-12, "scale homogeneity dV")


ALL_BWD_CHECKS = [check_bwd_against_autograd, check_bwd_finite_differences,
                  check_bwd_closed_forms, check_bwd_invariants]
