"""Pins for the oracle's Based linear attention: facts fixed by the definition
and by the feature-map identity, not by the oracle itself.

Each ``check_*`` takes ``based(q, k, v, scale, rows=None) -> (O, DEN)`` so the
same checks run on the real oracle and on copies with a planted mistake.
Definition pinned (causal, per head): s_ij = scale <q_i, k_j>,
w_ij = 1 + s_ij + s_ij^2 / 2, DEN_i = sum_{j<=i} w_ij, O_i = sum_{j<=i} w_ij v_j / DEN_i
(the Based feature map, the second-order Taylor expansion of exp; the kernel is
listed as "Based Linear Attention" among the new kernels on thebeat.tech
"ThunderKittens 2.0").
"""
from __future__ import annotations

import math

import numpy as np
import torch

from tests.oracle_pins import bf


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def _qkv(B, H, N, Dqk, Dv, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, N, Dqk), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, N, Dqk), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, N, Dv), generator=g).to(torch.bfloat16)
    return q, k, v


def check_zero_queries(based):
    """Q = 0: every weight is 1, so DEN_i = i + 1 and O_i is the prefix mean
    of V (pins the causal direction and the normalisation)."""
    _, k, v = _qkv(1, 2, 23, 16, 8, 1)
    q = torch.zeros_like(k)
    O, DEN = based(q, k, v, 0.25)
    n = np.arange(1, 24, dtype=np.float64)
    _close(DEN, np.broadcast_to(n, DEN.shape), 1e-13, "Q=0 DEN")
    _close(O, np.cumsum(v.double().numpy(), axis=2) / n[None, None, :, None], 1e-13, "Q=0 O")


def check_first_row_and_constant_v(based):
    """Row 0 sees key 0 only: O_0 = V_0, DEN_0 = 1 + s + s^2/2; and with every
    V row equal to v, O_i = v for every row."""
    q, k, v = _qkv(1, 1, 9, 16, 4, 2)
    O, DEN = based(q, k, v, 0.3)
    s = 0.3 * float((q[0, 0, 0].double() @ k[0, 0, 0].double()))
    _close(O[0, 0, 0], v[0, 0, 0].double().numpy(), 1e-15, "row 0 output")
    _close(DEN[0, 0, 0], 1.0 + s + 0.5 * s * s, 1e-13, "row 0 DEN")
    vc = v[:, :, :1].expand(1, 1, 9, 4).contiguous()
    O, _ = based(q, k, vc, 0.3)
    _close(O, np.broadcast_to(vc.double().numpy(), O.shape), 1e-13, "constant V")


def check_two_keys_by_hand(based):
    """N = 2, Dqk = 1 with small integers: row 1 has s = (q1 k0, q1 k1) * scale
    = (2, -1) * 0.5 = (1, -0.5): w = (2.5, 0.625), DEN = 3.125,
    O = (2.5 * 3 + 0.625 * 7) / 3.125 = 3.8 for v = (3, 7)."""
    q = bf(np.array([1.0, 2.0]).reshape(1, 1, 2, 1))
    k = bf(np.array([1.0, -0.5]).reshape(1, 1, 2, 1))
    v = bf(np.array([3.0, 7.0]).reshape(1, 1, 2, 1))
    O, DEN = based(q, k, v, 0.5)
    _close(DEN[0, 0, 1], 3.125, 1e-15, "two keys DEN")
    _close(O[0, 0, 1, 0], 3.8, 1e-14, "two keys O")


def _phi(x, scale):
    """Explicit Taylor feature map: phi(x) . phi(y) = 1 + s + s^2/2 with
    s = scale <x, y>: [1, sqrt(scale) x, scale / sqrt(2) * vec(x x^T)]."""
    n, d = x.shape
    quad = np.einsum("ni,nj->nij", x, x).reshape(n, d * d)
    return np.concatenate([np.ones((n, 1)), math.sqrt(scale) * x, scale / math.sqrt(2.0) * quad], axis=1)


def check_recurrent_form(based):
    """The linear (recurrent) evaluation through the explicit feature map:
    running state S_i = sum_{j<=i} phi(k_j) v_j^T and z_i = sum_{j<=i} phi(k_j),
    O_i = phi(q_i)^T S_i / phi(q_i)^T z_i.  A different algorithm (prefix sums
    of outer products) for the same quantity."""
    q, k, v = _qkv(1, 2, 40, 16, 8, 3)
    scale = 0.25
    O, DEN = based(q, k, v, scale)
    for h in range(2):
        pq = _phi(q[0, h].double().numpy(), scale)
        pk = _phi(k[0, h].double().numpy(), scale)
        S = np.cumsum(np.einsum("nf,nd->nfd", pk, v[0, h].double().numpy()), axis=0)
        z = np.cumsum(pk, axis=0)
        den = np.einsum("nf,nf->n", pq, z)
        num = np.einsum("nf,nfd->nd", pq, S)
        _close(DEN[0, h], den, 1e-10 * np.abs(den).max(), "recurrent form DEN")
        _close(O[0, h], num / den[:, None], 1e-11, "recurrent form O")


def check_rows_entry_and_heads(based):
    """The rows entry computes the same rows as the whole problem, head by head."""
    q, k, v = _qkv(2, 2, 30, 16, 8, 4)
    O, DEN = based(q, k, v, 0.2)
    for b, h in [(0, 1), (1, 0)]:
        rows = [0, 5, 29]
        Or, Dr = based(q[b, h], k[b, h], v[b, h], 0.2, rows=rows)
        _close(Or, O[b, h, rows], 0.0, "rows entry O")
        _close(Dr, DEN[b, h, rows], 0.0, "rows entry DEN")


def check_scale_homogeneity(based):
    """Scores depend on scale * q only: (2q, scale/2) equals (q, scale)."""
    q, k, v = _qkv(1, 1, 17, 16, 8, 5)
    O1, D1 = based(q, k, v, 0.5)
    O2, D2 = based((q.float() * 2).to(torch.bfloat16), k, v, 0.25)
    _close(O2, O1, 1e-13, "scale homogeneity O")
    _close(D2, D1, 1e-12, "scale homogeneity DEN")


BASED_CHECKS = [check_zero_queries, check_first_row_and_constant_v, check_two_keys_by_hand,
                check_recurrent_form, check_rows_entry_and_heads, check_scale_homogeneity]
