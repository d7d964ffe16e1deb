"""Pins for the oracle's Hedgehog linear attention: facts fixed by the
definition, not by the oracle itself.

Each ``check_*`` takes ``hedgehog(q, k, v, wq, wk, rows=None) -> (O, DEN)`` (one
head) so the same checks run on the real oracle and on copies with a planted
mistake.  Definition pinned: phi(x) = [softmax(x W), softmax(-x W)],
w_ij = phi_q(q_i) . phi_k(k_j), causal, O_i = sum_{j<=i} w_ij v_j / DEN_i (the
Hedgehog feature map; the kernel is listed as "LoLCATS Hedgehog Linear
Attention" among the new kernels on thebeat.tech "ThunderKittens 2.0").
"""
from __future__ import annotations

import numpy as np
import torch
from scipy.special import softmax

from tests.oracle_pins import bf


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def _inputs(N, d, f, Dv, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((N, d), generator=g).to(torch.bfloat16)
    k = torch.randn((N, d), generator=g).to(torch.bfloat16)
    v = torch.randn((N, Dv), generator=g).to(torch.bfloat16)
    wq = (torch.randn((d, f), generator=g) * 0.2).to(torch.bfloat16)
    wk = (torch.randn((d, f), generator=g) * 0.2).to(torch.bfloat16)
    return q, k, v, wq, wk


def check_zero_projection(hh):
    """W = 0: both softmaxes are uniform, phi = [1/f ...], so w_ij = 2/f for
    every pair: DEN_i = 2 (i+1) / f and O_i is the prefix mean of V."""
    q, k, v, wq, _ = _inputs(19, 8, 4, 5, 1)
    z = torch.zeros_like(wq)
    O, DEN = hh(q, k, v, z, z)
    n = np.arange(1, 20, dtype=np.float64)
    _close(DEN, 2.0 * n / 4, 1e-14, "W=0 DEN")
    _close(O, np.cumsum(v.double().numpy(), axis=0) / n[:, None], 1e-13, "W=0 O")


def check_one_feature(hh):
    """f = 1: each softmax over one entry is 1, so phi = [1, 1] and w_ij = 2
    whatever q, k and W are (pins the normalisation over the features)."""
    q, k, v, wq, wk = _inputs(11, 8, 1, 3, 2)
    O, DEN = hh(q, k, v, wq, wk)
    _close(DEN, 2.0 * np.arange(1, 12), 1e-13, "f=1 DEN")
    _close(O, np.cumsum(v.double().numpy(), axis=0) / np.arange(1, 12)[:, None], 1e-13, "f=1 O")


def check_against_scipy(hh):
    """The feature maps from scipy's softmax of the fp64 projections and the
    causal weighted mean written with numpy (a different route to each step)."""
    q, k, v, wq, wk = _inputs(30, 16, 8, 6, 3)
    qd, kd, vd, wqd, wkd = (t.double().numpy() for t in (q, k, v, wq, wk))
    zq, zk = qd @ wqd, kd @ wkd
    pq = np.concatenate([softmax(zq, axis=1), softmax(-zq, axis=1)], axis=1)
    pk = np.concatenate([softmax(zk, axis=1), softmax(-zk, axis=1)], axis=1)
    w = np.tril(pq @ pk.T)
    den = w.sum(axis=1)
    O, DEN = hh(q, k, v, wq, wk)
    _close(DEN, den, 1e-13, "scipy DEN")
    _close(O, (w @ vd) / den[:, None], 1e-13, "scipy O")


def check_shift_invariance(hh):
    """softmax(z + c) = softmax(z): adding a column vector u to W changes
    z = x W by the same amount c = x.u in every feature of a row, so phi (and
    everything after it) is unchanged.  Small integers keep W exact."""
    g = torch.Generator().manual_seed(4)
    q = torch.randint(-2, 3, (9, 6), generator=g).double()
    k = torch.randint(-2, 3, (9, 6), generator=g).double()
    v = torch.randint(-3, 4, (9, 4), generator=g).double()
    w = torch.randint(-2, 3, (6, 5), generator=g).double() * 0.25
    u = torch.randint(-2, 3, (6, 1), generator=g).double() * 0.25
    O1, D1 = hh(bf(q), bf(k), bf(v), bf(w), bf(w))
    O2, D2 = hh(bf(q), bf(k), bf(v), bf(w + u), bf(w + u))
    _close(O2, O1, 1e-13, "shift invariance O")
    _close(D2, D1, 1e-13, "shift invariance DEN")


def check_rows_entry(hh):
    q, k, v, wq, wk = _inputs(25, 8, 4, 3, 5)
    O, DEN = hh(q, k, v, wq, wk)
    rows = [0, 7, 24]
    Or, Dr = hh(q, k, v, wq, wk, rows=rows)
    _close(Or, O[rows], 0.0, "rows entry O")
    _close(Dr, DEN[rows], 0.0, "rows entry DEN")


HEDGEHOG_CHECKS = [check_zero_projection, check_one_feature, check_against_scipy, check_shift_invariance,
                   check_rows_entry]
