"""Pins for the oracle's GEMM (C = A op(B) in fp64): facts fixed by the
definition of a matrix product, not by the oracle itself.

Each ``check_*`` takes ``gemm(a, b, b_kmajor, rows=None) -> C`` so the same
checks run on the real oracle and on copies of it with a planted mistake
(tests/test_oracle_mutants.py).  Definition pinned: C[m,n] = sum_k A[m,k] B'[k,n]
with B' = B^T for B stored [N,K] and B' = B for B stored [K,N]
(10100.com/article/71410160, section on grid-level abstraction, names GEMM as the
workload the tile abstractions are built around).
"""
from __future__ import annotations

import numpy as np
import torch

from tests.oracle_pins import bf


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def check_hand_example(gemm):
    """A 2x3 by 3x2 product with small integers, worked by hand:
    [[1,2,3],[4,5,6]] @ [[7,8],[9,10],[11,12]] = [[58,64],[139,154]]."""
    a = bf([[1, 2, 3], [4, 5, 6]])
    b_kn = bf([[7, 8], [9, 10], [11, 12]])
    expect = [[58, 64], [139, 154]]
    _close(gemm(a, b_kn, False), expect, 0.0, "hand example, B [K,N]")
    _close(gemm(a, b_kn.T.contiguous(), True), expect, 0.0, "hand example, B [N,K]")


def check_identity(gemm):
    """A I = A, for I stored either way (a square identity is its own
    transpose, so this also pins the inner index)."""
    g = torch.Generator().manual_seed(8)
    a = torch.randn((5, 7), generator=g).to(torch.bfloat16)
    eye = torch.eye(7).to(torch.bfloat16)
    for kmajor in (False, True):
        _close(gemm(a, eye, kmajor), a.double().numpy(), 0.0, f"A I = A (b_kmajor={kmajor})")


def check_permutation_columns(gemm):
    """B' a permutation matrix picks columns of A: C[:, n] = A[:, pi(n)].
    Stored [K,N] the 1s sit at (pi(n), n); stored [N,K] at (n, pi(n)).  A
    transposed B index fails this."""
    g = torch.Generator().manual_seed(9)
    K, N = 6, 4
    a = torch.randn((3, K), generator=g).to(torch.bfloat16)
    pi = [4, 0, 5, 2]
    b_kn = torch.zeros((K, N))
    for n, k in enumerate(pi):
        b_kn[k, n] = 1.0
    expect = a.double().numpy()[:, pi]
    _close(gemm(a, b_kn.to(torch.bfloat16), False), expect, 0.0, "permutation, B [K,N]")
    _close(gemm(a, b_kn.T.contiguous().to(torch.bfloat16), True), expect, 0.0, "permutation, B [N,K]")


def check_against_numpy(gemm):
    """float64 numpy matmul of the bf16 values, both layouts, odd sizes."""
    g = torch.Generator().manual_seed(10)
    for M, N, K in [(7, 9, 13), (33, 16, 40), (1, 5, 300)]:
        a = torch.randn((M, K), generator=g).to(torch.bfloat16)
        b = torch.randn((K, N), generator=g).to(torch.bfloat16)
        ref = np.matmul(a.double().numpy(), b.double().numpy())
        tol = 1e-12 * max(1.0, np.abs(ref).max())
        _close(gemm(a, b, False), ref, tol, f"vs numpy {M,N,K} B [K,N]")
        _close(gemm(a, b.T.contiguous(), True), ref, tol, f"vs numpy {M,N,K} B [N,K]")


def check_rows_entry(gemm):
    """Selected rows equal the same rows of the whole product."""
    g = torch.Generator().manual_seed(11)
    a = torch.randn((20, 24), generator=g).to(torch.bfloat16)
    b = torch.randn((12, 24), generator=g).to(torch.bfloat16)
    whole = gemm(a, b, True)
    rows = [0, 3, 19, 7]
    _close(gemm(a, b, True, rows=rows), whole[rows], 0.0, "rows entry")


def check_linearity(gemm):
    """(A1 + A2) B = A1 B + A2 B with small integers (every value exact)."""
    g = torch.Generator().manual_seed(12)
    a1 = torch.randint(-4, 5, (6, 10), generator=g).double()
    a2 = torch.randint(-4, 5, (6, 10), generator=g).double()
    b = torch.randint(-4, 5, (10, 8), generator=g).double()
    lhs = gemm(bf(a1 + a2), bf(b), False)
    rhs = gemm(bf(a1), bf(b), False) + gemm(bf(a2), bf(b), False)
    _close(lhs, rhs, 0.0, "linearity in A")


GEMM_CHECKS = [check_hand_example, check_identity, check_permutation_columns, check_against_numpy,
               check_rows_entry, check_linearity]
