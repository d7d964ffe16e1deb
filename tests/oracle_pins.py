"""Pins for the fp64 oracle: checks against facts fixed by the definition of
softmax attention, not against the oracle itself.

Each ``check_*`` takes ``fwd(q, k, v, causal, scale) -> (O, LSE)`` so the same
checks run on the real oracle (tests/test_oracle_pins.py) and on copies of it
with a planted mistake (tests/test_oracle_mutants.py), which every mistake
must fail.

Definition pinned (the "ThunderKittens" attention forward on
10100.com/article/71410160, section "writing a kernel with TK",
attn_fwd_template consumer::compute and consumer::finish; the inner loop on
alanwu.xyz/posts/thunderkittens): O_i = sum_j softmax_j(scale <Q_i,K_j>) V_j,
LSE_i = ln sum_j exp(scale <Q_i,K_j>), j over all keys, or j <= i (causal).
With Nq queries against Nkv >= Nq keys the causal queries stand at the end
of the key sequence: j <= i + Nkv - Nq (attention inference over a cache,
listed on the groovesquid.com summary of the ThunderKittens paper).
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F
from scipy.special import logsumexp, softmax

from tiled_attention_tk_gb300.inputs import make_qkv


def bf(x) -> torch.Tensor:
    """Exactly representable values as a bf16 tensor (asserts exactness)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float64), dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), "value not exactly representable in bf16"
    return b


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


# --- special cases with closed forms ---------------------------------------

def check_constant_values(fwd):
    """Every key row carries the same value vector v -> O_i = v for every row,
    whatever the scores (the weights of a row sum to one)."""
    g = torch.Generator().manual_seed(3)
    for causal in (False, True):
        B, H, N, D = 2, 2, 19, 8
        q, k, _ = make_qkv(B, H, N, D, 41)
        vrow = torch.randn((B, H, 1, D), generator=g).to(torch.bfloat16)
        v = vrow.expand(B, H, N, D).contiguous()
        O, _ = fwd(q, k, v, causal, 0.5)
        _close(O, np.broadcast_to(vrow.double().numpy(), (B, H, N, D)), 1e-12,
               f"constant V (causal={causal})")


def check_single_key(fwd):
    """N = 1: the only key takes all the weight.  O = V_0 and
    LSE = scale * <q_0, k_0>."""
    q = bf([[[[1.5, -2.0, 0.25, 3.0]]]])
    k = bf([[[[0.5, 1.0, -4.0, 2.0]]]])
    v = bf([[[[7.0, -1.0, 0.125, 2.5]]]])
    scale = 0.75
    dot = math.fsum([1.5 * 0.5, -2.0 * 1.0, 0.25 * -4.0, 3.0 * 2.0])
    for causal in (False, True):
        O, L = fwd(q, k, v, causal, scale)
        _close(O, v.double().numpy(), 0.0, "N=1 output")
        _close(L, np.array([[[scale * dot]]]), 1e-15, "N=1 LSE")


def check_causal_first_row(fwd):
    """Causal row 0 sees key 0 only: O_0 = V_0, LSE_0 = scale * <q_0, k_0>."""
    q, k, v = make_qkv(1, 3, 23, 16, 77)
    scale = 0.3
    O, L = fwd(q, k, v, True, scale)
    qd, kd = q.double().numpy(), k.double().numpy()
    for h in range(3):
        _close(O[0, h, 0], v.double().numpy()[0, h, 0], 1e-15, "causal row 0 output")
        dot = math.fsum((qd[0, h, 0] * kd[0, h, 0]).tolist())
        _close(L[0, h, 0], scale * dot, 1e-13, "causal row 0 LSE")


def check_zero_queries(fwd):
    """Q = 0 makes every score 0, so each allowed key weighs 1/|J_i|:
    LSE_i = ln |J_i| (ln N, or ln(i+1) under the causal mask) and O_i is the
    mean of V over J_i (the prefix mean under the causal mask).  This fixes
    the causal direction, the tail and the natural-log LSE convention."""
    B, H, N, D = 1, 2, 37, 16
    _, k, v = make_qkv(B, H, N, D, 5)
    q = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    vd = v.double().numpy()
    O, L = fwd(q, k, v, False, 0.9)
    _close(L, np.full((B, H, N), math.log(N)), 1e-13, "Q=0 LSE non-causal")
    _close(O, np.broadcast_to(vd.mean(axis=2, keepdims=True), O.shape), 1e-13,
           "Q=0 output non-causal")
    O, L = fwd(q, k, v, True, 0.9)
    counts = np.arange(1, N + 1, dtype=np.float64)
    _close(L, np.broadcast_to(np.log(counts), (B, H, N)), 1e-13, "Q=0 LSE causal")
    prefix_mean = np.cumsum(vd, axis=2) / counts[None, None, :, None]
    _close(O, prefix_mean, 1e-13, "Q=0 output causal")


def check_two_keys(fwd):
    """D = 1, N = 2, scores chosen so the two-way softmax has a closed form:
    w_1 = 1 / (1 + exp(s_0 - s_1)), LSE = max(s) + ln(1 + exp(-|s_0 - s_1|)).
    Includes logits near 2e4, where an exponential without the max
    subtracted overflows, and scores 2000 apart within one row, where
    subtracting anything but the maximum overflows."""
    cases = [  # (q rows, k rows, v rows, scale)
        ([1.0, -2.0], [0.5, 1.5], [3.0, -1.0], 1.0),
        ([200.0, -100.0], [100.0, 99.0], [1.0, 2.0], 1.0),
        ([200.0, -100.0], [100.0, 90.0], [1.0, 2.0], 1.0),  # scores 2000 apart
        ([0.0625, 3.0], [-8.0, 8.0], [0.5, -0.25], 0.5),
    ]
    for qs, ks, vs, scale in cases:
        q = bf(np.array(qs).reshape(1, 1, 2, 1))
        k = bf(np.array(ks).reshape(1, 1, 2, 1))
        v = bf(np.array(vs).reshape(1, 1, 2, 1))
        O, L = fwd(q, k, v, False, scale)
        for i in range(2):
            s0, s1 = scale * qs[i] * ks[0], scale * qs[i] * ks[1]
            w1 = 1.0 / (1.0 + math.exp(min(s0 - s1, 700.0)))
            o = vs[0] * (1.0 - w1) + vs[1] * w1
            lse = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
            _close(O[0, 0, i, 0], o, 1e-12 * max(1.0, abs(o)), "two-key output")
            _close(L[0, 0, i], lse, 1e-12 * max(1.0, abs(lse)), "two-key LSE")
        # causal: row 0 sees key 0 only, row 1 both keys
        O, L = fwd(q, k, v, True, scale)
        _close(O[0, 0, 0, 0], vs[0], 0.0, "two-key causal row 0")
        _close(L[0, 0, 0], scale * qs[0] * ks[0], 1e-12 * max(1.0, abs(scale * qs[0] * ks[0])),
               "two-key causal row 0 LSE")


# --- library routines --------------------------------------------------------

def check_against_library(fwd):
    """fp64 PyTorch scaled_dot_product_attention for O and scipy's
    logsumexp of the masked score matrix for LSE, on small seeded inputs
    (square causal masks in PyTorch are top-left aligned: key j <= query i)."""
    shapes = [(1, 2, 7, 4, False), (2, 1, 9, 8, True), (1, 1, 33, 64, True),
              (1, 1, 20, 128, False), (1, 3, 5, 3, True), (1, 1, 130, 64, False)]
    for idx, (B, H, N, D, causal) in enumerate(shapes):
        q, k, v = make_qkv(B, H, N, D, 300 + idx)
        scale = 1.0 / math.sqrt(D) * (1.0 + 0.1 * idx)
        O, L = fwd(q, k, v, causal, scale)
        qd, kd, vd = q.double(), k.double(), v.double()
        O_ref = F.scaled_dot_product_attention(qd, kd, vd, is_causal=causal, scale=scale)
        S = (scale * torch.matmul(qd, kd.transpose(-1, -2))).numpy()
        if causal:
            S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
        L_ref = logsumexp(S, axis=-1)
        _close(O, O_ref.numpy(), 1e-12, f"O vs torch SDPA fp64 {B,H,N,D,causal}")
        _close(L, L_ref, 1e-12, f"LSE vs scipy logsumexp {B,H,N,D,causal}")


# --- invariants ----------------------------------------------------------------

def check_key_permutation(fwd):
    """Without a mask the keys form a set: permuting K and V rows together
    leaves O and LSE unchanged."""
    q, k, v = make_qkv(1, 2, 29, 16, 88)
    perm = torch.randperm(29, generator=torch.Generator().manual_seed(1))
    O1, L1 = fwd(q, k, v, False, 0.25)
    O2, L2 = fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, 0.25)
    _close(O2, O1, 1e-13, "key permutation O")
    _close(L2, L1, 1e-13, "key permutation LSE")


def check_head_independence(fwd):
    """Each (b,h) head is its own problem: a head computed alone equals the
    same head inside a larger batch."""
    q, k, v = make_qkv(2, 3, 17, 8, 99)
    for causal in (False, True):
        O, L = fwd(q, k, v, causal, 0.4)
        for b, h in [(0, 0), (1, 2), (0, 1)]:
            o1, l1 = fwd(q[b:b + 1, h:h + 1].contiguous(), k[b:b + 1, h:h + 1].contiguous(),
                         v[b:b + 1, h:h + 1].contiguous(), causal, 0.4)
            _close(o1[0, 0], O[b, h], 0.0, "head independence O")
            _close(l1[0, 0], L[b, h], 0.0, "head independence LSE")


def check_scale_homogeneity(fwd):
    """Scores depend on scale*Q only: (2Q, scale/2) gives the same result as
    (Q, scale).  Doubling a bf16 value is exact."""
    q, k, v = make_qkv(1, 1, 21, 16, 12)
    for causal in (False, True):
        O1, L1 = fwd(q, k, v, causal, 0.5)
        O2, L2 = fwd((q.float() * 2).to(torch.bfloat16), k, v, causal, 0.25)
        _close(O2, O1, 1e-13, "scale homogeneity O")
        _close(L2, L1, 1e-13, "scale homogeneity LSE")


def check_key_shift(fwd):
    """Adding one vector c to every key adds scale*<q_i, c> to every score of
    row i: O is unchanged and LSE_i grows by exactly that amount.  Small
    integers keep every input exact in bf16."""
    g = torch.Generator().manual_seed(5)
    N, D = 13, 8
    qi = torch.randint(-3, 4, (1, 1, N, D), generator=g).double()
    ki = torch.randint(-3, 4, (1, 1, N, D), generator=g).double()
    vi = torch.randint(-5, 6, (1, 1, N, D), generator=g).double()
    c = torch.randint(-4, 5, (D,), generator=g).double()
    scale = 0.125
    for causal in (False, True):
        O1, L1 = fwd(bf(qi), bf(ki), bf(vi), causal, scale)
        O2, L2 = fwd(bf(qi), bf(ki + c), bf(vi), causal, scale)
        shift = scale * (qi[0, 0] @ c).numpy()
        _close(O2, O1, 1e-12, "key shift O")
        _close(L2[0, 0], L1[0, 0] + shift, 1e-12, "key shift LSE")


# --- queries against a longer key sequence (Nq != Nkv) ------------------------

def check_rect_zero_queries(fwd):
    """Q = 0 with Nq = 7 queries over Nkv = 20 keys: every allowed key weighs
    1/|J_i|.  Non-causal: LSE_i = ln 20 and O_i = mean of all V rows.
    Causal, queries at the end of the key sequence: query i sees keys
    0..i+13, so LSE_i = ln(i + 14) and O_i is the mean of V_0..V_{i+13}."""
    B, H, Nq, Nkv, D = 1, 2, 7, 20, 16
    _, k, v = make_qkv(B, H, Nkv, D, 6)
    q = torch.zeros((B, H, Nq, D), dtype=torch.bfloat16)
    vd = v.double().numpy()
    O, L = fwd(q, k, v, False, 0.7)
    _close(L, np.full((B, H, Nq), math.log(Nkv)), 1e-13, "rect Q=0 LSE non-causal")
    _close(O, np.broadcast_to(vd.mean(axis=2, keepdims=True), O.shape), 1e-13,
           "rect Q=0 output non-causal")
    O, L = fwd(q, k, v, True, 0.7)
    counts = np.arange(Nkv - Nq + 1, Nkv + 1, dtype=np.float64)
    _close(L, np.broadcast_to(np.log(counts), (B, H, Nq)), 1e-13, "rect Q=0 LSE causal")
    prefix_mean = (np.cumsum(vd, axis=2) / np.arange(1, Nkv + 1)[None, None, :, None])[:, :, Nkv - Nq:]
    _close(O, prefix_mean, 1e-13, "rect Q=0 output causal")


def check_rect_against_library(fwd):
    """Non-causal Nq != Nkv (both Nq < Nkv and Nq > Nkv) against fp64 PyTorch
    scaled_dot_product_attention and scipy's logsumexp; and one query
    against Nkv keys under the causal mask, which sees every key, against the
    same routines without a mask."""
    cases = [(1, 2, 5, 23, 8, False), (2, 1, 31, 9, 16, False), (1, 1, 1, 37, 64, True),
             (1, 2, 1, 130, 128, True)]
    for idx, (B, H, Nq, Nkv, D, causal) in enumerate(cases):
        q = make_qkv(B, H, Nq, D, 500 + idx)[0]
        _, k, v = make_qkv(B, H, Nkv, D, 600 + idx)
        scale = 1.0 / math.sqrt(D)
        O, L = fwd(q, k, v, causal, scale)
        qd, kd, vd = q.double(), k.double(), v.double()
        O_ref = F.scaled_dot_product_attention(qd, kd, vd, scale=scale)
        L_ref = logsumexp((scale * torch.matmul(qd, kd.transpose(-1, -2))).numpy(), axis=-1)
        _close(O, O_ref.numpy(), 1e-12, f"rect O vs torch SDPA {B,H,Nq,Nkv,D,causal}")
        _close(L, L_ref, 1e-12, f"rect LSE vs scipy logsumexp {B,H,Nq,Nkv,D,causal}")


def check_rect_is_suffix_of_square(fwd):
    """Causal queries at the end of the key sequence are the last Nq rows of
    the square causal problem whose first Nkv - Nq queries are anything:
    row i of the rectangular problem equals row i + Nkv - Nq of the square
    one, computed with the same arithmetic (exactly equal)."""
    B, H, Nq, Nkv, D = 1, 2, 9, 30, 16
    _, k, v = make_qkv(B, H, Nkv, D, 71)
    qfull = make_qkv(B, H, Nkv, D, 72)[0]
    q = qfull[:, :, Nkv - Nq:].contiguous()
    O, L = fwd(q, k, v, True, 0.3)
    Of, Lf = fwd(qfull, k, v, True, 0.3)
    _close(O, Of[:, :, Nkv - Nq:], 0.0, "rect causal rows = square causal suffix (O)")
    _close(L, Lf[:, :, Nkv - Nq:], 0.0, "rect causal rows = square causal suffix (LSE)")


ALL_CHECKS = [check_constant_values, check_single_key, check_causal_first_row,
              check_zero_queries, check_two_keys, check_against_library,
              check_key_permutation, check_head_independence, check_scale_homogeneity,
              check_key_shift, check_rect_zero_queries, check_rect_against_library,
              check_rect_is_suffix_of_square]


def check_weights(weights_fn):
    """The weight matrix of one head: rows are probability vectors (sum 1,
    non-negative), masked keys weigh exactly 0, and it equals scipy's
    softmax of the masked score matrix."""
    for causal in (False, True):
        q, k, _ = make_qkv(1, 1, 11, 8, 123)
        scale = 0.35
        P = weights_fn(q[0, 0], k[0, 0], causal, scale)
        assert np.all(P >= 0.0)
        _close(P.sum(axis=1), np.ones(11), 1e-12, "weights sum to one")
        S = scale * (q[0, 0].double() @ k[0, 0].double().T).numpy()
        if causal:
            assert np.all(P[np.triu_indices(11, 1)] == 0.0), "masked weights must be 0"
            S = np.where(np.tril(np.ones((11, 11), dtype=bool)), S, -np.inf)
        _close(P, softmax(S, axis=1), 1e-13, "weights vs scipy softmax")
