"""Parity of the GEMM (tk_gemm, through the C ABI) with the fp64 oracle.

Bar, per element: |C_gpu - C_ref| <= 2^-8 |C_ref| + 2^-20 (|A| |B'|)[m,n].
The first term is one bf16 ulp of the result (the rounding of C is half an
ulp; an fp32 sum that lands next to a rounding boundary may round to the
neighbour); the second bounds the fp32 accumulation error by a margin of
about 16x over K * 2^-24 * sum |a b| / sqrt(K) for these sizes.  Shapes cover
one tile, ragged M, N and K, both B layouts, data-parallel-only schedules
(fewer tiles than SMs among them), a stream-K schedule with a partial last
wave, the CTA-pair path (ragged and whole-wave shapes, both B layouts) and
the benchmark's 8192^3 launch (pairs) on sampled rows.
"""
import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, b_kmajor, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((M, K), generator=g).to(torch.bfloat16)
    b = torch.randn((N, K) if b_kmajor else (K, N), generator=g).to(torch.bfloat16)
    return a, b


def _check(oracle_mod, a, b, b_kmajor, c, rows=None, what=""):
    ref = oracle_mod.gemm(a, b, b_kmajor, rows=rows)
    ad, bd = a.double().abs().numpy(), b.double().abs().numpy()
    if rows is not None:
        ad = ad[rows]
    mag = ad @ (bd.T if b_kmajor else bd)
    got = c.double().cpu().numpy() if rows is None else c.double().cpu().numpy()[rows]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * mag
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{what}: error {err[worst]:.3e} > bound {bound[worst]:.3e} "
                                  f"at {worst} (ref {ref[worst]:.4e})")


def _run(a, b, b_kmajor, stream_k):
    c = tk.gemm(a.cuda(), b.cuda(), b_kmajor=b_kmajor, stream_k=stream_k)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"
    return c.cpu()


@pytest.mark.parametrize("b_kmajor", [True, False])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (1, 8, 8), (130, 264, 72), (256, 512, 1024),
                                   (1000, 1000, 520), (300, 136, 2056)])
def test_gemm_small(oracle_mod, M, N, K, b_kmajor):
    a, b = _inputs(M, N, K, b_kmajor, M + N + K)
    for stream_k in (True, False):
        c = _run(a, b, b_kmajor, stream_k)
        _check(oracle_mod, a, b, b_kmajor, c, what=f"{M}x{N}x{K} kmajor={b_kmajor} sk={stream_k}")


@pytest.mark.parametrize("b_kmajor", [True, False])
def test_gemm_fewer_tiles_than_sms(oracle_mod, b_kmajor):
    """4 x 8 = 32 output tiles: one wave, whole tiles (stream-K does not pay
    here and the schedule leaves it out)."""
    M, N, K = 512, 2048, 4096
    a, b = _inputs(M, N, K, b_kmajor, 21)
    assert tk.gemm_workspace_bytes(M, N, K, True) == 0
    c = _run(a, b, b_kmajor, True)
    _check(oracle_mod, a, b, b_kmajor, c, what="32 tiles")


@pytest.mark.parametrize("b_kmajor", [True, False])
def test_gemm_stream_k_partial_wave(oracle_mod, b_kmajor):
    """12 x 20 = 240 pair tiles, K = 4096: whole-tile waves, then the partial
    wave plus one wave split in K over the pairs (each CTA of a pair writes its
    128 rows of the partial).  Checked on two rows of every 128-row block (so
    every tile and both CTAs' halves), for stream-K on and off."""
    M, N, K = 3000, 5120, 4096
    a, b = _inputs(M, N, K, b_kmajor, 22)
    assert tk.gemm_workspace_bytes(M, N, K, True) > 0
    # 12 x 20 = 240 pair tiles: 3.2 waves over the pairs, the last partial
    # wave plus one split in K
    assert tk.gemm_uses_pairs(M, N, K, True) and tk.gemm_uses_pairs(M, N, K, False)
    rows = sorted({r for blk in range(0, M, 128) for r in (blk + 3, min(blk + 127, M - 1))})
    for stream_k in (True, False):
        c = _run(a, b, b_kmajor, stream_k)
        _check(oracle_mod, a, b, b_kmajor, c, rows=rows, what=f"3000x5120x4096 sk={stream_k}")


def test_gemm_deterministic():
    a, b = _inputs(3000, 5120, 4096, True, 23)
    c1 = _run(a, b, True, True)
    c2 = _run(a, b, True, True)
    assert torch.equal(c1, c2)


def test_gemm_bench_shape_sampled(oracle_mod):
    """The benchmark's 8192 x 8192 x 8192 launch (CTA pairs), checked on sampled rows."""
    M = N = K = 8192
    assert tk.gemm_uses_pairs(M, N, K, True)
    a, b = _inputs(M, N, K, True, 24)
    c = _run(a, b, True, True)
    rows = [0, 1, 127, 128, 4095, 4096, 8190, 8191]
    _check(oracle_mod, a, b, True, c, rows=rows, what="8192^3")


# ---------------------------------------------------------------- CTA pairs
# At least one wave of 256 x 256 tiles over the SM pairs and K >= 768 run on
# pairs of CTAs: the leader's MMAs read both CTAs' halves of A and B, and each
# CTA writes its own 128 rows of every tile.

def _pair_shape_rows(M):
    """Two rows of every 128-row half of every 256-row pair tile."""
    return sorted({r for blk in range(0, M, 128) for r in (blk + 5, min(blk + 126, M - 1))})


@pytest.mark.parametrize("b_kmajor", [True, False])
@pytest.mark.parametrize("M,N,K", [(2148, 2632, 1032), (2304, 2064, 776)])
def test_gemm_pairs_ragged(oracle_mod, b_kmajor, M, N, K):
    """9 x 11 pair tiles with M, N and K all ragged (the last tile's second
    CTA holds no row of C), and 9 x 9 with ragged N and the shortest K that
    takes pairs; against the oracle on two rows of every 128-row block;
    stream-K on or off takes the same path."""
    assert tk.gemm_uses_pairs(M, N, K, True) and tk.gemm_uses_pairs(M, N, K, False)
    assert tk.gemm_workspace_bytes(M, N, K, True) == 0 and tk.gemm_workspace_bytes(M, N, K, False) == 0
    a, b = _inputs(M, N, K, b_kmajor, 31 + K)
    rows = _pair_shape_rows(M)
    c1 = _run(a, b, b_kmajor, True)
    _check(oracle_mod, a, b, b_kmajor, c1, rows=rows, what=f"pairs {M}x{N}x{K} kmajor={b_kmajor}")
    c2 = _run(a, b, b_kmajor, False)
    assert torch.equal(c1, c2)


def test_gemm_pairs_full_wave_multiple(oracle_mod):
    """4864 x 4096 x 2048: 19 x 16 = 304 pair tiles, four whole waves over 76
    pairs; two rows of every 128-row block."""
    M, N, K = 4864, 4096, 2048
    assert tk.gemm_uses_pairs(M, N, K, True) and tk.gemm_workspace_bytes(M, N, K, True) == 0
    a, b = _inputs(M, N, K, True, 32)
    c = _run(a, b, True, True)
    _check(oracle_mod, a, b, True, c, rows=_pair_shape_rows(M)[::3], what="pairs 4864x4096x2048")


def test_gemm_pairs_second_cta_empty(oracle_mod):
    """M = 100: every pair tile's second CTA lies wholly past M (its loads read
    zeros, its stores are clipped away), across 76 pair tiles of N; every row
    against the oracle."""
    M, N, K = 100, 76 * 256, 1024
    assert tk.gemm_uses_pairs(M, N, K, True)
    a, b = _inputs(M, N, K, True, 34)
    c = _run(a, b, True, True)
    _check(oracle_mod, a, b, True, c, what="pairs M=100")


def test_gemm_pairs_deterministic():
    a, b = _inputs(2148, 2632, 1032, True, 33)
    c1 = _run(a, b, True, True)
    c2 = _run(a, b, True, True)
    assert torch.equal(c1, c2)


def test_gemm_rejects_small_workspace():
    a, b = _inputs(3000, 5120, 4096, True, 25)
    a, b = a.cuda(), b.cuda()
    need = tk.gemm_workspace_bytes(3000, 5120, 4096, True)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(tk.TkError) as e:
        tk.gemm(a, b, workspace=ws)
    assert e.value.name == "TK_ERR_WORKSPACE"
