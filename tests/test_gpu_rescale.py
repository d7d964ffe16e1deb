"""The forward's lazy O rescale, driven on every key tile of every checked row.

The kernel keeps a per-row reference maximum of the raw scores and rescales
the partial output O (and the row sum l) only when a key tile's maximum
exceeds that reference by more than 2^24 in the exp2 domain, i.e. when
(max_tile - m_ref) * scale * log2(e) > 24.  Random inputs reach that branch
on about one row in a hundred, so these inputs are built to reach it on
every tile: keys carry a component 512 * (t + 1) for key tile t and queries
a per-row factor a_i in [1, 2) on it, all exact in bf16, so each 128-key
tile raises every row's maximum score by at least 512 * a_i minus the noise
of the other components.  A host-side check computes, in float64, each
checked row's maximum over the keys it sees in every tile and asserts that
each rise clears the threshold, so the rescale runs on every tile after the
first.  The output is compared element by element with the fp64 oracle at
the forward's bars (O max-abs 2e-2, mean-abs 2e-3; LSE max-abs 1e-3).

Head dims 64, 128 and 256; without and with the causal mask; queries as
long as the keys and fewer queries than keys (queries at the end of the key
sequence under the causal mask).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_tk_gb300 as tk

pytestmark = pytest.mark.gpu

TAU_LOG2 = 24.0   # the kernel's rescale threshold in powers of two
BN = 128          # keys per key tile
STEP = 512.0      # rise of the key component per key tile


def _inputs(B, H, Nq, Nkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Nq, D), generator=g) * 0.5
    k = torch.randn((B, H, Nkv, D), generator=g) * 0.5
    v = torch.randn((B, H, Nkv, D), generator=g)
    # a_i in [1, 2) on multiples of 1/8 (exact in bf16)
    q[..., 0] = 1.0 + (torch.randint(0, 8, (B, H, Nq), generator=g).float() / 8.0)
    tiles = torch.arange(Nkv) // BN
    k[..., 0] = (STEP * (tiles + 1).float()).expand(B, H, Nkv)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def _assert_rescale_every_tile(q, k, causal, scale):
    """Each checked row's maximum over the keys it sees rises by more than
    the threshold from every key tile to the next (it visits them in order)."""
    c = scale * math.log2(math.e)
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    offset = Nkv - Nq
    transitions = 0
    for b in range(B):
        for h in range(H):
            s = q[b, h].double().numpy() @ k[b, h].double().numpy().T  # raw scores [Nq, Nkv]
            for i in range(Nq):
                last = min(i + offset, Nkv - 1) if causal else Nkv - 1
                n_t = last // BN + 1
                prev = None
                for t in range(n_t):
                    m = s[i, t * BN:min((t + 1) * BN, last + 1)].max()
                    if prev is not None:
                        assert (m - prev) * c > TAU_LOG2, (b, h, i, t, (m - prev) * c)
                        transitions += 1
                    prev = m
    return transitions


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nkv", [(1024, 1024), (300, 1024)])
def test_rescale_on_every_key_tile(D, causal, Nq, Nkv):
    B, H = 1, 2
    scale = 1.0 / math.sqrt(D)
    q, k, v = _inputs(B, H, Nq, Nkv, D, 7000 + D + 2 * causal + (Nq != Nkv))
    transitions = _assert_rescale_every_tile(q, k, causal, scale)
    assert transitions >= B * H * Nq  # every row rescales at least once past its first tile
    o, lse = tk.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} ({detail:#x})"
    O_ref, L_ref = oracle.attn_fwd(q, k, v, causal, scale)
    err = np.abs(o.cpu().double().numpy() - O_ref)
    lerr = np.abs(lse.cpu().double().numpy() - L_ref)
    assert err.max() <= 2e-2, err.max()
    assert err.mean() <= 2e-3, err.mean()
    assert lerr.max() <= 1e-3, lerr.max()
