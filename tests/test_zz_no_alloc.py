"""tk_attn_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (it uses a fixed 32 MiB workspace built into the library).

The GPU test calls the new entry point through the C ABI and compares it
with tk_attn_bwd (same kernels, caller-provided workspace) on two calls in a
row with different inputs, so that whatever the first call leaves in the
shared workspace cannot leak into the second.  Bar: the backward parity bar
(max-abs <= 0.02 * max|ref| + 1e-4, mean-abs <= 0.01 * mean|ref| + 1e-5),
with tk_attn_bwd's output as the reference.

This file sorts last so that a run stopping at its first failure has already
run every other test.
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import make_qkv


def test_noalloc_rejects_problems_beyond_the_fixed_workspace():
    """Host-side: a problem whose workspace exceeds 32 MiB is refused before
    any pointer is looked at (fake, never dereferenced addresses)."""
    lib = tk.load()
    B, H, N, D = 1, 16, 8192, 128  # 131072 rows -> about 64 MiB of workspace
    assert lib.tk_attn_bwd_workspace_bytes(B, H, N, D) > 32 << 20
    a = 0x10000000
    rc = lib.tk_attn_bwd_noalloc(a, a + 2**28, a + 2**29, a + 3 * 2**28, a + 2**30, a + 5 * 2**28,
                                 a + 6 * 2**28, a + 7 * 2**28, a + 2**31, B, H, N, D, 0, 0.08, None)
    assert rc == tk.STATUS["TK_ERR_NOALLOC_TOO_LARGE"]
    assert "32 MiB" in tk.strerror(rc)


def _noalloc(q, k, v, o, lse, do, causal, scale):
    B, H, N, D = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    rc = tk.load().tk_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                       dv.data_ptr(), B, H, N, D, int(causal), float(scale),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, tk.strerror(rc)
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    for call, (B, H, N, D, causal, seed) in enumerate([(2, 3, 300, 128, True, 11),
                                                       (1, 4, 257, 64, False, 23)]):
        scale = 1.0 / math.sqrt(D)
        q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, 31000 + seed))
        do = make_qkv(B, H, N, D, 32000 + seed)[0].cuda()
        o, lse = tk.fwd(q, k, v, causal=causal, scale=scale)
        got = _noalloc(q, k, v, o, lse, do, causal, scale)
        ref = tk.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert tk.device_status()[0] == 0
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            g = g.double().cpu().numpy()
            r = r.double().cpu().numpy()
            err = np.abs(g - r)
            assert np.all(np.isfinite(g)), f"call {call} {name}: non-finite"
            assert err.max() <= 0.02 * np.abs(r).max() + 1e-4, f"call {call} {name}: max err {err.max():.3e}"
            assert err.mean() <= 0.01 * np.abs(r).mean() + 1e-5, f"call {call} {name}: mean err {err.mean():.3e}"
