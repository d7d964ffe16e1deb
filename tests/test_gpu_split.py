"""The forward's tail split (tk_attn_fwd_ws, through the C ABI).

Without the causal mask every work unit (a head's pair of 128-row query
tiles) costs the same, so the only imbalance is the last round of units on
the SMs.  When that round is at most half full, each of its units runs as two
pieces over the two halves of the key tiles, and the piece that publishes
second merges the two by their LSE (the same combination of partial softmax
sums the online softmax makes across key tiles).

The shapes here are chosen from this device's SM count so that the split is
taken (tk_attn_fwd_workspace_bytes > 0): head dims 32, 64, 96 and 128, equal
lengths, a ragged key tail that falls in the second piece, more keys than
queries, ragged queries.  Checked: parity with the fp64 oracle at the
forward's bars (O max-abs 2e-2, mean-abs 2e-3; LSE max-abs 1e-3); the heads
outside the tail bitwise equal to the unsplit entry point (tk_attn_fwd_kv);
two split launches bitwise equal, also after the workspace served another
shape; a too-small, misaligned or missing workspace refused before anything
runs; no workspace for the causal mask, head dim 256 or a full last round.
"""
import math

import numpy as np
import pytest
import torch

import tiled_attention_tk_gb300 as tk
from tiled_attention_tk_gb300.inputs import make_qkv_rect

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _pairs(Nq):
    return ((Nq + 127) // 128 + 1) // 2


def _heads_with_tail(Nq, want_tail):
    """The smallest head count above one round whose last round holds
    `want_tail` units or, failing that, any count whose last round is at most
    half full."""
    sms, n_pairs = _sms(), _pairs(Nq)
    fallback = None
    for bh in range(1, 8 * sms):
        units = bh * n_pairs
        tail = units % sms
        if units > sms and 0 < tail <= sms // 2:
            if tail == want_tail:
                return bh
            fallback = fallback or bh
    return fallback


def _split_run(q, k, v, causal, scale, ws=None):
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    need = tk.fwd_workspace_bytes(B, H, Nq, Nkv, D, causal)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    tk.fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                  ws.numel(), B, H, Nq, Nkv, D, causal, scale, int(torch.cuda.current_stream().cuda_stream))
    return o, lse


def _plain_run(q, k, v, causal, scale):
    B, H, Nq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    tk.fwd_kv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, k.shape[2], D,
                  causal, scale, int(torch.cuda.current_stream().cuda_stream))
    return o, lse


def _status_ok():
    torch.cuda.synchronize()
    status, detail = tk.device_status()
    assert status == 0, f"device status {status} detail {detail:#x}"


CASES = [
    (512, 512, 128, 10),    # two pairs per head, four key tiles: pieces of two
    (512, 512, 64, 6),
    (512, 700, 96, 8),      # six key tiles; the ragged key tail is in the second piece
    (200, 1000, 32, 7),     # one pair per head, eight key tiles
    (1000, 1000, 128, 4),   # ragged queries and keys
]


@pytest.mark.parametrize("Nq,Nkv,D,want_tail", CASES)
def test_split_parity(oracle_mod, Nq, Nkv, D, want_tail):
    H = _heads_with_tail(Nq, want_tail)
    assert H is not None
    assert tk.fwd_workspace_bytes(1, H, Nq, Nkv, D, False) > 0, "the split is not taken for this shape"
    q, k, v = make_qkv_rect(1, H, Nq, Nkv, D, 9100 + Nq + Nkv + D)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = _split_run(qd, kd, vd, False, scale)
    _status_ok()
    O_ref, L_ref = oracle_mod.attn_fwd(q, k, v, False, scale)
    on, ln = o.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.all(np.isfinite(on)) and np.all(np.isfinite(ln))
    err, lerr = np.abs(on - O_ref), np.abs(ln - L_ref)
    assert err.max() <= O_MAX, f"O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"O mean-abs {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"LSE max-abs {lerr.max():.3e}"
    # the tail heads alone meet the bar too (they are few among all heads)
    sms, n_pairs = _sms(), _pairs(Nq)
    first_tail_head = ((H * n_pairs) // sms) * sms // n_pairs
    t_err = np.abs(on[:, first_tail_head:] - O_ref[:, first_tail_head:])
    t_lerr = np.abs(ln[:, first_tail_head:] - L_ref[:, first_tail_head:])
    assert t_err.max() <= O_MAX and t_err.mean() <= O_MEAN, (t_err.max(), t_err.mean())
    assert t_lerr.max() <= LSE_MAX, t_lerr.max()


@pytest.mark.parametrize("Nq,Nkv,D,want_tail", CASES[:3])
def test_split_matches_unsplit_outside_tail_and_is_deterministic(Nq, Nkv, D, want_tail):
    H = _heads_with_tail(Nq, want_tail)
    q, k, v = make_qkv_rect(1, H, Nq, Nkv, D, 9200 + Nq + D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(D)
    need = tk.fwd_workspace_bytes(1, H, Nq, Nkv, D, False)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o1, l1 = _split_run(qd, kd, vd, False, scale, ws)
    # the same workspace serves another split shape in between
    H2 = _heads_with_tail(512, 3)
    q2, k2, v2 = make_qkv_rect(1, H2, 512, 512, 64, 9300)
    ws2_need = tk.fwd_workspace_bytes(1, H2, 512, 512, 64, False)
    ws_big = torch.empty(max(need, ws2_need), dtype=torch.uint8, device="cuda")
    _split_run(q2.cuda(), k2.cuda(), v2.cuda(), False, 0.125, ws_big)
    o2, l2 = _split_run(qd, kd, vd, False, scale, ws_big)
    op, lp = _plain_run(qd, kd, vd, False, scale)
    _status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2), "two split launches differ"
    sms, n_pairs = _sms(), _pairs(Nq)
    first_tail_head = ((H * n_pairs) // sms) * sms // n_pairs
    assert first_tail_head > 0
    assert torch.equal(o1[:, :first_tail_head], op[:, :first_tail_head])
    assert torch.equal(l1[:, :first_tail_head], lp[:, :first_tail_head])
    # the tail heads differ from the unsplit ones only by the merge's rounding
    assert (o1[:, first_tail_head:].float() - op[:, first_tail_head:].float()).abs().max().item() <= 1e-2
    assert (l1[:, first_tail_head:] - lp[:, first_tail_head:]).abs().max().item() <= 1e-4


def test_split_workspace_checks():
    Nq = Nkv = 512
    D = 128
    H = _heads_with_tail(Nq, 10)
    need = tk.fwd_workspace_bytes(1, H, Nq, Nkv, D, False)
    assert need > 0
    q = torch.zeros((1, H, Nq, D), dtype=torch.bfloat16, device="cuda")
    k, v = torch.zeros_like(q), torch.zeros_like(q)
    o, lse = torch.empty_like(q), torch.empty((1, H, Nq), dtype=torch.float32, device="cuda")
    sh = int(torch.cuda.current_stream().cuda_stream)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    with pytest.raises(tk.TkError) as e:
        tk.fwd_ws_raw(*ptrs, ws.data_ptr(), need - 1, 1, H, Nq, Nkv, D, False, 0.1, sh)
    assert e.value.name == "TK_ERR_WORKSPACE"
    with pytest.raises(tk.TkError) as e:
        tk.fwd_ws_raw(*ptrs, ws.data_ptr() + 16, need, 1, H, Nq, Nkv, D, False, 0.1, sh)
    assert e.value.name == "TK_ERR_WORKSPACE"
    with pytest.raises(tk.TkError) as e:
        tk.fwd_ws_raw(*ptrs, None, need, 1, H, Nq, Nkv, D, False, 0.1, sh)
    assert e.value.name == "TK_ERR_NULL_PTR"
    with pytest.raises(tk.TkError) as e:  # the workspace over the output
        tk.fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), o.data_ptr(), need,
                      1, H, Nq, Nkv, D, False, 0.1, sh)
    assert e.value.name == "TK_ERR_ALIAS"
    _status_ok()


def test_no_split_where_it_does_not_apply():
    sms = _sms()
    H = _heads_with_tail(512, 10)
    assert tk.fwd_workspace_bytes(1, H, 512, 512, 128, True) == 0     # causal: the schedule is balanced otherwise
    assert tk.fwd_workspace_bytes(1, H, 512, 512, 256, False) == 0    # head dim 256: its own kernel
    assert tk.fwd_workspace_bytes(1, H, 512, 384, 128, False) == 0    # three key tiles: pieces too short
    assert tk.fwd_workspace_bytes(1, sms, 256, 512, 128, False) == 0  # a full last round
    assert tk.fwd_workspace_bytes(1, 3, 512, 512, 128, False) == 0    # fewer units than SMs
    # a last round more than half full
    assert tk.fwd_workspace_bytes(1, sms + sms // 2 + 1, 256, 512, 128, False) == 0
