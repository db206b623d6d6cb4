"""Failure paths on the GPU: bounded device-side waits that run out report
ATTN_ERR_TIMEOUT through the status word and leave the context usable; a
block mask that does not match the call is rejected before launching.

The timeout is provoked on the host's request: with ATTN_FAULT_NO_LOADS the
load warp issues no copy, so the other warps wait for data that never comes
and their bounded waits run out (a 20 ms limit here). No GPU fault is raised:
the kernel drains, frees its tensor memory and returns, and the status word
reports ATTN_ERR_TIMEOUT.
"""
import numpy as np
import pytest

from oracle import attention_forward
from synth import make_workload
from tests.helpers import DeviceRun, oracle_spec

pytestmark = pytest.mark.gpu


def workload():
    return make_workload(0, seed=41, B=1, Hq=4, Hkv=2, S=2048, D=128, causal=True,
                         backward=True)


def test_forward_timeout_reports_status_and_recovers():
    import torch
    import masked_attention_gb300 as M
    w = workload()
    g = DeviceRun(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.empty_like(g.q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device="cuda")
    M.attn_fwd(g.q, g.k, g.v, o, lse, g.variant, block_mask=g.bm, status=status,
               timeout_ns=20_000_000, fault_inject=M.FAULT_NO_LOADS)
    assert M.attn_check_status(status) == M.ATTN_ERR_TIMEOUT
    assert int(status.item()) == 0  # attn_check_status clears it
    # the context still works: a normal call afterwards is correct
    O, L = g.fwd()
    torch.cuda.synchronize()
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, oracle_spec(w), heads=[(0, 0), (0, 3)])
    for b, h in [(0, 0), (0, 3)]:
        assert np.abs(O[b, h].float().cpu().numpy() - O_ref[b, h]).max() < 2e-2
    assert M.attn_check_status() == M.ATTN_OK


def test_backward_timeout_reports_status_and_recovers():
    import torch
    import masked_attention_gb300 as M
    w = workload()
    g = DeviceRun(w, transposed=True)
    O, L = g.fwd()
    dq, dk, dv = torch.empty_like(g.q), torch.empty_like(g.k), torch.empty_like(g.v)
    ws = torch.empty(M.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq), dtype=torch.uint8,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.attn_bwd(g.q, g.k, g.v, O, L, g.do, dq, dk, dv, ws, g.variant, block_mask=g.bm,
               status=status, timeout_ns=20_000_000, fault_inject=M.FAULT_NO_LOADS)
    assert M.attn_check_status(status) == M.ATTN_ERR_TIMEOUT
    M.attn_bwd(g.q, g.k, g.v, O, L, g.do, dq, dk, dv, ws, g.variant, block_mask=g.bm)
    assert M.attn_check_status() == M.ATTN_OK


def test_mismatched_block_mask_is_rejected():
    import torch
    import masked_attention_gb300 as M
    w = workload()
    g = DeviceRun(w)  # block mask built for the causal mask
    o = torch.empty_like(g.q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device="cuda")
    with pytest.raises(M.AttnError) as e:
        M.attn_fwd(g.q, g.k, g.v, o, lse, M.MASK_CAUSAL | M.MASK_WINDOW, window=64,
                   block_mask=g.bm)
    assert e.value.status == M.ATTN_ERR_INVALID_ARG
    # the backward needs the transposed lists
    ws = torch.empty(M.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(M.AttnError) as e:
        M.attn_bwd(g.q, g.k, g.v, o, lse, g.do, torch.empty_like(g.q), torch.empty_like(g.k),
                   torch.empty_like(g.v), ws, g.variant, block_mask=g.bm)
    assert e.value.status == M.ATTN_ERR_INVALID_ARG


def test_small_workspace_is_rejected():
    import torch
    import masked_attention_gb300 as M
    w = workload()
    g = DeviceRun(w, transposed=True)
    O, L = g.fwd()
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.AttnError) as e:
        M.attn_bwd(g.q, g.k, g.v, O, L, g.do, torch.empty_like(g.q), torch.empty_like(g.k),
                   torch.empty_like(g.v), ws, g.variant, block_mask=g.bm)
    assert e.value.status == M.ATTN_ERR_WORKSPACE_TOO_SMALL
