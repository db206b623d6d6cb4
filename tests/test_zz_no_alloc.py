"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers are handed their tensors but have no way to obtain a workspace:
code running inside a framework that owns every device allocation and forbids
raw cudaMalloc, or a plug-in that receives tensors without an allocator. For
them the library offers attn_bwd_noalloc, which keeps the backward's row
terms in a fixed array inside the library instead of a caller-provided
workspace. These tests call it through the C ABI and check that it gives the
same gradients as attn_bwd with a caller workspace, on two calls in a row
(the array is shared and keeps the previous call's contents), and that a
problem too large for the fixed array is refused before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from synth import make_workload
from tests.helpers import DeviceRun

pytestmark = pytest.mark.gpu


def bf16_grad_tol(ref):
    a = np.abs(ref)
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-30))) - 7), 0.0)
    return 1e-2 + 0.5 * ulp


def test_noalloc_backward_matches_workspace_backward_twice():
    import torch
    import masked_attention_gb300 as M
    cases = [
        dict(B=2, Hq=4, Hkv=2, S=512, D=128, causal=True, prefix=True, softcap=30.0,
             prefix_lo=64, prefix_hi=300),
        dict(B=1, Hq=2, Hkv=2, S=768, D=64, causal=True, alibi=True),
    ]
    for n, case in enumerate(cases):  # two calls in a row, different shapes and variants
        w = make_workload(0, seed=900 + n, backward=True, **case)
        g = DeviceRun(w, transposed=True)
        O, L = g.fwd()
        ref = [torch.empty_like(t) for t in (g.q, g.k, g.v)]
        ws = torch.empty(M.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq), dtype=torch.uint8,
                         device="cuda")
        M.attn_bwd(g.q, g.k, g.v, O, L, g.do, *ref, ws, g.variant, **g.kwargs())
        got = [torch.empty_like(t) for t in (g.q, g.k, g.v)]
        M.attn_bwd_noalloc(g.q, g.k, g.v, O, L, g.do, *got, g.variant, **g.kwargs())
        torch.cuda.synchronize()
        assert M.attn_check_status() == M.ATTN_OK
        for a, b in zip(got, ref):
            a = a.float().cpu().numpy().astype(np.float64)
            b = b.float().cpu().numpy().astype(np.float64)
            assert (np.abs(a - b) <= bf16_grad_tol(b)).all()


def test_noalloc_backward_refuses_problems_beyond_its_array():
    import masked_attention_gb300 as M
    p = M._params(M.BF16, 0.0, 0, 0.0, None, None, None, None, None, 0)
    # B * Hq * Sq = 2 * 16 * 131072 = 4,194,304 rows > 2,097,152: refused before any launch
    dummy = 0x100000
    st = M.lib().attn_bwd_noalloc(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                  2, 16, 16, 131072, 131072, 128, M.MASK_CAUSAL,
                                  ctypes.byref(p), None)
    assert st == M.ATTN_ERR_WORKSPACE_TOO_SMALL
