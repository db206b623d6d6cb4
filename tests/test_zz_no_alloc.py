"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers are handed their tensors but have no way to obtain a workspace:
code running inside a framework that owns every device allocation and forbids
raw cudaMalloc, or a plug-in that receives tensors without an allocator. For
them the library offers attn_bwd_noalloc, which keeps the backward's row
terms in a fixed array inside the library instead of a caller-provided
workspace. These tests call it through the C ABI and check:

* that it gives the same gradients as attn_bwd with a caller workspace, bit
  for bit (the same deterministic kernels read the same row terms), on two
  calls in a row, the second covering more rows of the shared array than the
  first, so a stale entry left by the first call would show;
* that a call allocates nothing: the device's free memory and torch's
  allocated bytes are the same before and after it (the first call on a
  device loads the library module that holds the array; it is made before
  the measured calls);
* that a problem too large for the fixed array is refused before anything
  runs.

This file is named so that pytest collects it last.
"""
import ctypes
import gc

import pytest

from synth import make_workload
from tests.helpers import DeviceRun

pytestmark = pytest.mark.gpu

# Two problems of different shapes and variants; the second has more rows
# (B * Hq * Sq = 4096) than the first (1536).
CASES = [
    dict(B=1, Hq=2, Hkv=2, S=768, D=64, causal=True, alibi=True),
    dict(B=2, Hq=4, Hkv=2, S=512, D=128, causal=True, prefix=True, softcap=30.0,
         prefix_lo=64, prefix_hi=300),
]


def test_noalloc_backward_equals_workspace_backward_twice():
    import torch
    import masked_attention_gb300 as M
    prepared = []
    for n, case in enumerate(CASES):
        w = make_workload(0, seed=900 + n, backward=True, **case)
        g = DeviceRun(w, transposed=True)
        O, L = g.fwd()
        ref = [torch.empty_like(t) for t in (g.q, g.k, g.v)]
        ws = torch.empty(M.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq), dtype=torch.uint8,
                         device="cuda")
        M.attn_bwd(g.q, g.k, g.v, O, L, g.do, *ref, ws, g.variant, **g.kwargs())
        got = [torch.empty_like(t) for t in (g.q, g.k, g.v)]
        prepared.append((g, O, L, ref, got))
    torch.cuda.synchronize()
    assert M.attn_check_status() == M.ATTN_OK

    # set-up call: the first call on the device looks up the array's address
    g, O, L, _, got = prepared[0]
    M.attn_bwd_noalloc(g.q, g.k, g.v, O, L, g.do, *got, g.variant, **g.kwargs())
    torch.cuda.synchronize()

    for g, O, L, ref, got in prepared:  # two calls in a row
        for t in got:
            t.fill_(float("nan"))
        kw = g.kwargs()
        torch.cuda.synchronize()
        # the garbage collector would free earlier tests' tensors at random
        # points and move torch's allocated bytes: off around the measured call
        gc.collect()
        gc.disable()
        try:
            free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
            M.attn_bwd_noalloc(g.q, g.k, g.v, O, L, g.do, *got, g.variant, **kw)
            torch.cuda.synchronize()
            free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        finally:
            gc.enable()
        assert M.attn_check_status() == M.ATTN_OK
        assert free1 == free0 and alloc1 == alloc0, (free0, free1, alloc0, alloc1)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), name


def test_noalloc_backward_refuses_problems_beyond_its_array():
    import masked_attention_gb300 as M
    p = M._params(M.BF16, 0.0, 0, 0.0, None, None, None, None, None, 0)
    # B * Hq * Sq = 2 * 16 * 131072 = 4,194,304 rows > 2,097,152: refused before any launch
    dummy = 0x100000
    st = M.lib().attn_bwd_noalloc(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                  2, 16, 16, 131072, 131072, 128, M.MASK_CAUSAL,
                                  ctypes.byref(p), None)
    assert st == M.ATTN_ERR_WORKSPACE_TOO_SMALL
