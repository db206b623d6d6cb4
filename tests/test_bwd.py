"""Backward parity: dQ, dK, dV of the CUDA path against the oracle's analytic
fp64 gradients (FlexAttention page, "Performance": a deterministic backward
that recomputes intermediates).

Tolerance: the flat bound max|g - g_ref| <= 1e-2 on the bf16 outputs dQ, dK
and dV. Rounding an output to bf16 alone costs half an ulp, 0.0156 once
|g_ref| >= 4; only such elements, and only within one bf16 ulp of g_ref, are
exempt, and they are counted, printed and capped (tests/helpers.py,
check_bf16).
"""
import numpy as np
import pytest

from oracle import attention_backward
from synth import make_workload
from tests.helpers import (DeviceRun, check_bf16, check_canaries, guarded_empty,
                           guarded_like, oracle_spec, variant_bits)

pytestmark = pytest.mark.gpu


def run_bwd(w, use_block_mask=True, f16=False):
    """f16: a workspace with room for the fp16 path's copies (used where the
    lengths are whole tiles and the inputs in range; else the bf16 path)."""
    import torch
    import masked_attention_gb300 as M
    g = DeviceRun(w, use_block_mask=use_block_mask, transposed=True)
    O, L = g.fwd()
    dq = guarded_like(g.q)
    dk = guarded_like(g.k)
    dv = guarded_like(g.v)
    nbytes = (M.attn_bwd_workspace_bytes_f16(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D) if f16
              else M.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq))
    ws = guarded_empty((nbytes,), torch.uint8)
    M.attn_bwd(g.q, g.k, g.v, O, L, g.do, dq, dk, dv, ws, g.variant, **g.kwargs())
    torch.cuda.synchronize()
    assert M.attn_check_status() == M.ATTN_OK
    check_canaries()
    return g, dq, dk, dv


def check_grads(w, dq, dk, dv, heads=None):
    dQ, dK, dV, _, _ = attention_backward(w.q, w.k, w.v, w.do, oracle_spec(w), heads=heads)
    out = {}
    for name, got, ref in (("dq", dq, dQ), ("dk", dk, dK), ("dv", dv, dV)):
        got = got.float().cpu().numpy().astype(np.float64)
        if heads is not None:
            sel = [(b, h if name == "dq" else h // (w.Hq // w.Hkv)) for b, h in heads]
            got = np.stack([got[b, h] for b, h in sel])
            ref = np.stack([ref[b, h] for b, h in sel])
        out[name] = check_bf16(got, ref, f"{name} {w.name}")["max_err"]
    return out


CASES = {
    "causal_d128": dict(B=2, Hq=2, Hkv=2, S=512, D=128, causal=True),
    "causal_alibi_d64": dict(B=1, Hq=4, Hkv=4, S=768, D=64, causal=True, alibi=True),
    "gqa_prefix_softcap_d128": dict(B=1, Hq=4, Hkv=2, S=512, D=128, causal=True, prefix=True,
                                    softcap=20.0, prefix_lo=100, prefix_hi=300),
    "doc_window_causal_d128": dict(B=1, Hq=2, Hkv=2, S=1024, D=128, causal=True, window=300,
                                   document=True, doc_lo=100, doc_hi=500),
    "full_d64": dict(B=1, Hq=2, Hkv=1, S=384, D=64),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bwd_reduced(name):
    """Both paths on whole tiles: bf16 operands with their rounding remainders,
    and fp16 operands (a workspace with the fp16 copies), against one oracle
    result."""
    w = make_workload(0, seed=500 + sorted(CASES).index(name), backward=True, **CASES[name])
    dQ, dK, dV, _, _ = attention_backward(w.q, w.k, w.v, w.do, oracle_spec(w))
    for f16 in (False, True):
        _, dq, dk, dv = run_bwd(w, f16=f16)
        for nm, got, ref in (("dq", dq, dQ), ("dk", dk, dK), ("dv", dv, dV)):
            check_bf16(got.float().cpu().numpy(), ref, f"{nm} {w.name} f16={f16}")


def test_bwd_f16_out_of_range_takes_the_bf16_path():
    """Values whose products would leave fp16's range (2 D max|dO| max|V| >
    60000) with the fp16 path's workspace: the call converts, finds them out of
    range and runs the bf16 kernels; the gradients still match the oracle and
    equal those of the bf16 path bit for bit."""
    import torch
    w = make_workload(0, seed=509, backward=True, B=1, Hq=2, Hkv=2, S=256, D=64, causal=True)
    w.v = (w.v.float() * 8.0).to(w.v.dtype)
    w.do = (w.do.float() * 4.0).to(w.do.dtype)
    _, dq1, dk1, dv1 = run_bwd(w, f16=False)
    _, dq2, dk2, dv2 = run_bwd(w, f16=True)
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    check_grads(w, dq2, dk2, dv2)


# Lengths that are not multiples of the 128-row tile: the last query and key
# tiles run past Sq and Skv (zero-filled rows, padding keys masked, padding
# rows not stored); Sq != Skv; a prefix longer than the keys; one position;
# and the relative-position bias (which runs the same general kernels).
RAGGED = {
    "ragged_full_d64": dict(B=2, Hq=2, Hkv=1, Sq=200, Skv=333, D=64),
    "ragged_causal_d128": dict(B=1, Hq=2, Hkv=2, S=300, D=128, causal=True),
    "ragged_causal_alibi_softcap_d128": dict(B=1, Hq=4, Hkv=2, S=451, D=128, causal=True,
                                             alibi=True, softcap=30.0),
    "ragged_doc_window_d64": dict(B=2, Hq=2, Hkv=2, S=517, D=64, causal=True, window=150,
                                  document=True, doc_lo=60, doc_hi=200),
    "ragged_prefix_past_keys_d128": dict(B=1, Hq=2, Hkv=1, Sq=130, Skv=390, D=128,
                                         causal=True, prefix=True, prefix_len=[450]),
    "single_position_d64": dict(B=1, Hq=1, Hkv=1, S=1, D=64, causal=True),
    # the relative-position bias table (a constant of the call: no gradient to it)
    "relbias_causal_d128": dict(B=1, Hq=2, Hkv=2, S=384, D=128, causal=True, relbias=True),
    "relbias_alibi_softcap_gqa_ragged_d64": dict(B=2, Hq=4, Hkv=2, S=300, D=64, causal=True,
                                                 alibi=True, softcap=15.0, relbias=True),
    "relbias_full_d128": dict(B=1, Hq=2, Hkv=1, Sq=200, Skv=256, D=128, relbias=True),
}


@pytest.mark.parametrize("use_block_mask", [True, False])
@pytest.mark.parametrize("name", sorted(RAGGED))
def test_bwd_ragged(name, use_block_mask):
    w = make_workload(0, seed=600 + sorted(RAGGED).index(name), backward=True, **RAGGED[name])
    _, dq, dk, dv = run_bwd(w, use_block_mask=use_block_mask)
    check_grads(w, dq, dk, dv)


@pytest.mark.parametrize("name", ["causal_d128", "doc_window_causal_d128"])
def test_bwd_without_block_mask(name):
    w = make_workload(0, seed=500 + sorted(CASES).index(name), backward=True, **CASES[name])
    _, dq, dk, dv = run_bwd(w, use_block_mask=False)
    check_grads(w, dq, dk, dv)


@pytest.mark.parametrize("f16", [False, True])
def test_bwd_full_size_workload5_sampled_heads(f16):
    """The training-step workload at full size, on both paths; every gradient
    of three (b, h) heads is checked (heads are independent under MHA)."""
    w = make_workload(5)
    _, dq, dk, dv = run_bwd(w, f16=f16)
    check_grads(w, dq, dk, dv, heads=[(0, 0), (3, 7), (7, 15)])


@pytest.mark.parametrize("f16", [False, True])
def test_bwd_deterministic(f16):
    import torch
    w = make_workload(0, seed=77, backward=True, **CASES["gqa_prefix_softcap_d128"])
    _, a, b, c = run_bwd(w, f16=f16)
    for _ in range(2):
        _, a2, b2, c2 = run_bwd(w, f16=f16)
        assert torch.equal(a, a2) and torch.equal(b, b2) and torch.equal(c, c2)


# One query shard against one key shard of a longer sequence (context
# parallelism): the call's rows and keys sit at absolute positions
# q_offset + i and kv_offset + j of the whole sequence, which every mask
# term, ALiBi and the document ids use. The gradients are those of this
# call's partial attention (its own O and LSE), against the oracle's with the
# same offsets. (whole-sequence overrides, (q_lo, q_hi), (kv_lo, kv_hi))
SHARDS = {
    "doc_window_causal_d128": (dict(B=1, Hq=2, Hkv=2, S=1024, D=128, causal=True, window=300,
                                    document=True, doc_lo=100, doc_hi=400), (512, 1024), (256, 768)),
    "causal_alibi_softcap_ragged_d64": (dict(B=1, Hq=2, Hkv=1, S=800, D=64, causal=True,
                                             alibi=True, softcap=20.0), (300, 700), (100, 600)),
    "gqa_prefix_causal_d128": (dict(B=2, Hq=4, Hkv=2, S=600, D=128, causal=True, prefix=True,
                                    prefix_len=[250, 420]), (200, 456), (0, 333)),
    "full_alibi_keys_after_queries_d64": (dict(B=1, Hq=2, Hkv=2, S=640, D=64, alibi=True),
                                          (128, 256), (384, 640)),
}


@pytest.mark.parametrize("use_block_mask", [True, False])
@pytest.mark.parametrize("name", sorted(SHARDS))
def test_bwd_position_offsets(name, use_block_mask):
    import dataclasses
    import torch
    import masked_attention_gb300 as M
    over, (qa, qb), (ka, kb) = SHARDS[name]
    w = make_workload(0, seed=650 + sorted(SHARDS).index(name), backward=True, **over)
    dev = "cuda"
    q = w.q[:, :, qa:qb].contiguous()
    do = w.do[:, :, qa:qb].contiguous()
    k = w.k[:, :, ka:kb].contiguous()
    v = w.v[:, :, ka:kb].contiguous()
    variant = variant_bits(w)
    doc = torch.from_numpy(w.doc_id).to(dev) if w.document else None
    pre = torch.from_numpy(w.prefix_len).to(dev) if w.prefix else None
    kw = dict(window=w.window or 0, softcap=w.softcap or 0.0, doc_id=doc, prefix_len=pre,
              q_offset=qa, kv_offset=ka)
    bm = None
    if use_block_mask:
        bm = M.build_block_mask(variant & 0xF, w.B, qb - qa, kb - ka, window=w.window or 0,
                                doc_id=doc, prefix_len=pre, q_offset=qa, kv_offset=ka,
                                transposed=True)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = guarded_like(qd)
    lse = guarded_empty((w.B, w.Hq, qb - qa), torch.float32)
    M.attn_fwd(qd, kd, vd, o, lse, variant, block_mask=bm, **kw)
    dq, dk, dv = guarded_like(qd), guarded_like(kd), guarded_like(vd)
    ws = guarded_empty((M.attn_bwd_workspace_bytes(w.B, w.Hq, qb - qa),), torch.uint8)
    M.attn_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, variant, block_mask=bm, **kw)
    torch.cuda.synchronize()
    assert M.attn_check_status() == M.ATTN_OK
    check_canaries()
    spec = dataclasses.replace(oracle_spec(w), q_offset=qa, kv_offset=ka)
    dQ, dK, dV, _, _ = attention_backward(q, k, v, do, spec)
    for nm, got, ref in (("dq", dq, dQ), ("dk", dk, dK), ("dv", dv, dV)):
        check_bf16(got.float().cpu().numpy(), ref, f"{nm} shard {name}")


def test_bwd_f16_workspace_on_ragged_lengths_takes_the_general_path():
    """A workspace with room for the fp16 copies on lengths that are not whole
    tiles: the fp16 path does not apply (whole tiles at offset 0 only) and the
    general bf16 kernels give the same bits as with the minimal workspace."""
    import torch
    w = make_workload(0, seed=610, backward=True, **RAGGED["ragged_causal_alibi_softcap_d128"])
    _, dq1, dk1, dv1 = run_bwd(w, f16=False)
    _, dq2, dk2, dv2 = run_bwd(w, f16=True)
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    check_grads(w, dq2, dk2, dv2)
