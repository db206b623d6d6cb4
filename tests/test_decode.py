"""Decode against a key/value cache (FlexAttention page, variant list:
PagedAttention, alone and with a sliding window): attn_decode against the
fp64 oracle on the same seeded inputs, for contiguous and paged caches, GQA
groups whose query heads share one tile, every mask and score term, new
tokens placed at the end of the cache with q_offset, with and without
splitting the keys across CTAs (the split results merged by the
online-softmax merge), ragged key counts, empty rows and out-of-range pages.
Outputs are held to the flat bf16 bound (tests/helpers.py, check_bf16) and
guarded by canaries."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import attention_forward
from synth import make_workload
from tests.helpers import (check_bf16, check_canaries, guarded_empty, max_abs, oracle_spec,
                           variant_bits)
from tests.test_fwd import lse_tol
from tests.test_paged import paged_pools

pytestmark = pytest.mark.gpu

# (workload overrides, q_offset rule, page size or 0)
CASES = {
    # one new token per sequence, causal, GQA group 4, D = 128, ragged cache
    "causal_gqa4_d128": (dict(B=3, Hq=8, Hkv=2, Sq=1, Skv=1000, D=128, causal=True), "end", 0),
    # sliding window + causal + ALiBi, group 8 x 2 rows = 16 rows, paged by 16
    "window_alibi_gqa8_sq2_d64_ps16": (dict(B=2, Hq=16, Hkv=2, Sq=2, Skv=777, D=64, causal=True,
                                            window=200, alibi=True), "end", 16),
    # document + prefix + soft-cap, paged by 64
    "doc_prefix_softcap_d128_ps64": (dict(B=2, Hq=4, Hkv=2, Sq=1, Skv=1300, D=128, causal=True,
                                          document=True, doc_lo=100, doc_hi=500, prefix=True,
                                          prefix_lo=50, prefix_hi=400, softcap=20.0), "end", 64),
    # relative-position bias, full attention, group 4 x 4 rows
    "relbias_full_sq4_d64": (dict(B=1, Hq=4, Hkv=1, Sq=4, Skv=300, D=64, relbias=True), "zero", 0),
    # MHA with 16 query rows, full attention, paged by 32
    "mha_sq16_d128_ps32": (dict(B=2, Hq=3, Hkv=3, Sq=16, Skv=513, D=128), "zero", 32),
    # the new token far past a short window: rows see keys of the window only
    "window_far_d64": (dict(B=1, Hq=2, Hkv=1, Sq=1, Skv=2000, D=64, causal=True, window=64),
                       "end", 0),
}


def run_decode(w, q_off, page_size, split):
    import masked_attention_gb300 as M
    dev = "cuda"
    q, k, v = (t.to(dev).contiguous() for t in (w.q, w.k, w.v))
    kw = dict(window=w.window or 0, softcap=w.softcap or 0.0, q_offset=q_off)
    if w.document:
        kw["doc_id"] = torch.from_numpy(w.doc_id).to(dev)
    if w.prefix:
        kw["prefix_len"] = torch.from_numpy(w.prefix_len).to(dev)
    if w.relbias:
        kw["rel_bias"] = w.rel_bias.to(dev).contiguous()
    if page_size:
        kp, vp, table = paged_pools(w.k, w.v, page_size, seed=w.seed + 7)
        k, v = kp.to(dev), vp.to(dev)
        kw.update(page_table=table.to(dev), page_size=page_size, Skv=w.Skv)
    ws = None
    nbytes = M.attn_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D)
    if split and nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    o = guarded_empty((w.B, w.Hq, w.Sq, w.D), torch.bfloat16)
    lse = guarded_empty((w.B, w.Hq, w.Sq), torch.float32)
    M.attn_decode(q, k, v, o, lse, variant_bits(w), workspace=ws, **kw)
    check_canaries()
    assert M.attn_check_status() == M.ATTN_OK
    return o, lse, nbytes


def q_offset_for(w, rule):
    return w.Skv - w.Sq if rule == "end" else 0


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_matches_oracle(name, split):
    over, rule, ps = CASES[name]
    w = make_workload(0, seed=880 + sorted(CASES).index(name), **over)
    q_off = q_offset_for(w, rule)
    o, lse, _ = run_decode(w, q_off, ps, split)
    spec = dataclasses.replace(oracle_spec(w), q_offset=q_off)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, spec)
    check_bf16(o.float().cpu().numpy(), O_ref, f"decode O {name} split={split}")
    assert max_abs(lse.cpu().numpy(), L_ref) <= lse_tol(w, L_ref)


def test_decode_splits_the_keys_when_few_ctas():
    """One sequence, two key/value heads, a long cache: the keys are split
    (a workspace is asked for) and the merged result equals the unsplit one
    within the bound."""
    import masked_attention_gb300 as M
    w = make_workload(0, seed=890, B=1, Hq=8, Hkv=2, Sq=1, Skv=8192, D=128, causal=True)
    assert M.attn_decode_workspace_bytes(1, 8, 2, 1, 8192, 128) > 0
    o1, l1, _ = run_decode(w, w.Skv - 1, 0, False)
    o2, l2, _ = run_decode(w, w.Skv - 1, 0, True)
    check_bf16(o2.float().cpu().numpy(), o1.float().cpu().numpy(), "decode split vs one split")
    assert max_abs(l1.cpu().numpy(), l2.cpu().numpy()) <= 1e-4


def test_decode_equals_forward_kernel():
    """The decode kernel and the tensor-core forward compute the same
    attention (different kernels, same bound)."""
    import masked_attention_gb300 as M
    w = make_workload(0, seed=891, B=2, Hq=8, Hkv=2, Sq=2, Skv=640, D=128, causal=True,
                      alibi=True)
    o, lse, _ = run_decode(w, w.Skv - 2, 0, True)
    q, k, v = (t.cuda() for t in (w.q, w.k, w.v))
    o2 = torch.empty_like(q)
    l2 = torch.empty(w.B, w.Hq, w.Sq, device="cuda")
    M.attn_fwd(q, k, v, o2, l2, variant_bits(w), q_offset=w.Skv - 2)
    torch.cuda.synchronize()
    check_bf16(o.float().cpu().numpy(), o2.float().cpu().numpy(), "decode vs forward")
    assert max_abs(lse.cpu().numpy(), l2.cpu().numpy()) <= 2e-3


def test_decode_empty_rows():
    """Keys all before the window of the query: O = 0 and LSE = -inf."""
    w = make_workload(0, seed=892, B=1, Hq=2, Hkv=1, Sq=1, Skv=100, D=64, causal=True, window=5)
    o, lse, _ = run_decode(w, 500, 0, True)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_decode_page_outside_the_pool_reads_zeros():
    """A page index outside [0, num_pages) reads as zero keys and values
    (nothing is read): the result equals the oracle's on a cache whose keys
    and values of that page are zero."""
    w = make_workload(0, seed=893, B=1, Hq=4, Hkv=1, Sq=1, Skv=96, D=64)
    import masked_attention_gb300 as M
    kp, vp, table = paged_pools(w.k, w.v, 32, seed=894)
    table[0, 1] = kp.shape[0] + 5  # second page out of range
    o = guarded_empty((w.B, w.Hq, w.Sq, w.D), torch.bfloat16)
    lse = guarded_empty((w.B, w.Hq, w.Sq), torch.float32)
    M.attn_decode(w.q.cuda(), kp.cuda(), vp.cuda(), o, lse, 0, page_table=table.cuda(),
                  page_size=32, Skv=w.Skv)
    check_canaries()
    k0, v0 = w.k.clone(), w.v.clone()
    k0[:, :, 32:64] = 0
    v0[:, :, 32:64] = 0
    O_ref, L_ref = attention_forward(w.q, k0, v0, oracle_spec(w))
    check_bf16(o.float().cpu().numpy(), O_ref, "decode zero page")
    assert max_abs(lse.cpu().numpy(), L_ref) <= 2e-3


def test_decode_argument_checks():
    import masked_attention_gb300 as M
    w = make_workload(0, seed=895, B=1, Hq=32, Hkv=1, Sq=1, Skv=64, D=64)
    q, k, v = (t.cuda() for t in (w.q, w.k, w.v))
    o = torch.empty_like(q)
    lse = torch.empty(1, 32, 1, device="cuda")
    with pytest.raises(M.AttnError) as e:  # 32 query heads per key/value head > 16 rows
        M.attn_decode(q, k, v, o, lse, 0)
    assert e.value.status == M.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("split", [False, True])
def test_decode_scores_far_above_the_running_max(split):
    """Keys of one late block score far above the rest (a large component
    shared with the queries): the running maximum of the split that reaches
    it jumps by far more than the exponent range there, and the merged result
    still equals the oracle's."""
    w = make_workload(0, seed=896, B=2, Hq=8, Hkv=2, Sq=1, Skv=3000, D=128, causal=True)
    g = torch.Generator().manual_seed(897)
    u = torch.randn(w.D, generator=g)
    u = u / u.norm() * 30.0
    w.q = (w.q.float() + u).to(w.q.dtype)
    k = w.k.float()
    k[:, :, 2500:2628] += u
    w.k = k.to(w.k.dtype)
    q_off = w.Skv - w.Sq
    o, lse, _ = run_decode(w, q_off, 0, split)
    spec = dataclasses.replace(oracle_spec(w), q_offset=q_off)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, spec)
    check_bf16(o.float().cpu().numpy(), O_ref, f"decode large scores split={split}")
    assert max_abs(lse.cpu().numpy(), L_ref) <= lse_tol(w, L_ref)
