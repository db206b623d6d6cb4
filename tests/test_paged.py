"""Paged K/V cache (FlexAttention page, variant list: PagedAttention): the
keys and values sit in pages of a shared pool, mapped per sequence by a page
table. The forward over the paged cache must give the same bits as over the
contiguous K/V (same kernel arithmetic; the rows of the last page past Skv
are masked) and match the oracle."""
import numpy as np
import pytest
import torch

from oracle import attention_forward
from synth import make_workload
from tests.helpers import (DeviceRun, check_bf16, check_canaries, guarded_empty, guarded_like,
                           oracle_spec)

pytestmark = pytest.mark.gpu

CASES = {
    "full_gqa_d128_ps16": (dict(B=2, Hq=4, Hkv=2, Sq=128, Skv=700, D=128), 16),
    "window_alibi_d64_ps64": (dict(B=1, Hq=2, Hkv=2, Sq=300, Skv=1000, D=64, window=200,
                                   alibi=True), 64),
    "decode_softcap_d128_ps32": (dict(B=3, Hq=8, Hkv=2, Sq=1, Skv=517, D=128, softcap=30.0), 32),
    "causal_doc_d64_ps128": (dict(B=2, Hq=2, Hkv=1, S=640, D=64, causal=True, document=True,
                                  doc_lo=100, doc_hi=300), 128),
}


def paged_pools(k, v, page_size, seed):
    """Pools [num_pages, Hkv, page_size, D] and a shuffled page table holding
    k and v; unreferenced pages hold NaN (never read), rows of the last page
    past Skv hold finite noise (read, then masked)."""
    B, Hkv, Skv, D = k.shape
    pps = (Skv + page_size - 1) // page_size
    num_pages = B * pps + 5
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)[:B * pps]
    table = torch.from_numpy(perm.reshape(B, pps).astype(np.int32))
    kp = torch.full((num_pages, Hkv, page_size, D), float("nan"), dtype=k.dtype)
    vp = torch.full((num_pages, Hkv, page_size, D), float("nan"), dtype=v.dtype)
    g = torch.Generator().manual_seed(seed)
    for b in range(B):
        for lp in range(pps):
            phys = int(table[b, lp])
            kp[phys] = torch.randn(Hkv, page_size, D, generator=g).to(k.dtype)
            vp[phys] = torch.randn(Hkv, page_size, D, generator=g).to(v.dtype)
            rows = min(page_size, Skv - lp * page_size)
            kp[phys, :, :rows] = k[b, :, lp * page_size:lp * page_size + rows]
            vp[phys, :, :rows] = v[b, :, lp * page_size:lp * page_size + rows]
    return kp, vp, table


@pytest.mark.parametrize("name", sorted(CASES))
def test_paged_forward_matches_contiguous_and_oracle(name):
    import masked_attention_gb300 as M
    spec, page_size = CASES[name]
    w = make_workload(0, seed=700 + sorted(CASES).index(name), **spec)
    g = DeviceRun(w)
    O_ref_gpu, L_ref_gpu = g.fwd()
    kp, vp, table = paged_pools(w.k, w.v, page_size, seed=710 + sorted(CASES).index(name))
    kp, vp, table = kp.cuda(), vp.cuda(), table.cuda()
    o = guarded_like(g.q)
    lse = guarded_empty((w.B, w.Hq, w.Sq), torch.float32)
    M.attn_fwd(g.q, kp, vp, o, lse, g.variant, Skv=w.Skv, page_table=table,
               page_size=page_size, **g.kwargs())
    check_canaries()
    assert torch.equal(o, O_ref_gpu) and torch.equal(lse, L_ref_gpu)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, oracle_spec(w))
    check_bf16(o.float().cpu().numpy(), O_ref, f"paged O {name}")


def test_paged_arguments_are_checked():
    import masked_attention_gb300 as M
    w = make_workload(0, seed=720, B=1, Hq=2, Hkv=2, Sq=128, Skv=300, D=64)
    g = DeviceRun(w, use_block_mask=False)
    kp, vp, table = (t.cuda() for t in paged_pools(w.k, w.v, 32, seed=721))
    o = torch.empty_like(g.q)
    lse = torch.empty(1, 2, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(M.AttnError) as e:  # page size not in {16, 32, 64, 128}
        M.attn_fwd(g.q, kp, vp, o, lse, 0, Skv=300, page_table=table, page_size=48)
    assert e.value.status == M.ATTN_ERR_UNSUPPORTED
    with pytest.raises(M.AttnError) as e:  # table too short for Skv
        M.attn_fwd(g.q, kp, vp, o, lse, 0, Skv=300 + 32 * 20, page_table=table, page_size=32)
    assert e.value.status == M.ATTN_ERR_INVALID_ARG
