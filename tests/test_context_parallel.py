"""Context parallelism on one GPU: a sequence cut into query and key/value
shards, every (query shard, key shard) pair run as its own forward call with
its absolute position offsets, the key shards' partial results merged with
attn_combine, compared with the oracle's attention over the whole sequence.
The exchange of key/value shards between GPUs is not part of this library
(one GPU); what each GPU computes, and the merge, are.

Tolerances (bf16): the merged O is held to the same flat 1e-2 bound as a
single call (tests/helpers.py, check_bf16); LSE merges by a log-sum-exp,
which moves by at most the largest error of its inputs, so the single-call
LSE bound holds.
"""
import numpy as np
import pytest

from oracle import attention_forward, block_mask, combine_partials
from synth import make_workload
from tests.helpers import (check_bf16, check_canaries, guarded_empty, max_abs, oracle_spec,
                           variant_bits)
from tests.test_fwd import lse_tol

pytestmark = pytest.mark.gpu

CASES = {
    # document + window + causal (the long-context mix), uneven cuts
    "doc_window_causal_d128": (dict(B=1, Hq=4, Hkv=2, S=1024, D=128, causal=True, window=300,
                                    document=True, doc_lo=90, doc_hi=400),
                               [0, 256, 512, 1024], [0, 384, 640, 1024]),
    # ALiBi + causal at D = 64, cut points off the 128 grid (ragged shards)
    "causal_alibi_d64_ragged": (dict(B=2, Hq=2, Hkv=2, S=600, D=64, causal=True, alibi=True),
                                [0, 200, 600], [0, 77, 330, 600]),
    # GQA PrefixLM + soft-cap
    "prefix_softcap_gqa_d128": (dict(B=2, Hq=4, Hkv=1, S=512, D=128, causal=True, prefix=True,
                                     softcap=20.0, prefix_lo=60, prefix_hi=400),
                                [0, 256, 512], [0, 128, 256, 384, 512]),
    # fp32 path
    "f32_doc_causal": (dict(B=1, Hq=2, Hkv=2, S=300, D=64, dtype="f32", causal=True,
                            document=True, doc_lo=40, doc_hi=120),
                       [0, 150, 300], [0, 100, 300]),
}


def run_shards(w, q_cuts, kv_cuts, use_block_mask=True):
    import torch
    import masked_attention_gb300 as M
    dev = "cuda"
    q, k, v = (t.to(dev).contiguous() for t in (w.q, w.k, w.v))
    doc = torch.from_numpy(w.doc_id).to(dev) if w.document else None
    pre = torch.from_numpy(w.prefix_len).to(dev) if w.prefix else None
    variant = variant_bits(w)
    kw = dict(window=w.window or 0, doc_id=doc, prefix_len=pre)
    outs = []
    for qa, qb in zip(q_cuts[:-1], q_cuts[1:]):
        qs = q[:, :, qa:qb].contiguous()
        o_parts = torch.empty((len(kv_cuts) - 1,) + tuple(qs.shape), dtype=qs.dtype, device=dev)
        l_parts = torch.empty(len(kv_cuts) - 1, w.B, w.Hq, qb - qa, device=dev)
        for n, (ka, kb) in enumerate(zip(kv_cuts[:-1], kv_cuts[1:])):
            ks, vs = k[:, :, ka:kb].contiguous(), v[:, :, ka:kb].contiguous()
            bm = None
            if use_block_mask:
                bm = M.build_block_mask(variant & 0xF, w.B, qb - qa, kb - ka, q_offset=qa,
                                        kv_offset=ka, **kw)
            M.attn_fwd(qs, ks, vs, o_parts[n], l_parts[n], variant, softcap=w.softcap or 0.0,
                       block_mask=bm, q_offset=qa, kv_offset=ka, **kw)
        o = torch.empty_like(qs)
        lse = torch.empty(w.B, w.Hq, qb - qa, device=dev)
        M.attn_combine(o_parts, l_parts, o, lse)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert M.attn_check_status() == 0
    O = torch.cat([o for o, _ in outs], dim=2)
    L = torch.cat([l for _, l in outs], dim=2)
    return O, L


def check_merged(w, O, L, O_ref, L_ref):
    O = O.float().cpu().numpy().astype(np.float64)
    L = L.cpu().numpy().astype(np.float64)
    err = np.abs(O - O_ref)
    if w.dtype == "f32":
        assert err.max() <= 2e-4, err.max()
    else:
        check_bf16(O, O_ref, f"merged O {w.name}")
    assert max_abs(L, L_ref) <= lse_tol(w, L_ref), max_abs(L, L_ref)


@pytest.mark.parametrize("name", sorted(CASES))
def test_sharded_forward_merges_to_full_attention(name):
    spec, q_cuts, kv_cuts = CASES[name]
    w = make_workload(0, seed=900 + sorted(CASES).index(name), **spec)
    O, L = run_shards(w, q_cuts, kv_cuts)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, oracle_spec(w))
    check_merged(w, O, L, O_ref, L_ref)


def test_sharded_forward_without_block_mask():
    """The causal bound of the call without lists uses the offsets too (the
    key tiles past the shard's last allowed key are not visited)."""
    spec, q_cuts, kv_cuts = CASES["causal_alibi_d64_ragged"]
    w = make_workload(0, seed=950, **spec)
    O, L = run_shards(w, q_cuts, kv_cuts, use_block_mask=False)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, oracle_spec(w))
    check_merged(w, O, L, O_ref, L_ref)


@pytest.mark.parametrize("qa,qb,ka,kb", [(256, 512, 128, 384), (300, 700, 0, 450),
                                         (0, 333, 500, 1000), (640, 1000, 600, 1000)])
def test_block_mask_with_offsets_is_exact(qa, qb, ka, kb):
    """The device block mask of a shard pair equals the oracle's brute-force
    classification with the same offsets, bit for bit."""
    import dataclasses
    import torch
    import masked_attention_gb300 as M
    w = make_workload(0, seed=960, B=2, Hq=1, Hkv=1, S=1000, D=64, causal=True, window=350,
                      document=True, doc_lo=60, doc_hi=300, prefix=True, prefix_lo=0,
                      prefix_hi=200, with_tensors=False)
    doc = torch.from_numpy(w.doc_id).cuda()
    pre = torch.from_numpy(w.prefix_len).cuda()
    for variant in (M.MASK_CAUSAL | M.MASK_WINDOW | M.MASK_DOCUMENT,
                    M.MASK_CAUSAL | M.MASK_PREFIX, M.MASK_CAUSAL):
        bm = M.build_block_mask(variant, w.B, qb - qa, kb - ka, window=350, doc_id=doc,
                                prefix_len=pre, q_offset=qa, kv_offset=ka, transposed=True)
        got = bm.to_host()
        spec = oracle_spec(w)
        spec = dataclasses.replace(
            spec, causal=True, window=350 if variant & M.MASK_WINDOW else None,
            doc_id=w.doc_id if variant & M.MASK_DOCUMENT else None,
            prefix_len=w.prefix_len if variant & M.MASK_PREFIX else None,
            q_offset=qa, kv_offset=ka)
        ref = block_mask(spec, w.B, qb - qa, kb - ka)
        assert np.array_equal(got["full_cnt"], ref.full_cnt)
        assert np.array_equal(got["part_cnt"], ref.part_cnt)
        for b in range(w.B):
            for qt in range(ref.full_cnt.shape[1]):
                assert list(got["full_idx"][b, qt, :ref.full_cnt[b, qt]]) == ref.full_idx[b][qt]
                assert list(got["part_idx"][b, qt, :ref.part_cnt[b, qt]]) == ref.part_idx[b][qt]
        assert np.array_equal(got["t_full_cnt"], ref.t_full_cnt)
        assert np.array_equal(got["t_part_cnt"], ref.t_part_cnt)


@pytest.mark.parametrize("D,dtype,n,rows", [(64, "bf16", 5, 3000), (128, "bf16", 5, 3000),
                                            (128, "f32", 3, 3001), (64, "f32", 2, 2998),
                                            (128, "bf16", 32, 1027), (64, "bf16", 40, 517)])
def test_combine_matches_oracle_merge(D, dtype, n, rows):
    """attn_combine on random parts (with empty parts and rows empty in every
    part) against the oracle's merge of the same stored values; row counts
    that are not a multiple of the rows a warp merges at once, and more parts
    than a warp has lanes."""
    import torch
    import masked_attention_gb300 as M
    g = torch.Generator().manual_seed(970 + D + n)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o_parts = torch.randn(n, rows, D, generator=g).to(tdt)
    l_parts = (torch.randn(n, rows, generator=g) * 4.0).float()
    empty = torch.rand(n, rows, generator=g) < 0.3
    l_parts[empty] = -float("inf")
    o_parts[empty] = 0
    l_parts[:, :17] = -float("inf")   # rows with no kept key anywhere
    o_parts[:, :17] = 0
    o = guarded_empty((rows, D), tdt)
    lse = guarded_empty((rows,), torch.float32)
    M.attn_combine(o_parts.cuda(), l_parts.cuda(), o, lse)
    check_canaries()
    O_ref, L_ref = combine_partials([(o_parts[k], l_parts[k]) for k in range(n)])
    O = o.float().cpu().numpy()
    L = lse.cpu().numpy()
    if dtype == "bf16":
        check_bf16(O, O_ref, f"combine D={D} parts={n}")
    else:
        assert np.all(np.abs(O - O_ref) <= 1e-5)
    assert max_abs(L, L_ref) <= 1e-5
    assert np.all(O[:17] == 0) and np.all(np.isneginf(L[:17]))
