"""Block-mask builder on the GPU against the oracle's brute-force tile
classification: bit-exact counts and lists (FlexAttention page, item on
exploiting mask sparsity)."""
import numpy as np
import pytest

from oracle import block_mask as oracle_block_mask
from synth import make_workload
from tests.helpers import oracle_spec

pytestmark = pytest.mark.gpu


def compare(w, transposed=True):
    import torch
    import masked_attention_gb300 as M
    from tests.helpers import variant_bits
    doc = torch.from_numpy(w.doc_id).cuda() if w.document else None
    pre = torch.from_numpy(w.prefix_len).cuda() if w.prefix else None
    bm = M.build_block_mask(variant_bits(w) & 0xF, w.B, w.Sq, w.Skv, window=w.window or 0,
                            doc_id=doc, prefix_len=pre, transposed=transposed)
    torch.cuda.synchronize()
    got = bm.to_host()
    ref = oracle_block_mask(oracle_spec(w), w.B, w.Sq, w.Skv)
    assert np.array_equal(got["full_cnt"], ref.full_cnt)
    assert np.array_equal(got["part_cnt"], ref.part_cnt)
    for b in range(w.B):
        for qt in range(bm.nq):
            nf, np_ = ref.full_cnt[b, qt], ref.part_cnt[b, qt]
            assert list(got["full_idx"][b, qt, :nf]) == list(ref.full_idx[b][qt])
            assert list(got["part_idx"][b, qt, :np_]) == list(ref.part_idx[b][qt])
    # order: a permutation of the rows, by descending visited tiles, ties ascending
    cost = (ref.full_cnt + ref.part_cnt).reshape(-1)
    order = got["order"]
    assert sorted(order) == list(range(w.B * bm.nq))
    keys = [(-cost[r], r) for r in order]
    assert keys == sorted(keys)
    if transposed:
        assert np.array_equal(got["t_full_cnt"], ref.t_full_cnt)
        assert np.array_equal(got["t_part_cnt"], ref.t_part_cnt)
        for b in range(w.B):
            for kt in range(bm.nkv):
                nf, np_ = ref.t_full_cnt[b, kt], ref.t_part_cnt[b, kt]
                assert list(got["t_full_idx"][b, kt, :nf]) == list(ref.t_full_idx[b][kt])
                assert list(got["t_part_idx"][b, kt, :np_]) == list(ref.t_part_idx[b][kt])
        tcost = (ref.t_full_cnt + ref.t_part_cnt).reshape(-1)
        assert sorted(got["t_order"]) == list(range(w.B * bm.nkv))
        # t_order: batch element by batch element, longest first within each
        tkeys = [(r // bm.nkv, -tcost[r], r) for r in got["t_order"]]
        assert tkeys == sorted(tkeys)
    return ref


@pytest.mark.parametrize("number", [2, 3, 4, 5])
def test_block_mask_full_size_workloads(number):
    w = make_workload(number, with_tensors=False)
    compare(w, transposed=number in (3, 5))


EDGE = [
    dict(B=1, Hq=1, D=64, Sq=300, Skv=520, causal=True, window=200, document=True,
         doc_lo=20, doc_hi=150),                      # ragged tiles, window not a tile multiple
    dict(B=2, Hq=1, D=64, Sq=640, Skv=384, prefix=True, causal=True, prefix_lo=1, prefix_hi=700),
    dict(B=1, Hq=1, D=64, S=1024),                   # no mask bits: every tile full
    dict(B=3, Hq=1, D=64, S=777, document=True, doc_lo=1, doc_hi=40),   # many tiny documents
    dict(B=1, Hq=1, D=64, Sq=128, Skv=2048, causal=True),  # keys beyond every query: empty
    dict(B=1, Hq=1, D=64, S=1, causal=True),          # a single position
]


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_block_mask_edges(case):
    w = make_workload(0, seed=100 + case, with_tensors=False, **EDGE[case])
    compare(w)


def test_block_mask_scrambled_document_ids():
    """Document ids that are not contiguous runs (the bounds test only proves
    emptiness from disjoint id ranges, so this exercises the pair scan)."""
    w = make_workload(0, seed=7, with_tensors=False, B=1, Hq=1, D=64, S=1024, document=True,
                      doc_lo=5, doc_hi=60, causal=True)
    rng = np.random.default_rng(3)
    w.doc_id = rng.integers(0, 4, size=w.doc_id.shape).astype(np.int32)
    compare(w)
