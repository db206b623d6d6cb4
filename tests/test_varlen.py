"""Jagged batches (FlexAttention page, variant list: irregular tensors):
sequences packed with no padding, described by cumulative lengths. The
packed attention must equal each sequence's own attention computed
separately by the oracle (a definition independent of the document-mask
code path), forward and backward."""
import numpy as np
import pytest
import torch

from oracle import Spec, attention_backward, attention_forward
from synth import make_workload
from tests.helpers import DeviceRun, check_bf16

LENGTHS = [100, 300, 57, 1, 400, 166]   # total 1024: several tiles, ragged seams


def packed_workload(D, backward=False, seed=600, lengths=LENGTHS):
    total = sum(lengths)
    w = make_workload(0, seed=seed, B=1, Hq=4, Hkv=2, S=total, D=D, causal=True,
                      document=True, doc_lengths=[lengths], backward=backward)
    return w


def per_sequence(w, lengths, backward=False):
    """Oracle on each sequence alone (its own slice of q, k, v), stitched."""
    outs = []
    cu = np.concatenate([[0], np.cumsum(lengths)])
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        q = w.q[:, :, a:b].double().numpy()
        k = w.k[:, :, a:b].double().numpy()
        v = w.v[:, :, a:b].double().numpy()
        if backward:
            do = w.do[:, :, a:b].double().numpy()
            outs.append(attention_backward(q, k, v, do, Spec(causal=True)))
        else:
            outs.append(attention_forward(q, k, v, Spec(causal=True)))
    return [np.concatenate([o[t] for o in outs], axis=2) for t in range(len(outs[0]))]


@pytest.mark.gpu
def test_doc_ids_from_seqlens_matches_numpy():
    import masked_attention_gb300 as M
    cu = torch.tensor(np.concatenate([[0], np.cumsum(LENGTHS)]), dtype=torch.int32,
                      device="cuda")
    ids = M.doc_ids_from_seqlens(cu).cpu().numpy()[0]
    ref = np.repeat(np.arange(len(LENGTHS)), LENGTHS)
    assert np.array_equal(ids, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_packed_forward_equals_per_sequence(D):
    import masked_attention_gb300 as M
    w = packed_workload(D)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(LENGTHS)]), dtype=torch.int32,
                      device="cuda")
    g = DeviceRun(w, use_block_mask=False)
    g.doc_id = M.doc_ids_from_seqlens(cu)
    g.bm = M.build_block_mask(g.variant & 0xF, 1, w.Sq, w.Skv, doc_id=g.doc_id)
    O, L = g.fwd()
    torch.cuda.synchronize()
    O_ref, L_ref = per_sequence(w, LENGTHS)
    O = O.float().cpu().numpy()
    L = L.cpu().numpy()
    check_bf16(O, O_ref, f"packed O D={D}")
    assert np.abs(L - L_ref).max() <= 2e-3


@pytest.mark.gpu
def test_packed_backward_equals_per_sequence():
    import masked_attention_gb300 as M
    lengths = [128, 384, 256, 256]  # the bf16 backward needs 128-multiple totals
    w = packed_workload(128, backward=True, seed=610, lengths=lengths)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32,
                      device="cuda")
    g = DeviceRun(w, use_block_mask=False)
    g.doc_id = M.doc_ids_from_seqlens(cu)
    g.bm = M.build_block_mask(g.variant & 0xF, 1, w.Sq, w.Skv, doc_id=g.doc_id,
                              transposed=True)
    O, L = g.fwd()
    dq, dk, dv = torch.empty_like(g.q), torch.empty_like(g.k), torch.empty_like(g.v)
    ws = torch.empty(M.attn_bwd_workspace_bytes(1, w.Hq, w.Sq), dtype=torch.uint8,
                     device="cuda")
    M.attn_bwd(g.q, g.k, g.v, O, L, g.do, dq, dk, dv, ws, g.variant, **g.kwargs())
    torch.cuda.synchronize()
    ref = per_sequence(w, lengths, backward=True)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref[:3]):
        check_bf16(got.float().cpu().numpy(), want, f"packed {name}")


def test_doc_ids_from_seqlens_rejects_bad_arguments():
    import masked_attention_gb300 as M
    L = M.lib()
    assert L.attn_doc_ids_from_seqlens(0x10000, 0, 10, 0x20000, None) == M.ATTN_ERR_INVALID_ARG
    assert L.attn_doc_ids_from_seqlens(0x10000, 3, -1, 0x20000, None) == M.ATTN_ERR_INVALID_ARG
    assert L.attn_doc_ids_from_seqlens(None, 3, 10, 0x20000, None) == M.ATTN_ERR_INVALID_ARG
    assert L.attn_doc_ids_from_seqlens(0x10000, 3, 0, 0x20000, None) == M.ATTN_OK
