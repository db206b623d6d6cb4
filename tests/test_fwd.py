"""Forward parity: the CUDA path against the fp64 CPU oracle on the same
seeded inputs.

Tolerances (1e-2 on bf16 O and 1e-4 on fp32 O are the stated bounds; the
derivation of the others is beside each constant):
* bf16 O: max|O - O_ref| <= 1e-2 (flat). Rounding O to bf16 alone costs half
  an ulp, which exceeds 1e-2 once |O_ref| >= 4: such elements are exempt when
  they lie within one bf16 ulp of O_ref, and they are counted, printed and
  capped (tests/helpers.py, check_bf16).
* bf16 LSE: 2e-3 without soft-capping; with it, the hardware tanh (relative
  error below 2^-10.9) adds up to |s'| * 2^-10.9 <= 50 * tanh(|s|/50) * 5.3e-4,
  bounded here per row through the oracle's largest |s'|.
* fp32 O: 1e-4; fp32 LSE: 1e-5.
"""
import math

import numpy as np
import pytest

from oracle import attention_forward
from synth import make_workload
from tests.helpers import DeviceRun, check_bf16, oracle_spec

pytestmark = pytest.mark.gpu

TANH_REL = 2.0 ** -10.9


def lse_tol(w, ref_lse):
    if w.dtype == "f32":
        return 1e-5
    tol = 2e-3
    if w.softcap is not None:
        tol += w.softcap * TANH_REL  # |s'| <= softcap
    return tol


def check(w, O, L, O_ref, L_ref, rows=None):
    O = O.float().cpu().numpy().astype(np.float64)
    L = L.cpu().numpy().astype(np.float64)
    if rows is not None:
        O, L = O[:, :, rows], L[:, :, rows]
        O_ref, L_ref = O_ref[:, :, rows], L_ref[:, :, rows]
    mask = ~np.isnan(L_ref)
    if w.dtype == "f32":
        err = np.abs(O - O_ref)[mask]
        assert err.max() <= 1e-4, err.max()
    else:
        check_bf16(O, O_ref, f"O {w.name}", valid=mask[..., None])
    both_inf = np.isneginf(L) & np.isneginf(L_ref)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(L - L_ref))[mask]
    assert lerr.max() <= lse_tol(w, L_ref), lerr.max()


def run_and_check(w, use_block_mask=True, rows=None, heads=None):
    import torch
    g = DeviceRun(w, use_block_mask=use_block_mask)
    O, L = g.fwd()
    torch.cuda.synchronize()
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, oracle_spec(w), rows=rows, heads=heads)
    check(w, O, L, O_ref, L_ref, rows=rows)
    return g, O, L


def test_workload1_fp32_full():
    run_and_check(make_workload(1))


def test_workload1_fp32_without_block_mask():
    run_and_check(make_workload(1), use_block_mask=False)


FP32_CASES = [
    dict(B=2, Hq=4, Hkv=2, Sq=200, Skv=333, D=128, causal=True, alibi=True),
    dict(B=1, Hq=2, Hkv=1, S=300, D=64, causal=True, window=50, document=True, doc_lo=10,
         doc_hi=120, softcap=3.0),
    dict(B=2, Hq=2, Hkv=2, S=257, D=64, prefix=True, causal=True, prefix_lo=0, prefix_hi=300),
    dict(B=1, Hq=1, Hkv=1, Sq=40, Skv=5, D=64, causal=True, window=2),  # empty rows
]


@pytest.mark.parametrize("case", range(len(FP32_CASES)))
def test_fp32_ragged(case):
    w = make_workload(0, seed=200 + case, dtype="f32", **FP32_CASES[case])
    run_and_check(w)


# Reduced sizes of the bf16 workloads: every element is checked. They span
# several tiles per side so the full, partial and empty paths all run.
BF16_CASES = {
    "causal_alibi_d64": dict(B=2, Hq=4, Hkv=4, S=1024, D=64, causal=True, alibi=True),
    "doc_window_causal_d128": dict(B=1, Hq=4, Hkv=4, S=2048, D=128, causal=True, window=300,
                                   document=True, doc_lo=100, doc_hi=900),
    "gqa_prefix_softcap_d128": dict(B=2, Hq=8, Hkv=2, S=1024, D=128, causal=True, prefix=True,
                                    softcap=50.0, prefix_lo=64, prefix_hi=700),
    "causal_d128": dict(B=2, Hq=2, Hkv=2, S=1024, D=128, causal=True),
    "full_d64": dict(B=1, Hq=2, Hkv=1, S=512, D=64),
    "alibi_softcap_window_d64": dict(B=1, Hq=2, Hkv=2, S=768, D=64, causal=True, window=130,
                                     alibi=True, softcap=5.0),
    "odd_heads_gqa_d128": dict(B=1, Hq=3, Hkv=1, S=512, D=128, causal=True),
    "cross_lengths_d64": dict(B=1, Hq=2, Hkv=2, Sq=256, Skv=768, D=64, causal=True,
                              prefix=True, prefix_lo=300, prefix_hi=500),
    # Soft-caps small against the scores: |s / cap| > 1 in many or most
    # 32-row groups of a tile, so the tanh.approx form runs beside (cap 3) or
    # instead of (cap 1) the polynomial one.
    "softcap1_causal_d128": dict(B=1, Hq=2, Hkv=2, S=512, D=128, causal=True, softcap=1.0),
    "softcap3_gqa_d64": dict(B=1, Hq=4, Hkv=2, S=640, D=64, causal=True, softcap=3.0),
}


# bf16 with sequence lengths that are not multiples of the 128-row tile: the
# last query tile runs past Sq (rows not stored) and the last key tile past
# Skv (zero-filled keys masked), for every mask term and score_mod.
BF16_RAGGED = {
    "causal_alibi_d64_s300": dict(B=2, Hq=2, Hkv=2, S=300, D=64, causal=True, alibi=True),
    "full_d128_q100_k389": dict(B=1, Hq=2, Hkv=1, Sq=100, Skv=389, D=128),
    "doc_window_d128_s333": dict(B=1, Hq=2, Hkv=2, S=333, D=128, causal=True, window=90,
                                 document=True, doc_lo=20, doc_hi=150),
    "prefix_softcap_gqa_d64_q257_k129": dict(B=2, Hq=4, Hkv=2, Sq=257, Skv=129, D=64,
                                             causal=True, prefix=True, softcap=5.0,
                                             prefix_lo=60, prefix_hi=300),
    "single_row_d128": dict(B=1, Hq=1, Hkv=1, Sq=1, Skv=1, D=128, causal=True),
    "window_empty_rows_d64": dict(B=1, Hq=2, Hkv=2, Sq=140, Skv=7, D=64, causal=True,
                                  window=3),
    # Document masking alone with a last key tile that the block mask calls
    # full (one document over its keys and the last query tile's rows) but
    # that runs past Skv: the kernel masks it element by element and needs
    # its keys' document ids, which differ from 0 here.
    "doc_full_tail_d64_s200": dict(B=2, Hq=2, Hkv=2, S=200, D=64, document=True,
                                   doc_lengths=[[128, 72], [50, 78, 72]]),
    "doc_full_tail_gqa_d128_q300_k200": dict(B=1, Hq=4, Hkv=2, Sq=300, Skv=200, D=128,
                                             document=True, doc_lengths=[[100, 28, 172]]),
}


# Relative-position bias (a per-head table indexed by the query-key distance),
# alone and with every other term, at both head dims and a ragged length.
BF16_RELBIAS = {
    "causal_d64": dict(B=2, Hq=2, Hkv=2, S=512, D=64, causal=True, relbias=True),
    "doc_window_d128": dict(B=1, Hq=2, Hkv=2, S=768, D=128, causal=True, window=200,
                            document=True, doc_lo=60, doc_hi=400, relbias=True),
    "gqa_prefix_softcap_d128": dict(B=1, Hq=4, Hkv=2, S=512, D=128, causal=True, prefix=True,
                                    softcap=20.0, prefix_lo=50, prefix_hi=300, relbias=True),
    "alibi_softcap_full_d64": dict(B=1, Hq=2, Hkv=1, S=384, D=64, alibi=True, softcap=5.0,
                                   relbias=True),
    "ragged_causal_d128_q200_k333": dict(B=1, Hq=2, Hkv=2, Sq=200, Skv=333, D=128,
                                         causal=True, relbias=True),
}


@pytest.mark.parametrize("name", sorted(BF16_RELBIAS))
def test_bf16_rel_bias(name):
    w = make_workload(0, seed=500 + sorted(BF16_RELBIAS).index(name), **BF16_RELBIAS[name])
    run_and_check(w)


def test_fp32_rel_bias():
    w = make_workload(0, seed=520, dtype="f32", B=1, Hq=2, Hkv=1, Sq=150, Skv=211, D=64,
                      causal=True, window=90, alibi=True, relbias=True)
    run_and_check(w)


@pytest.mark.parametrize("name", sorted(BF16_RAGGED))
def test_bf16_ragged(name):
    w = make_workload(0, seed=400 + sorted(BF16_RAGGED).index(name), **BF16_RAGGED[name])
    run_and_check(w)


@pytest.mark.parametrize("name", ["causal_alibi_d64_s300", "full_d128_q100_k389"])
def test_bf16_ragged_without_block_mask(name):
    w = make_workload(0, seed=400 + sorted(BF16_RAGGED).index(name), **BF16_RAGGED[name])
    run_and_check(w, use_block_mask=False)


@pytest.mark.parametrize("name", sorted(BF16_CASES))
def test_bf16_reduced(name):
    w = make_workload(0, seed=300 + sorted(BF16_CASES).index(name), **BF16_CASES[name])
    run_and_check(w)


@pytest.mark.parametrize("name", ["causal_alibi_d64", "doc_window_causal_d128",
                                  "gqa_prefix_softcap_d128"])
def test_bf16_reduced_without_block_mask(name):
    w = make_workload(0, seed=300 + sorted(BF16_CASES).index(name), **BF16_CASES[name])
    run_and_check(w, use_block_mask=False)


def sample_rows(S, step=61):
    rows = set(range(0, 128)) | set(range(S - 128, S)) | set(range(0, S, step))
    return np.array(sorted(rows))


@pytest.mark.parametrize("number", [2, 3, 4, 5])
def test_full_size_workloads_sampled(number):
    """The full workloads in the launch configuration the benchmark times,
    checked on sampled rows of a few heads (rows are independent, so the
    sampled oracle rows are exact)."""
    w = make_workload(number)
    rows = sample_rows(w.Sq)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (w.B // 2, w.Hq // 2 + 1)]
    import torch
    g = DeviceRun(w)
    O, L = g.fwd()
    torch.cuda.synchronize()
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, oracle_spec(w), rows=rows, heads=heads)
    sel = np.zeros(w.Sq, bool)
    sel[rows] = True
    Oc = O.float().cpu().numpy()
    Lc = L.cpu().numpy()
    for b, h in heads:
        check_bf16(Oc[b, h, sel], O_ref[b, h, sel], f"O workload {number} head {(b, h)}")
        lerr = np.abs(Lc[b, h, sel] - L_ref[b, h, sel])
        assert lerr.max() <= lse_tol(w, None), lerr.max()
    assert np.isfinite(Lc).all() and np.isfinite(Oc).all()


def test_zero_query_gives_mean_of_kept_values():
    """Closed form on the GPU: Q = 0 gives the plain mean of the kept value
    rows (document + window + causal)."""
    import torch
    w = make_workload(0, seed=5, B=1, Hq=2, Hkv=2, S=1024, D=128, causal=True, window=200,
                      document=True, doc_lo=50, doc_hi=400)
    w.q = torch.zeros_like(w.q)
    run_and_check(w)


def test_deterministic():
    import torch
    w = make_workload(0, seed=9, **BF16_CASES["gqa_prefix_softcap_d128"])
    g = DeviceRun(w)
    O1, L1 = g.fwd()
    O2, L2 = g.fwd()
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_status_clean_after_runs():
    import masked_attention_gb300 as M
    assert M.attn_check_status() == M.ATTN_OK


# Multi-head attention at D = 128 without a block mask runs units of two query
# tiles of one head (2q, 2q + 1) over the union of their key tiles. Odd tile
# counts leave a last unit with one row; with a query offset (new tokens after
# a cached prefix) the two rows' causal ranges differ by a tile, and the
# earlier row's first visited tile is wholly masked for it.
PAIR_CASES = {
    "causal_odd_tiles_q300": dict(B=2, Hq=3, Hkv=3, Sq=300, Skv=300, D=128, causal=True),
    "causal_offset_q333_k700": dict(B=1, Hq=2, Hkv=2, Sq=333, Skv=700, D=128, causal=True,
                                    alibi=True),
    "window_offset_q384_k900": dict(B=1, Hq=2, Hkv=2, Sq=384, Skv=900, D=128, causal=True,
                                    window=200),
    "full_q200_k129": dict(B=1, Hq=1, Hkv=1, Sq=200, Skv=129, D=128),
}


@pytest.mark.parametrize("name", sorted(PAIR_CASES))
def test_bf16_query_tile_pairs(name):
    import dataclasses
    import torch
    import masked_attention_gb300 as M
    from tests.helpers import guarded_empty, check_canaries, variant_bits
    w = make_workload(0, seed=560 + sorted(PAIR_CASES).index(name), **PAIR_CASES[name])
    q_off = max(0, w.Skv - w.Sq)
    q, k, v = (t.cuda().contiguous() for t in (w.q, w.k, w.v))
    o = guarded_empty((w.B, w.Hq, w.Sq, w.D), torch.bfloat16)
    lse = guarded_empty((w.B, w.Hq, w.Sq), torch.float32)
    M.attn_fwd(q, k, v, o, lse, variant_bits(w), window=w.window or 0, q_offset=q_off)
    check_canaries()
    assert M.attn_check_status() == M.ATTN_OK
    spec = dataclasses.replace(oracle_spec(w), q_offset=q_off)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, spec)
    check(w, o, lse, O_ref, L_ref)


# Scores that jump far above a row's running reference: the keys of the first
# key tile (visited last: tiles go from the largest index down) and every query
# share a large component, so their scores exceed the reference taken from the
# later tiles by far more than 64 (log2 units). The tile's weights overflow the
# 2^64 bound, and the kernel redoes it with its true maximum, rescaling l and O.
# With the soft-cap the shared component also pushes |s / cap| past 1, which
# sends the polynomial form's columns back to tanh.approx.
REDO_CASES = {
    "causal_d128": dict(B=1, Hq=2, Hkv=2, S=768, D=128, causal=True),
    "gqa_softcap_d128": dict(B=1, Hq=4, Hkv=2, S=640, D=128, causal=True, softcap=50.0),
    "alibi_d64": dict(B=1, Hq=2, Hkv=2, S=512, D=64, causal=True, alibi=True),
    "prefix_gqa_d128": dict(B=1, Hq=2, Hkv=1, S=600, D=128, causal=True, prefix=True,
                            prefix_lo=100, prefix_hi=300),
}


@pytest.mark.parametrize("use_block_mask", [True, False])
@pytest.mark.parametrize("name", sorted(REDO_CASES))
def test_bf16_redo_after_large_scores(name, use_block_mask):
    import torch
    w = make_workload(0, seed=600 + sorted(REDO_CASES).index(name), **REDO_CASES[name])
    g = torch.Generator().manual_seed(601)
    u = torch.randn(w.D, generator=g)
    u = u / u.norm() * 30.0
    w.q = (w.q.float() + u).to(w.q.dtype)
    k = w.k.float()
    k[:, :, :128] += u
    w.k = k.to(w.k.dtype)
    run_and_check(w, use_block_mask=use_block_mask)
