"""Seeded sweeps of random backward and decode configurations against the
oracle. Backward: head dim, GQA grouping, any Sq and Skv, every combination
of mask terms and score terms (the relative-position bias included), with and
without the block mask, gradients held to the flat bf16 bound. Decode: a few
query rows of a GQA group at the end of a contiguous or paged cache of any
length, every mask and score term, with and without key splits. Each case is
small enough for the fp64 oracle to check every element."""
import dataclasses

import numpy as np
import pytest

from oracle import attention_forward
from synth import make_workload
from tests.helpers import check_bf16, max_abs, oracle_spec
from tests.test_bwd import check_grads, run_bwd
from tests.test_decode import run_decode
from tests.test_fwd import lse_tol

pytestmark = pytest.mark.gpu


def _terms(rng, spec, S_hi):
    if rng.random() < 0.6:
        spec["causal"] = True
    if rng.random() < 0.3:
        spec["window"] = int(rng.integers(1, S_hi))
    if rng.random() < 0.3:
        spec.update(document=True, doc_lo=int(rng.integers(1, 40)),
                    doc_hi=int(rng.integers(41, S_hi)))
    if rng.random() < 0.25:
        spec.update(prefix=True, prefix_lo=0, prefix_hi=int(rng.integers(1, S_hi)))
    if rng.random() < 0.4:
        spec["alibi"] = True
    if rng.random() < 0.3:
        spec["softcap"] = float(rng.choice([2.0, 10.0, 50.0]))
    return spec


def bwd_cases(n=16, seed=3031):
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(n):
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2]))
        Hq = Hkv * int(rng.choice([1, 2, 4]))
        Sq = int(rng.integers(1, 400))
        Skv = Sq if rng.random() < 0.5 else int(rng.integers(1, 400))
        spec = _terms(rng, dict(B=int(rng.integers(1, 3)), Hq=Hq, Hkv=Hkv, Sq=Sq, Skv=Skv, D=D),
                      400)
        if rng.random() < 0.2:
            spec["relbias"] = True
        cases.append((c, spec, bool(rng.random() < 0.75)))
    return cases


@pytest.mark.parametrize("case", bwd_cases(), ids=lambda c: f"case{c[0]}")
def test_backward_sweep(case):
    idx, spec, use_bm = case
    w = make_workload(0, seed=3100 + idx, backward=True, **spec)
    _, dq, dk, dv = run_bwd(w, use_block_mask=use_bm)
    check_grads(w, dq, dk, dv)


def decode_cases(n=16, seed=4041):
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(n):
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2, 4]))
        group = int(rng.choice([1, 2, 4, 8]))
        Sq = int(rng.integers(1, 16 // group + 1))
        Skv = int(rng.integers(Sq, 3000))
        spec = _terms(rng, dict(B=int(rng.integers(1, 4)), Hq=Hkv * group, Hkv=Hkv, Sq=Sq,
                                Skv=Skv, D=D), 2000)
        page = int(rng.choice([0, 16, 32, 64, 128]))
        cases.append((c, spec, page, bool(rng.random() < 0.5)))
    return cases


@pytest.mark.parametrize("case", decode_cases(), ids=lambda c: f"case{c[0]}")
def test_decode_sweep(case):
    idx, spec, page, split = case
    w = make_workload(0, seed=4100 + idx, **spec)
    q_off = w.Skv - w.Sq  # the new rows at the end of the cache
    o, lse, _ = run_decode(w, q_off, page, split)
    ref_spec = dataclasses.replace(oracle_spec(w), q_offset=q_off)
    O_ref, L_ref = attention_forward(w.q, w.k, w.v, ref_spec)
    check_bf16(o.float().cpu().numpy(), O_ref, f"decode sweep {idx}")
    assert max_abs(lse.cpu().numpy(), L_ref) <= lse_tol(w, L_ref)
