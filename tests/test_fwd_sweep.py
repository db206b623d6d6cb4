"""A seeded sweep of random forward configurations against the oracle: head
dim, GQA grouping, ragged lengths, every combination of mask terms and
score terms, with and without the block mask. Each case is small enough for
the fp64 oracle to check every element."""
import numpy as np
import pytest

from synth import make_workload
from tests.test_fwd import run_and_check

pytestmark = pytest.mark.gpu


def sweep_cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(n):
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2]))
        Hq = Hkv * int(rng.choice([1, 2, 3]))
        Sq = int(rng.integers(1, 420))
        Skv = Sq if rng.random() < 0.5 else int(rng.integers(1, 420))
        spec = dict(B=int(rng.integers(1, 3)), Hq=Hq, Hkv=Hkv, Sq=Sq, Skv=Skv, D=D)
        if rng.random() < 0.6:
            spec["causal"] = True
        if rng.random() < 0.3:
            spec["window"] = int(rng.integers(1, 300))
        if rng.random() < 0.3:
            spec.update(document=True, doc_lo=int(rng.integers(1, 40)),
                        doc_hi=int(rng.integers(41, 300)))
        if rng.random() < 0.25:
            spec.update(prefix=True, prefix_lo=0, prefix_hi=int(rng.integers(1, 450)))
        if rng.random() < 0.4:
            spec["alibi"] = True
        if rng.random() < 0.3:
            spec["softcap"] = float(rng.choice([2.0, 10.0, 50.0]))
        if rng.random() < 0.2:
            spec["relbias"] = True
        cases.append((c, spec, bool(rng.random() < 0.75)))
    return cases


@pytest.mark.parametrize("case", sweep_cases(), ids=lambda c: f"case{c[0]}")
def test_forward_sweep(case):
    idx, spec, use_bm = case
    w = make_workload(0, seed=900 + idx, **spec)
    run_and_check(w, use_block_mask=use_bm)
