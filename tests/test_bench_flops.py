"""The benchmark's FLOP count (the numerator of its metric): 4 * D * kept
(query, key) pairs. Its own mask count must agree with the oracle's and with
closed forms; no GPU needed."""
import numpy as np
import pytest

import bench
from oracle import block_mask, kept_per_row
from synth import make_workload
from tests.helpers import oracle_spec

SMALL = [
    dict(B=2, Hq=2, Hkv=2, S=300, D=64, causal=True, alibi=True),
    dict(B=1, Hq=2, Hkv=2, S=700, D=128, causal=True, window=100, document=True, doc_lo=50,
         doc_hi=200),
    dict(B=2, Hq=4, Hkv=1, S=500, D=128, causal=True, prefix=True, prefix_lo=10, prefix_hi=400),
    dict(B=1, Hq=1, Hkv=1, Sq=130, Skv=260, D=64),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_kept_pairs_match_oracle(case):
    w = make_workload(0, seed=30 + case, with_tensors=False, **SMALL[case])
    ref = int(kept_per_row(oracle_spec(w), w.B, w.Sq, w.Skv).sum())
    assert bench.kept_pairs(w) == ref


def test_bench_workload_flops_closed_form():
    """Causal, B=4, S=2048: every batch element keeps S(S+1)/2 pairs per head;
    16 heads at D = 64 make 34.36 GFLOP per forward."""
    w = make_workload(2, with_tensors=False)
    S = w.Sq
    assert bench.kept_pairs(w) == w.B * S * (S + 1) // 2
    flops = 4.0 * w.D * bench.kept_pairs(w) * w.Hq
    assert flops == 4 * 64 * 4 * 2048 * 2049 // 2 * 16
    assert abs(flops / 1e9 - 34.3765) < 1e-3


def test_window_workload_density():
    """Document + window 1024 + causal at S = 16384: every row keeps at most
    1024 keys, so the density is below 1024 / S."""
    w = make_workload(3, with_tensors=False)
    kept = bench.kept_pairs(w)
    assert 0 < kept <= w.B * w.Sq * 1024
    assert kept / (w.B * w.Sq * w.Skv) < 1024 / w.Skv


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_visited_pairs_match_oracle_tiles(case):
    """Executed work: the in-bounds area of every tile the oracle's brute-force
    classification calls full or partial."""
    w = make_workload(0, seed=30 + case, with_tensors=False, **SMALL[case])
    bm = block_mask(oracle_spec(w), w.B, w.Sq, w.Skv)
    area = 0
    for b, qt, kt in zip(*np.nonzero(bm.state)):
        rows = min(128, w.Sq - 128 * qt)
        cols = min(128, w.Skv - 128 * kt)
        area += rows * cols
    assert bench.visited_pairs(w) == area
    assert bench.kept_pairs(w) <= area


def test_bench_workload_executed_over_algorithmic():
    """Causal S = 2048: 136 of 256 tiles per head are visited (16 of them on
    the diagonal, a little over half kept there): 1.062 times the kept pairs."""
    w = make_workload(2, with_tensors=False)
    ratio = bench.visited_pairs(w) / bench.kept_pairs(w)
    assert bench.visited_pairs(w) == w.B * 136 * 128 * 128
    assert abs(ratio - (136 * 128 * 128) / (2048 * 2049 / 2)) < 1e-12
