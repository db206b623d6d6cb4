"""Context-parallel ring schedule on CPU ranks (gloo).

The ring module (``masked_attention_gb300/context_parallel.py``) is host
logic: which key/value shard a rank holds at each step, the shard exchange
along the ring, the skip of pairs the mask empties, and the merge. Here it
runs on 2 and 3 gloo ranks with the oracle as the per-shard compute and the
oracle's merge, and every rank's merged result is compared with the
oracle's attention over the whole sequence (FlexAttention page, variant
list: ... + context parallel; Online-Softmax/FlashAttention page, the merge
of partial maxima and sums). No GPU is involved.
"""
import os
import socket

import numpy as np
import pytest

from masked_attention_gb300.context_parallel import (pair_may_keep, ring_order,
                                                     shard_cuts)

CASES = {
    # document + sliding window + causal (the page's composed mask)
    "doc_window_causal": dict(B=1, Hq=2, Hkv=1, S=300, D=16, causal=True, window=70,
                              document=True, doc_lo=30, doc_hi=120),
    # PrefixLM + causal + soft-cap + GQA: the prefix keeps later shards' pairs
    "prefix_causal_softcap": dict(B=2, Hq=4, Hkv=2, S=257, D=16, causal=True, prefix=True,
                                  prefix_lo=20, prefix_hi=150, softcap=5.0),
    # full attention + ALiBi: no pair is skipped
    "full_alibi": dict(B=1, Hq=2, Hkv=2, S=100, D=8, alibi=True),
}


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, name, out_dir):
    import torch
    import torch.distributed as dist

    from masked_attention_gb300.context_parallel import ring_forward
    from oracle import attention_forward, combine_partials
    from synth import make_workload
    from tests.helpers import oracle_spec

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = make_workload(0, seed=40 + sorted(CASES).index(name), **CASES[name])
        spec = oracle_spec(w)
        cuts = shard_cuts(w.Sq, world)
        lo, hi = cuts[rank], cuts[rank + 1]
        q = w.q[:, :, lo:hi].double().contiguous()
        k = w.k[:, :, lo:hi].double().contiguous()
        v = w.v[:, :, lo:hi].double().contiguous()

        def shard_forward(qs, ks, vs, q_offset, kv_offset):
            import dataclasses
            s = dataclasses.replace(spec, q_offset=q_offset, kv_offset=kv_offset)
            O, L = attention_forward(qs, ks, vs, s)
            return torch.from_numpy(O), torch.from_numpy(L)

        trace = []
        O, L = ring_forward(q, k, v, rank=rank, world=world, cuts=cuts,
                            shard_forward=shard_forward, merge=combine_partials,
                            causal=w.causal, window=w.window or 0,
                            prefix_max=int(w.prefix_len.max()) if w.prefix else None,
                            trace=trace)
        O_ref, L_ref = attention_forward(w.q, w.k, w.v, spec, rows=np.arange(lo, hi))
        O_ref, L_ref = O_ref[:, :, lo:hi], L_ref[:, :, lo:hi]
        err_o = float(np.abs(np.asarray(O) - O_ref).max())
        both_inf = np.isneginf(np.asarray(L)) & np.isneginf(L_ref)
        err_l = float(np.where(both_inf, 0.0, np.abs(np.asarray(L) - L_ref)).max())
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([err_o, err_l, len(trace), sum(r for _, _, r in trace)]))
        with open(os.path.join(out_dir, f"trace{rank}.txt"), "w") as f:
            f.write(repr(trace))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name", sorted(CASES))
def test_ring_forward_on_gloo_ranks_equals_whole_sequence(name, world, tmp_path):
    import torch.multiprocessing as mp
    mp.start_processes(_rank_main, args=(world, _free_port(), name, str(tmp_path)),
                       nprocs=world, start_method="spawn", join=True)
    w_causal = CASES[name].get("causal", False)
    for r in range(world):
        err_o, err_l, steps, computed = np.load(tmp_path / f"rank{r}.npy")
        assert err_o <= 1e-12 and err_l <= 1e-12, (r, err_o, err_l)
        assert steps == world  # one step per key/value shard
        trace = eval(open(tmp_path / f"trace{r}.txt").read())
        assert [j for _, j, _ in trace] == ring_order(r, world)
        if w_causal and not CASES[name].get("prefix"):
            # key shards after the query shard are skipped (causal); the own
            # shard always runs
            assert all(run for _, j, run in trace if j == r), trace
            assert not any(run for _, j, run in trace if j > r), trace
        if name == "doc_window_causal" and world == 3 and r == 2:
            # shard 0 (positions 0..99) lies wholly outside the 70-token window
            # of queries 200..299
            assert (2, 0, False) in trace, trace


def test_shard_cuts_cover_the_sequence():
    for S, world in [(10, 3), (128, 4), (5, 5), (0, 2), (7, 1)]:
        c = shard_cuts(S, world)
        assert c[0] == 0 and c[-1] == S and len(c) == world + 1
        sizes = np.diff(c)
        assert sizes.max() - sizes.min() <= 1


def test_ring_order_visits_every_shard_once():
    for world in (1, 2, 5):
        for r in range(world):
            o = ring_order(r, world)
            assert o[0] == r and sorted(o) == list(range(world))


def test_pair_may_keep_is_exact_on_small_ranges():
    """Brute force: pair_may_keep is False only when no pair is kept, for the
    causal, window and prefix terms (the document term is never used)."""
    rng = np.random.default_rng(3)
    for _ in range(400):
        q_lo, kv_lo = int(rng.integers(0, 40)), int(rng.integers(0, 40))
        q_hi, kv_hi = q_lo + int(rng.integers(1, 12)), kv_lo + int(rng.integers(1, 12))
        causal = bool(rng.random() < 0.7)
        window = int(rng.integers(1, 20)) if rng.random() < 0.5 else 0
        prefix = int(rng.integers(0, 50)) if rng.random() < 0.4 else None
        i = np.arange(q_lo, q_hi)[:, None]
        j = np.arange(kv_lo, kv_hi)[None, :]
        keep = np.ones((q_hi - q_lo, kv_hi - kv_lo), bool)
        if causal:
            keep &= j <= i
        if window:
            keep &= (i - j) < window
        if prefix is not None:
            keep |= j < prefix
        got = pair_may_keep(causal, window, prefix, q_lo, q_hi, kv_lo, kv_hi)
        assert got == bool(keep.any())
