"""CPU oracle for masked attention (fp64, numpy). TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call this module. The CUDA library never imports, links or
runs it, and it shares no code, table or constant with the CUDA library.

What it computes (FlexAttention page, "FlexAttention" section and its
``score_mod`` loop; Online-Softmax/FlashAttention page, abstract):

    s[b,h,i,j]  = scale * <q[b,h,i,:], k[b,hk,j,:]>           (hk = h // (Hq/Hkv))
    s'[b,h,i,j] = score_mod(s[b,h,i,j], b, h, i, j)            (applied element-wise)
    keep        = mask_mod(b, h, i, j)
    O[b,h,i,:]  = sum_j softmax_j(s' over kept j) * v[b,hk,j,:]
    LSE[b,h,i]  = log sum_{kept j} exp(s'[b,h,i,j])           (natural log)

The softmax is the 3-pass safe softmax named in the Online-Softmax /
FlashAttention page abstract: pass 1 takes the row maximum over kept entries,
pass 2 the sum of exp(s' - max), pass 3 normalises and multiplies by V. The
full score matrix of every (b, h) is materialised (in row slabs only to bound
memory; every row is always computed over all keys).

Readings taken where the pages are silent:

* scale defaults to 1/sqrt(D) and multiplies QK^T before score_mod;
* ALiBi adds ``-slope_h * (i - j)`` with ``slope_h = 2**(-8 (h+1) / Hq)``
  (h is the 0-based query head);
* soft-capping replaces the score by ``c * tanh(s / c)`` and, when ALiBi is
  also on, acts after the ALiBi bias;
* the mask is ``(causal AND window AND document) OR prefix`` over the terms
  that are switched on (absent AND-terms are true, an absent prefix is false):
  causal ``j <= i``, window ``i - j < W``, document ``doc[b,i] == doc[b,j]``,
  prefix ``j < P_b``; indices are absolute positions (top-left aligned);
* a row with no kept key has O = 0 and LSE = -inf;
* a call may be one shard of a longer sequence: query row r and key column c
  stand for absolute positions q_offset + r and kv_offset + c, and results
  over disjoint key shards merge by the online-softmax merge
  (``combine_partials``);
* GQA groups consecutive query heads: query head h reads KV head h // (Hq/Hkv).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

NEG_INF = -np.inf


@dataclasses.dataclass
class Spec:
    """Which score_mod / mask_mod terms are on, and their parameters."""
    causal: bool = False
    window: Optional[int] = None            # sliding window W (keys with i - j < W)
    doc_id: Optional[np.ndarray] = None     # int [B, L], L >= max(Sq, Skv)
    prefix_len: Optional[np.ndarray] = None  # int [B]
    alibi: bool = False
    alibi_slopes: Optional[np.ndarray] = None  # [Hq]; None -> 2**(-8(h+1)/Hq)
    softcap: Optional[float] = None
    scale: Optional[float] = None           # None -> 1/sqrt(D)
    # relative-position bias table [Hq, Sq + Skv - 1]; entry d + rel_bias_zero
    # is added for query-key distance d = i - j (rel_bias_zero = Skv - 1)
    rel_bias: Optional[np.ndarray] = None
    rel_bias_zero: int = 0
    # Absolute position of query row 0 and of key 0 (a shard of a longer
    # sequence, as in context-parallel attention): every mask term, the ALiBi
    # bias and the document ids use absolute positions q_offset + i and
    # kv_offset + j; doc_id then covers max(q_offset + Sq, kv_offset + Skv).
    q_offset: int = 0
    kv_offset: int = 0


def alibi_slopes(Hq: int) -> np.ndarray:
    """Geometric ALiBi slopes 2**(-8 (h+1) / Hq), h = 0..Hq-1."""
    h = np.arange(Hq, dtype=np.float64)
    return np.exp2(-8.0 * (h + 1.0) / Hq)


def mask_mod(spec: Spec, b: int, i: np.ndarray, j: np.ndarray) -> np.ndarray:
    """Boolean keep-mask for query positions ``i`` and key positions ``j``
    (broadcast against each other). FlexAttention page, "Causal Mask" and
    "Sliding Window + Causal" sections, and its list of variants (document
    masking, PrefixLM)."""
    i = np.asarray(i, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    keep = np.ones(np.broadcast_shapes(i.shape, j.shape), dtype=bool)
    if spec.causal:
        keep &= j <= i
    if spec.window is not None:
        keep &= (i - j) < spec.window
    if spec.doc_id is not None:
        doc = np.asarray(spec.doc_id[b], dtype=np.int64)
        keep &= doc[i] == doc[j]
    if spec.prefix_len is not None:
        keep |= j < int(spec.prefix_len[b])
    return keep


def score_mod(spec: Spec, s: np.ndarray, h: int, Hq: int, i: np.ndarray,
              j: np.ndarray) -> np.ndarray:
    """Element-wise score modification applied before the softmax
    (FlexAttention page, "FlexAttention" section: score_mod(score, b, h,
    q_idx, kv_idx); "Soft-capping" and relative-position sections)."""
    out = s
    if spec.alibi:
        slopes = spec.alibi_slopes if spec.alibi_slopes is not None else alibi_slopes(Hq)
        out = out - float(slopes[h]) * (np.asarray(i, np.float64) - np.asarray(j, np.float64))
    if spec.rel_bias is not None:
        out = out + rel_bias_term(spec, h, i, j)
    if spec.softcap is not None:
        c = float(spec.softcap)
        out = c * np.tanh(out / c)
    return out


def rel_bias_term(spec: Spec, h: int, i: np.ndarray, j: np.ndarray) -> np.ndarray:
    """Relative-position bias: a per-head table indexed by the query-key
    distance i - j (FlexAttention page, relative position encoding: the score
    is adjusted by the distance between query and key, computed in the kernel
    without an S x S tensor). The table is a captured buffer of the call."""
    d = np.asarray(i, np.int64) - np.asarray(j, np.int64)
    return np.asarray(spec.rel_bias[h], np.float64)[d + spec.rel_bias_zero]


def score_mod_grad(spec: Spec, s: np.ndarray, h: int, Hq: int, i: np.ndarray,
                   j: np.ndarray) -> np.ndarray:
    """d score_mod / d s (chain rule: the ALiBi bias has slope 1 in s; the
    soft-cap c*tanh(x/c) has derivative 1 - tanh(x/c)**2)."""
    if spec.softcap is None:
        return np.ones_like(s)
    x = s
    if spec.alibi:
        slopes = spec.alibi_slopes if spec.alibi_slopes is not None else alibi_slopes(Hq)
        x = x - float(slopes[h]) * (np.asarray(i, np.float64) - np.asarray(j, np.float64))
    if spec.rel_bias is not None:
        x = x + rel_bias_term(spec, h, i, j)
    t = np.tanh(x / float(spec.softcap))
    return 1.0 - t * t


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: bf16 widens to fp64 exactly
        x = x.detach().to("cpu")
        import torch  # local: the oracle itself needs only numpy
        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _scale(spec: Spec, D: int) -> float:
    return float(spec.scale) if spec.scale is not None else 1.0 / math.sqrt(D)


def _slab_rows(Skv: int, budget_bytes: int = 256 << 20) -> int:
    return max(1, budget_bytes // (8 * 4 * max(Skv, 1)))


def attention_forward(q, k, v, spec: Spec, rows: Optional[Sequence[int]] = None,
                      heads: Optional[Sequence[tuple]] = None):
    """Oracle forward. Returns ``(O, LSE)`` in fp64.

    ``q`` [B,Hq,Sq,D], ``k``/``v`` [B,Hkv,Skv,D] (numpy or torch; widened to
    fp64). ``rows`` restricts the query rows computed (other rows stay NaN);
    ``heads`` restricts the (b, h) pairs computed. Rows are independent, so a
    restricted run gives exactly the same values on the rows it computes.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    assert Hq % Hkv == 0, "Hq must be a multiple of Hkv"
    group = Hq // Hkv
    scale = _scale(spec, D)
    O = np.full((B, Hq, Sq, v.shape[3]), np.nan)
    LSE = np.full((B, Hq, Sq), np.nan)
    row_idx = np.arange(Sq) if rows is None else np.asarray(rows, dtype=np.int64)
    pairs = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    j = np.arange(Skv)[None, :]
    ja = j + spec.kv_offset  # absolute key positions
    slab = _slab_rows(Skv)
    for b, h in pairs:
        hk = h // group
        for start in range(0, len(row_idx), slab):
            i = row_idx[start:start + slab][:, None]
            ia = i + spec.q_offset  # absolute query positions
            s = scale * (q[b, h, i[:, 0], :] @ k[b, hk].T)
            s = score_mod(spec, s, h, Hq, ia, ja)
            keep = mask_mod(spec, b, ia, ja)
            # pass 1: row maximum over kept entries
            m = np.where(keep, s, NEG_INF).max(axis=1)
            m_safe = np.where(np.isfinite(m), m, 0.0)
            # pass 2: sum of exponentials relative to the maximum
            e = np.exp(np.where(keep, s - m_safe[:, None], -np.inf))
            l = e.sum(axis=1)
            # pass 3: normalise and weight the values
            with np.errstate(invalid="ignore", divide="ignore"):
                p = np.where(l[:, None] > 0, e / np.where(l > 0, l, 1.0)[:, None], 0.0)
                O[b, h, i[:, 0], :] = p @ v[b, hk]
                LSE[b, h, i[:, 0]] = np.where(l > 0, m_safe + np.log(np.where(l > 0, l, 1.0)),
                                              NEG_INF)
    return O, LSE


def attention_backward(q, k, v, do, spec: Spec, heads: Optional[Sequence[tuple]] = None):
    """Analytic gradients of ``sum(dO * O)`` with respect to q, k, v (fp64).

    The FlexAttention page ("Performance" section) describes a deterministic
    backward that recomputes intermediates; here everything is recomputed from
    scratch in fp64:

        P      = exp(s' - LSE) on kept entries, else 0
        dV_j   = sum_i P_ij dO_i
        dP_ij  = <dO_i, v_j>
        Delta_i= <dO_i, O_i>
        dS_ij  = P_ij (dP_ij - Delta_i) * score_mod'(s_ij)
        dQ_i   = scale * sum_j dS_ij k_j
        dK_j   = scale * sum_i dS_ij q_i

    With GQA, dK and dV of a KV head sum over the query heads of its group.
    Returns ``(dQ, dK, dV, O, LSE)``; with ``heads`` given, only those (b, h)
    contribute (other entries of dQ stay NaN, dK/dV hold partial sums).
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    group = Hq // Hkv
    scale = _scale(spec, D)
    O, LSE = attention_forward(q, k, v, spec, heads=heads)
    dQ = np.full_like(q, np.nan)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    pairs = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    i = np.arange(Sq)[:, None] + spec.q_offset   # absolute positions
    j = np.arange(Skv)[None, :] + spec.kv_offset
    for b, h in pairs:
        hk = h // group
        s = scale * (q[b, h] @ k[b, hk].T)
        t = score_mod(spec, s, h, Hq, i, j)
        keep = mask_mod(spec, b, i, j)
        lse = LSE[b, h][:, None]
        with np.errstate(invalid="ignore"):
            P = np.where(keep & np.isfinite(lse), np.exp(t - np.where(np.isfinite(lse), lse, 0.0)),
                         0.0)
        dV[b, hk] += P.T @ do[b, h]
        dP = do[b, h] @ v[b, hk].T
        delta = np.sum(do[b, h] * O[b, h], axis=1)
        dS = P * (dP - delta[:, None]) * score_mod_grad(spec, s, h, Hq, i, j)
        dQ[b, h] = scale * (dS @ k[b, hk])
        dK[b, hk] += scale * (dS.T @ q[b, h])
    return dQ, dK, dV, O, LSE


@dataclasses.dataclass
class BlockMask:
    """Tile classification (exploiting mask sparsity: FlexAttention page,
    list item on sparsity). Tile (qt, kt) covers query rows
    [qt*BM, min((qt+1)*BM, Sq)) and key columns [kt*BN, min((kt+1)*BN, Skv)).
    A tile is full if every pair in it is kept, empty if none is, else partial.
    Lists are ascending."""
    full_cnt: np.ndarray   # int32 [B, nq]
    part_cnt: np.ndarray   # int32 [B, nq]
    full_idx: list         # [B][nq] -> list of kt
    part_idx: list
    t_full_cnt: np.ndarray  # int32 [B, nkv] (transposed: per KV tile, its q tiles)
    t_part_cnt: np.ndarray
    t_full_idx: list
    t_part_idx: list
    state: np.ndarray      # int8 [B, nq, nkv]: 0 empty, 1 partial, 2 full


def block_mask(spec: Spec, B: int, Sq: int, Skv: int, BM: int = 128, BN: int = 128) -> BlockMask:
    """Brute-force tile classification: evaluates mask_mod on every (i, j)."""
    nq = (Sq + BM - 1) // BM
    nkv = (Skv + BN - 1) // BN
    state = np.zeros((B, nq, nkv), dtype=np.int8)
    for b in range(B):
        for qt in range(nq):
            i = np.arange(qt * BM, min((qt + 1) * BM, Sq))[:, None] + spec.q_offset
            j = np.arange(Skv)[None, :] + spec.kv_offset
            keep = mask_mod(spec, b, i, j)
            for kt in range(nkv):
                tile = keep[:, kt * BN:min((kt + 1) * BN, Skv)]
                if tile.all():
                    state[b, qt, kt] = 2
                elif tile.any():
                    state[b, qt, kt] = 1
    full_idx = [[list(np.nonzero(state[b, qt] == 2)[0]) for qt in range(nq)] for b in range(B)]
    part_idx = [[list(np.nonzero(state[b, qt] == 1)[0]) for qt in range(nq)] for b in range(B)]
    t_full_idx = [[list(np.nonzero(state[b, :, kt] == 2)[0]) for kt in range(nkv)] for b in range(B)]
    t_part_idx = [[list(np.nonzero(state[b, :, kt] == 1)[0]) for kt in range(nkv)] for b in range(B)]
    return BlockMask(
        full_cnt=(state == 2).sum(axis=2).astype(np.int32),
        part_cnt=(state == 1).sum(axis=2).astype(np.int32),
        full_idx=full_idx, part_idx=part_idx,
        t_full_cnt=(state == 2).sum(axis=1).astype(np.int32),
        t_part_cnt=(state == 1).sum(axis=1).astype(np.int32),
        t_full_idx=t_full_idx, t_part_idx=t_part_idx, state=state)


def kept_per_row(spec: Spec, B: int, Sq: int, Skv: int) -> np.ndarray:
    """Number of kept keys of every query row, int64 [B, Sq]."""
    out = np.zeros((B, Sq), dtype=np.int64)
    j = np.arange(Skv)[None, :] + spec.kv_offset
    slab = _slab_rows(Skv, 64 << 20)
    for b in range(B):
        for start in range(0, Sq, slab):
            i = np.arange(start, min(start + slab, Sq))[:, None] + spec.q_offset
            out[b, start:start + slab] = mask_mod(spec, b, i, j).sum(axis=1)
    return out


def combine_partials(parts):
    """Merges attention results over disjoint key sets into the result over
    their union. ``parts`` is a sequence of ``(O_k, LSE_k)``, each the output
    and log-sum-exp of the same queries against one key shard (fp64 or
    widened to it; LSE_k = -inf where a row kept no key of that shard).

    This is the merge step of the online softmax (Online-Softmax/FlashAttention
    page, the 2-pass online softmax: two partial maxima and sums combine as
    m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m)) applied to whole partial
    results, as context-parallel attention does with key/value shards
    (FlexAttention page, variant list: sliding window + document masking +
    causal + context parallel). Because O_k is normalised by its own sum,
    O = sum_k e^(LSE_k - LSE) O_k with LSE = ln sum_k e^(LSE_k). A row with no
    kept key in any shard gets O = 0 and LSE = -inf.
    """
    Os = [_as_f64(o) for o, _ in parts]
    Ls = [_as_f64(l) for _, l in parts]
    L = np.stack(Ls)                       # [K, ...rows]
    m = L.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(L - m_safe)                 # e^(LSE_k - m); 0 for empty parts
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, m_safe + np.log(np.where(tot > 0, tot, 1.0)), NEG_INF)
        frac = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0)
    # a part with weight 0 contributes nothing (its O row may be anything)
    O = sum(np.where(frac[k][..., None] > 0, frac[k][..., None] * Os[k], 0.0) for k in range(len(Os)))
    return O, lse
