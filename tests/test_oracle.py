"""Pins for the CPU oracle: brute force, a library special case, closed forms,
invariants and finite differences. None of these re-uses the oracle's own
vectorised code path, so a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.

Pages cited: the FlexAttention page (sections "FlexAttention", "Causal Mask",
"Sliding Window + Causal", "Soft-capping", the variant list and the sparsity
item) and the Online-Softmax/FlashAttention page (abstract: 3-pass safe
softmax, 2-pass online softmax, 1-pass FlashAttention).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (Spec, alibi_slopes, attention_backward, attention_forward, block_mask,
                    combine_partials, kept_per_row)
from synth import doc_ids_from_lengths, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------------------
# Brute force: the element-by-element score_mod loop of the FlexAttention page
# ("FlexAttention" section), with the softmax written out per row in pure
# Python floats.
# ---------------------------------------------------------------------------

def brute_force(q, k, v, causal=False, window=None, doc=None, prefix=None, alibi=False,
                softcap=None, table=None):
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    group = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    O = np.zeros((B, Hq, Sq, D))
    LSE = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            slope = 2.0 ** (-8.0 * (h + 1) / Hq)
            for qi in range(Sq):
                scores = []
                for kj in range(Skv):
                    dot = 0.0
                    for d in range(D):
                        dot += float(q[b, h, qi, d]) * float(k[b, hk, kj, d])
                    sc = dot * scale
                    if alibi:
                        sc = sc + slope * (kj - qi)
                    if table is not None:  # bias by the query-key distance
                        sc = sc + float(table[h][qi - kj + Skv - 1])
                    if softcap is not None:
                        sc = softcap * math.tanh(sc / softcap)
                    ok = True
                    if causal and not (kj <= qi):
                        ok = False
                    if window is not None and not (qi - kj < window):
                        ok = False
                    if doc is not None and doc[b][qi] != doc[b][kj]:
                        ok = False
                    if prefix is not None and kj < prefix[b]:
                        ok = True
                    if ok:
                        scores.append((kj, sc))
                if not scores:
                    LSE[b, h, qi] = -math.inf
                    continue
                top = max(sc for _, sc in scores)
                den = sum(math.exp(sc - top) for _, sc in scores)
                for kj, sc in scores:
                    w = math.exp(sc - top) / den
                    for d in range(D):
                        O[b, h, qi, d] += w * float(v[b, hk, kj, d])
                LSE[b, h, qi] = top + math.log(den)
    return O, LSE


BF_CASES = [
    dict(),
    dict(causal=True),
    dict(causal=True, alibi=True),
    dict(causal=True, window=3),
    dict(causal=True, window=4, doc=[[0, 0, 0, 1, 1, 1, 1, 2, 2, 2]] * 2),
    dict(causal=True, prefix=[4, 7], softcap=2.0),
    dict(alibi=True, softcap=1.5),
    dict(window=2),
    dict(causal=True, table="rel"),
    dict(alibi=True, softcap=2.5, table="rel", window=5),
]


@pytest.mark.parametrize("case", BF_CASES)
@pytest.mark.parametrize("heads", [(2, 2), (4, 2)])
def test_oracle_matches_brute_force(case, heads):
    Hq, Hkv = heads
    B, S, D = 2, 10, 4
    q = rnd((B, Hq, S, D), 1)
    k = rnd((B, Hkv, S, D), 2)
    v = rnd((B, Hkv, S, D), 3)
    case = dict(case)
    table = None
    if case.pop("table", None):
        table = rnd((Hq, 2 * S - 1), 11)
    O_ref, L_ref = brute_force(q, k, v, table=table, **case)
    spec = Spec(causal=case.get("causal", False), window=case.get("window"),
                doc_id=np.array(case["doc"]) if "doc" in case else None,
                prefix_len=np.array(case["prefix"]) if "prefix" in case else None,
                alibi=case.get("alibi", False), softcap=case.get("softcap"),
                rel_bias=table, rel_bias_zero=S - 1)
    O, L = attention_forward(q, k, v, spec)
    assert np.max(np.abs(O - O_ref)) < 1e-12
    assert np.max(np.abs(L - L_ref)) < 1e-12


# ---------------------------------------------------------------------------
# Library special case: PyTorch's scaled_dot_product_attention in fp64 on the
# CPU (mask-only variants have the identity score_mod).
# ---------------------------------------------------------------------------

def test_oracle_matches_sdpa_causal_flag():
    q, k, v = rnd((2, 3, 33, 8), 4), rnd((2, 3, 33, 8), 5), rnd((2, 3, 33, 8), 6)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True).numpy()
    O, _ = attention_forward(q, k, v, Spec(causal=True))
    assert np.max(np.abs(O - ref)) < 1e-12


def test_oracle_matches_sdpa_gqa():
    q, k, v = rnd((1, 8, 20, 8), 7), rnd((1, 2, 20, 8), 8), rnd((1, 2, 20, 8), 9)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), enable_gqa=True).numpy()
    O, _ = attention_forward(q, k, v, Spec())
    assert np.max(np.abs(O - ref)) < 1e-12


def test_oracle_matches_sdpa_boolean_mask():
    S = 40
    doc = np.array([doc_ids_from_lengths([13, 9, 18], S)])
    q, k, v = rnd((1, 2, S, 16), 10), rnd((1, 2, S, 16), 11), rnd((1, 2, S, 16), 12)
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    mask = (j <= i) & (i - j < 7) & (doc[0][i] == doc[0][j])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask)).numpy()
    O, _ = attention_forward(q, k, v, Spec(causal=True, window=7, doc_id=doc))
    assert np.max(np.abs(O - ref)) < 1e-12


# ---------------------------------------------------------------------------
# Closed forms.
# ---------------------------------------------------------------------------

def test_zero_query_gives_mean_of_kept_values():
    """Q = 0 makes every kept score 0: O_i is the plain mean of the kept value
    rows and LSE_i = ln(#kept). The kept sets are written as index ranges."""
    S, D, W, P = 50, 4, 6, 17
    lengths = [12, 20, 18]
    doc = np.array([doc_ids_from_lengths(lengths, S)])
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    doc_start = np.array([starts[d] for d in doc[0]])
    v = rnd((1, 1, S, D), 13)
    k = rnd((1, 1, S, D), 14)
    q = np.zeros((1, 1, S, D))
    cases = {
        "causal": (Spec(causal=True), lambda i: range(0, i + 1)),
        "window": (Spec(causal=True, window=W), lambda i: range(max(0, i - W + 1), i + 1)),
        "prefix": (Spec(causal=True, prefix_len=np.array([P])), lambda i: range(0, max(i + 1, P))),
        "document": (Spec(causal=True, doc_id=doc), lambda i: range(doc_start[i], i + 1)),
        "doc+window": (Spec(causal=True, window=W, doc_id=doc),
                       lambda i: range(max(doc_start[i], i - W + 1), i + 1)),
        "full": (Spec(), lambda i: range(0, S)),
    }
    for name, (spec, kept) in cases.items():
        O, L = attention_forward(q, k, v, spec)
        for i in range(S):
            js = list(kept(i))
            assert np.allclose(O[0, 0, i], v[0, 0, js].mean(axis=0), atol=1e-13), name
            assert abs(L[0, 0, i] - math.log(len(js))) < 1e-13, name
        counts = kept_per_row(spec, 1, S, S)[0]
        assert list(counts) == [len(list(kept(i))) for i in range(S)], name


def test_alibi_geometric_series():
    """Q = 0 with causal ALiBi: row i weights key i-d by exp(-m_h d), so
    LSE_i = ln((1 - exp(-m_h (i+1))) / (1 - exp(-m_h))) with m_h = 2^(-8(h+1)/H)."""
    H, S, D = 4, 24, 4
    v = rnd((1, H, S, D), 15)
    O, L = attention_forward(np.zeros((1, H, S, D)), rnd((1, H, S, D), 16), v,
                             Spec(causal=True, alibi=True))
    for h in range(H):
        m = 2.0 ** (-8.0 * (h + 1) / H)
        for i in range(S):
            lse = math.log((1 - math.exp(-m * (i + 1))) / (1 - math.exp(-m)))
            assert abs(L[0, h, i] - lse) < 1e-12
            w = np.exp(-m * np.arange(i + 1))
            w /= w.sum()
            expect = sum(w[d] * v[0, h, i - d] for d in range(i + 1))
            assert np.allclose(O[0, h, i], expect, atol=1e-12)
    assert np.allclose(alibi_slopes(8), [2.0 ** -(x + 1) for x in range(8)])


def test_softcap_closed_form():
    """Every key equal, so every score is the same t = scale*<q,k>; the capped
    score is c*tanh(t/c) and LSE = c*tanh(t/c) + ln(#kept)."""
    S, D, c = 12, 16, 50.0
    k = np.tile(rnd((1, 1, 1, D), 17), (1, 1, S, 1))
    kk = k[0, 0, 0]
    q = np.zeros((1, 1, S, D))
    for i in range(S):  # t_i grows from -200 to +200: beyond the cap
        q[0, 0, i] = kk * ((-200 + 400 * i / (S - 1)) * math.sqrt(D) / kk.dot(kk))
    _, L = attention_forward(q, k, rnd((1, 1, S, D), 18), Spec(causal=True, softcap=c))
    for i in range(S):
        t = -200 + 400 * i / (S - 1)
        assert abs(L[0, 0, i] - (c * math.tanh(t / c) + math.log(i + 1))) < 1e-11


def test_causal_first_rows():
    """Causal row 0 sees only key 0: O_0 = v_0, LSE_0 = <q_0,k_0>/sqrt(D).
    Row 1 mixes v_0 and v_1 with weight sigmoid((<q_1,k_0> - <q_1,k_1>)/sqrt(D))."""
    D = 32
    q, k, v = rnd((1, 1, 6, D), 19), rnd((1, 1, 6, D), 20), rnd((1, 1, 6, D), 21)
    O, L = attention_forward(q, k, v, Spec(causal=True))
    assert np.allclose(O[0, 0, 0], v[0, 0, 0], atol=1e-15)
    assert abs(L[0, 0, 0] - q[0, 0, 0].dot(k[0, 0, 0]) / math.sqrt(D)) < 1e-13
    a = (q[0, 0, 1].dot(k[0, 0, 0]) - q[0, 0, 1].dot(k[0, 0, 1])) / math.sqrt(D)
    w0 = 1.0 / (1.0 + math.exp(-a))
    assert np.allclose(O[0, 0, 1], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1], atol=1e-13)


def test_empty_rows_give_zero_and_minus_inf():
    """Causal + window 2 with fewer keys than queries: rows i >= Skv + 1 keep
    no key, so O = 0 and LSE = -inf there."""
    q, k, v = rnd((1, 1, 16, 4), 22), rnd((1, 1, 4, 4), 23), rnd((1, 1, 4, 4), 24)
    O, L = attention_forward(q, k, v, Spec(causal=True, window=2))
    assert np.all(O[0, 0, 5:] == 0.0) and np.all(np.isneginf(L[0, 0, 5:]))
    assert np.all(np.isfinite(L[0, 0, :5]))


def test_page_window_is_1024_recent_tokens():
    """Golden fact from the FlexAttention page ("Sliding Window + Causal"):
    a query attends to the most recent 1024 tokens. With W = 1024, every row
    past the first 1023 keeps exactly 1024 keys, itself included."""
    with open(os.path.join(GOLDEN, "flexattention_page_facts.json")) as f:
        facts = json.load(f)
    W = facts["sliding_window_tokens"]["value"]
    counts = kept_per_row(Spec(causal=True, window=W), 1, 3000, 3000)[0]
    assert np.all(counts[W - 1:] == W)
    assert list(counts[:5]) == [1, 2, 3, 4, 5]


# ---------------------------------------------------------------------------
# Invariants.
# ---------------------------------------------------------------------------

def test_window_at_least_S_equals_causal():
    q, k, v = rnd((1, 2, 40, 8), 25), rnd((1, 2, 40, 8), 26), rnd((1, 2, 40, 8), 27)
    a = attention_forward(q, k, v, Spec(causal=True, window=40))
    b = attention_forward(q, k, v, Spec(causal=True))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_document_mask_equals_independent_documents():
    lengths = [9, 14, 1, 16]
    S = sum(lengths)
    doc = np.array([doc_ids_from_lengths(lengths, S)])
    q, k, v = rnd((1, 2, S, 8), 28), rnd((1, 2, S, 8), 29), rnd((1, 2, S, 8), 30)
    O, L = attention_forward(q, k, v, Spec(causal=True, doc_id=doc, alibi=True))
    start = 0
    for n in lengths:
        sl = slice(start, start + n)
        o, l = attention_forward(q[:, :, sl], k[:, :, sl], v[:, :, sl],
                                 Spec(causal=True, alibi=True))
        assert np.allclose(O[:, :, sl], o, atol=1e-13) and np.allclose(L[:, :, sl], l, atol=1e-13)
        start += n


def test_gqa_equals_repeated_kv():
    q = rnd((2, 8, 16, 8), 31)
    k, v = rnd((2, 2, 16, 8), 32), rnd((2, 2, 16, 8), 33)
    spec = Spec(causal=True, softcap=3.0, prefix_len=np.array([3, 9]))
    a = attention_forward(q, k, v, spec)
    b = attention_forward(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), spec)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_huge_softcap_is_identity():
    q, k, v = rnd((1, 2, 20, 8), 34), rnd((1, 2, 20, 8), 35), rnd((1, 2, 20, 8), 36)
    a = attention_forward(q, k, v, Spec(causal=True, softcap=1e9))
    b = attention_forward(q, k, v, Spec(causal=True))
    assert np.max(np.abs(a[0] - b[0])) < 1e-12 and np.max(np.abs(a[1] - b[1])) < 1e-12


def test_alibi_row_constant_does_not_change_output():
    """softmax is shift-invariant per row, so ALiBi's O equals attention with
    the bias +slope*j alone (written out here with an explicit softmax)."""
    H, S, D = 2, 18, 8
    q, k, v = rnd((1, H, S, D), 37), rnd((1, H, S, D), 38), rnd((1, H, S, D), 39)
    O, _ = attention_forward(q, k, v, Spec(causal=True, alibi=True))
    for h in range(H):
        m = 2.0 ** (-8.0 * (h + 1) / H)
        s = q[0, h] @ k[0, h].T / math.sqrt(D) + m * np.arange(S)[None, :]
        s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        assert np.allclose(O[0, h], p @ v[0, h], atol=1e-13)


def test_prefix_extremes():
    q, k, v = rnd((1, 2, 30, 8), 40), rnd((1, 2, 30, 8), 41), rnd((1, 2, 30, 8), 42)
    zero = attention_forward(q, k, v, Spec(causal=True, prefix_len=np.array([0])))
    causal = attention_forward(q, k, v, Spec(causal=True))
    assert np.array_equal(zero[0], causal[0])
    full = attention_forward(q, k, v, Spec(causal=True, prefix_len=np.array([30])))
    bidir = attention_forward(q, k, v, Spec())
    assert np.array_equal(full[0], bidir[0])


def test_online_softmax_equals_three_pass():
    """The 2-pass online softmax / 1-pass FlashAttention recurrence (running
    max m, running sum l, rescaled accumulator), with tiles of 16 keys, gives
    the 3-pass result (Online-Softmax/FlashAttention page, abstract)."""
    B, H, S, D, T = 1, 2, 70, 8, 16
    q, k, v = rnd((B, H, S, D), 43), rnd((B, H, S, D), 44), rnd((B, H, S, D), 45)
    doc = np.array([doc_ids_from_lengths([30, 40], S)])
    spec = Spec(causal=True, doc_id=doc, softcap=2.0, alibi=True)
    O_ref, L_ref = attention_forward(q, k, v, spec)
    for h in range(H):
        slope = 2.0 ** (-8.0 * (h + 1) / H)
        for i in range(S):
            m, l, acc = -np.inf, 0.0, np.zeros(D)
            for j0 in range(0, S, T):
                js = np.arange(j0, min(j0 + T, S))
                s = k[0, h, js] @ q[0, h, i] / math.sqrt(D) - slope * (i - js)
                s = 2.0 * np.tanh(s / 2.0)
                ok = (js <= i) & (doc[0][js] == doc[0][i])
                if not ok.any():
                    continue
                s = np.where(ok, s, -np.inf)
                m_new = max(m, s.max())
                corr = math.exp(m - m_new) if np.isfinite(m) else 0.0
                p = np.exp(s - m_new)
                l = l * corr + p.sum()
                acc = acc * corr + p @ v[0, h, js]
                m = m_new
            assert np.allclose(acc / l, O_ref[0, h, i], atol=1e-12)
            assert abs(m + math.log(l) - L_ref[0, h, i]) < 1e-12


# ---------------------------------------------------------------------------
# Backward: finite differences and closed forms.
# ---------------------------------------------------------------------------

GRAD_SPECS = [
    Spec(causal=True),
    Spec(causal=True, alibi=True),
    Spec(causal=True, softcap=1.5),
    Spec(causal=True, window=3, alibi=True, softcap=2.0),
    Spec(causal=True, prefix_len=np.array([4])),
    Spec(),
]


@pytest.mark.parametrize("spec", GRAD_SPECS)
def test_backward_matches_finite_differences(spec):
    B, Hq, Hkv, S, D = 1, 4, 2, 7, 3
    q, k, v = rnd((B, Hq, S, D), 46), rnd((B, Hkv, S, D), 47), rnd((B, Hkv, S, D), 48)
    do = rnd((B, Hq, S, D), 49)
    dQ, dK, dV, _, _ = attention_backward(q, k, v, do, spec)

    def loss(q_, k_, v_):
        return float(np.sum(attention_forward(q_, k_, v_, spec)[0] * do))

    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy()
            xm = x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            pos = "qkv".index(name)
            args_p[pos] = xp
            args_m[pos] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(num - g)) < 1e-6 * max(1.0, np.max(np.abs(g))), name


# Shards of a longer sequence (context parallelism): the queries and keys sit
# at absolute positions q_offset + i and kv_offset + j, Sq != Skv, and every
# position-dependent term (causal, window, prefix, document ids, ALiBi) uses
# the absolute positions.
OFFSET_GRAD_SPECS = [
    Spec(causal=True, q_offset=9, kv_offset=6),
    Spec(causal=True, window=4, alibi=True, softcap=2.0, q_offset=9, kv_offset=6),
    Spec(causal=True, prefix_len=np.array([8]), q_offset=9, kv_offset=6),
    Spec(causal=True, doc_id=np.array([[0] * 11 + [1] * 5]), q_offset=9, kv_offset=6),
    Spec(alibi=True, q_offset=2, kv_offset=11),
]


@pytest.mark.parametrize("spec", OFFSET_GRAD_SPECS)
def test_backward_with_offsets_matches_finite_differences(spec):
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 5, 7, 3
    q, k, v = rnd((B, Hq, Sq, D), 146), rnd((B, Hkv, Skv, D), 147), rnd((B, Hkv, Skv, D), 148)
    do = rnd((B, Hq, Sq, D), 149)
    dQ, dK, dV, _, _ = attention_backward(q, k, v, do, spec)

    def loss(q_, k_, v_):
        O = attention_forward(q_, k_, v_, spec)[0]
        return float(np.sum(np.where(np.isfinite(O), O, 0.0) * do))

    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p, args_m = [q, k, v], [q, k, v]
            pos = "qkv".index(name)
            args_p[pos], args_m[pos] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(num - g)) < 1e-6 * max(1.0, np.max(np.abs(g))), name


def test_backward_identical_keys_give_zero_dq():
    """With the identity score_mod every row of dS sums to zero, so if all keys
    are the same vector, dQ_i = scale * (sum_j dS_ij) k = 0."""
    S, D = 12, 8
    k = np.tile(rnd((1, 1, 1, D), 50), (1, 1, S, 1))
    dQ, _, _, _, _ = attention_backward(rnd((1, 1, S, D), 51), k, rnd((1, 1, S, D), 52),
                                        rnd((1, 1, S, D), 53), Spec(causal=True))
    assert np.max(np.abs(dQ)) < 1e-13


def test_backward_uniform_weights_dv():
    """Q = 0 and causal: P_ij = 1/(i+1) for j <= i, so dV_j = sum_{i>=j} dO_i/(i+1)."""
    S, D = 10, 4
    do = rnd((1, 1, S, D), 54)
    _, _, dV, _, _ = attention_backward(np.zeros((1, 1, S, D)), rnd((1, 1, S, D), 55),
                                        rnd((1, 1, S, D), 56), do, Spec(causal=True))
    for j in range(S):
        expect = sum(do[0, 0, i] / (i + 1) for i in range(j, S))
        assert np.allclose(dV[0, 0, j], expect, atol=1e-13)


# ---------------------------------------------------------------------------
# Block mask (exploiting sparsity: the FlexAttention page's sparsity item).
# ---------------------------------------------------------------------------

def test_block_mask_causal_closed_form():
    bm = block_mask(Spec(causal=True), 1, 1024, 1024)
    for qt in range(8):
        assert bm.full_idx[0][qt] == list(range(qt)) and bm.part_idx[0][qt] == [qt]
        assert bm.t_full_idx[0][qt] == list(range(qt + 1, 8)) and bm.t_part_idx[0][qt] == [qt]


def test_block_mask_window_closed_form():
    """Causal + window W (a multiple of the tile): tile (qt, kt) is full for
    qt - W/128 < kt < qt, partial at kt = qt and kt = qt - W/128, else empty."""
    W = 512
    bm = block_mask(Spec(causal=True, window=W), 1, 2048, 2048)
    r = W // 128
    for qt in range(16):
        assert bm.full_idx[0][qt] == list(range(max(0, qt - r + 1), qt))
        assert bm.part_idx[0][qt] == ([qt - r] if qt - r >= 0 else []) + [qt]


def test_block_mask_prefix_closed_form():
    """Prefix 300 OR causal: key tiles 0 and 1 are visible to every query; key
    tile 2 is visible to all queries only up to key 299, so query tiles 0..2
    see it partially; from query tile 3 on, causality covers it fully."""
    P = 300
    bm = block_mask(Spec(causal=True, prefix_len=np.array([P])), 1, 1024, 1024)
    for qt in range(8):
        if qt <= 2:
            assert bm.full_idx[0][qt] == [0, 1] and bm.part_idx[0][qt] == [2]
        else:
            assert bm.full_idx[0][qt] == list(range(qt)) and bm.part_idx[0][qt] == [qt]


def test_block_mask_ragged_and_documents():
    """Tiles past the end cover only the valid rows/columns; a document tile
    is empty exactly when the two position ranges share no document."""
    lengths = [200, 60, 500]
    S = sum(lengths)  # 760: the last tile is ragged (760 - 640 = 120 rows)
    doc = np.array([doc_ids_from_lengths(lengths, S)])
    bm = block_mask(Spec(doc_id=doc), 1, S, S)
    assert bm.state.shape == (1, 6, 6)
    for qt in range(6):
        for kt in range(6):
            dq = set(doc[0][qt * 128:(qt + 1) * 128])
            dk = set(doc[0][kt * 128:(kt + 1) * 128])
            if not (dq & dk):
                assert bm.state[0, qt, kt] == 0
            elif len(dq) == 1 and dq == dk:
                assert bm.state[0, qt, kt] == 2
            else:
                assert bm.state[0, qt, kt] == 1


def test_workload_recipe_shapes():
    w = make_workload(3, with_tensors=False)
    assert sum(w.doc_lengths[0]) == 16384 and w.doc_id.shape == (1, 16384)
    assert all(256 <= n <= 4096 for n in w.doc_lengths[0][:-1])
    w4 = make_workload(4, with_tensors=False)
    assert w4.prefix_len.shape == (2,) and all(512 <= p <= 4096 for p in w4.prefix_len)


# ---------------------------------------------------------------------------
# Relative-position bias (FlexAttention page, relative position encoding):
# special cases and invariants of the distance-indexed table.
# ---------------------------------------------------------------------------

def test_rel_bias_table_of_alibi_equals_alibi():
    """ALiBi is the table T[h][d] = -slope_h * d over the distance d = i - j."""
    B, Hq, Sq, Skv, D = 1, 4, 23, 31, 8
    q, k, v = rnd((B, Hq, Sq, D), 21), rnd((B, Hq, Skv, D), 22), rnd((B, Hq, Skv, D), 23)
    d = np.arange(-(Skv - 1), Sq)
    table = -alibi_slopes(Hq)[:, None] * d[None, :]
    for causal in (False, True):
        O1, L1 = attention_forward(q, k, v, Spec(causal=causal, alibi=True))
        O2, L2 = attention_forward(q, k, v, Spec(causal=causal, rel_bias=table,
                                                 rel_bias_zero=Skv - 1))
        assert np.max(np.abs(O1 - O2)) < 1e-12
        assert np.max(np.abs(L1 - L2)) < 1e-12


def test_rel_bias_constant_table_shifts_lse_only():
    """A constant bias c leaves O unchanged and adds c to the LSE (softmax is
    shift-invariant)."""
    q, k, v = rnd((2, 2, 17, 8), 24), rnd((2, 2, 17, 8), 25), rnd((2, 2, 17, 8), 26)
    c = 1.75
    O1, L1 = attention_forward(q, k, v, Spec(causal=True))
    O2, L2 = attention_forward(q, k, v, Spec(causal=True, rel_bias=np.full((2, 33), c),
                                             rel_bias_zero=16))
    assert np.max(np.abs(O1 - O2)) < 1e-12
    assert np.max(np.abs(L2 - L1 - c)) < 1e-12


def test_rel_bias_gradient_matches_finite_differences():
    """The table is a constant of the call: dQ, dK, dV follow from the biased
    scores (central differences of the forward)."""
    B, H, S, D = 1, 2, 6, 3
    q, k, v, do = (rnd((B, H, S, D), 30 + t) for t in range(4))
    spec = Spec(causal=True, softcap=2.0, rel_bias=rnd((H, 2 * S - 1), 34), rel_bias_zero=S - 1)
    dq, dk, dv, _, _ = attention_backward(q, k, v, do, spec)

    def loss(q_, k_, v_):
        O, _ = attention_forward(q_, k_, v_, spec)
        return float(np.sum(O * do))

    h = 1e-6
    for X, G, idx in ((q, dq, (0, 1, 4, 2)), (k, dk, (0, 0, 2, 1)), (v, dv, (0, 1, 3, 0))):
        Xp, Xm = X.copy(), X.copy()
        Xp[idx] += h
        Xm[idx] -= h
        args_p = [Xp if Y is X else Y for Y in (q, k, v)]
        args_m = [Xm if Y is X else Y for Y in (q, k, v)]
        fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert abs(fd - G[idx]) < 1e-6 * max(1.0, abs(fd))


# ---------------------------------------------------------------------------
# Shards of a longer sequence (absolute positions) and the merge of partial
# results: together they must reproduce attention over the whole sequence.
# ---------------------------------------------------------------------------

def _shard_spec(spec: Spec, q_off: int, kv_off: int) -> Spec:
    import dataclasses
    return dataclasses.replace(spec, q_offset=q_off, kv_offset=kv_off)


SHARD_SPECS = {
    "doc_window_causal_alibi_softcap": lambda doc, pre: Spec(
        causal=True, window=23, doc_id=doc, alibi=True, softcap=3.0),
    "prefix_causal": lambda doc, pre: Spec(causal=True, prefix_len=pre),
    "full_alibi": lambda doc, pre: Spec(alibi=True),
}


@pytest.mark.parametrize("name", sorted(SHARD_SPECS))
def test_sharded_attention_merges_to_full_attention(name):
    """Queries and keys cut into shards at uneven points: each (query shard,
    key shard) pair computed with its absolute offsets, the key shards merged
    by the log-sum-exp rule, equals attention over the whole sequence (the
    merge is exact in real arithmetic: the online-softmax merge of partial
    maxima and sums). A missing or mis-signed offset moves the mask or the
    ALiBi bias; a wrong merge weight changes O or LSE."""
    B, Hq, Hkv, S, D = 2, 4, 2, 90, 8
    q, k, v = rnd((B, Hq, S, D), 71), rnd((B, Hkv, S, D), 72), rnd((B, Hkv, S, D), 73)
    doc = np.stack([doc_ids_from_lengths([17, 40, 33], S), doc_ids_from_lengths([60, 30], S)])
    pre = np.array([12, 47])
    spec = SHARD_SPECS[name](doc, pre)
    O_ref, L_ref = attention_forward(q, k, v, spec)
    q_cuts, kv_cuts = [0, 41, 90], [0, 25, 61, 90]
    for qa, qb in zip(q_cuts[:-1], q_cuts[1:]):
        parts = []
        for ka, kb in zip(kv_cuts[:-1], kv_cuts[1:]):
            parts.append(attention_forward(q[:, :, qa:qb], k[:, :, ka:kb], v[:, :, ka:kb],
                                           _shard_spec(spec, qa, ka)))
        O, L = combine_partials(parts)
        assert np.allclose(O, O_ref[:, :, qa:qb], atol=1e-12, rtol=0)
        fin = np.isfinite(L_ref[:, :, qa:qb])
        assert np.array_equal(np.isfinite(L), fin)
        assert np.allclose(L[fin], L_ref[:, :, qa:qb][fin], atol=1e-12, rtol=0)


def test_merge_special_cases():
    """Merging: one part is the identity; a part with no kept key (O = 0,
    LSE = -inf) contributes nothing; only empty parts give O = 0, LSE = -inf;
    two parts with equal LSE average their outputs, and the merged LSE is
    ln 2 larger."""
    rng = np.random.default_rng(5)
    O1, L1 = rng.standard_normal((3, 4)), rng.standard_normal(3)
    O0, L0 = np.zeros((3, 4)), np.full(3, -np.inf)
    O, L = combine_partials([(O1, L1)])
    assert np.array_equal(O, O1) and np.array_equal(L, L1)
    O, L = combine_partials([(O0, L0), (O1, L1), (O0, L0)])
    assert np.allclose(O, O1, atol=1e-15) and np.allclose(L, L1, atol=1e-15)
    O, L = combine_partials([(O0, L0), (O0, L0)])
    assert np.array_equal(O, O0) and np.all(L == -np.inf)
    O2 = rng.standard_normal((3, 4))
    O, L = combine_partials([(O1, L1), (O2, L1)])
    assert np.allclose(O, (O1 + O2) / 2, atol=1e-15)
    assert np.allclose(L, L1 + math.log(2.0), atol=1e-15)


def test_block_mask_of_a_shard_is_a_window_of_the_full_block_mask():
    """With offsets that are multiples of the tile size, the tiles of a
    (query shard, key shard) pair are the full problem's tiles at the shifted
    tile indices."""
    S = 640
    doc = np.array([doc_ids_from_lengths([200, 300, 140], S)])
    spec = Spec(causal=True, window=300, doc_id=doc)
    full = block_mask(spec, 1, S, S)
    shard = block_mask(_shard_spec(spec, 256, 128), 1, 384, 256)
    assert np.array_equal(shard.state[0], full.state[0, 2:5, 1:3])
