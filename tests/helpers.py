"""Glue shared by the tests: turns a synthetic workload into the oracle's
description of it. Holds no attention arithmetic."""
import numpy as np

from oracle import Spec


def oracle_spec(w, **extra) -> Spec:
    return Spec(causal=w.causal, window=w.window,
                doc_id=w.doc_id if w.document else None,
                prefix_len=w.prefix_len if w.prefix else None,
                alibi=w.alibi, softcap=w.softcap,
                rel_bias=w.rel_bias.double().numpy() if w.rel_bias is not None else None,
                rel_bias_zero=w.Skv - 1, **extra)


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nanmax(d)) if d.size else 0.0


def variant_bits(w) -> int:
    """The library's variant bitmask for a synthetic workload."""
    import masked_attention_gb300 as M
    v = 0
    if w.causal:
        v |= M.MASK_CAUSAL
    if w.window is not None:
        v |= M.MASK_WINDOW
    if w.document:
        v |= M.MASK_DOCUMENT
    if w.prefix:
        v |= M.MASK_PREFIX
    if w.alibi:
        v |= M.SCORE_ALIBI
    if w.softcap is not None:
        v |= M.SCORE_SOFTCAP
    if w.relbias:
        v |= M.SCORE_RELBIAS
    return v


class DeviceRun:
    """Uploads a workload and runs the library's forward on it."""

    def __init__(self, w, use_block_mask=True, transposed=False):
        import torch
        import masked_attention_gb300 as M
        self.w = w
        self.M = M
        dev = "cuda"
        self.q, self.k, self.v = (t.to(dev).contiguous() for t in (w.q, w.k, w.v))
        self.do = w.do.to(dev).contiguous() if w.do is not None else None
        self.doc_id = torch.from_numpy(w.doc_id).to(dev) if w.document else None
        self.prefix_len = torch.from_numpy(w.prefix_len).to(dev) if w.prefix else None
        self.variant = variant_bits(w)
        self.window = w.window or 0
        self.softcap = w.softcap or 0.0
        self.rel_bias = w.rel_bias.to(dev).contiguous() if w.rel_bias is not None else None
        self.bm = None
        if use_block_mask:
            self.bm = M.build_block_mask(self.variant & 0xF, w.B, w.Sq, w.Skv,
                                         window=self.window, doc_id=self.doc_id,
                                         prefix_len=self.prefix_len, transposed=transposed)

    def kwargs(self):
        kw = dict(window=self.window, softcap=self.softcap, doc_id=self.doc_id,
                  prefix_len=self.prefix_len, block_mask=self.bm)
        if self.rel_bias is not None:
            kw["rel_bias"] = self.rel_bias
        return kw

    def fwd(self, o=None, lse=None):
        import torch
        w = self.w
        if o is None:
            o = torch.empty_like(self.q)
        if lse is None:
            lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device="cuda")
        self.M.attn_fwd(self.q, self.k, self.v, o, lse, self.variant, **self.kwargs())
        return o, lse
