"""Glue shared by the tests: turns a synthetic workload into the oracle's
description of it. Holds no attention arithmetic."""
import numpy as np

from oracle import Spec


def oracle_spec(w, **extra) -> Spec:
    return Spec(causal=w.causal, window=w.window,
                doc_id=w.doc_id if w.document else None,
                prefix_len=w.prefix_len if w.prefix else None,
                alibi=w.alibi, softcap=w.softcap, **extra)


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nanmax(d)) if d.size else 0.0
