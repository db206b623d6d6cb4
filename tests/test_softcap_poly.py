"""The soft-cap's polynomial form in the bf16 forward (fwd_tc_kernel.cuh,
tanh_poly_coeffs): cap * log2(e) * tanh(s / cap) is evaluated as s * Q(s^2)
for |s / cap| <= 1 instead of with tanh.approx (FlexAttention page, the
soft-capping score_mod). Pinned here on the CPU against numpy's tanh, with
the coefficients read from the kernel source and the kernel's operation
order (fp32, Horner in u = y^2): the relative error stays within the bound
the source states (8.2e-5) and below tanh.approx's 2^-10.9, the bound the
forward's LSE tolerance already allows for."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "masked_attention_gb300", "csrc",
                   "fwd_tc_kernel.cuh")


def coefficients():
    text = open(SRC).read()
    body = text[text.index("tanh_poly_coeffs("):]
    body = body[:body.index("}")]
    found = dict(re.findall(r"a\[(\d)\] = (-?[0-9.]+)f \* f\1;", body))
    assert sorted(found) == ["0", "1", "2", "3"], found
    return np.array([float(found[str(k)]) for k in range(4)], dtype=np.float32)


def poly_tanh_f32(y):
    """tanh(y) ~ y * (c0 + u (c1 + u (c2 + u c3))), u = y^2, all in fp32."""
    c = coefficients()
    y = np.asarray(y, dtype=np.float32)
    u = (y * y).astype(np.float32)
    q = np.float32(c[3])
    for k in (2, 1, 0):
        q = (q * u + c[k]).astype(np.float32)
    return (q * y).astype(np.float32)


def test_polynomial_error_bound_on_the_range():
    y = np.linspace(-1.0, 1.0, 400001, dtype=np.float32)
    y = y[y != 0]
    ref = np.tanh(y.astype(np.float64))
    rel = np.abs(poly_tanh_f32(y) - ref) / np.abs(ref)
    assert rel.max() <= 8.2e-5, rel.max()
    assert rel.max() < 2.0 ** -10.9


def test_polynomial_is_odd_and_exact_at_zero():
    y = np.linspace(0.0, 1.0, 1001, dtype=np.float32)
    assert np.array_equal(poly_tanh_f32(-y), -poly_tanh_f32(y))
    assert poly_tanh_f32(np.float32(0.0)) == 0.0


def test_folded_coefficients_match_the_plain_form():
    """The kernel folds the scale into the coefficients: with sc = scale / cap
    and cl2 = cap * log2(e), s * sum_k a_k (s^2)^k where a_k = c_k sc^(2k+1)
    cl2 equals cl2 * P(s * sc): checked in fp64 for the bench workload's cap
    and scale and for a small cap."""
    c = coefficients().astype(np.float64)
    for cap, scale in ((50.0, 128 ** -0.5), (1.0, 64 ** -0.5)):
        sc, cl2 = scale / cap, cap * np.log2(np.e)
        a = np.array([c[k] * sc ** (2 * k + 1) * cl2 for k in range(4)])
        s = np.linspace(-cap / scale, cap / scale, 2001)
        folded = s * sum(a[k] * (s * s) ** k for k in range(4))
        y = s * sc
        plain = cl2 * y * sum(c[k] * (y * y) ** k for k in range(4))
        assert np.allclose(folded, plain, rtol=1e-12, atol=1e-12)
