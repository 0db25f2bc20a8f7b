"""The polynomial exp2 of the prefill softmax, checked against exp2 in double
precision through an fp32 emulation of the device steps."""

import numpy as np

from paged_kv_cache_forward_gb300 import exp2_fit as E


def test_refit_reproduces_the_compiled_coefficients():
    c = E.fit()
    assert np.allclose(c, E.COEFFS, rtol=1e-5, atol=1e-7)


def test_relative_error_bound_on_the_used_range():
    xs = np.concatenate([np.linspace(-125, 8, 500001), np.arange(-125, 9)]).astype(np.float32)
    got = E.emulate(xs).astype(np.float64)
    ref = 2.0 ** xs.astype(np.float64)
    rel = np.abs(got - ref) / ref
    assert rel.max() < 8e-5           # far below bf16's relative spacing 2^-8
    # what the kernel keeps is bf16: the rounded value is within one bf16 step
    assert rel.max() < 2.0 ** -9


def test_special_values():
    assert E.emulate(np.float32(-np.inf)) == 0.0
    assert E.emulate(np.float32(-200.0)) == 0.0
    assert abs(float(E.emulate(np.float32(0.0))) - 1.0) < 1e-4
    assert abs(float(E.emulate(np.float32(8.0))) - 256.0) < 256.0 * 1e-4
