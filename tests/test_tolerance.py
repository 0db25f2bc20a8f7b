"""The GPU parity bound (tests/gpu_util.py) on the CPU: 1.5e-2 max-abs, except
that an element whose exact value cannot be written in bf16 within 1.5e-2
(magnitude >= 4) is held to half a bf16 ulp of it plus 1e-3."""

import numpy as np
import torch

from gpu_util import TOL_MAX, bf16_half_ulp, max_abs_bound


def test_half_ulp_of_known_binades():
    # bf16 keeps 8 significant bits: in [2^k, 2^(k+1)) its spacing is 2^(k-7)
    cases = {0.3: 2.0 ** -10, 1.0: 2.0 ** -8, 1.99: 2.0 ** -8, 2.5: 2.0 ** -7, 4.0: 2.0 ** -6,
             4.07: 2.0 ** -6, 7.9: 2.0 ** -6, 9.0: 2.0 ** -5, -5.5: 2.0 ** -6}
    for x, half in cases.items():
        assert bf16_half_ulp(np.array([x]))[0] == half, x


def test_bound_is_the_stated_one_below_magnitude_4():
    ref = np.linspace(-3.99, 3.99, 2001)
    assert np.all(max_abs_bound(ref) == TOL_MAX)


def test_bound_covers_exact_bf16_rounding_everywhere():
    rng = np.random.default_rng(0)
    ref = rng.normal(0.0, 3.0, 200000)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert np.all(np.abs(rounded - ref) <= max_abs_bound(ref))


def test_bound_still_catches_a_real_error():
    ref = np.array([0.5, 1.0, 5.0])
    assert 0.02 > max_abs_bound(ref)[0]  # 0.02 at 0.5
    assert 0.02 > max_abs_bound(ref)[2]  # 0.02 at 5: more than half an ulp (0.0156) + 1e-3
