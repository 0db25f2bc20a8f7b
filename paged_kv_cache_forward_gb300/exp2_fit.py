"""Coefficients of the polynomial exp2 used for part of the softmax in the
prefill kernel, and the fp32 emulation the tests check them with.

Method (Cody-Waite range reduction, with the round-to-nearest done by adding
1.5 * 2^23, the exponent-field construction of Schraudolph's "A fast, compact
approximation of the exponential function", 1999):
    n = rint(x)               (x + 1.5*2^23, then subtract it back)
    f = x - n                 in [-0.5, 0.5]
    2^f ~ c0 + c1 f + c2 f^2 + c3 f^3
    2^x = that value with n added to its exponent field
The cubic is fitted here by iteratively reweighted least squares (Lawson's
algorithm) towards the minimax relative error on [-0.5, 0.5].  The kernel uses
it for arguments in [-125, 8] (softmax exponents after the running-max shift,
which the lazy rescale bounds by 8); below -125 it returns 0.  Its result is
rounded to bf16 (relative spacing 2^-8), so a relative error of ~1e-4 is far
inside what the output can show.

    python -m paged_kv_cache_forward_gb300.exp2_fit
"""

import numpy as np

# The values compiled into csrc/pa_device.cuh (poly_exp2).
COEFFS = (0.9999282956123352, 0.693260908126831, 0.24260765314102173, 0.0551702119410038)
MAGIC = np.float32(12582912.0)  # 1.5 * 2^23


def fit(deg: int = 3, iters: int = 80):
    x = np.linspace(-0.5, 0.5, 40001)
    y = 2.0 ** x
    w = 1 / y
    for _ in range(iters):
        A = np.vander(x, deg + 1, increasing=True) * w[:, None]
        c, *_ = np.linalg.lstsq(A, y * w, rcond=None)
        err = (np.polyval(c[::-1], x) - y) / y
        w = w * (np.abs(err) + 1e-12) ** 0.3
        w /= w.max()
    return tuple(float(v) for v in c.astype(np.float32))


def emulate(x: np.ndarray, coeffs=COEFFS) -> np.ndarray:
    """The device computation, step by step in fp32."""
    x = np.asarray(x, dtype=np.float32)
    c = [np.float32(v) for v in coeffs]
    with np.errstate(invalid="ignore", over="ignore"):
        return _emulate(x, c)


def _emulate(x, c):
    t = (x + MAGIC).astype(np.float32)
    n_int = t.view(np.int32) - np.int32(0x4B400000)
    n = (t - MAGIC).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = c[3]
    for k in (2, 1, 0):
        p = (p * f + c[k]).astype(np.float32)
    out = (p.view(np.int32) + (n_int << 23)).view(np.float32)
    return np.where(x < np.float32(-125.0), np.float32(0.0), out)


if __name__ == "__main__":
    print("fitted:", fit())
    xs = np.linspace(-125, 8, 2000001).astype(np.float32)
    rel = np.abs(emulate(xs).astype(np.float64) - 2.0 ** xs.astype(np.float64)) / 2.0 ** xs.astype(np.float64)
    print("compiled coefficients: max relative error on [-125, 8]:", rel.max())
