"""Fit of the odd polynomial the kernel evaluates for tanh(u), 0 <= u <= 1.

tanh(u) = u + u z Q(z), z = u^2, with Q of degree 5 in z.  Q approximates
g(z) = (tanh(u) / u - 1) / z; the fit minimizes the relative error of tanh,
whose sensitivity to an error in Q is u z / tanh(u):
  * points: 20000 values of u spaced evenly on [2^-12, 1];
  * weighted least squares (float64) with weights u z / tanh(u), reweighted
    60 times toward the minimax solution (Lawson's iteration: each weight is
    multiplied by the point's current absolute weighted error, then all are
    normalized to sum 1);
  * the six coefficients are rounded to nearest binary32.
The kernel evaluates Q by Horner's rule with fused multiply-adds, then
t = fma(u z, Q, u).  Printed here: the constants (kTanhQ0 .. kTanhQ5) and the
largest error in binary32 ulps over a sample; the exhaustive bound (1.7 ulp on
every float in [1/4, 1] and every 64th below) is checked by the test suite.

    python -m nvfp4_quantization_grouped_gb300.fit_tanh
"""
import numpy as np


def fit(n_iter: int = 60, npts: int = 20000, lo: float = 2.0 ** -12) -> np.ndarray:
    u = np.linspace(lo, 1.0, npts)
    z = u * u
    g = (np.tanh(u) / u - 1.0) / z
    a = np.vander(z, 6, increasing=True)
    wrel = u * z / np.tanh(u)
    lw = np.ones_like(u)
    c = None
    for _ in range(n_iter):
        w = wrel * lw
        c, *_ = np.linalg.lstsq(a * w[:, None], g * w, rcond=None)
        lw = lw * np.abs((a @ c - g) * wrel)
        lw /= lw.sum()
    return np.asarray(c, dtype=np.float32)


def max_ulp_error(c32: np.ndarray, u: np.ndarray) -> float:
    """Largest |t - tanh(u)| in binary32 ulps of tanh(u), t evaluated as the
    kernel does (each fused multiply-add rounded once to binary32)."""
    u = u.astype(np.float32)
    z = (u * u).astype(np.float32)

    def fma(x, y, w):
        return (x.astype(np.float64) * y.astype(np.float64) + np.asarray(w, np.float64)).astype(np.float32)

    q = fma(np.full_like(z, c32[5]), z, c32[4])
    for k in (3, 2, 1, 0):
        q = fma(q, z, c32[k])
    t = fma((u * z).astype(np.float32), q, u)
    ref = np.tanh(u.astype(np.float64))
    rf = np.abs(ref).astype(np.float32)
    ulp = np.nextafter(rf, np.float32(np.inf)).astype(np.float64) - rf.astype(np.float64)
    return float(np.max(np.abs(t.astype(np.float64) - ref) / ulp))


if __name__ == "__main__":
    c32 = fit()
    for k, v in enumerate(c32):
        print(f"kTanhQ{k} = {float(v).hex().replace('0000000p', 'p')}f")
    us = np.concatenate([np.arange(0x3E800000, 0x3F800001, 7, dtype=np.uint32).view(np.float32),
                         np.arange(1, 0x3E800000, 4096, dtype=np.uint32).view(np.float32)])
    print(f"max error over the sample: {max_ulp_error(c32, us):.3f} ulp")
