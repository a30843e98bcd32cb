"""The kernels' fast exponential and sigmoid (exp_neg, sigmoid_fast in
gsa_kernel.cuh) at every BF16 input, against the exact functions (float64).

exp_neg(t) computes e^-t as 2^(-t log2 e) with the hardware's approximate
base-2 exponential (no flush to zero); its relative error is the exponential's
own plus the rounding of the product, bounded here by (4 + 1.25 t) 2^-24.
sigmoid_fast takes 1 / (1 + E) or E / (1 + E) with E = e^-|x| and the
approximate divide (divisor in [1, 2]): within (12 + 2 |x|) 2^-24, and 0
where 1 / (1 + e^-x) overflows in FP32 (x below -88.72283..., as the FP32
oracle gives).  The SwiGLU gate is a BF16 value, so these inputs are every
argument the SwiGLU kernels give them.  The dprobs tolerance of the SiLU-based
activations (gpu_util.act_rel_err) is derived from these bounds."""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
U = 2.0 ** -24
EXP_OVERFLOW = float.fromhex("0x1.62e42ep+6")   # largest x with e^x finite in FP32
SUB = 2.0 ** -149                               # the smallest subnormal


def exp_bound(t):
    return (4 + 1.25 * t) * U


def sigmoid_bound(x):
    return (12 + 2 * np.abs(x)) * U


@pytest.fixture(scope="module")
def probe():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tempfile.mkdtemp()
    exe = os.path.join(d, "act_probe")
    subprocess.run([nvcc, "-std=c++17", "-O3", "-fmad=false", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(ROOT, "nvfp4_quantization_grouped_gb300", "csrc"),
                    "-o", exe, os.path.join(ROOT, "tests", "native", "act_probe.cu"), "-lcuda"], check=True)
    out = subprocess.run([exe], capture_output=True, check=True).stdout
    shutil.rmtree(d, ignore_errors=True)
    r = np.frombuffer(out, dtype=np.float32).reshape(6, 65536).astype(np.float64)
    with np.errstate(invalid="ignore"):   # the NaN patterns
        x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    return x, r


def _check(got, exact, bound, what):
    """|got - exact| <= bound * |exact| where the exact value is normal, and
    within that plus one subnormal step where it is not; returns the worst
    ratio of the error to the bound over the normal range."""
    err = np.abs(got - exact)
    normal = np.abs(exact) >= 2.0 ** -126
    ratio = err[normal] / (bound[normal] * np.abs(exact[normal]))
    assert np.all(err[normal] <= bound[normal] * np.abs(exact[normal])), (what, ratio.max())
    assert np.all(err[~normal] <= bound[~normal] * np.abs(exact[~normal]) + SUB), what
    return ratio.max()


def test_exp_neg_every_bf16_input(probe):
    x, r = probe
    ok = np.isfinite(x)
    t = np.abs(x[ok])
    exact = np.exp(-t)
    worst = _check(r[0][ok], exact, exp_bound(t), "exp_neg")
    print(f"exp_neg: worst {worst:.2f} of the bound")
    # no flush to zero: every value the exact function keeps above half the smallest subnormal is nonzero
    assert np.all(r[0][ok][exact >= 2.0 ** -148] > 0)
    # an infinite argument gives 0
    assert np.all(r[0][~np.isnan(x) & ~ok] == 0)


def test_sigmoid_fast_every_bf16_input(probe):
    x, r = probe
    ok = np.isfinite(x)
    xs = x[ok]
    with np.errstate(over="ignore"):
        exact = np.where(xs < -EXP_OVERFLOW, 0.0, 1.0 / (1.0 + np.exp(-xs)))
    worst = _check(r[1][ok], exact, sigmoid_bound(xs), "sigmoid_fast")
    print(f"sigmoid_fast: worst {worst:.2f} of the bound")
    assert np.all(r[1][ok][xs < -EXP_OVERFLOW] == 0)


def test_swiglu_value_and_derivatives_every_bf16_gate(probe):
    """v = a sigmoid(a), da = sigmoid(a) + a sigmoid(a) (1 - sigmoid(a)),
    db = v at b = 1: within the sigmoid's bound plus the roundings of the
    products (da against the size of its two terms, which can cancel)."""
    x, r = probe
    ok = np.isfinite(x)
    a = x[ok]
    with np.errstate(over="ignore"):
        s = np.where(a < -EXP_OVERFLOW, 0.0, 1.0 / (1.0 + np.exp(-a)))
    v = a * s
    t2 = a * s * (1.0 - s)
    wv = _check(r[2][ok], v, sigmoid_bound(a) + U, "swiglu v")
    assert np.array_equal(r[4][ok], r[2][ok])
    scale = np.abs(s) + np.abs(t2)
    err = np.abs(r[3][ok] - (s + t2))
    big = scale >= 2.0 ** -120
    # sg's absolute error (a few units near sg ~ 1) enters a sg (1 - sg) multiplied by |a|
    bd = (sigmoid_bound(a) + 4 * U) * scale + 4 * U * np.abs(a)
    assert np.all(err[big] <= bd[big])
    print(f"swiglu: v worst {wv:.2f}, da worst {(err[big] / bd[big]).max():.2f} of the bound")


def test_sigmoid_val_equals_sigmoid_fast(probe):
    """The SwiGLU values' sigmoid (the approximate divide) gives the
    reciprocal instruction's value at every BF16 argument, NaN patterns
    aside: the forward, its regeneration and the backward agree."""
    x, r = probe
    ok = ~np.isnan(x)
    assert np.array_equal(r[5][ok].astype(np.float32).view(np.uint32), r[1][ok].astype(np.float32).view(np.uint32))
