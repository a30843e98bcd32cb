"""Exhaustive host-side proofs of arithmetic shortcuts the CUDA kernel takes
in place of an IEEE operation, so that its results stay bit-identical to the
plain definition.  Each check enumerates every binary32 input of the range
where the kernel uses the shortcut."""
import os
import platform
import subprocess
import tempfile

import pytest

# NVFP4 block scale needs amax_b / 6 rounded to nearest even.  The kernel
# computes q = a * RN(1/6), then one correction q + r * RN(1/6) with the
# exact remainder r = a - 6 q (both steps fused multiply-adds), for every
# a >= 2^-118, and divides below that.
DIV6_SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
int main(void) {
    const float y = 0.16666667163372040f;
    unsigned long long bad = 0;
    for (uint32_t u = 0x04800000u; u < 0x7f800000u; ++u) {   /* 2^-118 .. FLT_MAX, every positive float */
        float a; memcpy(&a, &u, 4);
        volatile float six = 6.0f;
        float ref = a / six;
        float q = a * y;
        float r = fmaf(-q, 6.0f, a);
        float q1 = fmaf(r, y, q);
        if (memcmp(&q1, &ref, 4) != 0) ++bad;
    }
    printf("%llu\n", bad);
    return 0;
}
"""


def test_division_by_six_shortcut_is_correctly_rounded():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "div6.c")
        exe = os.path.join(d, "div6")
        with open(src, "w") as f:
            f.write(DIV6_SRC)
        flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
        if platform.machine() in ("x86_64", "AMD64"):
            flags.append("-mfma")
        subprocess.run(["gcc", *flags, "-o", exe, src, "-lm"], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
        assert out.strip() == "0"


# TanhSReLU evaluates tanh(u), 0 <= u <= 1, with a degree-5 polynomial in u^2
# (the kernel's kTanhQ0..5, FP32 fused multiply-adds) and the library tanhf
# above 1.  The activation's tolerance (2 BF16 ulp, rare code flips) needs an
# FP32 result about as close to tanh as tanhf's own (documented at 2 ulp):
# every float in [1/4, 1] and every 64th below are held to 1.7 ulp of tanh
# evaluated in double.
TANH_SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static double err_ulp(uint32_t b, float c0, float c1, float c2, float c3, float c4, float c5) {
    float u; memcpy(&u, &b, 4);
    float z = u * u;
    float q = fmaf(c5, z, c4); q = fmaf(q, z, c3); q = fmaf(q, z, c2); q = fmaf(q, z, c1); q = fmaf(q, z, c0);
    float uz = u * z;
    float t = fmaf(uz, q, u);
    double ref = tanh((double)u);
    float rf = fabsf((float)ref);
    double ulp = (double)nextafterf(rf, INFINITY) - (double)rf;
    return fabs((double)t - ref) / ulp;
}
int main(void) {
    const float c0 = %s, c1 = %s, c2 = %s, c3 = %s, c4 = %s, c5 = %s;
    double worst = 0;
    for (uint32_t b = 0x3e800000u; b <= 0x3f800000u; ++b) {
        double e = err_ulp(b, c0, c1, c2, c3, c4, c5);
        if (e > worst) worst = e;
    }
    for (uint32_t b = 1; b < 0x3e800000u; b += 64) {
        double e = err_ulp(b, c0, c1, c2, c3, c4, c5);
        if (e > worst) worst = e;
    }
    printf("%%.4f\n", worst);
    return 0;
}
"""


def _kernel_tanh_coefficients():
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "nvfp4_quantization_grouped_gb300", "csrc", "gsa_kernel.cuh")
    src = open(path).read()
    vals = {}
    for k in range(6):
        m = re.search(r"kTanhQ%d = (-?0x[0-9a-fA-F.]+p-?[0-9]+f)" % k, src)
        assert m, f"kTanhQ{k} not found"
        vals[k] = m.group(1)
    return [vals[k] for k in range(6)]


def test_tanh_polynomial_within_1p7_ulp():
    coeffs = _kernel_tanh_coefficients()
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "tanhq.c")
        exe = os.path.join(d, "tanhq")
        with open(src, "w") as f:
            f.write(TANH_SRC % tuple(coeffs))
        flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
        if platform.machine() in ("x86_64", "AMD64"):
            flags.append("-mfma")
        subprocess.run(["gcc", *flags, "-o", exe, src, "-lm"], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
        assert float(out.strip()) <= 1.7, out


def test_tanh_coefficients_are_the_committed_fit():
    # the kernel's constants are exactly what the fit script prints
    import numpy as np
    from nvfp4_quantization_grouped_gb300 import fit_tanh
    fitted = fit_tanh.fit()
    kernel = np.array([float.fromhex(c.rstrip("f")) for c in _kernel_tanh_coefficients()], np.float32)
    assert np.array_equal(fitted, kernel), (fitted, kernel)


# With the expert's tensor scale S <= 2^100 the kernel takes the corrected
# product for every block amax, including those below 2^-118 where it is not
# the IEEE quotient: the product with S then stays below 2^-10, half the
# smallest E4M3 subnormal, so the block scale code is 0 either way.
DIV6_TINY_SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
int main(void) {
    const float y = 0.16666667163372040f;
    const float S = 0x1p100f;
    unsigned long long bad = 0;
    for (uint32_t u = 0; u < 0x04800000u; ++u) {   /* every float in [0, 2^-118) */
        float a; memcpy(&a, &u, 4);
        float q0 = a * y;
        float q = fmaf(fmaf(-q0, 6.0f, a), y, q0);
        volatile float six = 6.0f;
        float ref = a / six;
        if (!(q * S < 0x1p-10f) || !(ref * S < 0x1p-10f)) ++bad;
    }
    printf("%llu\n", bad);
    return 0;
}
"""


def test_division_by_six_below_range_gives_zero_scale_code():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "div6t.c")
        exe = os.path.join(d, "div6t")
        with open(src, "w") as f:
            f.write(DIV6_TINY_SRC)
        flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
        if platform.machine() in ("x86_64", "AMD64"):
            flags.append("-mfma")
        subprocess.run(["gcc", *flags, "-o", exe, src, "-lm"], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
        assert out.strip() == "0"
