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
