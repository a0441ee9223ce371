"""The kernels divide row sums by the row length with a reciprocal computed once and one
Markstein correction step (RowDivisor in csrc/ln_device.cuh): q0 = a * inv, r = fma(-q0, n, a),
q = fma(r, inv, q0), with inv = 1/n rounded.  Those are IEEE fp32 operations rounded to
nearest, the same on the host as on the GPU, so the claim that q is the correctly rounded
a / n, bit for bit what a division gives, is checked here in C on the host CPU over every
row length up to 2048, a spread of longer ones, and random magnitudes and signs."""
import os
import shutil
import subprocess

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static uint64_t s = 88172645463325252ull;
static uint64_t xr(void) { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return s; }
static float rnd(void) {  /* random sign, exponent 2^-60 .. 2^60, random mantissa */
    uint32_t m = (uint32_t)(xr() & 0x7fffff);
    uint32_t e = (uint32_t)(xr() % 121) + 67;
    uint32_t b = ((uint32_t)(xr() & 1) << 31) | (e << 23) | m;
    float f;
    memcpy(&f, &b, 4);
    return f;
}
int main(void) {
    long bad = 0, n = 0;
    for (int cols = 1; cols <= 16384; cols += (cols < 2048 ? 1 : 7)) {
        const float c = (float)cols, inv = 1.0f / c;
        for (int i = 0; i < 200; ++i, ++n) {
            const float a = i == 0 ? 0.0f : (i == 1 ? c * 3.0f : rnd());
            const float q = a * inv;
            const float r = fmaf(-q, c, a);
            const float q1 = fmaf(r, inv, q);
            const float ref = a / c;
            if (memcmp(&q1, &ref, 4) != 0) ++bad;
        }
    }
    printf("%ld %ld\n", bad, n);
    return 0;
}
"""


def test_corrected_quotient_equals_division(tmp_path):
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "div.c"
    exe = tmp_path / "div"
    src.write_text(SRC)
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", str(exe), str(src), "-lm"], check=True)
    bad, n = map(int, subprocess.run([str(exe)], check=True, capture_output=True,
                                     text=True).stdout.split())
    assert n > 800000
    assert bad == 0
