"""The residual passes of the stochastic verifier divide by the normaliser Z
with Markstein's sequence instead of an IEEE division instruction:
y = RN(1/Z), q = RN(d*y), r = fma(-q, Z, d), result fma(r, y, q).  Markstein's
theorem makes the result the correctly rounded d/Z when no quantity
underflows or overflows; the kernel takes this path only for d in [2^-100, 1]
and Z in [2^-46, 2^17].  This test checks the sequence against IEEE fp32
division on the CPU over that domain (random, power-of-two edges, and Z of
the form fp32(S) * 2^-46), so the verifier's bit-exact contract does not rest
on the theorem alone."""
import os
import subprocess
import tempfile

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static uint64_t st = 0x9E3779B97F4A7C15ull;
static uint64_t next(void) { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return st; }
static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t b_of(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* log-uniform fp32 in [2^lo, 2^hi) with a uniform 23-bit significand */
static float logu(int lo, int hi) {
    int e = lo + (int)(next() % (uint64_t)(hi - lo));
    return ldexpf(f_of(0x3f800000u | (uint32_t)(next() & 0x7fffffu)), e);
}

static int check(float d, float Z) {
    if (!(d >= 0x1p-100f && d <= 1.0f)) return 0;
    volatile float y = 1.0f / Z;           /* RN(1/Z) */
    volatile float q = d * y;
    volatile float r = fmaf(-q, Z, d);
    volatile float m = fmaf(r, y, q);
    volatile float ref = d / Z;
    if (b_of(m) != b_of(ref)) {
        printf("mismatch d=%a Z=%a got %a want %a\n", d, Z, m, ref);
        return 1;
    }
    return 0;
}

int main(void) {
    long bad = 0, n = 0;
    for (long i = 0; i < 4000000; i++, n++) bad += check(logu(-100, 0), logu(-46, 17));
    for (long i = 0; i < 2000000; i++, n++) {   /* Z = fp32(S) * 2^-46, S up to 2^63 */
        uint64_t S = next() >> (next() % 64);
        if (S == 0) S = 1;
        bad += check(logu(-40, 0), (float)S * 0x1p-46f);
    }
    for (int e = -46; e < 17; e++)              /* Z at and next to powers of two */
        for (int k = -64; k <= 64; k++) {
            float Z = f_of(b_of(ldexpf(1.0f, e)) + (uint32_t)k);
            for (int j = 0; j < 2000; j++, n++) bad += check(logu(-100, 0), Z);
        }
    for (int k = 0; k < 4096; k++)              /* d next to 1 and to powers of two */
        for (int j = 0; j < 200; j++, n++) {
            float d = f_of(0x3f800000u - (uint32_t)k);
            bad += check(d, logu(-46, 17));
            bad += check(ldexpf(f_of(0x3f800000u + (uint32_t)k), -(int)(next() % 100)), logu(-46, 17));
        }
    printf("checked %ld bad %ld\n", n, bad);
    return bad != 0;
}
"""


def test_markstein_division_equals_ieee_division_on_the_kernel_domain():
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        exe = os.path.join(d, "m")
        open(c, "w").write(SRC)
        try:
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", c, "-o", exe,
                                   "-lm"])
        except (OSError, subprocess.CalledProcessError):
            pytest.skip("no C compiler")
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stdout[-2000:]
        assert "bad 0" in r.stdout
