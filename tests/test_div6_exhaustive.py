"""The NVFP4 quantizers divide a block's amax by 6 with a product and one FMA correction step
(``div6_rn`` in ``csrc/quant.cu``: q0 = fl(x * fl(1/6)), q = fma(fma(-q0, 6, x), fl(1/6), q0))
instead of the full IEEE division, for every x >= 2^-125.  This test runs that sequence on the
host over every non-negative finite float (C with ``fmaf``, which C requires to round once) and
checks it against the host's IEEE quotient: equal for all x >= 2^-125, and the inputs below,
which the kernel sends to the full division, are the only ones where it can differ."""
import os
import shutil
import subprocess
import tempfile

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float asf(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t asu(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
int main(void) {
  const float c = 0x1.555556p-3f;
  const uint32_t lo = 0x01000000u;                  /* 2^-125 */
  unsigned long long bad_hi = 0, bad_lo = 0;
  if (asu(1.0f / 6.0f) != asu(c)) { printf("constant\n"); return 2; }
#pragma omp parallel for reduction(+ : bad_hi, bad_lo) schedule(static)
  for (long long i = 0; i <= 0x7F7FFFFFLL; ++i) {
    const float x = asf((uint32_t)i);
    volatile float ref = x / 6.0f;
    const float q0 = x * c;
    const float q = fmaf(fmaf(-q0, 6.0f, x), c, q0);
    if (asu(q) != asu(ref)) { if ((uint32_t)i >= lo) ++bad_hi; else ++bad_lo; }
  }
  printf("%llu %llu\n", bad_hi, bad_lo);
  return 0;
}
"""


def test_div6_equals_ieee_division_above_2_pow_minus_125():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "div6.c"), os.path.join(d, "div6")
        open(src, "w").write(SRC)
        flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
        r = subprocess.run([gcc, *flags, "-fopenmp", src, "-o", exe, "-lm"], capture_output=True, text=True)
        if r.returncode != 0:   # no OpenMP runtime: one thread (about half a minute)
            r = subprocess.run([gcc, *flags, src, "-o", exe, "-lm"], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert out.returncode == 0, out.stdout + out.stderr
        bad_hi, bad_lo = (int(v) for v in out.stdout.split())
        assert bad_hi == 0
        assert bad_lo > 0   # the full division below 2^-125 is needed, not just cautious
