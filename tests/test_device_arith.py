"""Arithmetic identities the CUDA kernels rely on, checked exactly on the CPU.

The NVFP4 row quantiser obtains the IEEE single-precision quotient fp32(b / 6)
of a block max b (a bf16 value) without a division: q1 = fp32(b * fp32(1/6)),
then q = fp32(fma(fp32(fma(-6, q1, b)), fp32(1/6), q1)).  This test evaluates
that sequence with exact rational arithmetic (each fma rounded once) for every
positive finite bf16 value and compares it with numpy's IEEE float32 quotient.
"""
from fractions import Fraction

import numpy as np


def rn32(x: Fraction) -> Fraction:
    """Round an exact rational to the nearest float32 (ties to even), with
    subnormals; overflow is not reached by the values checked here."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    q = x / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_division_by_six_via_residual_correction():
    mags = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    want = (mags / np.float32(6.0)).astype(np.float64)
    r6 = Fraction(float(np.float32(1.0) / np.float32(6.0)))
    bad = []
    for b32, w in zip(mags.tolist(), want.tolist()):
        b = Fraction(b32)
        q1 = rn32(b * r6)
        r = rn32(b - 6 * q1)
        q = rn32(r * r6 + q1)
        if q != Fraction(w):
            bad.append(b32)
    assert not bad, bad[:5]
    # the plain product alone is not enough (so the correction step matters)
    assert np.count_nonzero((mags * np.float32(1.0 / 6.0)) != (mags / np.float32(6.0))) > 0


C_DIV6 = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
/* every positive float b in [2^-125, FLT_MAX]: fp32(b * fp32(1/6)) with one
   residual correction against the IEEE quotient b / 6 */
int main(void) {
  const float r6 = 1.0f / 6.0f;
  long long bad = 0, n = 0;
#pragma omp parallel for reduction(+:bad,n) schedule(static)
  for (long long u = 0x01000000LL; u <= 0x7F7FFFFFLL; ++u) {
    uint32_t w = (uint32_t)u;
    float b;
    memcpy(&b, &w, 4);
    float q1 = b * r6;
    float q = fmaf(fmaf(-6.0f, q1, b), r6, q1);
    bad += (q != b / 6.0f);
    n += 1;
  }
  /* below 2^-125 the quotient is subnormal and the shortcut can be off: the
     kernel divides there */
  long long below = 0;
  for (uint32_t w = 1; w < 0x01000000u; ++w) {
    float b;
    memcpy(&b, &w, 4);
    float q1 = b * r6;
    below += (fmaf(fmaf(-6.0f, q1, b), r6, q1) != b / 6.0f);
  }
  printf("%lld %lld %lld\n", n, bad, below);
  return 0;
}
"""


def test_division_by_six_for_every_float_block_max(tmp_path):
    """The columnwise NVFP4 cast's block max is any FP32 value (the RHT output),
    so its division-free fp32(b / 6) is checked for every float in the range
    where the kernel uses it, [2^-125, FLT_MAX], against C's IEEE float
    division (gcc, no FMA contraction; fmaf is the correctly rounded fused
    multiply-add)."""
    import subprocess
    src, exe = tmp_path / "div6.c", tmp_path / "div6"
    src.write_text(C_DIV6)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-std=c11", str(src), "-o",
                    str(exe), "-lm"], check=True)
    n, bad, below = map(int, subprocess.run([str(exe)], capture_output=True, text=True, check=True,
                                            timeout=600).stdout.split())
    assert n == 0x7F7FFFFF - 0x01000000 + 1
    assert bad == 0
    assert below > 0          # the guard is needed
