"""The append kernels form x / s (and the scale m / FMAX) as a corrected
product with a correctly rounded reciprocal instead of an IEEE division
(Markstein's final correction step: y = rn(x r), q = rn(y - (y s - x) r)).
This checks, in plain C on the host, that the identity gives the IEEE
quotient bit for bit over the inputs the kernels feed it -- every bf16 row
absmax m, the scale s = max(rn(m / FMAX), 1e-12), and (a stride of m values)
every bf16 x with |x| <= m -- or, where the residual underflows, a quotient
that is also below 2^-60 with the same sign, whose FP8 and INT8 codes are
zero either way."""
import os
import shutil
import subprocess
import tempfile

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
static float bf(uint32_t b) { uint32_t u = b << 16; float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float quot(float x, float s, float r) {
  volatile float y = x * r;
  volatile float e = fmaf(y, s, -x);
  volatile float q = fmaf(-e, r, y);
  return q;
}
int main(int argc, char** argv) {
  const int stride = atoi(argv[1]);
  const float fms[3] = {448.0f, 57344.0f, 127.0f};
  long bad = 0, pairs = 0, tiny = 0;
  for (int k = 0; k < 3; ++k) {
    volatile float fm = fms[k];
    const float rf = 1.0f / fm;
    for (uint32_t mb = 0; mb < 0x7F80; ++mb) {       /* every finite bf16 absmax */
      const float m = bf(mb);
      float s = quot(m, fm, rf);
      if (!(s >= 1e-12f)) s = 1e-12f;
      float sref = m / fm;
      if (!(sref >= 1e-12f)) sref = 1e-12f;
      if (bits(s) != bits(sref)) { printf("scale m %a: %a vs %a\n", m, s, sref); ++bad; }
      if (mb % stride) continue;
      const float r = 1.0f / s;
      for (uint32_t xb = 0; xb <= mb; ++xb) {
        for (int sg = 0; sg < 2; ++sg) {
          const float x = bf(xb | (sg ? 0x8000u : 0u));
          const float q = quot(x, s, r), ref = x / s;
          ++pairs;
          if (bits(q) == bits(ref)) continue;
          if (fabsf(q) < 0x1p-60f && fabsf(ref) < 0x1p-60f && signbit(q) == signbit(ref)) {
            ++tiny;
            continue;
          }
          if (bad < 10) printf("fmax %g m %a x %a: %a vs %a\n", fms[k], m, x, q, ref);
          ++bad;
        }
      }
    }
  }
  printf("pairs %ld tiny %ld bad %ld\n", pairs, tiny, bad);
  return bad != 0;
}
"""


def test_corrected_product_equals_ieee_quotient():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "q.c")
        exe = os.path.join(d, "q")
        with open(src, "w") as f:
            f.write(SRC)
        subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", exe, src, "-lm"], check=True)
        r = subprocess.run([exe, "53"], capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-2000:]
        assert "bad 0" in r.stdout
