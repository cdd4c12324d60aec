"""The e4m3 requantisation quotient of the routed L1 epilogues, checked on the host.

The kernels take x / s (s = fp32(amax) / 448) without a full-range divide per element:
q0 = x * inv, r = fma(-q0, s, x), q = fma(r, inv, q0) with inv = 1/s (Markstein's
correction).  With inv correctly rounded this is the correctly rounded fp32 quotient, the
same value the oracle's fp32 division gives, so the e4m3 code decisions agree.  With inv
from a fast reciprocal refined by one Newton step (the per-token scale path) it must agree
on all but a vanishing fraction of quotients.  Both claims are checked here in C with fmaf
(correctly rounded by C99) over random requantisation inputs.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

C_SRC = r"""
#include <math.h>
#include <stdint.h>
#include <string.h>
static float quot(float x, float s, float inv) {
  float q0 = x * inv;
  float r = fmaf(-q0, s, x);
  return fmaf(r, inv, q0);
}
static float nudge(float v, int ulps) {  /* v moved by `ulps` units in the last place */
  uint32_t b; memcpy(&b, &v, 4); b = (uint32_t)((int32_t)b + ulps); memcpy(&v, &b, 4);
  return v;
}
/* mode 0: inv = 1/s correctly rounded; mode 1: inv from a reciprocal `err` ulps off,
   refined by one Newton step.  Returns the number of quotients that differ from x / s. */
long count_mismatch(const float* x, const float* amax, long n, int mode, int err) {
  long bad = 0;
  for (long i = 0; i < n; ++i) {
    volatile float a = amax[i];
    float s = a / 448.0f;
    float inv;
    if (mode == 0) {
      inv = 1.0f / s;
    } else {
      float y0 = nudge(1.0f / s, err);
      inv = fmaf(fmaf(-s, y0, 1.0f), y0, y0);
    }
    volatile float ref = x[i] / s;
    float q = quot(x[i], s, inv);
    if (memcmp(&q, (const void*)&ref, 4) != 0) ++bad;
  }
  return bad;
}
"""


@pytest.fixture(scope="module")
def lib():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    d = tempfile.mkdtemp()
    src = os.path.join(d, "q.c")
    so = os.path.join(d, "q.so")
    with open(src, "w") as f:
        f.write(C_SRC)
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-shared", "-fPIC", src, "-o", so, "-lm"],
                   check=True)
    L = ctypes.CDLL(so)
    L.count_mismatch.restype = ctypes.c_long
    L.count_mismatch.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long, ctypes.c_int,
                                 ctypes.c_int]
    yield L
    shutil.rmtree(d, ignore_errors=True)


def _inputs(n, seed):
    rng = np.random.default_rng(seed)
    # activations over many magnitudes; amax >= |x| as in a quantisation group
    x = (rng.standard_normal(n) * np.exp(rng.uniform(-20, 20, n))).astype(np.float32)
    amax = (np.abs(x) * (1.0 + rng.exponential(1.0, n))).astype(np.float32)
    amax = np.maximum(amax, np.float32(1e-30))
    return np.ascontiguousarray(x), np.ascontiguousarray(amax)


def test_correction_with_rounded_reciprocal_equals_fp32_division(lib):
    x, amax = _inputs(2_000_000, 0)
    bad = lib.count_mismatch(x.ctypes.data, amax.ctypes.data, x.size, 0, 0)
    assert bad == 0


@pytest.mark.parametrize("err", [-2, -1, 1, 2])
def test_correction_with_refined_fast_reciprocal_is_almost_always_exact(lib, err):
    x, amax = _inputs(1_000_000, 10 + err)
    bad = lib.count_mismatch(x.ctypes.data, amax.ctypes.data, x.size, 1, err)
    assert bad <= 10, bad  # at most ten in a million quotients one ulp away


def test_quotient_check_detects_a_plain_product(lib):
    # the check has teeth: dropping the correction (q = x * inv) is visibly inexact
    x, amax = _inputs(200_000, 9)
    s = (amax / np.float32(448.0)).astype(np.float32)
    inv = (np.float32(1.0) / s).astype(np.float32)
    plain = (x * inv).astype(np.float32)
    ref = (x / s).astype(np.float32)
    assert np.count_nonzero(plain != ref) > 1000
