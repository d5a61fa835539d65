"""Helpers shared by the GPU parity tests: seeded inputs, uploads, tolerance checks.

Tolerance for floating-point outputs (r the oracle's exact fp64 value, cond the
sum of absolute products of that output, scale * sum |w| |x|):

    elementwise  |y - r| <= rho * |r| + alpha * cond (+ extra)
    normwise     ||y - r||_2 <= nu * ||r||_2 (+ ||extra||_2)

The two elementwise terms separate the two error sources of every kernel here:
- rho * |r| is the rounding of the output itself.  A bf16 output is rounded
  once, to nearest even, which moves it by at most 2^-8 |r| (half an ulp of
  an 8-bit significand at the bottom of a binade); rho = 2^-7 is twice that,
  so that the correct rounding uses at most half of the bound.  For fp32
  outputs rho = 1e-5, the relative error the hot-path contract states.
- alpha * cond bounds the accumulation and conversion error before that
  rounding.  The kernels form exact integer dots (group or slice sums) and
  add a few hundred fp32 terms at most, so the error is a few times
  2^-24 * cond; alpha = 1e-5 covers it with margin.  The tensor-core paths
  with an fp32 accumulator (TQ2_0 x int8, W1A8 with M > 8) round once per
  16-element MMA step, so their alpha grows with K (tol_tc).
- extra is a per-element bound that a kernel states for inputs outside its
  exact range (the GEMV's per-group fixed point with an extreme in-group
  dynamic range); only the tests that probe that range pass it.

With these bounds an output missing one 128-element group, one 32-element
shift class or a 16-row tile's group fails (tests/test_parity_checker.py
plants such errors on the CPU).  The normwise bound nu is 1e-5 for fp32
outputs and 2^-8 for bf16 outputs.
"""
import math

import numpy as np
import torch


class Tol:
    """Elementwise rho (output rounding) and alpha (accumulation), normwise nu."""

    def __init__(self, rho, alpha, nu):
        self.rho, self.alpha, self.nu = float(rho), float(alpha), float(nu)

    def __repr__(self):
        return "Tol(rho=%g, alpha=%g, nu=%g)" % (self.rho, self.alpha, self.nu)


TOL_F32 = Tol(1e-5, 1e-5, 1e-5)
TOL_BF16 = Tol(2.0 ** -7, 1e-5, 2.0 ** -8)


def tol_tc(base, K):
    """Tolerance of a tensor-core product whose fp32 accumulator is rounded
    (at most 2^-23 relative, truncation included) once per 16-element MMA
    step: alpha = max(base alpha, 2^-23 * ceil(K / 16))."""
    return Tol(base.rho, max(base.alpha, 2.0 ** -23 * math.ceil(K / 16)), base.nu)


def assert_close(y, ref, cond, tol, what="", extra=None):
    y = np.asarray(y, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    cond = np.asarray(cond, np.float64).ravel()
    assert y.shape == ref.shape == cond.shape, "%s: shapes %s %s %s" % (what, y.shape, ref.shape, cond.shape)
    assert np.all(np.isfinite(y)), "%s: non-finite output" % what
    err = np.abs(y - ref)
    bound = tol.rho * np.abs(ref) + tol.alpha * cond
    if extra is not None:
        bound = bound + np.asarray(extra, np.float64).ravel()
    bad = np.nonzero(err > bound)[0]
    if bad.size:
        i = bad[np.argmax(err[bad] / np.maximum(bound[bad], 1e-300))]
        raise AssertionError("%s: %d of %d elements out of tolerance %r; worst at %d: got %r want %r (bound %r)" %
                             (what, bad.size, y.size, tol, i, y[i], ref[i], bound[i]))
    rn = np.linalg.norm(ref)
    if rn > 0:
        # a stated per-element bound loosens the norm by its own norm
        xn = 0.0 if extra is None else np.linalg.norm(np.asarray(extra, np.float64).ravel()) / rn
        rel = np.linalg.norm(y - ref) / rn
        assert rel <= tol.nu + xn, "%s: normwise error %g > %g" % (what, rel, tol.nu + xn)


def fixed_point_bound(w, x, scale, D, G=128):
    """The i2_s GEMV's stated error for activations outside the exact range
    (include/bl.h, bl_gemv_i2s): each 128-element group of x is carried as an
    integer with 8D - 1 magnitude bits relative to the group's max|x|, so an
    element's absolute error is at most 2^-(8D-1) times that maximum.  Per
    output: |scale| * sum_g 2^-(8D-1) max|x_g| * sum_{k in g} |w[n,k]|.
    D = 2 for bf16 x and y, 3 otherwise (4 for fp32 x on the tiled fallback)."""
    w = np.asarray(w)
    N, K = w.shape
    gmax = np.abs(np.asarray(x, np.float64)).reshape(K // G, G).max(axis=1)
    wabs = np.abs(w.astype(np.float64)).reshape(N, K // G, G).sum(axis=2)
    return abs(float(scale)) * (wabs @ (gmax * 2.0 ** -(8 * D - 1)))


def to_gpu(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_gpu(bits):
    """uint16 bf16 bit patterns -> torch.bfloat16 CUDA tensor."""
    return to_gpu(np.ascontiguousarray(bits, np.uint16).view(np.int16), torch.bfloat16)


def fp16_gpu(bits):
    return to_gpu(np.ascontiguousarray(bits, np.uint16).view(np.int16), torch.float16)


def bits16(t):
    """bf16/fp16 CUDA tensor -> uint16 numpy bit patterns."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def x_f64(x, dtype):
    """Exact fp64 values of an fp32 array or of bf16 bit patterns."""
    if dtype == "f32":
        return np.asarray(x, np.float32).astype(np.float64)
    return bf16_to_f64(x)
