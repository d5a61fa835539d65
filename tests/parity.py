"""Helpers shared by the GPU parity tests: seeded inputs, uploads, tolerance checks.

Tolerance (for floating-point outputs): every element must satisfy
    |y - r| <= tol * (cond + |r|)
where r is the oracle's exact (fp64) value and cond the sum of absolute
products of that output (scale * sum |w| |x|), and the whole vector must
satisfy ||y - r||_2 <= tol * ||r||_2.  tol = 1e-5 for fp32 outputs and
2e-2 for bf16 outputs.
"""
import numpy as np
import torch

TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def assert_close(y, ref, cond, tol, what=""):
    y = np.asarray(y, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    cond = np.asarray(cond, np.float64).ravel()
    err = np.abs(y - ref)
    bound = tol * (cond + np.abs(ref))
    bad = np.nonzero(err > bound)[0]
    if bad.size:
        i = bad[np.argmax(err[bad] / np.maximum(bound[bad], 1e-300))]
        raise AssertionError("%s: %d of %d elements out of tolerance; worst at %d: got %r want %r (bound %r)" %
                             (what, bad.size, y.size, i, y[i], ref[i], bound[i]))
    rn = np.linalg.norm(ref)
    if rn > 0:
        rel = np.linalg.norm(y - ref) / rn
        assert rel <= tol, "%s: normwise error %g > %g" % (what, rel, tol)


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
