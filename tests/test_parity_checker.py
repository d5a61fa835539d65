"""The tolerance check the GPU parity tests rely on (tests/parity.py), run on
the CPU against planted errors: it must reject an error just above either
bound and accept one just inside both."""
import numpy as np
import pytest

from parity import TOL_BF16, TOL_F32, assert_close, bf16_to_f64, x_f64


@pytest.mark.parametrize("tol", [TOL_F32, TOL_BF16])
def test_elementwise_bound(tol):
    g = np.random.Generator(np.random.PCG64(41))
    ref = g.standard_normal(1000)
    cond = np.abs(ref) * 3 + 1.0
    bound = tol * (cond + np.abs(ref))
    y = ref.copy()
    y[17] += 0.99 * bound[17]               # one element just inside its own bound
    assert_close(y, ref, cond, tol)
    y[17] = ref[17] + 1.01 * bound[17]      # and just outside it
    with pytest.raises(AssertionError, match="out of tolerance"):
        assert_close(y, ref, cond, tol)


@pytest.mark.parametrize("tol", [TOL_F32, TOL_BF16])
def test_normwise_bound(tol):
    g = np.random.Generator(np.random.PCG64(43))
    ref = g.standard_normal(1000)
    cond = np.full(1000, 1e9)                # elementwise bound far away: only the norm can fail
    d = g.standard_normal(1000)
    d *= 1.01 * tol * np.linalg.norm(ref) / np.linalg.norm(d)
    with pytest.raises(AssertionError, match="normwise"):
        assert_close(ref + d, ref, cond, tol)
    assert_close(ref + d * (0.99 / 1.01), ref, cond, tol)


def test_every_element_is_checked():
    ref = np.ones(4097)
    y = ref.copy()
    y[-1] = 1.5                              # the last element of a ragged length
    with pytest.raises(AssertionError):
        assert_close(y, ref, np.zeros_like(ref), TOL_F32)


def test_exact_decoders():
    assert list(bf16_to_f64(np.array([0x3F80, 0xBF80, 0x0001, 0x7F7F], np.uint16))) == \
        [1.0, -1.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127]
    x = np.array([1.0, 2.0 ** -140, -3.25], np.float32)
    assert list(x_f64(x, "f32")) == [1.0, 2.0 ** -140, -3.25]
