"""The tolerance check the GPU parity tests rely on (tests/parity.py), run on
the CPU against planted errors: it must reject an error just above either
bound and accept one just inside both, and it must reject the localized
mistakes a tile-edge or decode bug makes (a dropped 128-element group in a
few rows, a dropped group in one 16-row tile, one shift class of one group
decoded from the wrong bit pair) at the BitNet-2B MLP and LM-head shapes,
while accepting the oracle's own result rounded to the output type."""
import numpy as np
import pytest

from gemm_bl_gemv_gb300 import synth
from oracle import oracle as O
from parity import TOL_BF16, TOL_F32, Tol, assert_close, bf16_to_f64, tol_tc, x_f64


def bound_of(tol, ref, cond):
    return tol.rho * np.abs(ref) + tol.alpha * cond


@pytest.mark.parametrize("tol", [TOL_F32, TOL_BF16])
def test_elementwise_bound(tol):
    g = np.random.Generator(np.random.PCG64(41))
    ref = g.standard_normal(1000) + 3.0
    cond = np.abs(ref) * 3 + 1.0
    bound = bound_of(tol, ref, cond)
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
    d *= 1.01 * tol.nu * np.linalg.norm(ref) / np.linalg.norm(d)
    with pytest.raises(AssertionError, match="normwise"):
        assert_close(ref + d, ref, cond, tol)
    assert_close(ref + d * (0.99 / 1.01), ref, cond, tol)


def test_extra_term_and_tc_alpha():
    ref = np.ones(10)
    cond = np.ones(10)
    y = ref.copy()
    y[3] += 0.5
    with pytest.raises(AssertionError):
        assert_close(y, ref, cond, Tol(1e-5, 1e-5, 1.0))
    assert_close(y, ref, cond, Tol(1e-5, 1e-5, 1.0), extra=np.full(10, 0.5))
    assert tol_tc(TOL_F32, 16).alpha == TOL_F32.alpha
    assert tol_tc(TOL_F32, 16384).alpha == pytest.approx(2.0 ** -23 * 1024)


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


# ---------------------------------------------------------------------------
# localized mistakes at the workload shapes
# ---------------------------------------------------------------------------

def as_bf16(v):
    """fp64 -> the value of its bf16 rounding (nearest even), as fp64."""
    return bf16_to_f64(O.round_bf16(np.asarray(v, np.float64)))


def group_cols(g, G=128):
    return np.arange(g * G, (g + 1) * G)


def shift_class_cols(g, t):
    """Elements of shift class t of i2_s group g: 32 consecutive elements."""
    return np.arange(g * 128 + 32 * t, g * 128 + 32 * t + 32)


@pytest.fixture(scope="module")
def mlp_gate():
    """The BitNet-2B gate product (6912 x 2560, bf16 in and out): weights,
    x, scale, the oracle's r and cond."""
    wl = synth.WORKLOADS["i2s_mlp_bitnet2b"]
    N, K = wl.extra["gate"]
    w = synth.weight_matrix(wl.index, "w_gate", N, K, "ternary", wl.p_zero)
    xb = synth.activations(wl.index, 1, K, "bf16")[0]
    s = synth.tensor_scale(wl.index, "scale_gate")
    x = x_f64(xb, "bf16")
    r, cond = O.gemv_i2s(O.pack_i2s(w, s), x, N, K)
    return w, x, float(s), r, cond


def mutated(w, x, s, r, rows, cols):
    """r with the products of (rows, cols) left out, as a kernel that skipped them would give."""
    out = r.copy()
    for row in rows:
        out[row] -= s * float(w[row, cols].astype(np.float64) @ x[cols])
    return out


def test_mlp_correct_result_passes(mlp_gate):
    _, _, _, r, cond = mlp_gate
    assert_close(as_bf16(r), r, cond, TOL_BF16, "bf16(oracle)")


def test_mlp_dropped_group_in_one_percent_of_rows(mlp_gate):
    w, x, s, r, cond = mlp_gate
    rows = np.arange(0, w.shape[0], 100)
    with pytest.raises(AssertionError):
        assert_close(as_bf16(mutated(w, x, s, r, rows, group_cols(5))), r, cond, TOL_BF16, "dropped group")


def test_mlp_dropped_group_in_one_tile(mlp_gate):
    w, x, s, r, cond = mlp_gate
    rows = np.arange(1600, 1616)
    y = as_bf16(mutated(w, x, s, r, rows, group_cols(0)))
    with pytest.raises(AssertionError):
        assert_close(y, r, cond, TOL_BF16, "tile group")
    # every row of the tile is flagged, not just a few
    err = np.abs(y - r)[rows]
    assert np.count_nonzero(err > bound_of(TOL_BF16, r[rows], cond[rows])) >= 14


def test_mlp_one_row_wrong_shift_class(mlp_gate):
    """Row 777, group 7: shift class 1 decoded from class 2's bit pair."""
    w, x, s, r, cond = mlp_gate
    row, c1, c2 = 777, shift_class_cols(7, 1), shift_class_cols(7, 2)
    y = r.copy()
    y[row] += s * float((w[row, c2] - w[row, c1]).astype(np.float64) @ x[c1])
    with pytest.raises(AssertionError):
        assert_close(as_bf16(y), r, cond, TOL_BF16, "shift class")


@pytest.fixture(scope="module")
def lmhead_rows():
    """2048 sampled rows of the W1A8 LM head (5120 -> 248320, G = 128), M = 4."""
    wl = synth.WORKLOADS["w1a8_lmhead_248320"]
    N, K, G = wl.N, wl.K, wl.group
    rows = np.sort(np.random.Generator(np.random.PCG64(5)).choice(N, 2048, replace=False))
    w = synth.weight_rows(wl.index, "w", N, K, rows, "signs")
    ws = synth.block_scale_rows(wl.index, N, K // G, rows, 0.02, "group_scale")
    q, sm = O.quantize_act_absmax_int8(synth.activations(wl.index, 4, K, "bf16"), "bf16")
    _, y, cond = O.gemm_w1a8(q, sm, O.pack_w1(w), ws, None, K, G)
    return w, ws, q, sm, y, cond


def w1a8_contrib(w, ws, q, sm, row, cols, G=128):
    """[M] contributions of (row, cols) to y (cols inside one group)."""
    g = int(cols[0]) // G
    d = O.fp16_to_f64(ws[row, g])
    return sm.astype(np.float64) * d * (q[:, cols].astype(np.float64) @ w[row, cols].astype(np.float64))


def test_lmhead_correct_result_passes(lmhead_rows):
    _, _, _, _, y, cond = lmhead_rows
    assert_close(as_bf16(y), y, cond, TOL_BF16, "bf16(oracle)")


@pytest.mark.parametrize("kind", ["one_percent_rows", "tile", "bit_class"])
def test_lmhead_localized_mistakes(lmhead_rows, kind):
    w, ws, q, sm, y, cond = lmhead_rows
    yb = y.copy()                                  # [M, rows]
    if kind == "one_percent_rows":
        for row in range(0, w.shape[0], 100):
            yb[:, row] -= w1a8_contrib(w, ws, q, sm, row, group_cols(11))
    elif kind == "tile":
        for row in range(512, 528):
            yb[:, row] -= w1a8_contrib(w, ws, q, sm, row, group_cols(0))
    else:
        # one row, one group: the 16 elements of one bit class of a byte read with flipped signs
        cols = np.arange(17 * 128 + 3, 18 * 128, 8)
        yb[:, 901] -= 2 * w1a8_contrib(w, ws, q, sm, 901, cols)
    with pytest.raises(AssertionError):
        assert_close(as_bf16(yb), y, cond, TOL_BF16, kind)


# ---------------------------------------------------------------------------
# the GEMV's stated fixed-point bound (the `extra` term), checked by emulation
# ---------------------------------------------------------------------------

def emulate_fixed_point(w, x, scale, D, G=128):
    """y as the GEMV's stated arithmetic forms it: per group, X = rint(x 2^F)
    with 2^(8D-2) <= max|x_g| 2^F < 2^(8D-1), exact integer dots, fp64 sums."""
    N, K = w.shape
    y = np.zeros(N)
    for g in range(K // G):
        xg = x[g * G:(g + 1) * G]
        m = np.abs(xg).max()
        if m == 0:
            continue
        e = np.frexp(m)[1]                      # 2^(e-1) <= m < 2^e
        F = (8 * D - 1) - e
        X = np.rint(np.ldexp(xg, F))
        y += np.ldexp(w[:, g * G:(g + 1) * G].astype(np.float64) @ X, -F)
    return scale * y


@pytest.mark.parametrize("D,outlier", [(2, 1e6), (3, 1e6), (4, 1e7)])
def test_fixed_point_bound_holds_and_is_needed(D, outlier):
    """An outlier on a zero weight sets its group's exponent without adding
    to cond: the emulated kernel arithmetic then leaves the rho/alpha bound
    for some outputs, and stays within it once the stated bound is added."""
    from parity import fixed_point_bound
    g = np.random.Generator(np.random.PCG64(300 + D))
    N, K = 64, 512
    w = synth.ternary(g, (N, K), 0.4)
    x = synth.normal_f32(g, (K,)).astype(np.float64)
    if D < 4:
        x = bf16_to_f64(synth.f32_to_bf16_bits(x.astype(np.float32)))
    x[7] = outlier
    w[:, 7] = 0
    r = 1.25 * (w.astype(np.float64) @ x)
    cond = 1.25 * (np.abs(w.astype(np.float64)) @ np.abs(x))
    y = emulate_fixed_point(w, x, 1.25, D)
    tol = TOL_BF16 if D == 2 else TOL_F32
    extra = fixed_point_bound(w, x, 1.25, D)
    assert np.all(np.abs(y - r) <= extra * (1 + 1e-12))
    assert_close(y, r, cond, tol, "emulated", extra=extra)
    with pytest.raises(AssertionError):
        assert_close(y, r, cond, tol, "emulated without the stated bound")
