"""The seeded input generator (gemm_bl_gemv_gb300/synth.py) that the oracle and
the GPU path share: it holds no BitLinear arithmetic, but the full-size parity
tests rely on it drawing the same rows whether asked for a sample or the whole
matrix, and on its value distributions being the stated ones."""
import numpy as np

from gemm_bl_gemv_gb300 import synth


def test_sampled_rows_equal_full_matrix_rows():
    N, K = 3 * synth.ROW_BLOCK + 17, 256
    full = synth.weight_matrix(5, "w", N, K, "ternary", 0.4)
    rows = np.array([0, 1, synth.ROW_BLOCK - 1, synth.ROW_BLOCK, 2 * synth.ROW_BLOCK + 3, N - 1])
    assert np.array_equal(synth.weight_rows(5, "w", N, K, rows, "ternary", 0.4), full[rows])
    assert np.array_equal(synth.weight_rows(5, "w", N, K, rows[::-1], "ternary", 0.4), full[rows[::-1]])
    sc = synth.block_scale_matrix(5, N, K // 256)
    assert np.array_equal(synth.block_scale_rows(5, N, K // 256, rows), sc[rows])


def test_draws_are_deterministic_and_distinct_per_tensor():
    a = synth.weight_matrix(1, "w_gate", 64, 256, "ternary", 0.4)
    assert np.array_equal(a, synth.weight_matrix(1, "w_gate", 64, 256, "ternary", 0.4))
    assert not np.array_equal(a, synth.weight_matrix(1, "w_up", 64, 256, "ternary", 0.4))
    assert not np.array_equal(a, synth.weight_matrix(2, "w_gate", 64, 256, "ternary", 0.4))


def test_value_sets_and_rates():
    t = synth.weight_matrix(3, "w", 2048, 1024, "ternary", 0.4)
    assert set(np.unique(t)) <= {-1, 0, 1}
    p0 = np.mean(t == 0)
    assert abs(p0 - 0.4) < 0.01 and abs(np.mean(t == 1) - np.mean(t == -1)) < 0.01
    s = synth.weight_matrix(3, "w", 512, 1024, "signs")
    assert set(np.unique(s)) == {-1, 1} and abs(np.mean(s == 1) - 0.5) < 0.01
    d = synth.block_scale_matrix(3, 512, 20).view(np.float16).astype(np.float64)
    assert (d >= 0).all() and abs(np.mean(d) - 0.02 * np.sqrt(2 / np.pi)) < 0.002  # E|N(0, s)| = s sqrt(2/pi)
    x = synth.activations(3, 4, 4096, "f32")
    assert x.dtype == np.float32 and abs(x.mean()) < 0.05 and abs(x.std() - 1) < 0.05
    xb = synth.activations(3, 4, 4096, "bf16")
    assert xb.dtype == np.uint16
