"""GPU path (libbl through its C ABI) against the CPU oracle, element by element.

Integer and byte results (packed bytes, int8 activations, int32 group dots and
accumulators) must be bit-exact; floating-point results must meet the
tolerance in tests/parity.py.  Shapes span several tiles and a ragged tail;
the full-size workloads are checked on sampled rows, in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from gemm_bl_gemv_gb300 import synth
from oracle import oracle as O
from parity import (TOL_BF16, TOL_F32, assert_close, bf16_gpu, bits16, fixed_point_bound, fp16_gpu, to_gpu,
                    tol_tc, x_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from gemm_bl_gemv_gb300 import build
    build.build()
    from gemm_bl_gemv_gb300 import binding
    binding.set_overlap(False)
    binding.device_error(clear=True)
    yield binding
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0, "a kernel recorded a device-side wait timeout"


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def ternary(g, N, K, p0=1 / 3):
    return synth.ternary(g, (N, K), p0)


def rand_x(g, K, dtype, M=None):
    shape = (K,) if M is None else (M, K)
    x = synth.normal_f32(g, shape)
    return x if dtype == "f32" else synth.f32_to_bf16_bits(x)


def x_gpu(x, dtype):
    return to_gpu(x) if dtype == "f32" else bf16_gpu(x)


# ---------------------------------------------------------------------------
# packing: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (33, 2560), (64, 6912)])
def test_pack_i2s_bit_exact(B, N, K):
    g = rng(N * 1000 + K)
    w = ternary(g, N, K)
    w[0, :] = 0
    if N > 2:
        w[1, :] = 1
        w[2, :] = -1
    got = B.bl_pack_i2s(to_gpu(w), 1.5).cpu().numpy()
    assert np.array_equal(got, O.pack_i2s(w, np.float32(1.5)))


@pytest.mark.parametrize("N,K", [(1, 256), (5, 512), (33, 5120)])
def test_pack_tq2_0_bit_exact(B, N, K):
    g = rng(N * 7 + K)
    w = ternary(g, N, K)
    d = synth.abs_normal_fp16_bits(g, (N, K // 256), 0.02)
    got = B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d)).cpu().numpy()
    assert np.array_equal(got, O.pack_tq2_0(w, d))


@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (17, 5120)])
def test_pack_w1_bit_exact(B, N, K):
    g = rng(N * 11 + K)
    w = ternary(g, N, K)  # zeros must pack as -1
    got = B.bl_pack_w1(to_gpu(w)).cpu().numpy()
    assert np.array_equal(got, O.pack_w1(w))


# ---------------------------------------------------------------------------
# activation quantization: bit-exact q and s
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,K", [(1, 1), (3, 7), (8, 5120), (512, 2560), (2, 70000)])
def test_act_quant_bit_exact(B, dtype, M, K):
    g = rng(M * 31 + K)
    x = synth.normal_f32(g, (M, K)) * g.uniform(0.01, 100, (M, 1)).astype(np.float32)
    if M >= 3:
        x[1] = 0.0                                    # zero row
        x[2, : min(K, 4)] = [127.0, 0.5, 1.5, -2.5][: min(K, 4)]  # ties to even with amax 127
        if K > 4:
            x[2, 4:] = 0.0
    xin = x if dtype == "f32" else synth.f32_to_bf16_bits(x)
    q, s = B.bl_quantize_act_absmax_int8(x_gpu(xin, dtype))
    qo, so = O.quantize_act_absmax_int8(xin, dtype)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


# ---------------------------------------------------------------------------
# i2_s GEMV
# ---------------------------------------------------------------------------

def run_gemv_i2s(B, w, scale, x, xd, yd):
    N, K = w.shape
    packed = B.bl_pack_i2s(to_gpu(w), scale)
    y = B.bl_gemv_i2s(packed, x_gpu(x, xd), N, K, y_dtype=torch.float32 if yd == "f32" else torch.bfloat16)
    yv = y.cpu().numpy().astype(np.float64) if yd == "f32" else x_f64(bits16(y), "bf16")
    ref, cond = O.gemv_i2s(O.pack_i2s(w, scale), x_f64(x, xd), N, K)
    return yv, ref, cond


@pytest.mark.parametrize("xd,yd", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("N,K", [(1, 128), (3, 384), (31, 2560), (33, 2560), (100, 1024), (257, 6912)])
def test_gemv_i2s_small(B, xd, yd, N, K):
    g = rng(N + 13 * K)
    w = ternary(g, N, K)
    x = rand_x(g, K, xd)
    scale = np.float32(g.uniform(0.5, 2.0))
    y, ref, cond = run_gemv_i2s(B, w, scale, x, xd, yd)
    assert_close(y, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "gemv_i2s %dx%d %s->%s" % (N, K, xd, yd))


@pytest.mark.parametrize("xd,yd", [("f32", "f32"), ("bf16", "bf16")])
@pytest.mark.parametrize("N", [1, 20, 300])
def test_gemv_i2s_max_k(B, xd, yd, N):
    """K = 32768, the largest K bl_gemv_i2s accepts (256 groups per row)."""
    K = 32768
    g = rng(N + 7)
    w = ternary(g, N, K)
    x = rand_x(g, K, xd)
    y, ref, cond = run_gemv_i2s(B, w, np.float32(0.75), x, xd, yd)
    assert_close(y, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "gemv_i2s %dx%d" % (N, K))


def test_gemv_i2s_unaligned_x(B):
    """x at an element-aligned but not 16-byte-aligned address (plain loads)."""
    N, K = 70, 1024
    g = rng(99)
    w = ternary(g, N, K)
    for xd in ("f32", "bf16"):
        x = rand_x(g, K, xd)
        xg = x_gpu(x, xd)
        buf = torch.empty(K + 1, dtype=xg.dtype, device="cuda")
        buf[1:].copy_(xg)
        packed = B.bl_pack_i2s(to_gpu(w), np.float32(1.0))
        yv = B.bl_gemv_i2s(packed, buf[1:], N, K, y_dtype=torch.float32).cpu().numpy().astype(np.float64)
        ref, cond = O.gemv_i2s(O.pack_i2s(w, np.float32(1.0)), x_f64(x, xd), N, K)
        assert_close(yv, ref, cond, TOL_F32, "gemv_i2s unaligned x " + xd)


@pytest.mark.parametrize("xd,yd,D", [("f32", "f32", 3), ("f32", "bf16", 3), ("bf16", "bf16", 2), ("bf16", "f32", 3)])
def test_gemv_i2s_extreme_inputs(B, xd, yd, D):
    """Degenerate activations: all zero, tiny values (1e-30), all equal, and
    in-group outliers of 1e4 and 1e6 (1e7 for fp32 x) times the typical
    |x|, whose weight is zero in every other row: such an outlier sets its
    group's fixed-point exponent without adding to cond, so these cases are
    checked against the kernel's stated fixed-point bound as well; plus an
    all-zero weight row."""
    K, N = 512, 40
    g = rng(5)
    w = ternary(g, N, K)
    w[0] = 0
    w[1::2, 7] = 0
    base = synth.normal_f32(g, (K,))
    cases = [np.zeros(K, np.float32), (base * 1e-30).astype(np.float32), np.full(K, -1.0, np.float32)]
    for big in (1e4, 1e7 if xd == "f32" else 1e6):
        o = base.copy()
        o[7] = big
        cases.append(o)
    for x in cases:
        xx = x if xd == "f32" else synth.f32_to_bf16_bits(x)
        y, ref, cond = run_gemv_i2s(B, w, np.float32(1.25), xx, xd, yd)
        extra = fixed_point_bound(w, x_f64(xx, xd), 1.25, D)
        assert_close(y, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "gemv_i2s extreme", extra=extra)


def test_gemv_i2s_workload_2560(B):
    """i2_s GEMV 2560x2560, fp32 in/out (all rows)."""
    wl = synth.WORKLOADS["i2s_gemv_2560"]
    w = synth.weight_matrix(wl.index, "w", wl.N, wl.K, "ternary", wl.p_zero)
    x = synth.activations(wl.index, 1, wl.K, "f32")[0]
    y, ref, cond = run_gemv_i2s(B, w, synth.tensor_scale(wl.index), x, "f32", "f32")
    assert_close(y, ref, cond, TOL_F32, "i2s_gemv_2560")


@pytest.mark.parametrize("mat", ["gate", "up", "down"])
def test_gemv_i2s_workload_mlp(B, mat):
    """BitNet-2B MLP shapes, bf16 in/out (all rows)."""
    wl = synth.WORKLOADS["i2s_mlp_bitnet2b"]
    N, K = wl.extra[mat]
    w = synth.weight_matrix(wl.index, "w_" + mat, N, K, "ternary", wl.p_zero)
    x = synth.activations(wl.index, 1, K, "bf16", tensor="x" if mat != "down" else "x_down")[0]
    y, ref, cond = run_gemv_i2s(B, w, synth.tensor_scale(wl.index, "scale_" + mat), x, "bf16", "bf16")
    assert_close(y, ref, cond, TOL_BF16, "mlp " + mat)


# ---------------------------------------------------------------------------
# fused gate + up + ReLU^2 x mul
# ---------------------------------------------------------------------------

def run_gate_up(B, wg, wu, sg, su, x, xd, hd):
    N, K = wg.shape
    pg, pu = B.bl_pack_i2s(to_gpu(wg), sg), B.bl_pack_i2s(to_gpu(wu), su)
    h = B.bl_gemv_i2s_gate_up(pg, pu, x_gpu(x, xd), N, K, h_dtype=torch.float32 if hd == "f32" else torch.bfloat16)
    hv = h.cpu().numpy().astype(np.float64) if hd == "f32" else x_f64(bits16(h), "bf16")
    ref, cond = O.gemv_i2s_gate_up(O.pack_i2s(wg, sg), O.pack_i2s(wu, su), x_f64(x, xd), N, K)
    return hv, ref, cond


@pytest.mark.parametrize("xd,hd", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (33, 2560), (100, 1024), (257, 6912), (20, 32768)])
def test_gemv_i2s_gate_up_small(B, xd, hd, N, K):
    g = rng(3 * N + K)
    wg, wu = ternary(g, N, K), ternary(g, N, K)
    x = rand_x(g, K, xd)
    h, ref, cond = run_gate_up(B, wg, wu, np.float32(g.uniform(0.5, 2)), np.float32(g.uniform(0.5, 2)), x, xd, hd)
    assert_close(h, ref, cond, TOL_F32 if hd == "f32" else TOL_BF16, "gate_up %dx%d %s->%s" % (N, K, xd, hd))


def test_gemv_i2s_gate_up_workload(B):
    """BitNet-2B MLP gate/up shapes (6912 x 2560), bf16 in/out, all rows."""
    wl = synth.WORKLOADS["i2s_mlp_bitnet2b"]
    N, K = wl.extra["gate"]
    wg = synth.weight_matrix(wl.index, "w_gate", N, K, "ternary", wl.p_zero)
    wu = synth.weight_matrix(wl.index, "w_up", N, K, "ternary", wl.p_zero)
    x = synth.activations(wl.index, 1, K, "bf16")[0]
    h, ref, cond = run_gate_up(B, wg, wu, synth.tensor_scale(wl.index, "scale_gate"),
                               synth.tensor_scale(wl.index, "scale_up"), x, "bf16", "bf16")
    assert_close(h, ref, cond, TOL_BF16, "gate_up workload")


def test_gemv_i2s_gate_up_matches_unfused(B):
    """With fp32 output the fused product equals relu(g)^2 * u formed on the
    host from two bl_gemv_i2s results (same per-row arithmetic)."""
    g = rng(77)
    N, K = 300, 2560
    wg, wu = ternary(g, N, K), ternary(g, N, K)
    x = rand_x(g, K, "f32")
    pg, pu = B.bl_pack_i2s(to_gpu(wg), np.float32(1.25)), B.bl_pack_i2s(to_gpu(wu), np.float32(0.5))
    xg = x_gpu(x, "f32")
    h = B.bl_gemv_i2s_gate_up(pg, pu, xg, N, K, h_dtype=torch.float32).cpu().numpy().astype(np.float64)
    gv = B.bl_gemv_i2s(pg, xg, N, K, y_dtype=torch.float32).cpu().numpy().astype(np.float64)
    uv = B.bl_gemv_i2s(pu, xg, N, K, y_dtype=torch.float32).cpu().numpy().astype(np.float64)
    ref = np.maximum(gv, 0) ** 2 * uv
    assert np.allclose(h, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())


# ---------------------------------------------------------------------------
# fused residual add, fused RMSNorm + residual
# ---------------------------------------------------------------------------

def res_gpu(r, yd):
    return to_gpu(r.astype(np.float32)) if yd == "f32" else bf16_gpu(synth.f32_to_bf16_bits(r.astype(np.float32)))


def res_f64(r, yd):
    return r.astype(np.float32).astype(np.float64) if yd == "f32" else x_f64(synth.f32_to_bf16_bits(r.astype(np.float32)), "bf16")


@pytest.mark.parametrize("xd,yd", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("N,K", [(1, 128), (33, 2560), (257, 6912), (20, 32768)])
def test_gemv_i2s_residual(B, xd, yd, N, K):
    g = rng(5 * N + K)
    w = ternary(g, N, K)
    x = rand_x(g, K, xd)
    r = synth.normal_f32(g, (N,)) * 4
    packed = B.bl_pack_i2s(to_gpu(w), np.float32(1.5))
    y = B.bl_gemv_i2s_residual(packed, x_gpu(x, xd), res_gpu(r, yd), N, K)
    yv = y.cpu().numpy().astype(np.float64) if yd == "f32" else x_f64(bits16(y), "bf16")
    ref, cond = O.gemv_i2s_norm_residual(O.pack_i2s(w, np.float32(1.5)), x_f64(x, xd), N, K, residual=res_f64(r, yd))
    assert_close(yv, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "residual %dx%d" % (N, K))


@pytest.mark.parametrize("xd,yd", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("N,K", [(1, 128), (33, 2560), (2560, 6912), (20, 32768)])
@pytest.mark.parametrize("with_residual", [True, False])
def test_gemv_i2s_rmsnorm(B, xd, yd, N, K, with_residual):
    g = rng(7 * N + K + with_residual)
    w = ternary(g, N, K)
    x = rand_x(g, K, xd)
    rw = (synth.normal_f32(g, (K,)) * 0.1 + 1.0).astype(np.float32)
    rw_in = rw if xd == "f32" else synth.f32_to_bf16_bits(rw)
    r = synth.normal_f32(g, (N,)) if with_residual else None
    packed = B.bl_pack_i2s(to_gpu(w), np.float32(0.75))
    y = B.bl_gemv_i2s_rmsnorm(packed, x_gpu(x, xd), x_gpu(rw_in, xd), N, K, eps=1e-5,
                              residual=res_gpu(r, yd) if with_residual else None,
                              y_dtype=torch.float32 if yd == "f32" else torch.bfloat16)
    yv = y.cpu().numpy().astype(np.float64) if yd == "f32" else x_f64(bits16(y), "bf16")
    ref, cond = O.gemv_i2s_norm_residual(O.pack_i2s(w, np.float32(0.75)), x_f64(x, xd), N, K,
                                         rms_w=x_f64(rw_in, xd), eps=1e-5,
                                         residual=res_f64(r, yd) if with_residual else None)
    assert_close(yv, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "rmsnorm %dx%d" % (N, K))


# ---------------------------------------------------------------------------
# TQ2_0 GEMV
# ---------------------------------------------------------------------------

def run_gemv_tq2(B, w, d, x, xd):
    N, K = w.shape
    packed = B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d))
    y = B.bl_gemv_tq2_0(packed, x_gpu(x, xd), N, K).cpu().numpy().astype(np.float64)
    ref, cond = O.gemv_tq2_0(O.pack_tq2_0(w, d), x_f64(x, xd), N, K)
    return y, ref, cond


@pytest.mark.parametrize("xd", ["f32", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 256), (5, 512), (31, 5120), (33, 5120), (70, 1792), (130, 256),
                                 (333, 768), (1000, 2560), (3, 22528)])
def test_gemv_tq2_0_small(B, xd, N, K):
    """Odd blocks 2 bytes past a 4-byte boundary, a tensor whose size is not
    a multiple of 16 bytes (333 x 768), a partial last tile, the longest row
    fp32 x supports (22528)."""
    g = rng(3 * N + K)
    w = ternary(g, N, K)
    d = synth.abs_normal_fp16_bits(g, (N, K // 256), 0.02)
    d[0, 0] = 0x0001          # an fp16 subnormal scale
    x = rand_x(g, K, xd)
    y, ref, cond = run_gemv_tq2(B, w, d, x, xd)
    assert_close(y, ref, cond, TOL_F32, "gemv_tq2_0 %dx%d %s" % (N, K, xd))


@pytest.mark.parametrize("xd", ["f32", "bf16"])
def test_gemv_tq2_0_unaligned_x(B, xd):
    """x one element past a 16-byte boundary (only element alignment is required)."""
    g = rng(777)
    N, K = 90, 1024
    w = ternary(g, N, K)
    d = synth.abs_normal_fp16_bits(g, (N, K // 256), 0.02)
    x = rand_x(g, K + 1, xd)
    xt = x_gpu(x, xd)[1:]
    y = B.bl_gemv_tq2_0(B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d)), xt, N, K).cpu().numpy().astype(np.float64)
    ref, cond = O.gemv_tq2_0(O.pack_tq2_0(w, d), x_f64(x[1:], xd), N, K)
    assert_close(y, ref, cond, TOL_F32, "gemv_tq2_0 unaligned x %s" % xd)


def test_gemv_tq2_0_many_rows(B):
    """30400 x 4096: 200 rows per SM, 25 eight-row tiles through each CTA's
    ring; sampled rows include the first and last of every 200-row share."""
    g = rng(9090)
    N, K = 30400, 4096
    w = ternary(g, N, K)
    d = synth.abs_normal_fp16_bits(g, (N, K // 256), 0.02)
    x = rand_x(g, K, "bf16")
    packed = B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d))
    y = B.bl_gemv_tq2_0(packed, x_gpu(x, "bf16"), N, K).cpu().numpy().astype(np.float64)
    edges = np.concatenate([np.arange(0, N, 200), np.arange(199, N, 200)])
    rows = np.unique(np.concatenate([edges, g.choice(N, 2000, replace=False)]))
    ref, cond = O.gemv_tq2_0(O.pack_tq2_0(w, d), x_f64(x, "bf16"), N, K, rows=rows)
    assert_close(y[rows], ref, cond, TOL_F32, "tq2_0 30400x4096")


def test_gemv_tq2_0_workload(B):
    wl = synth.WORKLOADS["tq2_0_gemv_5120x13824"]
    w = synth.weight_matrix(wl.index, "w", wl.N, wl.K, "ternary", wl.p_zero)
    d = synth.block_scale_matrix(wl.index, wl.N, wl.K // 256)
    x = synth.activations(wl.index, 1, wl.K, "bf16")[0]
    y, ref, cond = run_gemv_tq2(B, w, d, x, "bf16")
    assert_close(y, ref, cond, TOL_F32, "tq2_0 workload")


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (9, 70, 512), (128, 192, 1024), (130, 200, 2560),
                                   (512, 96, 768), (257, 389, 5120), (20, 1, 256), (130, 40, 16384)])
def test_gemm_tq2_0_int8(B, M, N, K):
    """TQ2_0 x int8 on the tensor cores: ragged M and N tails, N % 4 != 0
    (per-element stores), a negative, a zero and a subnormal block scale."""
    g = rng(5 * M + N + K)
    w = ternary(g, N, K)
    d = synth.abs_normal_fp16_bits(g, (N, K // 256), 0.02)
    d[0, 0] = 0x0001  # fp16 subnormal
    if N > 2:
        d[1, :] = 0x8000 | d[1, :]  # negative scales
        d[2, 0] = 0
    xb = synth.f32_to_bf16_bits(synth.normal_f32(g, (M, K)))
    q, s = O.quantize_act_absmax_int8(xb, "bf16")
    packed = B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d))
    y = B.bl_gemm_tq2_0_int8(to_gpu(q), to_gpu(s), packed, N).cpu().numpy().astype(np.float64)
    ref, cond = O.gemm_tq2_0_int8(q, s, O.pack_tq2_0(w, d), N, K)
    assert_close(y, ref, cond, tol_tc(TOL_F32, K), "tq2_0 int8 M=%d %dx%d" % (M, N, K))


def test_gemm_tq2_0_int8_scale_range_flag(B):
    """A block scale of 1024 or more is outside the kernel's exact range: the
    launch completes, flags BL_DEVERR_RANGE, and the other rows stay exact."""
    g = rng(4242)
    M, N, K = 130, 40, 512
    w = ternary(g, N, K)
    d = synth.abs_normal_fp16_bits(g, (N, K // 256), 0.02)
    d[7, 1] = 0x6800  # 2048
    q, s = O.quantize_act_absmax_int8(synth.f32_to_bf16_bits(synth.normal_f32(g, (M, K))), "bf16")
    B.device_error(clear=True)
    y = B.bl_gemm_tq2_0_int8(to_gpu(q), to_gpu(s), B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d)), N)
    torch.cuda.synchronize()
    assert B.device_error(clear=True) & B.BL_DEVERR_RANGE
    rows = np.array([r for r in range(N) if r != 7])
    ref, cond = O.gemm_tq2_0_int8(q, s, O.pack_tq2_0(w, d), N, K, rows=rows)
    assert_close(y.cpu().numpy().astype(np.float64)[:, rows], ref, cond, tol_tc(TOL_F32, K), "tq2_0 int8 other rows")


def test_gemm_tq2_0_int8_workload(B):
    """The 5120 -> 13824 TQ2_0 weights against 512 quantized tokens, sampled rows."""
    wl = synth.WORKLOADS["tq2_0_gemv_5120x13824"]
    M = 512
    w = synth.weight_matrix(wl.index, "w", wl.N, wl.K, "ternary", wl.p_zero)
    d = synth.block_scale_matrix(wl.index, wl.N, wl.K // 256)
    xb = synth.activations(wl.index, M, wl.K, "bf16")
    q, s = O.quantize_act_absmax_int8(xb, "bf16")
    packed = B.bl_pack_tq2_0(to_gpu(w), fp16_gpu(d))
    y = B.bl_gemm_tq2_0_int8(to_gpu(q), to_gpu(s), packed, wl.N).cpu().numpy().astype(np.float64)
    rows = np.unique(np.concatenate([[0, 1, wl.N - 1, wl.N - 2], rng(11).integers(0, wl.N, 40)]))
    ref, cond = O.gemm_tq2_0_int8(q, s, O.pack_tq2_0(w, d), wl.N, wl.K, rows=rows)
    assert_close(y[:, rows], ref, cond, tol_tc(TOL_F32, wl.K), "tq2_0 int8 workload")


# ---------------------------------------------------------------------------
# W1A8
# ---------------------------------------------------------------------------

def run_w1a8(B, w, ws, bias, q, s, G, rows=None, wq_gpu=None):
    N, K = w.shape if w is not None else (wq_gpu.shape[0], wq_gpu.shape[1] * 32)
    if wq_gpu is None:
        wq_gpu = B.bl_pack_w1(to_gpu(w))
    y, dots = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq_gpu, fp16_gpu(ws),
                             None if bias is None else bf16_gpu(bias), group=G, group_dots=True)
    yb = bits16(y)
    dots = dots.cpu().numpy()
    return yb, dots


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
@pytest.mark.parametrize("N,K", [(1, 256), (37, 512), (100, 5120)])
def test_gemm_w1a8_small(B, M, G, N, K):
    if K % G:
        pytest.skip("K not a multiple of G")
    g = rng(M * 100 + G + N + K)
    w = synth.signs(g, (N, K))
    xb = rand_x(g, K, "bf16", M)
    q, s = O.quantize_act_absmax_int8(xb, "bf16")
    ws = synth.abs_normal_fp16_bits(g, (N, K // G), 0.02)
    bias = synth.f32_to_bf16_bits(synth.normal_f32(g, (N,))) if (M + G) % 2 else None
    yb, dots = run_w1a8(B, w, ws, bias, q, s, G)
    wq = O.pack_w1(w)
    dref, yref, cond = O.gemm_w1a8(q, s, wq, ws, bias, K, G)
    assert np.array_equal(dots.astype(np.int64), dref), "group dots must be bit-exact"
    assert_close(x_f64(yb, "bf16"), yref, cond, TOL_BF16, "w1a8 M=%d G=%d %dx%d" % (M, G, N, K))


@pytest.mark.parametrize("N,K", [(14616, 1024), (1000, 5120), (64, 128), (7296, 2560), (8, 65536)])
def test_gemm_w1a8_one_token(B, N, K):
    """One token, 128-element groups (the activation-stationary kernel):
    several tiles per CTA with a ragged last tile, one group per row, the
    longest K it takes; exact group dots, y with and without the dots
    output identical, a bias, and the act quantization fused in equal to the
    two calls."""
    G = 128
    g = rng(N + K)
    w = synth.signs(g, (N, K))
    xb = rand_x(g, K, "bf16", 1)
    q, s = O.quantize_act_absmax_int8(xb, "bf16")
    ws = synth.abs_normal_fp16_bits(g, (N, K // G), 0.02)
    ws[0, 0] = 0x0001  # fp16 subnormal
    bias = synth.f32_to_bf16_bits(synth.normal_f32(g, (N,)))
    wq = B.bl_pack_w1(to_gpu(w))
    y, dots = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, fp16_gpu(ws), bf16_gpu(bias), group=G, group_dots=True)
    y2 = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, fp16_gpu(ws), bf16_gpu(bias), group=G)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    dref, yref, cond = O.gemm_w1a8(q, s, O.pack_w1(w), ws, bias, K, G)
    assert np.array_equal(dots.cpu().numpy().astype(np.int64), dref), "group dots must be bit-exact"
    assert_close(x_f64(bits16(y), "bf16"), yref, cond, TOL_BF16, "w1a8 one token %dx%d" % (N, K))
    y3 = B.bl_gemm_w1a8_act(bf16_gpu(xb), wq, fp16_gpu(ws), bf16_gpu(bias), group=G)
    assert torch.equal(y3.view(torch.int16), y2.view(torch.int16)), "fused quantization must equal the two calls"


def test_gemm_w1a8_no_dots_matches_dots_variant(B):
    g = rng(77)
    M, N, K, G = 4, 300, 1024, 128
    w = synth.signs(g, (N, K))
    q, s = O.quantize_act_absmax_int8(rand_x(g, K, "bf16", M), "bf16")
    ws = synth.abs_normal_fp16_bits(g, (N, K // G), 0.02)
    wq = B.bl_pack_w1(to_gpu(w))
    y1 = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, fp16_gpu(ws), group=G)
    y2, _ = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, fp16_gpu(ws), group=G, group_dots=True)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M", [9, 64, 130, 512])
@pytest.mark.parametrize("G", [32, 128, 256])
@pytest.mark.parametrize("N,K", [(200, 1024), (70, 2560), (1, 256), (33, 128)])
def test_gemm_w1a8_large_m_tensor_cores(B, M, G, N, K):
    """M > 8 runs on the tensor cores (B = +-group scale in fp16); with and
    without bias, against the oracle's fp64 product (N = 1, one K block)."""
    if K % G:
        pytest.skip("K not a multiple of G")
    g = rng(M * 31 + G + N + K)
    w = synth.signs(g, (N, K))
    xb = synth.f32_to_bf16_bits(synth.normal_f32(g, (M, K)))
    q, s = B.bl_quantize_act_absmax_int8(bf16_gpu(xb))
    qo, so = O.quantize_act_absmax_int8(xb, "bf16")
    ws = synth.abs_normal_fp16_bits(g, (N, K // G), 0.02)
    bias = synth.f32_to_bf16_bits(synth.normal_f32(g, (N,)) * 0.1) if G == 128 else None
    y = B.bl_gemm_w1a8(q, s, B.bl_pack_w1(to_gpu(w)), fp16_gpu(ws), bf16_gpu(bias) if bias is not None else None,
                       group=G)
    _, yref, cond = O.gemm_w1a8(qo, so, O.pack_w1(w), ws, bias, K, G)
    assert_close(x_f64(bits16(y), "bf16"), yref, cond, tol_tc(TOL_BF16, K), "w1a8 tc M=%d G=%d %dx%d" % (M, G, N, K))


@pytest.mark.parametrize("M", [1, 4, 8])
def test_gemm_w1a8_workload_lmhead(B, M):
    """LM head 5120 -> 248320: the benchmark's launch (no dot output) and the
    launch that also writes the int32 group dots give the same y bit for bit
    on all rows; sampled rows' dots are bit-exact and their y within tolerance."""
    wl = synth.WORKLOADS["w1a8_lmhead_248320"]
    N, K, G = wl.N, wl.K, wl.group
    wq = torch.empty((N, K // 32), dtype=torch.int32, device="cuda")
    for b in range((N + synth.ROW_BLOCK - 1) // synth.ROW_BLOCK):
        blk = synth.weight_block(wl.index, "w", N, K, b, "signs")
        r0 = b * synth.ROW_BLOCK
        B.bl_pack_w1(to_gpu(blk), out=wq[r0:r0 + blk.shape[0]])
    ws = synth.block_scale_matrix(wl.index, N, K // G, tensor="group_scale")
    xb = synth.activations(wl.index, M, K, "bf16")
    q, s = O.quantize_act_absmax_int8(xb, "bf16")
    y = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, fp16_gpu(ws), group=G)
    # the verification launch with the int32 group dots, on every row
    y2, dots = B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, fp16_gpu(ws), group=G, group_dots=True)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "y must not depend on the dots output"
    yb = bits16(y)
    rows = np.unique(np.concatenate([[0, 1, N - 1, N - 2], rng(M).integers(0, N, 60)]))
    wrows = synth.weight_rows(wl.index, "w", N, K, rows, "signs")
    dref, yref, cond = O.gemm_w1a8(q, s, O.pack_w1(wrows), ws[rows], None, K, G)
    got = dots[:, torch.from_numpy(rows).cuda(), :].cpu().numpy().astype(np.int64)
    assert np.array_equal(got, dref), "group dots must be bit-exact"
    del dots
    assert_close(x_f64(yb[:, rows], "bf16"), yref, cond, TOL_BF16, "lm head M=%d" % M)


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 5, 8])
@pytest.mark.parametrize("G,N,K", [(32, 37, 256), (128, 100, 1024), (256, 300, 4096), (128, 129, 2560),
                                   (64, 45, 1280), (32, 20, 96)])
def test_gemm_w1a8_act_fused(B, xdt, M, G, N, K):
    """Act quantization fused into the W1A8 prologue: the same bits as the two
    calls, and the oracle's quantization followed by its product.  The first
    three shapes take the lane-per-row kernel, the others the tiled one."""
    g = rng(M * 7 + G + N + K + (xdt == "f32"))
    w = synth.signs(g, (N, K))
    x = synth.normal_f32(g, (M, K))
    if M > 1:
        x[1, :] = 0  # an all-zero token: s = 0 and q = 0
    if M > 2:
        x[2, 5] = -1000.0  # one outlier sets the token's absmax
    if xdt == "bf16":
        x = synth.f32_to_bf16_bits(x)
    ws = synth.abs_normal_fp16_bits(g, (N, K // G), 0.02)
    bias = synth.f32_to_bf16_bits(synth.normal_f32(g, (N,))) if M % 2 else None
    wq = B.bl_pack_w1(to_gpu(w))
    biasg = None if bias is None else bf16_gpu(bias)
    xg = x_gpu(x, xdt)
    y = B.bl_gemm_w1a8_act(xg, wq, fp16_gpu(ws), biasg, group=G)
    q, s = B.bl_quantize_act_absmax_int8(xg)
    y2 = B.bl_gemm_w1a8(q, s, wq, fp16_gpu(ws), biasg, group=G)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "fused must equal the two-call sequence"
    qo, so = O.quantize_act_absmax_int8(x, xdt)
    _, yref, cond = O.gemm_w1a8(qo, so, O.pack_w1(w), ws, bias, K, G)
    assert_close(x_f64(bits16(y), "bf16"), yref, cond, TOL_BF16, "w1a8 act M=%d G=%d %dx%d" % (M, G, N, K))


@pytest.mark.parametrize("M", [1, 8])
def test_gemm_w1a8_act_workload_lmhead(B, M):
    """LM head 5120 -> 248320 with fused quantization, sampled rows."""
    wl = synth.WORKLOADS["w1a8_lmhead_248320"]
    N, K, G = wl.N, wl.K, wl.group
    wq = torch.empty((N, K // 32), dtype=torch.int32, device="cuda")
    for b in range((N + synth.ROW_BLOCK - 1) // synth.ROW_BLOCK):
        blk = synth.weight_block(wl.index, "w", N, K, b, "signs")
        r0 = b * synth.ROW_BLOCK
        B.bl_pack_w1(to_gpu(blk), out=wq[r0:r0 + blk.shape[0]])
    ws = synth.block_scale_matrix(wl.index, N, K // G, tensor="group_scale")
    xb = synth.activations(wl.index, M, K, "bf16")
    y = B.bl_gemm_w1a8_act(bf16_gpu(xb), wq, fp16_gpu(ws), group=G)
    yb = bits16(y)
    q, s = O.quantize_act_absmax_int8(xb, "bf16")
    rows = np.unique(np.concatenate([[0, 1, N - 1, N - 2], rng(M + 5).integers(0, N, 60)]))
    wrows = synth.weight_rows(wl.index, "w", N, K, rows, "signs")
    _, yref, cond = O.gemm_w1a8(q, s, O.pack_w1(wrows), ws[rows], None, K, G)
    assert_close(x_f64(yb[:, rows], "bf16"), yref, cond, TOL_BF16, "lm head act M=%d" % M)


# ---------------------------------------------------------------------------
# i2_s x int8 (prefill)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (5, 70, 256), (63, 40, 512), (64, 7, 128), (128, 128, 1024),
                                   (130, 200, 2560), (512, 96, 384), (200, 1, 256), (129, 385, 12800)])
def test_gemm_i2s_int8_small(B, M, N, K):
    """M < 64 runs on the CUDA cores, M >= 64 on the tensor cores (one K block,
    N = 1, N % 4 != 0 with per-element stores, a ragged M tail, a long K)."""
    g = rng(M + N + K)
    w = ternary(g, N, K)
    q, s = O.quantize_act_absmax_int8(rand_x(g, K, "bf16", M), "bf16")
    sw = np.float32(g.uniform(0.5, 2))
    packed = B.bl_pack_i2s(to_gpu(w), sw)
    y, acc = B.bl_gemm_i2s_int8(to_gpu(q), to_gpu(s), packed, N, acc=True)
    aref, yref, cond = O.gemm_i2s_int8(q, s, O.pack_i2s(w, sw), N, K)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), aref), "accumulators must be bit-exact"
    assert_close(y.cpu().numpy(), yref, cond, TOL_F32, "prefill %dx%dx%d" % (M, N, K))


def test_gemm_i2s_int8_workload_prefill(B):
    """M=512, 2560 -> 6912: all accumulators of sampled columns bit-exact; y within tolerance."""
    wl = synth.WORKLOADS["i2s_prefill_512"]
    M, N, K = wl.M, wl.N, wl.K
    w = synth.weight_matrix(wl.index, "w", N, K, "ternary", wl.p_zero)
    sw = synth.tensor_scale(wl.index)
    q, s = O.quantize_act_absmax_int8(synth.activations(wl.index, M, K, "bf16"), "bf16")
    packed = B.bl_pack_i2s(to_gpu(w), sw)
    y, acc = B.bl_gemm_i2s_int8(to_gpu(q), to_gpu(s), packed, N, acc=True)
    y2 = B.bl_gemm_i2s_int8(to_gpu(q), to_gpu(s), packed, N)
    assert torch.equal(y, y2), "the y-only launch must match the launch that also writes acc"
    rows = np.unique(np.concatenate([[0, N - 1], rng(9).integers(0, N, 62)]))
    aref, yref, cond = O.gemm_i2s_int8(q, s, O.pack_i2s(w, sw), N, K, rows=rows)
    assert np.array_equal(acc.cpu().numpy()[:, rows].astype(np.int64), aref)
    assert_close(y.cpu().numpy()[:, rows], yref, cond, TOL_F32, "prefill workload")


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("xd", ["bf16", "f32"])
@pytest.mark.parametrize("M,N,K", [(64, 200, 1024), (130, 385, 2560), (512, 96, 384), (5, 70, 256), (200, 1, 256)])
def test_gemm_i2s_int8_act_fused(B, xd, M, N, K, fuse):
    """The prefill from unquantized x in one call, as two launches or with
    the quantization fused into the product's launch: the workspace's codes
    and scales equal bl_quantize_act_absmax_int8's, y equals the two-call
    bl_gemm_i2s_int8 bit for bit and the oracle within tolerance; a second
    call on the same workspace (its barrier words reset by the first) gives
    the same bits.  M < 64 always takes the two launches."""
    g = rng(17 * M + N + K + (xd == "f32"))
    w = ternary(g, N, K)
    x = synth.normal_f32(g, (M, K)) * g.uniform(0.1, 10, (M, 1)).astype(np.float32)
    x[1, :] = 0.0                      # an all-zero token
    if xd == "bf16":
        x = synth.f32_to_bf16_bits(x)
    xg = x_gpu(x, xd)
    sw = np.float32(1.5)
    packed = B.bl_pack_i2s(to_gpu(w), sw)
    ws = B.gemm_i2s_int8_act_workspace(M, K)
    y = B.bl_gemm_i2s_int8_act(xg, packed, N, workspace=ws, fuse=fuse)
    torch.cuda.synchronize()
    q, s = B.bl_quantize_act_absmax_int8(xg)
    qo = ws[256:256 + M * K].view(M, K).view(torch.int8)
    so_off = 256 + (M * K + 255) // 256 * 256
    so = ws[so_off:so_off + 4 * M].view(torch.float32)
    assert torch.equal(qo, q) and torch.equal(so.view(torch.int32), s.view(torch.int32))
    y2 = B.bl_gemm_i2s_int8(q, s, packed, N)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32)), "fused must equal the two-call sequence"
    y3 = B.bl_gemm_i2s_int8_act(xg, packed, N, workspace=ws, fuse=fuse)
    assert torch.equal(y.view(torch.int32), y3.view(torch.int32))
    qr, sr = O.quantize_act_absmax_int8(x, xd)
    aref, yref, cond = O.gemm_i2s_int8(qr, sr, O.pack_i2s(w, sw), N, K)
    assert_close(y.cpu().numpy(), yref, cond, TOL_F32, "prefill act %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("fuse", [False, True])
def test_gemm_i2s_int8_act_workload_prefill(B, fuse):
    """The prefill workload (512 tokens, 2560 -> 6912) from bf16 x in one
    call: y equals the two-call sequence bit for bit; sampled columns within tolerance."""
    wl = synth.WORKLOADS["i2s_prefill_512"]
    M, N, K = wl.M, wl.N, wl.K
    w = synth.weight_matrix(wl.index, "w", N, K, "ternary", wl.p_zero)
    sw = synth.tensor_scale(wl.index)
    xb = synth.activations(wl.index, M, K, "bf16")
    packed = B.bl_pack_i2s(to_gpu(w), sw)
    xg = bf16_gpu(xb)
    y = B.bl_gemm_i2s_int8_act(xg, packed, N, fuse=fuse)
    q, s = B.bl_quantize_act_absmax_int8(xg)
    assert torch.equal(y.view(torch.int32), B.bl_gemm_i2s_int8(q, s, packed, N).view(torch.int32))
    rows = np.unique(np.concatenate([[0, N - 1], rng(19).integers(0, N, 40)]))
    qr, sr = O.quantize_act_absmax_int8(xb, "bf16")
    _, yref, cond = O.gemm_i2s_int8(qr, sr, O.pack_i2s(w, sw), N, K, rows=rows)
    assert_close(y.cpu().numpy()[:, rows], yref, cond, TOL_F32, "prefill act workload")


# ---------------------------------------------------------------------------
# determinism, overlap switch, error paths
# ---------------------------------------------------------------------------

def test_repeated_calls_bitwise_identical(B):
    g = rng(99)
    N, K = 3000, 2560
    w = ternary(g, N, K)
    packed = B.bl_pack_i2s(to_gpu(w), 1.0)
    x = x_gpu(rand_x(g, K, "bf16"), "bf16")
    ys = [B.bl_gemv_i2s(packed, x, N, K) for _ in range(3)]
    assert all(torch.equal(ys[0].view(torch.int16), t.view(torch.int16)) for t in ys[1:])
    wb = synth.signs(g, (N, K))
    wq = B.bl_pack_w1(to_gpu(wb))
    q, s = O.quantize_act_absmax_int8(rand_x(g, K, "bf16", 4), "bf16")
    ws = fp16_gpu(synth.abs_normal_fp16_bits(g, (N, K // 128), 0.02))
    outs = [B.bl_gemm_w1a8(to_gpu(q), to_gpu(s), wq, ws) for _ in range(3)]
    assert all(torch.equal(outs[0].view(torch.int16), t.view(torch.int16)) for t in outs[1:])


def test_overlap_mode_same_results(B):
    """With programmatic dependent launch enabled, back-to-back products give the same bits."""
    g = rng(123)
    N, K = 6912, 2560
    w = ternary(g, N, K, 0.4)
    packed = B.bl_pack_i2s(to_gpu(w), 0.75)
    x = x_gpu(rand_x(g, K, "bf16"), "bf16")
    torch.cuda.synchronize()
    ref = B.bl_gemv_i2s(packed, x, N, K)
    B.set_overlap(True)
    try:
        outs = [B.bl_gemv_i2s(packed, x, N, K) for _ in range(4)]
    finally:
        B.set_overlap(False)
    torch.cuda.synchronize()
    assert all(torch.equal(ref.view(torch.int16), t.view(torch.int16)) for t in outs)


@pytest.mark.parametrize("xd,yd,N,K,fused", [("bf16", "bf16", 152 * 48, 8192, False),   # K split over 2-CTA clusters
                                             ("f32", "f32", 152 * 40, 8192, False)])
def test_wait_timeout_path(B, xd, yd, N, K, fused):
    """The bounded-wait failure path on the GPU: with a 1 ns pipeline wait
    limit, weight waits that are not satisfied at once give up: the launch
    completes, BL_DEVERR_WAIT_TIMEOUT is recorded and the device stays
    usable; with the default limit restored the same call is correct again.
    (Each CTA's rows here, about 100 KB streamed from HBM after an L2 flush,
    take longer to arrive than the activation records take to build, so its
    first weight check fails.)"""
    g = rng(31337 + K + fused)
    w = ternary(g, N, K)
    wu = ternary(g, N, K) if fused else None
    x = rand_x(g, K, xd)
    packed = B.bl_pack_i2s(to_gpu(w), np.float32(1.25))
    pu = B.bl_pack_i2s(to_gpu(wu), np.float32(0.75)) if fused else None
    xg = x_gpu(x, xd)
    yt = torch.float32 if yd == "f32" else torch.bfloat16
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    flush = torch.empty(2 * int(getattr(props, "L2_cache_size", 0) or (129 << 20)) // 4, dtype=torch.float32,
                        device="cuda")
    flush.zero_()  # the freshly packed weights leave L2
    del flush
    torch.cuda.synchronize()
    B.device_error(clear=True)
    B.set_wait_limit(1)
    try:
        if fused:
            B.bl_gemv_i2s_gate_up(packed, pu, xg, N, K, h_dtype=yt)
        else:
            B.bl_gemv_i2s(packed, xg, N, K, y_dtype=yt)
        torch.cuda.synchronize()
    finally:
        B.set_wait_limit(0)
    assert B.device_error(clear=True) & B.BL_DEVERR_WAIT_TIMEOUT
    if fused:
        h = B.bl_gemv_i2s_gate_up(packed, pu, xg, N, K, h_dtype=yt)
        hv = h.cpu().numpy().astype(np.float64) if yd == "f32" else x_f64(bits16(h), "bf16")
        ref, cond = O.gemv_i2s_gate_up(O.pack_i2s(w, np.float32(1.25)), O.pack_i2s(wu, np.float32(0.75)),
                                       x_f64(x, xd), N, K)
        assert_close(hv, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "after timeout (gate/up)")
    else:
        y, ref, cond = run_gemv_i2s(B, w, np.float32(1.25), x, xd, yd)
        assert_close(y, ref, cond, TOL_F32 if yd == "f32" else TOL_BF16, "after timeout")
    torch.cuda.synchronize()
    assert B.device_error(clear=True) == 0


def test_error_paths(B):
    x = torch.zeros(100, dtype=torch.float32, device="cuda")
    p = torch.zeros(1000, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.BLError) as e:
        B.bl_gemv_i2s(p, x, 4, 100)
    assert e.value.status == B.BL_ERR_SHAPE
    with pytest.raises(B.BLError) as e:
        B.bl_gemv_i2s(p[1:], x, 4, 128)
    assert e.value.status == B.BL_ERR_ALIGN
    with pytest.raises(B.BLError) as e:
        B.bl_gemv_i2s_gate_up(p, p[1:], x, 4, 128)
    assert e.value.status == B.BL_ERR_ALIGN
    with pytest.raises(B.BLError) as e:
        B.bl_gemv_i2s_gate_up(p, p, x, 4, 96)
    assert e.value.status == B.BL_ERR_SHAPE
    with pytest.raises(B.BLError) as e:
        B.bl_gemv_i2s_rmsnorm(p, x[:1].expand(128).contiguous()[1:], x, 4, 96)
    assert e.value.status == B.BL_ERR_SHAPE
    q = torch.zeros((9, 128), dtype=torch.int8, device="cuda")
    with pytest.raises(B.BLError) as e:
        B.bl_gemm_w1a8(q, torch.ones(9, device="cuda"), torch.zeros((4, 4), dtype=torch.int32, device="cuda"),
                       torch.zeros((4, 1), dtype=torch.float16, device="cuda"), group_dots=True)
    assert e.value.status == B.BL_ERR_UNSUPPORTED
