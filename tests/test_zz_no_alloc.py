"""The allocation-free prefill entry point (bl_gemm_i2s_int8_act_noalloc),
for callers that cannot allocate device memory: code handed only its input
and output pointers by a host program that owns all device memory, or a loop
that must not call cudaMalloc.  Called through the C ABI, its output must
equal that of bl_gemm_i2s_int8_act with a caller workspace, on two calls in a
row with different inputs (the static workspace keeps the previous call's
contents), in both the two-launch and the single-launch form; a shape whose
workspace exceeds the static array is refused before any launch.

This file is collected last, so a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from gemm_bl_gemv_gb300 import synth
from oracle import oracle as O
from parity import TOL_F32, assert_close, bf16_gpu, to_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from gemm_bl_gemv_gb300 import build
    build.build()
    from gemm_bl_gemv_gb300 import binding
    binding.device_error(clear=True)
    yield binding
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0


def noalloc(B, x, packed, N, y, fuse):
    M, K = x.shape
    L = B.lib()
    st = L.bl_gemm_i2s_int8_act_noalloc(ctypes.c_void_p(x.data_ptr()), B.BL_BF16, ctypes.c_void_p(packed.data_ptr()),
                                        M, N, K, ctypes.c_void_p(y.data_ptr()), 1 if fuse else 0,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.BL_OK, L.bl_last_error().decode()


@pytest.mark.parametrize("fuse", [False, True])
def test_noalloc_matches_workspace_entry_point(B, fuse):
    M, N, K = 512, 6912, 2560
    g = np.random.Generator(np.random.PCG64(20261203 + fuse))
    w = synth.ternary(g, (N, K), 0.4)
    packed = B.bl_pack_i2s(to_gpu(w), np.float32(0.8))
    for call in range(2):
        xb = synth.f32_to_bf16_bits(synth.normal_f32(g, (M, K)) * np.float32(1 + 3 * call))
        xg = bf16_gpu(xb)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        noalloc(B, xg, packed, N, y, fuse)
        ref = B.bl_gemm_i2s_int8_act(xg, packed, N, fuse=fuse)
        torch.cuda.synchronize()
        qr, sr = O.quantize_act_absmax_int8(xb, "bf16")
        cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 24)]))
        _, _, cond = O.gemm_i2s_int8(qr, sr, O.pack_i2s(w, np.float32(0.8)), N, K, rows=cols)
        yc = y.cpu().numpy()[:, cols].astype(np.float64)
        rc = ref.cpu().numpy()[:, cols].astype(np.float64)
        assert_close(yc, rc, cond, TOL_F32, "no-alloc call %d" % call)
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), "the same arithmetic gives the same bits"


def test_noalloc_refuses_a_shape_beyond_the_static_workspace(B):
    L = B.lib()
    x = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    M, K = 4096, 4096  # 16 MiB of codes
    st = L.bl_gemm_i2s_int8_act_noalloc(ctypes.c_void_p(x.data_ptr()), B.BL_BF16, ctypes.c_void_p(x.data_ptr()), M, 128,
                                        K, ctypes.c_void_p(x.data_ptr()), 0, None)
    assert st == B.BL_ERR_UNSUPPORTED
    assert b"static" in L.bl_last_error()
