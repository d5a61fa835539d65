"""The C-ABI library builds, loads without a GPU, and exports every entry
point that include/bl.h declares (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bl.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(bl_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["bl_pack_i2s", "bl_pack_tq2_0", "bl_pack_w1", "bl_quantize_act_absmax_int8", "bl_gemv_i2s",
              "bl_gemv_tq2_0", "bl_gemm_w1a8", "bl_gemm_i2s_int8"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    from gemm_bl_gemv_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_lists_every_declared_symbol():
    from gemm_bl_gemv_gb300 import build
    build.build()
    from gemm_bl_gemv_gb300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


def test_host_checks_without_gpu():
    """Argument checks run before any CUDA call, so they work on a CPU-only box."""
    from gemm_bl_gemv_gb300 import build
    build.build()
    from gemm_bl_gemv_gb300 import binding as B
    L = B.lib()
    fake = ctypes.c_void_p(16 * 1024)  # never dereferenced: the checks fail first
    assert L.bl_gemv_i2s(None, fake, 0, fake, 0, 4, 128, None) == B.BL_ERR_NULL
    assert L.bl_gemv_i2s(fake, fake, 0, fake, 0, 4, 100, None) == B.BL_ERR_SHAPE
    assert L.bl_gemv_i2s(fake, fake, 7, fake, 0, 4, 128, None) == B.BL_ERR_DTYPE
    assert L.bl_gemv_i2s(ctypes.c_void_p(16 * 1024 + 8), fake, 0, fake, 0, 4, 128, None) == B.BL_ERR_ALIGN
    assert L.bl_gemv_tq2_0(fake, fake, 0, fake, 4, 128, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_w1a8(fake, fake, fake, fake, None, 9, 4, 128, 128, fake, fake, None) == B.BL_ERR_UNSUPPORTED
    assert L.bl_gemm_w1a8(fake, fake, fake, fake, None, 9, 4, 96, 32, fake, None, None) == B.BL_ERR_UNSUPPORTED
    assert L.bl_gemm_w1a8(fake, fake, fake, fake, None, 0, 4, 128, 128, fake, None, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_w1a8(fake, fake, fake, fake, None, 1, 4, 128, 48, fake, None, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_i2s_int8(fake, fake, fake, 4, 4, 132224, fake, None, None) == B.BL_ERR_UNSUPPORTED
    assert L.bl_gemm_w1a8_act(fake, 1, fake, fake, None, 9, 4, 1024, 128, fake, None) == B.BL_ERR_UNSUPPORTED
    assert L.bl_gemm_tq2_0_int8(fake, fake, fake, 4, 4, 384, fake, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_tq2_0_int8(fake, fake, fake, 0, 4, 256, fake, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_tq2_0_int8(None, fake, fake, 4, 4, 256, fake, None) == B.BL_ERR_NULL
    assert L.bl_gemm_tq2_0_int8(fake, fake, ctypes.c_void_p(16 * 1024 + 2), 4, 4, 256, fake, None) == B.BL_ERR_ALIGN
    assert L.bl_gemm_w1a8_act(fake, 1, fake, fake, None, 1, 4, 65536, 32, fake, None) == B.BL_ERR_UNSUPPORTED
    assert L.bl_gemm_w1a8_act(fake, 1, fake, fake, None, 1, 4, 1024, 48, fake, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_w1a8_act(fake, 5, fake, fake, None, 1, 4, 1024, 128, fake, None) == B.BL_ERR_DTYPE
    assert L.bl_gemm_w1a8_act(fake, 1, fake, fake, None, 0, 4, 1024, 128, fake, None) == B.BL_ERR_SHAPE
    assert L.bl_gemm_w1a8_act(None, 1, fake, fake, None, 1, 4, 1024, 128, fake, None) == B.BL_ERR_NULL
    assert L.bl_gemm_w1a8_act(ctypes.c_void_p(16 * 1024 + 4), 0, fake, fake, None, 1, 4, 1024, 128, fake,
                              None) == B.BL_ERR_ALIGN
    assert L.bl_pack_w1(fake, 4, 33, fake, None) == B.BL_ERR_SHAPE
    assert L.bl_quantize_act_absmax_int8(fake, 3, 1, 8, fake, fake, None) == B.BL_ERR_DTYPE
    assert b"K % 128" in L.bl_last_error() or b"bl_" in L.bl_last_error()
    assert L.bl_status_string(B.BL_ERR_ALIGN) == b"BL_ERR_ALIGN"


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No silent fallback: with libbl.so absent, importing the binding raises."""
    import shutil
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = tmp_path / "gemm_bl_gemv_gb300"
    pkg.mkdir()
    for f in ("__init__.py", "binding.py"):
        src = os.path.join(root, "gemm_bl_gemv_gb300", f)
        if os.path.exists(src):
            shutil.copy(src, pkg / f)
    r = subprocess.run([sys.executable, "-c", "import gemm_bl_gemv_gb300.binding"], cwd=str(tmp_path),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "ImportError" in r.stderr and "libbl.so" in r.stderr


def test_every_documented_rejection_without_gpu():
    """Each entry point's documented failure classes (include/bl.h), checked
    one by one on the host: a failing check returns its status before any CUDA
    call, so none of these touches a device."""
    from gemm_bl_gemv_gb300 import build
    build.build()
    from gemm_bl_gemv_gb300 import binding as B
    L = B.lib()
    A = 16 * 1024                # 16-byte aligned, never dereferenced
    P = ctypes.c_void_p
    a, o2, o4, o8 = P(A), P(A + 2), P(A + 4), P(A + 8)
    NULL, ERR, F32, BF16 = B.BL_ERR_NULL, B.BL_ERR_SHAPE, B.BL_F32, B.BL_BF16
    AL, DT, UN = B.BL_ERR_ALIGN, B.BL_ERR_DTYPE, B.BL_ERR_UNSUPPORTED
    cases = [
        # bl_device_error
        (L.bl_device_error, (None, 0), NULL),
        # packing
        (L.bl_pack_i2s, (None, 1.0, 4, 128, a, None), NULL),
        (L.bl_pack_i2s, (a, 1.0, 0, 128, a, None), ERR),
        (L.bl_pack_i2s, (a, 1.0, 4, 192, a, None), ERR),
        (L.bl_pack_i2s, (a, 1.0, 4, 128, o8, None), AL),
        (L.bl_pack_tq2_0, (a, None, 4, 256, a, None), NULL),
        (L.bl_pack_tq2_0, (a, a, 4, 384, a, None), ERR),
        (L.bl_pack_tq2_0, (a, P(A + 1), 4, 256, a, None), AL),
        (L.bl_pack_tq2_0, (a, a, 4, 256, P(A + 1), None), AL),
        (L.bl_pack_w1, (a, 4, 32, None, None), NULL),
        (L.bl_pack_w1, (a, 0, 32, a, None), ERR),
        (L.bl_pack_w1, (a, 4, 32, o2, None), AL),
        # act-quant
        (L.bl_quantize_act_absmax_int8, (a, F32, 1, 8, a, None, None), NULL),
        (L.bl_quantize_act_absmax_int8, (a, F32, 0, 8, a, a, None), ERR),
        (L.bl_quantize_act_absmax_int8, (a, F32, 1, 0, a, a, None), ERR),
        (L.bl_quantize_act_absmax_int8, (o2, F32, 1, 8, a, a, None), AL),
        (L.bl_quantize_act_absmax_int8, (a, BF16, 1, 8, a, o2, None), AL),
        # i2_s GEMV family
        (L.bl_gemv_i2s, (a, a, F32, a, 9, 4, 128, None), DT),
        (L.bl_gemv_i2s, (a, a, F32, a, F32, 0, 128, None), ERR),
        (L.bl_gemv_i2s, (a, a, F32, a, F32, 4, 32896, None), UN),
        (L.bl_gemv_i2s, (a, o2, F32, a, F32, 4, 128, None), AL),
        (L.bl_gemv_i2s_residual, (a, a, F32, None, a, F32, 4, 128, None), NULL),
        (L.bl_gemv_i2s_residual, (a, a, F32, o2, a, F32, 4, 128, None), AL),
        (L.bl_gemv_i2s_residual, (a, a, F32, a, a, F32, 4, 100, None), ERR),
        (L.bl_gemv_i2s_rmsnorm, (a, a, F32, None, 1e-6, None, a, F32, 4, 128, None), NULL),
        (L.bl_gemv_i2s_rmsnorm, (a, a, F32, a, -1.0, None, a, F32, 4, 128, None), ERR),
        (L.bl_gemv_i2s_rmsnorm, (a, a, F32, a, float("nan"), None, a, F32, 4, 128, None), ERR),
        (L.bl_gemv_i2s_rmsnorm, (a, a, BF16, P(A + 1), 1e-6, None, a, F32, 4, 128, None), AL),
        (L.bl_gemv_i2s_rmsnorm, (a, a, F32, a, 1e-6, o2, a, F32, 4, 128, None), AL),
        (L.bl_gemv_i2s_gate_up, (a, None, a, F32, a, F32, 4, 128, None), NULL),
        (L.bl_gemv_i2s_gate_up, (a, a, a, 2, a, F32, 4, 128, None), DT),
        (L.bl_gemv_i2s_gate_up, (a, a, a, F32, a, F32, 4, 65536, None), UN),
        (L.bl_gemv_i2s_gate_up, (a, o8, a, F32, a, F32, 4, 128, None), AL),
        # TQ2_0 GEMV
        (L.bl_gemv_tq2_0, (None, a, F32, a, 4, 256, None), NULL),
        (L.bl_gemv_tq2_0, (a, a, 3, a, 4, 256, None), DT),
        (L.bl_gemv_tq2_0, (a, a, F32, a, 4, 256 * 1025, None), UN),
        (L.bl_gemv_tq2_0, (a, a, F32, o2, 4, 256, None), AL),
        # W1A8
        (L.bl_gemm_w1a8, (a, a, a, a, None, 1, 4, 32 * 1025, 32, a, None, None), UN),
        (L.bl_gemm_w1a8, (a, a, a, a, None, 9, 4, 132224, 128, a, None, None), UN),
        (L.bl_gemm_w1a8, (a, a, a, a, None, 1, 0, 128, 128, a, None, None), ERR),
        (L.bl_gemm_w1a8, (a, a, a, a, None, 1, 4, 128, 96, a, None, None), ERR),
        (L.bl_gemm_w1a8, (o8, a, a, a, None, 1, 4, 128, 128, a, None, None), AL),
        (L.bl_gemm_w1a8, (a, a, a, o8, None, 1, 4, 128, 128, a, None, None), AL),
        (L.bl_gemm_w1a8, (a, a, a, a, P(A + 1), 1, 4, 128, 128, a, None, None), AL),
        (L.bl_gemm_w1a8, (a, None, a, a, None, 1, 4, 128, 128, a, None, None), NULL),
        (L.bl_gemm_w1a8_act, (a, F32, a, a, None, 1, 4, 128, 128, None, None), NULL),
        (L.bl_gemm_w1a8_act, (a, F32, a, a, None, 1, 4, 128, 128, P(A + 1), None), AL),
        # large-M products
        (L.bl_gemm_tq2_0_int8, (a, a, a, 4, 4, (1 << 24) + 256, a, None), UN),
        (L.bl_gemm_tq2_0_int8, (a, a, a, 4, 1 << 20, 1 << 16, a, None), UN),  # packed tensor >= 2 GiB
        (L.bl_gemm_tq2_0_int8, (a, o2, a, 4, 4, 256, a, None), AL),
        (L.bl_gemm_tq2_0_int8, (a, a, a, 4, 4, 256, o4, None), AL),
        (L.bl_gemm_i2s_int8, (a, a, None, 4, 4, 128, a, None, None), NULL),
        (L.bl_gemm_i2s_int8, (a, a, a, 64, 4, 131072 + 128, a, None, None), UN),  # 128 K > 2^24
        (L.bl_gemm_i2s_int8, (a, a, a, 4, 0, 128, a, None, None), ERR),
        (L.bl_gemm_i2s_int8, (a, a, a, 4, 4, 192, a, None, None), ERR),
        (L.bl_gemm_i2s_int8, (a, o4, a, 4, 4, 128, a, None, None), AL),
        (L.bl_gemm_i2s_int8, (a, a, a, 4, 4, 128, a, o4, None), AL),
        (L.bl_gemm_i2s_int8_act, (a, BF16, a, 4, 4, 128, a, None, 1 << 20, 0, None), NULL),
        (L.bl_gemm_i2s_int8_act, (a, 7, a, 4, 4, 128, a, a, 1 << 20, 0, None), DT),
        (L.bl_gemm_i2s_int8_act, (a, BF16, a, 4, 4, 192, a, a, 1 << 20, 0, None), ERR),
        (L.bl_gemm_i2s_int8_act, (a, BF16, a, 64, 4, 131072 + 128, a, a, 1 << 30, 0, None), UN),
        (L.bl_gemm_i2s_int8_act, (a, BF16, a, 4, 4, 128, a, a, 256, 0, None), ERR),    # workspace too small
        (L.bl_gemm_i2s_int8_act, (a, BF16, a, 4, 4, 128, a, P(A + 16), 1 << 20, 0, None), AL),
        (L.bl_gemm_i2s_int8_act, (P(A + 1), BF16, a, 4, 4, 128, a, a, 1 << 20, 0, None), AL),
    ]
    assert L.bl_gemm_i2s_int8_act_workspace(512, 2560) == 256 + 512 * 2560 + 2048
    assert L.bl_gemm_i2s_int8_act_workspace(0, 2560) == 0
    for fn, args, want in cases:
        got = fn(*args)
        assert got == want, (fn.__name__, args, B.status_name(got), B.status_name(want), L.bl_last_error())
        assert L.bl_last_error()  # every rejection leaves a message
