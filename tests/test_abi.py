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
