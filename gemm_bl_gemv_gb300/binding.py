"""Thin Python binding of libbl (include/bl.h) for torch CUDA tensors.

Argument marshalling only: every function checks tensor dtypes/devices,
allocates outputs with torch when none are given, and calls the C entry
point of the same name on the current CUDA stream.  All computation happens
in the library's kernels; there is no fallback.  A missing libbl.so raises
ImportError (build it with gemm_bl_gemv_gb300.build.build()).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbl.so")

BL_OK, BL_ERR_NULL, BL_ERR_SHAPE, BL_ERR_ALIGN, BL_ERR_DTYPE, BL_ERR_UNSUPPORTED, BL_ERR_CUDA = range(7)
BL_F32, BL_BF16 = 0, 1
BL_DEVERR_WAIT_TIMEOUT = 0x1
BL_DEVERR_RANGE = 0x2

EXPORTS = [
    "bl_status_string", "bl_last_error", "bl_device_error", "bl_set_overlap", "bl_get_overlap", "bl_set_wait_limit",
    "bl_pack_i2s", "bl_pack_tq2_0", "bl_pack_w1", "bl_quantize_act_absmax_int8",
    "bl_gemv_i2s", "bl_gemv_i2s_residual", "bl_gemv_i2s_rmsnorm", "bl_gemv_i2s_gate_up", "bl_gemv_tq2_0", "bl_gemm_w1a8", "bl_gemm_w1a8_act", "bl_gemm_i2s_int8",
    "bl_gemm_tq2_0_int8", "bl_gemm_i2s_int8_act", "bl_gemm_i2s_int8_act_workspace",
    "bl_gemm_i2s_int8_act_noalloc",
]


class BLError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (status_name(status), message))
        self.status = status


def _declare(L):
    p, i64, i32, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int
    sig = {
        "bl_status_string": ([st], ctypes.c_char_p),
        "bl_last_error": ([], ctypes.c_char_p),
        "bl_device_error": ([p, i32], st),
        "bl_set_overlap": ([i32], None),
        "bl_get_overlap": ([], i32),
        "bl_set_wait_limit": ([ctypes.c_uint64], st),
        "bl_pack_i2s": ([p, ctypes.c_float, i64, i64, p, p], st),
        "bl_pack_tq2_0": ([p, p, i64, i64, p, p], st),
        "bl_pack_w1": ([p, i64, i64, p, p], st),
        "bl_quantize_act_absmax_int8": ([p, i32, i64, i64, p, p, p], st),
        "bl_gemv_i2s": ([p, p, i32, p, i32, i64, i64, p], st),
        "bl_gemv_i2s_gate_up": ([p, p, p, i32, p, i32, i64, i64, p], st),
        "bl_gemv_i2s_residual": ([p, p, i32, p, p, i32, i64, i64, p], st),
        "bl_gemv_i2s_rmsnorm": ([p, p, i32, p, ctypes.c_float, p, p, i32, i64, i64, p], st),
        "bl_gemv_tq2_0": ([p, p, i32, p, i64, i64, p], st),
        "bl_gemm_w1a8": ([p, p, p, p, p, i64, i64, i64, i32, p, p, p], st),
        "bl_gemm_w1a8_act": ([p, i32, p, p, p, i64, i64, i64, i32, p, p], st),
        "bl_gemm_i2s_int8": ([p, p, p, i64, i64, i64, p, p, p], st),
        "bl_gemm_tq2_0_int8": ([p, p, p, i64, i64, i64, p, p], st),
        "bl_gemm_i2s_int8_act": ([p, i32, p, i64, i64, i64, p, p, ctypes.c_size_t, i32, p], st),
        "bl_gemm_i2s_int8_act_workspace": ([i64, i64], ctypes.c_size_t),
        "bl_gemm_i2s_int8_act_noalloc": ([p, i32, p, i64, i64, i64, p, i32, p], st),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libbl.so not built at %s; run gemm_bl_gemv_gb300.build.build()" % LIB_PATH)
    return _declare(ctypes.CDLL(LIB_PATH))


_lib = _load()


def lib():
    return _lib


def status_name(s):
    return _lib.bl_status_string(s).decode()


def _check(status):
    if status != BL_OK:
        raise BLError(status, _lib.bl_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return BL_F32
    if t.dtype == torch.bfloat16:
        return BL_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _cuda(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


_cudart = None


def cudart():
    """The CUDA runtime libbl.so is linked against (same process-wide library),
    with cudaMemcpyAsync declared, for callers that drive the C ABI directly."""
    global _cudart
    if _cudart is None:
        rt = ctypes.CDLL("libcudart.so.13")
        rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        rt.cudaMemcpyAsync.restype = ctypes.c_int
        _cudart = rt
    return _cudart


CUDA_MEMCPY_H2D, CUDA_MEMCPY_D2H = 1, 2


def set_overlap(enable: bool):
    _lib.bl_set_overlap(1 if enable else 0)


def get_overlap() -> bool:
    return bool(_lib.bl_get_overlap())


def set_wait_limit(ns: int):
    """Pipeline waits of later launches give up after ns nanoseconds (0: the default second); test aid."""
    _check(_lib.bl_set_wait_limit(int(ns)))


def device_error(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib.bl_device_error(ctypes.byref(v), 1 if clear else 0))
    return v.value


# ---- packing ---------------------------------------------------------------

def i2s_packed_bytes(N, K):
    return N * (K // 4) + 4


def tq2_0_packed_bytes(N, K):
    return N * (K // 256) * 66


def bl_pack_i2s(w, scale, out=None, stream=None):
    _cuda(w, "w")
    N, K = w.shape
    if out is None:
        out = torch.empty(i2s_packed_bytes(N, K), dtype=torch.uint8, device=w.device)
    _check(_lib.bl_pack_i2s(_ptr(w), ctypes.c_float(float(scale)), N, K, _ptr(_cuda(out, "out")), _stream(stream)))
    return out


def bl_pack_tq2_0(w, d_fp16_bits, out=None, stream=None):
    _cuda(w, "w")
    _cuda(d_fp16_bits, "d")
    N, K = w.shape
    if out is None:
        out = torch.empty(tq2_0_packed_bytes(N, K), dtype=torch.uint8, device=w.device)
    _check(_lib.bl_pack_tq2_0(_ptr(w), _ptr(d_fp16_bits), N, K, _ptr(_cuda(out, "out")), _stream(stream)))
    return out


def bl_pack_w1(w, out=None, stream=None):
    _cuda(w, "w")
    N, K = w.shape
    if out is None:
        out = torch.empty((N, K // 32), dtype=torch.int32, device=w.device)
    _check(_lib.bl_pack_w1(_ptr(w), N, K, _ptr(_cuda(out, "out")), _stream(stream)))
    return out


# ---- activation quantization -------------------------------------------------

def bl_quantize_act_absmax_int8(x, q=None, s=None, stream=None):
    _cuda(x, "x")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if s is None:
        s = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(_lib.bl_quantize_act_absmax_int8(_ptr(x), _dtype_code(x), M, K, _ptr(_cuda(q, "q")), _ptr(_cuda(s, "s")),
                                            _stream(stream)))
    return q, s


# ---- products --------------------------------------------------------------

def bl_gemv_i2s(packed, x, N, K, y=None, y_dtype=None, stream=None):
    _cuda(packed, "packed")
    _cuda(x, "x")
    if y is None:
        y = torch.empty(N, dtype=y_dtype or x.dtype, device=x.device)
    _check(_lib.bl_gemv_i2s(_ptr(packed), _ptr(x), _dtype_code(x), _ptr(_cuda(y, "y")), _dtype_code(y), N, K,
                            _stream(stream)))
    return y


def bl_gemv_i2s_residual(packed, x, residual, N, K, y=None, stream=None):
    """y = residual + scale * W x (y and residual share a dtype)."""
    _cuda(packed, "packed")
    _cuda(x, "x")
    _cuda(residual, "residual")
    if y is None:
        y = torch.empty(N, dtype=residual.dtype, device=x.device)
    if y.dtype != residual.dtype:
        raise TypeError("y and residual must share a dtype")
    _check(_lib.bl_gemv_i2s_residual(_ptr(packed), _ptr(x), _dtype_code(x), _ptr(residual), _ptr(_cuda(y, "y")),
                                     _dtype_code(y), N, K, _stream(stream)))
    return y


def bl_gemv_i2s_rmsnorm(packed, x, rms_weight, N, K, eps=1e-5, residual=None, y=None, y_dtype=None, stream=None):
    """y = residual + scale * W (x * rmsInv * rms_weight), rmsInv = 1/sqrt(mean(x^2) + eps)."""
    _cuda(packed, "packed")
    _cuda(x, "x")
    _cuda(rms_weight, "rms_weight")
    if rms_weight.dtype != x.dtype:
        raise TypeError("rms_weight must have x's dtype")
    if y is None:
        y = torch.empty(N, dtype=(residual.dtype if residual is not None else (y_dtype or x.dtype)), device=x.device)
    if residual is not None:
        _cuda(residual, "residual")
        if residual.dtype != y.dtype:
            raise TypeError("y and residual must share a dtype")
    _check(_lib.bl_gemv_i2s_rmsnorm(_ptr(packed), _ptr(x), _dtype_code(x), _ptr(rms_weight), float(eps),
                                    _ptr(residual) if residual is not None else None, _ptr(_cuda(y, "y")),
                                    _dtype_code(y), N, K, _stream(stream)))
    return y


def bl_gemv_i2s_gate_up(packed_gate, packed_up, x, N, K, h=None, h_dtype=None, stream=None):
    """h = max(0, scale_g * W_g x)^2 * (scale_u * W_u x), one token."""
    _cuda(packed_gate, "packed_gate")
    _cuda(packed_up, "packed_up")
    _cuda(x, "x")
    if h is None:
        h = torch.empty(N, dtype=h_dtype or x.dtype, device=x.device)
    _check(_lib.bl_gemv_i2s_gate_up(_ptr(packed_gate), _ptr(packed_up), _ptr(x), _dtype_code(x), _ptr(_cuda(h, "h")),
                                    _dtype_code(h), N, K, _stream(stream)))
    return h


def bl_gemv_tq2_0(packed, x, N, K, y=None, stream=None):
    _cuda(packed, "packed")
    _cuda(x, "x")
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=x.device)
    _check(_lib.bl_gemv_tq2_0(_ptr(packed), _ptr(x), _dtype_code(x), _ptr(_cuda(y, "y")), N, K, _stream(stream)))
    return y


def bl_gemm_w1a8(q, s, wq, ws_fp16_bits, bias_bf16_bits=None, group=128, y=None, group_dots=False, stream=None):
    for t, n in ((q, "q"), (s, "s"), (wq, "wq"), (ws_fp16_bits, "ws")):
        _cuda(t, n)
    M, K = q.shape
    N = wq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=q.device)
    dots = None
    if group_dots is True:
        dots = torch.empty((M, N, K // group), dtype=torch.int32, device=q.device)
    elif isinstance(group_dots, torch.Tensor):
        dots = group_dots
    _check(_lib.bl_gemm_w1a8(_ptr(q), _ptr(s), _ptr(wq), _ptr(ws_fp16_bits), _ptr(bias_bf16_bits), M, N, K, group,
                             _ptr(_cuda(y, "y")), _ptr(dots), _stream(stream)))
    return (y, dots) if dots is not None else y


def bl_gemm_w1a8_act(x, wq, ws_fp16_bits, bias_bf16_bits=None, group=128, y=None, stream=None):
    """bl_quantize_act_absmax_int8(x) then bl_gemm_w1a8, in one launch (M <= 8)."""
    for t, n in ((x, "x"), (wq, "wq"), (ws_fp16_bits, "ws")):
        _cuda(t, n)
    M, K = x.shape
    N = wq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(_lib.bl_gemm_w1a8_act(_ptr(x), _dtype_code(x), _ptr(wq), _ptr(ws_fp16_bits), _ptr(bias_bf16_bits), M, N, K,
                                 group, _ptr(_cuda(y, "y")), _stream(stream)))
    return y


def gemm_i2s_int8_act_workspace(M, K, device="cuda"):
    """A zero-filled workspace for bl_gemm_i2s_int8_act (uint8, 256-byte aligned by the allocator)."""
    n = int(_lib.bl_gemm_i2s_int8_act_workspace(int(M), int(K)))
    return torch.zeros(n, dtype=torch.uint8, device=device)


def bl_gemm_i2s_int8_act(x, packed, N, workspace=None, y=None, fuse=False, stream=None):
    """bl_quantize_act_absmax_int8(x) then bl_gemm_i2s_int8 in one call (fuse: one launch where it fits)."""
    for t, n in ((x, "x"), (packed, "packed")):
        _cuda(t, n)
    M, K = x.shape
    if workspace is None:
        workspace = gemm_i2s_int8_act_workspace(M, K, x.device)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(_lib.bl_gemm_i2s_int8_act(_ptr(x), _dtype_code(x), _ptr(packed), M, N, K, _ptr(_cuda(y, "y")),
                                     _ptr(workspace), workspace.numel(), 1 if fuse else 0, _stream(stream)))
    return y


def bl_gemm_i2s_int8(q, s, packed, N, y=None, acc=False, stream=None):
    for t, n in ((q, "q"), (s, "s"), (packed, "packed")):
        _cuda(t, n)
    M, K = q.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=q.device)
    a = None
    if acc is True:
        a = torch.empty((M, N), dtype=torch.int32, device=q.device)
    elif isinstance(acc, torch.Tensor):
        a = acc
    _check(_lib.bl_gemm_i2s_int8(_ptr(q), _ptr(s), _ptr(packed), M, N, K, _ptr(_cuda(y, "y")), _ptr(a),
                                 _stream(stream)))
    return (y, a) if a is not None else y


def bl_gemm_tq2_0_int8(q, s, packed, N, y=None, stream=None):
    """y[m, n] = s[m] * sum_b d[n,b] * (block dot of w and q), fp32 [M, N]."""
    for t, n in ((q, "q"), (s, "s"), (packed, "packed")):
        _cuda(t, n)
    M, K = q.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=q.device)
    _check(_lib.bl_gemm_tq2_0_int8(_ptr(q), _ptr(s), _ptr(packed), M, N, K, _ptr(_cuda(y, "y")), _stream(stream)))
    return y
