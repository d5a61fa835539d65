"""numpy front end of the C oracle (oracle/bl_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg; never by the product library.

All functions take and return numpy arrays.  bf16 and fp16 values travel as
their uint16 bit patterns.  Results of the products are fp64 (the exact
dot products, rounded once to fp64); ``cond`` is the matching sum of
absolute products, the scale used by the tolerance check.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def load(path):
    """Load an oracle shared library from `path` and declare its signatures."""
    L = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    sig = {
        "orc_set_threads": ([ctypes.c_int], ctypes.c_int),
        "orc_has_openmp": ([], ctypes.c_int),
        "orc_fp16_to_double": ([ctypes.c_uint16], ctypes.c_double),
        "orc_bf16_to_double": ([ctypes.c_uint16], ctypes.c_double),
        "orc_round_bf16": ([ctypes.c_double], ctypes.c_uint16),
        "orc_bf16_array_to_double": ([p, i64, p], None),
        "orc_fp16_array_to_double": ([p, i64, p], None),
        "orc_round_bf16_array": ([p, i64, p], None),
        "orc_i2s_packed_bytes": ([i64, i64], i64),
        "orc_pack_i2s": ([p, ctypes.c_float, i64, i64, p], ctypes.c_int),
        "orc_unpack_i2s": ([p, i64, i64, p, p], ctypes.c_int),
        "orc_gemv_i2s": ([p, p, i64, i64, p, i64, p, p], ctypes.c_int),
        "orc_gemv_i2s_gate_up": ([p, p, p, i64, i64, p, i64, p, p], ctypes.c_int),
        "orc_gemv_i2s_norm_residual": ([p, p, p, ctypes.c_double, p, i64, i64, p, i64, p, p], ctypes.c_int),
        "orc_gemm_i2s_int8": ([p, p, p, i64, i64, i64, p, i64, p, p, p], ctypes.c_int),
        "orc_tq2_0_packed_bytes": ([i64, i64], i64),
        "orc_pack_tq2_0": ([p, p, i64, i64, p], ctypes.c_int),
        "orc_unpack_tq2_0": ([p, i64, i64, p, p], ctypes.c_int),
        "orc_gemv_tq2_0": ([p, p, i64, i64, p, i64, p, p], ctypes.c_int),
        "orc_gemm_tq2_0_int8": ([p, p, p, i64, i64, i64, p, i64, p, p], ctypes.c_int),
        "orc_pack_w1": ([p, i64, i64, p], ctypes.c_int),
        "orc_unpack_w1": ([p, i64, i64, p], ctypes.c_int),
        "orc_gemm_w1a8": ([p, p, p, p, p, i64, i64, i64, i64, p, i64, p, p, p], ctypes.c_int),
        "orc_quantize_act_absmax_int8": ([p, p, i64, i64, p, p], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(_build.build())
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise OracleError("%s failed with %d" % (what, rc))


def _rows(rows, N):
    if rows is None:
        return None, N
    r = _c(rows, np.int64)
    return r, r.shape[0]


def set_threads(n: int) -> int:
    return lib().orc_set_threads(int(n))


def has_openmp() -> bool:
    return bool(lib().orc_has_openmp())


# ---- scalar formats -------------------------------------------------------

def bf16_to_f64(bits):
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().orc_bf16_array_to_double(_ptr(b), b.size, _ptr(out))
    return out


def fp16_to_f64(bits):
    h = _c(bits, np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().orc_fp16_array_to_double(_ptr(h), h.size, _ptr(out))
    return out


def round_bf16(x):
    d = _c(x, np.float64)
    out = np.empty(d.shape, np.uint16)
    lib().orc_round_bf16_array(_ptr(d), d.size, _ptr(out))
    return out


# ---- i2_s ------------------------------------------------------------------

def pack_i2s(w, scale):
    w = _c(w, np.int8)
    N, K = w.shape
    out = np.zeros(lib().orc_i2s_packed_bytes(N, K), np.uint8)
    _check(lib().orc_pack_i2s(_ptr(w), ctypes.c_float(scale), N, K, _ptr(out)), "pack_i2s")
    return out


def unpack_i2s(packed, N, K):
    p = _c(packed, np.uint8)
    w = np.empty((N, K), np.int8)
    s = ctypes.c_float()
    _check(lib().orc_unpack_i2s(_ptr(p), N, K, _ptr(w), ctypes.byref(s)), "unpack_i2s")
    return w, s.value


def gemv_i2s(packed, x, N, K, rows=None):
    p = _c(packed, np.uint8)
    x = _c(x, np.float64)
    r, nr = _rows(rows, N)
    y = np.empty(nr, np.float64)
    c = np.empty(nr, np.float64)
    _check(lib().orc_gemv_i2s(_ptr(p), _ptr(x), N, K, _ptr(r), nr, _ptr(y), _ptr(c)), "gemv_i2s")
    return y, c


def gemv_i2s_gate_up(packed_gate, packed_up, x, N, K, rows=None):
    """h = max(0, g)^2 * u with g, u the two i2_s GEMVs; returns (h, cond)."""
    pg = _c(packed_gate, np.uint8)
    pu = _c(packed_up, np.uint8)
    x = _c(x, np.float64)
    r, nr = _rows(rows, N)
    h = np.empty(nr, np.float64)
    c = np.empty(nr, np.float64)
    _check(lib().orc_gemv_i2s_gate_up(_ptr(pg), _ptr(pu), _ptr(x), N, K, _ptr(r), nr, _ptr(h), _ptr(c)),
           "gemv_i2s_gate_up")
    return h, c


def gemv_i2s_norm_residual(packed, x, N, K, rms_w=None, eps=1e-5, residual=None, rows=None):
    """y = residual + scale * W (x * rmsInv * rms_w)  (RMSNorm only when rms_w is given,
    residual 0 when None); returns (y, cond)."""
    p = _c(packed, np.uint8)
    x = _c(x, np.float64)
    w = None if rms_w is None else _c(rms_w, np.float64)
    res = None if residual is None else _c(residual, np.float64)
    r, nr = _rows(rows, N)
    y = np.empty(nr, np.float64)
    c = np.empty(nr, np.float64)
    _check(lib().orc_gemv_i2s_norm_residual(_ptr(p), _ptr(x), _ptr(w) if w is not None else None, float(eps),
                                            _ptr(res) if res is not None else None, N, K, _ptr(r), nr, _ptr(y),
                                            _ptr(c)), "gemv_i2s_norm_residual")
    return y, c


def gemm_i2s_int8(q, s_act, packed, N, K, rows=None):
    q = _c(q, np.int8)
    M = q.shape[0]
    s = _c(s_act, np.float32)
    p = _c(packed, np.uint8)
    r, nr = _rows(rows, N)
    acc = np.empty((M, nr), np.int64)
    y = np.empty((M, nr), np.float64)
    c = np.empty((M, nr), np.float64)
    _check(lib().orc_gemm_i2s_int8(_ptr(q), _ptr(s), _ptr(p), M, N, K, _ptr(r), nr, _ptr(acc), _ptr(y), _ptr(c)),
           "gemm_i2s_int8")
    return acc, y, c


# ---- TQ2_0 -----------------------------------------------------------------

def pack_tq2_0(w, d_bits):
    w = _c(w, np.int8)
    N, K = w.shape
    d = _c(d_bits, np.uint16)
    out = np.zeros(lib().orc_tq2_0_packed_bytes(N, K), np.uint8)
    _check(lib().orc_pack_tq2_0(_ptr(w), _ptr(d), N, K, _ptr(out)), "pack_tq2_0")
    return out


def unpack_tq2_0(packed, N, K):
    p = _c(packed, np.uint8)
    w = np.empty((N, K), np.int8)
    d = np.empty((N, K // 256), np.uint16)
    _check(lib().orc_unpack_tq2_0(_ptr(p), N, K, _ptr(w), _ptr(d)), "unpack_tq2_0")
    return w, d


def gemv_tq2_0(packed, x, N, K, rows=None):
    p = _c(packed, np.uint8)
    x = _c(x, np.float64)
    r, nr = _rows(rows, N)
    y = np.empty(nr, np.float64)
    c = np.empty(nr, np.float64)
    _check(lib().orc_gemv_tq2_0(_ptr(p), _ptr(x), N, K, _ptr(r), nr, _ptr(y), _ptr(c)), "gemv_tq2_0")
    return y, c


def gemm_tq2_0_int8(q, s_act, packed, N, K, rows=None):
    """y[m, r] = s_m * sum_b d[n,b] * (exact block dot of w and q); returns (y, cond), [M, nrows]."""
    q = _c(q, np.int8)
    M = q.shape[0]
    s = _c(s_act, np.float32)
    p = _c(packed, np.uint8)
    r, nr = _rows(rows, N)
    y = np.empty((M, nr), np.float64)
    c = np.empty((M, nr), np.float64)
    _check(lib().orc_gemm_tq2_0_int8(_ptr(q), _ptr(s), _ptr(p), M, N, K, _ptr(r), nr, _ptr(y), _ptr(c)),
           "gemm_tq2_0_int8")
    return y, c


# ---- W1A8 ------------------------------------------------------------------

def pack_w1(w):
    w = _c(w, np.int8)
    N, K = w.shape
    out = np.empty((N, K // 32), np.int32)
    _check(lib().orc_pack_w1(_ptr(w), N, K, _ptr(out)), "pack_w1")
    return out


def unpack_w1(wq, K):
    wq = _c(wq, np.int32)
    N = wq.shape[0]
    w = np.empty((N, K), np.int8)
    _check(lib().orc_unpack_w1(_ptr(wq), N, K, _ptr(w)), "unpack_w1")
    return w


def gemm_w1a8(q, s_act, wq, ws_bits, bias_bits, K, group, rows=None):
    q = _c(q, np.int8)
    M = q.shape[0]
    s = _c(s_act, np.float32)
    wq = _c(wq, np.int32)
    N = wq.shape[0]
    ws = _c(ws_bits, np.uint16)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    r, nr = _rows(rows, N)
    ng = K // group
    dots = np.empty((M, nr, ng), np.int64)
    y = np.empty((M, nr), np.float64)
    c = np.empty((M, nr), np.float64)
    _check(lib().orc_gemm_w1a8(_ptr(q), _ptr(s), _ptr(wq), _ptr(ws), _ptr(b), M, N, K, group, _ptr(r), nr,
                               _ptr(dots), _ptr(y), _ptr(c)), "gemm_w1a8")
    return dots, y, c


# ---- activation quantization --------------------------------------------------

def quantize_act_absmax_int8(x, dtype):
    """x: float32 array [M,K] (dtype 'f32') or uint16 bf16 bits [M,K] (dtype 'bf16')."""
    if dtype == "f32":
        x32, x16 = _c(x, np.float32), None
    elif dtype == "bf16":
        x32, x16 = None, _c(x, np.uint16)
    else:
        raise ValueError(dtype)
    src = x32 if x32 is not None else x16
    M, K = src.shape
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    _check(lib().orc_quantize_act_absmax_int8(_ptr(x32), _ptr(x16), M, K, _ptr(q), _ptr(s)), "quantize_act")
    return q, s
