"""Seeded synthetic inputs for the packed BitLinear workloads.

This module only draws random tensors of the workloads' shapes and value
distributions.  It holds none of the method's arithmetic: no packing, no
decoding, no products, no quantization.  Both the CUDA path (through the
library's pack kernels) and the CPU oracle (through its own packers) start
from these unpacked tensors.

Seeding: numpy ``Generator(PCG64)``.  Each tensor of each workload has its own
stream, and large matrices are drawn in row blocks of ``ROW_BLOCK`` rows, each
from its own stream, so any subset of rows can be regenerated without drawing
the whole matrix (the oracle checks sampled rows of the 248320-row LM head
this way).
"""
from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np

SEED_BASE = 20261202
ROW_BLOCK = 1024

_TENSOR_IDS = {"w": 1, "x": 2, "scale": 3, "block_scale": 4, "group_scale": 5, "bias": 6,
               "w_gate": 11, "w_up": 12, "w_down": 13, "x_down": 14,
               "scale_gate": 15, "scale_up": 16, "scale_down": 17}


def rng(workload_index: int, tensor: str, block: Optional[int] = None) -> np.random.Generator:
    key = (_TENSOR_IDS[tensor],) if block is None else (_TENSOR_IDS[tensor], 1 + int(block))
    ss = np.random.SeedSequence(SEED_BASE + int(workload_index), spawn_key=key)
    return np.random.Generator(np.random.PCG64(ss))


def ternary(g: np.random.Generator, shape, p_zero: float) -> np.ndarray:
    """i.i.d. values in {-1,0,+1}: P(0) = p_zero, P(-1) = P(+1) = (1-p_zero)/2."""
    p = (1.0 - p_zero) / 2.0
    return g.choice(np.array([-1, 0, 1], np.int8), size=shape, p=[p, p_zero, p])


def signs(g: np.random.Generator, shape) -> np.ndarray:
    """i.i.d. values in {-1,+1} with probability 1/2 each."""
    return (g.integers(0, 2, size=shape, dtype=np.int8) * 2 - 1).astype(np.int8)


def normal_f32(g: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)).astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return bit patterns.

    Used only to draw bf16-valued inputs (x ~ N(0,1) stored as bf16).
    """
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    return ((u + bias) >> 16).astype(np.uint16)


def abs_normal_fp16_bits(g: np.random.Generator, shape, sigma: float) -> np.ndarray:
    """|N(0, sigma)| rounded to float16 (numpy's conversion); return bit patterns."""
    v = np.abs(g.standard_normal(size=shape)) * sigma
    return v.astype(np.float16).view(np.uint16)


def uniform_f32(g: np.random.Generator, lo: float, hi: float, shape=None):
    v = g.uniform(lo, hi, size=shape)
    return np.float32(v) if shape is None else v.astype(np.float32)


# ---------------------------------------------------------------------------
# Workloads (shapes and distributions)
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    fmt: str               # "i2s", "tq2_0", "w1a8", "i2s_int8"
    M: int
    N: int
    K: int
    x_dtype: str           # "f32" or "bf16"
    y_dtype: str           # "f32" or "bf16"
    p_zero: float = 1.0 / 3.0
    group: int = 128
    extra: Dict[str, Tuple[int, int]] = field(default_factory=dict)


# The five workloads: index = seed offset.
WORKLOADS = {
    "i2s_gemv_2560": Workload(0, "i2s_gemv_2560", "i2s", 1, 2560, 2560, "f32", "f32"),
    # BitNet-2B-shaped MLP: gate and up 2560 -> 6912, down 6912 -> 2560.
    "i2s_mlp_bitnet2b": Workload(1, "i2s_mlp_bitnet2b", "i2s", 1, 6912, 2560, "bf16", "bf16", p_zero=0.4,
                                 extra={"gate": (6912, 2560), "up": (6912, 2560), "down": (2560, 6912)}),
    "tq2_0_gemv_5120x13824": Workload(2, "tq2_0_gemv_5120x13824", "tq2_0", 1, 13824, 5120, "bf16", "f32"),
    "w1a8_lmhead_248320": Workload(3, "w1a8_lmhead_248320", "w1a8", 8, 248320, 5120, "bf16", "bf16"),
    "i2s_prefill_512": Workload(4, "i2s_prefill_512", "i2s_int8", 512, 6912, 2560, "bf16", "f32"),
}


def weight_rows(workload_index: int, tensor: str, N: int, K: int, rows, kind: str, p_zero: float = 1.0 / 3.0):
    """Rows `rows` (sorted or not) of the [N,K] weight matrix `tensor` of a workload.

    kind: "ternary" (with p_zero) or "signs".  Rows are drawn block by block.
    """
    rows = np.asarray(rows, np.int64)
    out = np.empty((rows.shape[0], K), np.int8)
    blocks = np.unique(rows // ROW_BLOCK)
    for b in blocks:
        blk = weight_block(workload_index, tensor, N, K, int(b), kind, p_zero)
        sel = np.nonzero(rows // ROW_BLOCK == b)[0]
        out[sel] = blk[rows[sel] - b * ROW_BLOCK]
    return out


def weight_block(workload_index: int, tensor: str, N: int, K: int, block: int, kind: str,
                 p_zero: float = 1.0 / 3.0) -> np.ndarray:
    r0 = block * ROW_BLOCK
    nr = min(ROW_BLOCK, N - r0)
    g = rng(workload_index, tensor, block)
    if kind == "ternary":
        return ternary(g, (nr, K), p_zero)
    if kind == "signs":
        return signs(g, (nr, K))
    raise ValueError(kind)


def weight_matrix(workload_index: int, tensor: str, N: int, K: int, kind: str, p_zero: float = 1.0 / 3.0):
    nb = (N + ROW_BLOCK - 1) // ROW_BLOCK
    return np.concatenate([weight_block(workload_index, tensor, N, K, b, kind, p_zero) for b in range(nb)], axis=0)


def block_scale_rows(workload_index: int, N: int, nblocks: int, rows, sigma: float = 0.02, tensor="block_scale"):
    """fp16 bit patterns [len(rows), nblocks] of |N(0,sigma)| scales, drawn per row block."""
    rows = np.asarray(rows, np.int64)
    out = np.empty((rows.shape[0], nblocks), np.uint16)
    for b in np.unique(rows // ROW_BLOCK):
        r0 = int(b) * ROW_BLOCK
        nr = min(ROW_BLOCK, N - r0)
        blk = abs_normal_fp16_bits(rng(workload_index, tensor, int(b)), (nr, nblocks), sigma)
        sel = np.nonzero(rows // ROW_BLOCK == b)[0]
        out[sel] = blk[rows[sel] - r0]
    return out


def block_scale_matrix(workload_index: int, N: int, nblocks: int, sigma: float = 0.02, tensor="block_scale"):
    return block_scale_rows(workload_index, N, nblocks, np.arange(N), sigma, tensor)


def activations(workload_index: int, M: int, K: int, dtype: str, tensor: str = "x"):
    """x ~ N(0,1): float32 array, or bf16 bit patterns (uint16) when dtype == 'bf16'."""
    x = normal_f32(rng(workload_index, tensor), (M, K))
    return x if dtype == "f32" else f32_to_bf16_bits(x)


def tensor_scale(workload_index: int, tensor: str = "scale") -> np.float32:
    """One fp32 tensor scale ~ U(0.5, 2)."""
    return uniform_f32(rng(workload_index, tensor), 0.5, 2.0)
