"""Pins that tie the CPU oracle to the pages and to mathematics, not to itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something fixed independently of it:
  * hand-derived byte values (tests/golden/*.txt, each citing its passage);
  * a second decoder written here from the page's per-u32 formula;
  * the identities printed on the pages;
  * library routines (numpy matmul in fp64, numpy float16, torch bfloat16);
  * closed forms and brute force over every ternary quad.
The same functions run against mutated copies of the oracle in
test_oracle_mutants.py, which checks that every planted mistake is caught.
"""
import itertools
import os
import struct

import numpy as np

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# golden file parsing
# ---------------------------------------------------------------------------

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            yield [c.strip() for c in line.split("|")]


def _expand_bytes(spec):
    out = []
    for tok in spec.split():
        if "*" in tok:
            b, n = tok.split("*")
            out += [int(b, 16)] * int(n)
        else:
            out.append(int(tok, 16))
    return np.array(out, np.uint8)


def _matrix(N, K, spec, default=0):
    w = np.full((N, K), default, np.int8)
    for tok in spec.split():
        if tok.startswith("ALL="):
            w[:] = int(tok[4:])
            continue
        rc, v = tok.split("=")
        r, c = rc.split(":")
        w[int(r), int(c)] = int(v)
    return w


def golden_i2s():
    for name, nk, elems, scale, expected in _golden_lines("i2s_bytes.txt"):
        N, K = map(int, nk.split())
        yield name, _matrix(N, K, elems), np.float32(float(scale)), _expand_bytes(expected)


def golden_tq2_0():
    for name, nk, elems, scales, expected in _golden_lines("tq2_0_bytes.txt"):
        N, K = map(int, nk.split())
        d = np.array([int(s, 16) for s in scales.split()], np.uint16).reshape(N, K // 256)
        yield name, _matrix(N, K, elems), d, _expand_bytes(expected)


def golden_w1():
    for name, nk, elems, expected in _golden_lines("w1_words.txt"):
        N, K = map(int, nk.split())
        words = np.array([int(t, 16) for t in expected.split()], np.uint32).view(np.int32).reshape(N, K // 32)
        yield name, _matrix(N, K, elems), words


def golden_act_quant():
    for name, xs, qs, sbits in _golden_lines("act_quant.txt"):
        x = np.array([float(v) for v in xs.split()], np.float32)[None, :]
        q = np.array([int(v) for v in qs.split()], np.int8)[None, :]
        s = np.array([int(sbits, 16)], np.uint32).view(np.float32)
        yield name, x, q, s


# ---------------------------------------------------------------------------
# independent helpers (written from the pages, not from the oracle)
# ---------------------------------------------------------------------------

def i2s_decode_per_u32(packed, N, K):
    """Second i2_s decoder, from the page's per-u32 description
    ("Hesper/Layers/BitLinear", "Fused BitLinear Kernel"): a u32 never spans a
    32-byte group; group128 = u32Idx / 8, baseGroupPos = (u32Idx % 8) * 4; for
    byte b in 0..3 and shift s in [6,4,2,0], elemIdx = group128*128 +
    baseGroupPos + b + (3 - s/2)*32, value = ((byte >> s) & 3) - 1."""
    words = np.frombuffer(packed[: N * K // 4].tobytes(), dtype="<u4").reshape(N, K // 16)
    w = np.zeros((N, K), np.int8)
    for n in range(N):
        for u in range(K // 16):
            word = int(words[n, u])
            g, base = u // 8, (u % 8) * 4
            for b in range(4):
                byte = (word >> (8 * b)) & 0xFF
                for s in (6, 4, 2, 0):
                    e = g * 128 + base + b + (3 - s // 2) * 32
                    w[n, e] = ((byte >> s) & 3) - 1
    scale = struct.unpack("<f", packed[N * K // 4: N * K // 4 + 4].tobytes())[0]
    return w, scale


def w1_bits_numpy(wq, K):
    """Bits of int32 words, element k at bit k%32 of word k/32 (numpy unpackbits, little bit order)."""
    b = np.unpackbits(np.ascontiguousarray(wq).view(np.uint8), axis=-1, bitorder="little")
    return b.reshape(wq.shape[0], K).astype(np.int64)


def fp16_np(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16_torch(bits):
    import torch
    t = torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_i2s_golden_bytes():
    for name, w, scale, expected in golden_i2s():
        got = O.pack_i2s(w, scale)
        assert np.array_equal(got, expected), "i2s golden %s: %s" % (name, got.tobytes().hex())
        w2, s2 = O.unpack_i2s(expected, *w.shape)
        assert np.array_equal(w2, w) and np.float32(s2) == scale, "i2s golden unpack " + name


def pin_i2s_second_decoder():
    g = np.random.Generator(np.random.PCG64(7))
    for N, K in [(3, 128), (2, 384), (5, 256)]:
        w = g.integers(-1, 2, size=(N, K), dtype=np.int8)
        p = O.pack_i2s(w, np.float32(1.75))
        w_indep, s_indep = i2s_decode_per_u32(p, N, K)
        assert np.array_equal(w_indep, w), "i2s per-u32 decoder disagrees with the packer"
        w_orc, s_orc = O.unpack_i2s(p, N, K)
        assert np.array_equal(w_orc, w_indep) and s_orc == s_indep == np.float32(1.75)


def pin_i2s_gemv_matmul_and_identity():
    """y = scale * W x (numpy fp64 matmul) and y = scale*(sum_{w=+1} x - sum_{w=-1} x)
    ("Hesper/Layers/BitLinear", "BitLinear Mathematics")."""
    g = np.random.Generator(np.random.PCG64(11))
    for N, K in [(7, 128), (5, 512)]:
        w = g.integers(-1, 2, size=(N, K), dtype=np.int8)
        x = g.standard_normal(K)
        s = np.float32(0.8125)
        y, cond = O.gemv_i2s(O.pack_i2s(w, s), x, N, K)
        ref = float(s) * (w.astype(np.float64) @ x)
        ident = float(s) * (np.where(w == 1, x, 0.0).sum(1) - np.where(w == -1, x, 0.0).sum(1))
        assert np.allclose(y, ref, rtol=1e-13, atol=1e-12), "i2s gemv vs matmul"
        assert np.allclose(y, ident, rtol=1e-13, atol=1e-12), "i2s gemv vs identity"
        assert np.allclose(cond, abs(float(s)) * (np.abs(w) @ np.abs(x)), rtol=1e-13)
        rows = np.array([4, 0, 2])
        y2, _ = O.gemv_i2s(O.pack_i2s(w, s), x, N, K, rows=rows)
        assert np.allclose(y2, ref[rows], rtol=1e-13, atol=1e-12), "i2s gemv row selection"


def pin_i2s_brute_force_quads():
    """Every one of the 81 ternary quads placed on one byte (elements j, j+32,
    j+64, j+96 share byte j) against small integer x: exact integer result."""
    quads = np.array(list(itertools.product([-1, 0, 1], repeat=4)), np.int8)
    K = 128
    for j in (0, 13, 31):
        w = np.zeros((81, K), np.int8)
        w[:, [j, j + 32, j + 64, j + 96]] = quads
        x = np.zeros(K)
        x[[j, j + 32, j + 64, j + 96]] = [1.0, 10.0, 100.0, 1000.0]
        y, _ = O.gemv_i2s(O.pack_i2s(w, np.float32(1.0)), x, 81, K)
        ref = quads.astype(np.float64) @ np.array([1.0, 10.0, 100.0, 1000.0])
        assert np.array_equal(y, ref), "i2s brute force quads"


def pin_i2s_gate_up_worked_example():
    """Fused gate + up + ReLU^2 x mul ("Hesper/Layers/BitLinear", "Fused
    Gate+Up+ReLU²×Mul M=1 Kernel"): h = max(0, g)^2 * u with g, u each scaled
    by its own tensor scale.  Rows built so that with x = 1 the dots are the
    counts below; expected values worked out by hand:
      row 0: g = 0.5*6 = 3,   u = 2*(-1) = -2  -> h = 9 * -2 = -18
      row 1: g = 0.5*(-4) = -2, u = 2*7 = 14   -> h = 0 (ReLU)
      row 2: g = 0,           u = 2*4 = 8      -> h = 0
      row 3: g = 0.5*10 = 5,  u = 2*1 = 2      -> h = 25 * 2 = 50
      row 4: g = 0.5*2 = 1,   u = 2*(-3) = -6  -> h = -6"""
    K = 128

    def rows_with(counts):
        w = np.zeros((len(counts), K), np.int8)
        for i, c in enumerate(counts):
            if c > 0:
                w[i, :c] = 1
            elif c < 0:
                w[i, :-c] = -1
        return w

    wg = rows_with([6, -4, 0, 10, 2])
    wu = rows_with([-1, 7, 4, 1, -3])
    x = np.ones(K)
    h, cond = O.gemv_i2s_gate_up(O.pack_i2s(wg, np.float32(0.5)), O.pack_i2s(wu, np.float32(2.0)), x, 5, K)
    assert np.array_equal(h, [-18.0, 0.0, 0.0, 50.0, -6.0]), "gate_up worked example: %s" % h
    # cond: 2 a |u| cond_g + a^2 cond_u with cond_g = 0.5*|count_g|, cond_u = 2*|count_u|
    assert np.allclose(cond, [2 * 3 * 2 * 3 + 9 * 2, 0, 0, 2 * 5 * 2 * 5 + 25 * 2, 2 * 1 * 6 * 1 + 1 * 6]), cond


def pin_i2s_gate_up_composition():
    """On random inputs the fused result equals the two pinned GEMVs composed
    through numpy, row selection included."""
    g = np.random.Generator(np.random.PCG64(41))
    N, K = 9, 384
    wg = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    wu = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    x = g.standard_normal(K)
    pg, pu = O.pack_i2s(wg, np.float32(1.5)), O.pack_i2s(wu, np.float32(0.75))
    yg, _ = O.gemv_i2s(pg, x, N, K)
    yu, _ = O.gemv_i2s(pu, x, N, K)
    ref = np.maximum(yg, 0.0) ** 2 * yu
    h, _ = O.gemv_i2s_gate_up(pg, pu, x, N, K)
    assert np.allclose(h, ref, rtol=1e-13, atol=1e-12), "gate_up vs composition"
    rows = np.array([8, 1, 4])
    h2, _ = O.gemv_i2s_gate_up(pg, pu, x, N, K, rows=rows)
    assert np.allclose(h2, ref[rows], rtol=1e-13, atol=1e-12), "gate_up row selection"


def pin_i2s_norm_residual_worked_example():
    """Fused RMSNorm + BitLinear + residual ("Hesper/Layers/BitLinear",
    "Fused RMSNorm + BitLinear + Residual Add M=1 Kernel"):
    rmsInv = 1/sqrt(mean(x^2) + eps), x' = x * rmsInv * w_rms, y = res + s W x'.
    Worked by hand with K = 128, x = 1 everywhere, eps = 3: mean(x^2) = 1,
    rmsInv = 1/sqrt(4) = 0.5.  w_rms = 2 on elements 0..63, 1 elsewhere, so
    x' = 1 on 0..63 and 0.5 on 64..127.  Rows (s = 2, residual = 10, -3, 0):
      row 0: +1 on 0..9              -> dot = 10       -> y = 10 + 20 = 30
      row 1: +1 on 64..71            -> dot = 4        -> y = -3 + 8  = 5
      row 2: -1 on 0..3, +1 on 64..67 -> dot = -4 + 2 = -2 -> y = 0 - 4 = -4
    Without the norm (rms_w None) the same rows give 10, 8, 0 plus residual."""
    K = 128
    w = np.zeros((3, K), np.int8)
    w[0, :10] = 1
    w[1, 64:72] = 1
    w[2, :4] = -1
    w[2, 64:68] = 1
    x = np.ones(K)
    rms_w = np.where(np.arange(K) < 64, 2.0, 1.0)
    res = np.array([10.0, -3.0, 0.0])
    p = O.pack_i2s(w, np.float32(2.0))
    y, cond = O.gemv_i2s_norm_residual(p, x, 3, K, rms_w=rms_w, eps=3.0, residual=res)
    assert np.array_equal(y, [30.0, 5.0, -4.0]), "norm+residual worked example: %s" % y
    assert np.array_equal(cond, [20.0, 8.0, 12.0]), "norm+residual cond: %s" % cond
    y2, _ = O.gemv_i2s_norm_residual(p, x, 3, K, residual=res)
    assert np.array_equal(y2, [30.0, 13.0, 0.0]), "residual only: %s" % y2


def pin_i2s_norm_residual_composition():
    """Random inputs: the fused op equals numpy's RMSNorm (eps = 1e-5) fed to
    the pinned GEMV, plus the residual; row selection included."""
    g = np.random.Generator(np.random.PCG64(43))
    N, K = 11, 512
    w = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    x = g.standard_normal(K) * 3.0
    rw = g.uniform(0.5, 1.5, K)
    res = g.standard_normal(N)
    p = O.pack_i2s(w, np.float32(0.625))
    xn = x / np.sqrt(np.mean(x * x) + 1e-5) * rw
    ref, _ = O.gemv_i2s(p, xn, N, K)
    ref = ref + res
    y, _ = O.gemv_i2s_norm_residual(p, x, N, K, rms_w=rw, eps=1e-5, residual=res)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12), "norm+residual vs composition"
    rows = np.array([10, 0, 5])
    y2, _ = O.gemv_i2s_norm_residual(p, x, N, K, rms_w=rw, eps=1e-5, residual=res, rows=rows)
    assert np.allclose(y2, ref[rows], rtol=1e-12, atol=1e-12), "norm+residual row selection"


def pin_i2s_int8_gemm():
    """acc = q W^T exactly (numpy int64 matmul); y = acc * s_act * s_w."""
    g = np.random.Generator(np.random.PCG64(13))
    M, N, K = 6, 9, 256
    w = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    q = g.integers(-127, 128, size=(M, K), dtype=np.int8)
    sa = g.uniform(0.01, 0.1, M).astype(np.float32)
    sw = np.float32(1.25)
    acc, y, cond = O.gemm_i2s_int8(q, sa, O.pack_i2s(w, sw), N, K)
    ref = q.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(acc, ref), "i2s int8 acc"
    assert np.allclose(y, ref * sa[:, None].astype(np.float64) * float(sw), rtol=1e-14), "i2s int8 y"
    assert np.allclose(cond, (np.abs(q).astype(np.float64) @ np.abs(w).T) * np.abs(sa[:, None] * float(sw)))
    rows = np.array([8, 3])
    acc2, _, _ = O.gemm_i2s_int8(q, sa, O.pack_i2s(w, sw), N, K, rows=rows)
    assert np.array_equal(acc2, ref[:, rows])


def pin_tq2_0_golden_bytes():
    for name, w, d, expected in golden_tq2_0():
        got = O.pack_tq2_0(w, d)
        assert np.array_equal(got, expected), "tq2_0 golden %s: %s" % (name, got.tobytes().hex())
        w2, d2 = O.unpack_tq2_0(expected, *w.shape)
        assert np.array_equal(w2, w) and np.array_equal(d2, d), "tq2_0 golden unpack " + name


def pin_tq2_0_gemv():
    """y = sum_b d_b * (W_b . x_b) with d decoded by numpy float16, and the
    closed form y = 256 * sum_b d_b for W = +1, x = 1."""
    g = np.random.Generator(np.random.PCG64(17))
    N, K = 6, 768
    w = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    d = (np.abs(g.standard_normal((N, K // 256))) * 0.02).astype(np.float16).view(np.uint16)
    x = g.standard_normal(K)
    y, cond = O.gemv_tq2_0(O.pack_tq2_0(w, d), x, N, K)
    dd = fp16_np(d)
    ref = sum(dd[:, b] * (w[:, 256 * b:256 * (b + 1)].astype(np.float64) @ x[256 * b:256 * (b + 1)])
              for b in range(K // 256))
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14), "tq2_0 gemv vs blockwise matmul"
    refc = sum(dd[:, b] * (np.abs(w[:, 256 * b:256 * (b + 1)]) @ np.abs(x[256 * b:256 * (b + 1)]))
               for b in range(K // 256))
    assert np.allclose(cond, refc, rtol=1e-12)
    ones = np.ones((N, K), np.int8)
    y1, _ = O.gemv_tq2_0(O.pack_tq2_0(ones, d), np.ones(K), N, K)
    assert np.allclose(y1, 256.0 * dd.sum(1), rtol=1e-14), "tq2_0 closed form"
    yneg, _ = O.gemv_tq2_0(O.pack_tq2_0(-ones, d), np.ones(K), N, K)
    assert np.allclose(yneg, -256.0 * dd.sum(1), rtol=1e-14), "tq2_0 closed form (-1)"


def pin_tq2_0_int8_gemm():
    """y = s_m * sum_b d_b * (q_b W_b^T) with the block dots from numpy int64
    matmul and d decoded by numpy float16; the closed form y = 256 s sum_b d_b
    for W = +1, q = 1; and, with one scale for every block, the i2_s int8
    product of the same ternary matrix with that scale as its tensor scale."""
    g = np.random.Generator(np.random.PCG64(19))
    M, N, K = 5, 7, 768
    w = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    q = g.integers(-127, 128, size=(M, K), dtype=np.int8)
    sa = g.uniform(0.01, 0.1, M).astype(np.float32)
    d = (np.abs(g.standard_normal((N, K // 256))) * 0.02).astype(np.float16).view(np.uint16)
    d[0, 1] = 0x8000 | d[0, 1]  # a negative block scale
    y, cond = O.gemm_tq2_0_int8(q, sa, O.pack_tq2_0(w, d), N, K)
    dd = fp16_np(d)
    dots = [q[:, 256 * b:256 * (b + 1)].astype(np.int64) @ w[:, 256 * b:256 * (b + 1)].astype(np.int64).T
            for b in range(K // 256)]
    ref = sum(dd[None, :, b] * dots[b] for b in range(K // 256)) * sa[:, None].astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-300), "tq2_0 int8 vs blockwise int matmul"
    dabs = [np.abs(q[:, 256 * b:256 * (b + 1)]).astype(np.int64) @ np.abs(w[:, 256 * b:256 * (b + 1)]).T
            for b in range(K // 256)]
    refc = sum(np.abs(dd[None, :, b]) * dabs[b] for b in range(K // 256)) * sa[:, None]
    assert np.allclose(cond, refc, rtol=1e-12), "tq2_0 int8 cond"
    rows = np.array([6, 0])
    y2, _ = O.gemm_tq2_0_int8(q, sa, O.pack_tq2_0(w, d), N, K, rows=rows)
    assert np.array_equal(y2, y[:, rows])
    ones = np.ones((N, K), np.int8)
    y1, _ = O.gemm_tq2_0_int8(np.ones((1, K), np.int8), np.ones(1, np.float32), O.pack_tq2_0(ones, d), N, K)
    assert np.allclose(y1[0], 256.0 * dd.sum(1), rtol=1e-14), "tq2_0 int8 closed form"
    one_scale = np.full((N, K // 256), 0x3A00, np.uint16)  # 0.75 in every block
    yt, _ = O.gemm_tq2_0_int8(q, sa, O.pack_tq2_0(w, one_scale), N, K)
    _, yi, _ = O.gemm_i2s_int8(q, sa, O.pack_i2s(w, np.float32(0.75)), N, K)
    assert np.allclose(yt, yi, rtol=1e-14, atol=0), "tq2_0 int8 with one scale = i2_s int8"


def pin_w1_golden_words():
    for name, w, words in golden_w1():
        got = O.pack_w1(w)
        assert np.array_equal(got, words), "w1 golden %s: %s" % (name, got.view(np.uint32))
        back = O.unpack_w1(words, w.shape[1])
        assert np.array_equal(back, np.where(w > 0, 1, -1).astype(np.int8)), "w1 golden unpack " + name


def pin_w1_roundtrip_and_bits():
    """unpack(pack(W)) == W for +-1 ("binary-gemm", "Correctness"); zeros become
    -1; bits agree with numpy's little-endian unpackbits."""
    g = np.random.Generator(np.random.PCG64(19))
    N, K = 5, 320
    w = (g.integers(0, 2, size=(N, K), dtype=np.int8) * 2 - 1).astype(np.int8)
    wq = O.pack_w1(w)
    assert np.array_equal(O.unpack_w1(wq, K), w), "w1 roundtrip"
    assert np.array_equal(w1_bits_numpy(wq, K), (w > 0).astype(np.int64)), "w1 bit order"
    t = g.integers(-1, 2, size=(N, K), dtype=np.int8)
    assert np.array_equal(O.unpack_w1(O.pack_w1(t), K), np.where(t > 0, 1, -1)), "w1 zeros -> -1"


def pin_w1a8_identity_and_matmul():
    """dot(w, a) = 2 * sum_{b=1} a - sum a ("binary-gemm", "Method"), and
    y = s_act * sum_g ws_g * dot_g + bias against numpy fp64."""
    g = np.random.Generator(np.random.PCG64(23))
    for G in (32, 64, 128, 256):
        M, N, K = 3, 7, 512
        w = (g.integers(0, 2, size=(N, K), dtype=np.int8) * 2 - 1).astype(np.int8)
        wq = O.pack_w1(w)
        q = g.integers(-127, 128, size=(M, K), dtype=np.int8)
        s = g.uniform(0.005, 0.05, M).astype(np.float32)
        ws = (np.abs(g.standard_normal((N, K // G))) * 0.02).astype(np.float16).view(np.uint16)
        bias = (g.standard_normal(N).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        for b in (None, bias):
            dots, y, cond = O.gemm_w1a8(q, s, wq, ws, b, K, G)
            bits = w1_bits_numpy(wq, K)
            qq = q.astype(np.int64)
            for gi in range(K // G):
                sl = slice(gi * G, (gi + 1) * G)
                ident = 2 * (qq[:, None, sl] * bits[None, :, sl]).sum(-1) - qq[:, None, sl].sum(-1)
                assert np.array_equal(dots[:, :, gi], ident), "w1a8 binary identity, G=%d" % G
                assert np.array_equal(dots[:, :, gi], qq[:, sl] @ w[:, sl].astype(np.int64).T), "w1a8 dot"
            wsd = fp16_np(ws)
            ref = s[:, None].astype(np.float64) * np.einsum("mng,ng->mn", dots.astype(np.float64), wsd)
            if b is not None:
                ref = ref + bf16_torch(b)[None, :]
            assert np.allclose(y, ref, rtol=1e-13, atol=1e-15), "w1a8 y, G=%d" % G
            # the tolerance's condition number: |s| sum_k |ws_g(k)| |w_k| |q_k| + |bias| (|w| = 1)
            qabs = np.abs(q.astype(np.float64)).reshape(M, K // G, G).sum(-1)
            refc = np.abs(s[:, None].astype(np.float64)) * (qabs @ np.abs(wsd).T)
            if b is not None:
                refc = refc + np.abs(bf16_torch(b))[None, :]
            assert np.allclose(cond, refc, rtol=1e-13), "w1a8 cond, G=%d" % G


def pin_w1a8_unit_scales_exact():
    """With unit group scales and unit token scale the bf16 output equals the
    exact int32 accumulator wherever |acc| < 256 ("binary-gemm", "Correctness")."""
    g = np.random.Generator(np.random.PCG64(29))
    M, N, K, G = 2, 64, 128, 128
    w = (g.integers(0, 2, size=(N, K), dtype=np.int8) * 2 - 1).astype(np.int8)
    q = g.integers(-3, 4, size=(M, K), dtype=np.int8)
    ws = np.full((N, K // G), 0x3C00, np.uint16)
    dots, y, _ = O.gemm_w1a8(q, np.ones(M, np.float32), O.pack_w1(w), ws, None, K, G)
    acc = dots.sum(-1)
    sel = np.abs(acc) < 256
    assert sel.mean() > 0.9
    yb = O.bf16_to_f64(O.round_bf16(y))
    assert np.array_equal(yb[sel], acc[sel].astype(np.float64)), "w1a8 unit scales exact"


def pin_w1a8_full_path_within_bf16_step():
    """From unquantized activations: act-quant, the W1A8 product and the bf16
    output together stay within 2^-8 normwise of a dequantize-and-fp32
    reference (weights w*ws, activations q*s), the bf16 rounding step
    ("binary-gemm", "Correctness"); checked at group sizes 32 to 256."""
    g = np.random.Generator(np.random.PCG64(31))
    for G in (32, 64, 128, 256):
        M, N, K = 4, 96, 1024
        x = g.standard_normal((M, K)).astype(np.float32)
        q, s = O.quantize_act_absmax_int8(x, "f32")
        w = (g.integers(0, 2, size=(N, K), dtype=np.int8) * 2 - 1).astype(np.int8)
        ws = (np.abs(g.standard_normal((N, K // G))) * 0.02).astype(np.float16)
        _, y, _ = O.gemm_w1a8(q, s, O.pack_w1(w), ws.view(np.uint16), None, K, G)
        yb = O.bf16_to_f64(O.round_bf16(y))
        w_deq = w.astype(np.float32) * np.repeat(ws.astype(np.float32), G, axis=1)
        x_deq = q.astype(np.float32) * s[:, None]
        ref = (x_deq @ w_deq.T).astype(np.float64)
        err = np.linalg.norm(yb - ref) / np.linalg.norm(ref)
        assert err < 2.0 ** -8, "w1a8 full path normwise %.3g, G=%d" % (err, G)
        # and the bound is not vacuous: without the group scales it fails
        _, y1, _ = O.gemm_w1a8(q, s, O.pack_w1(w), np.full((N, K // G), 0x3C00, np.uint16), None, K, G)
        assert np.linalg.norm(y1 - ref) / np.linalg.norm(ref) > 1.0


def pin_fp16_decode_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = fp16_np(h)
    got = O.fp16_to_f64(h)
    ok = np.isnan(ref) == np.isnan(got)
    ok &= np.where(np.isnan(ref), True, got == ref)
    assert ok.all(), "fp16 decode"


def pin_bf16_decode_and_round():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_torch(b)
    got = O.bf16_to_f64(b)
    ok = (np.isnan(ref) == np.isnan(got)) & np.where(np.isnan(ref), True, got == ref)
    assert ok.all(), "bf16 decode"
    import torch
    g = np.random.Generator(np.random.PCG64(31))
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(2000) * 1e-39).astype(np.float32),      # float32 subnormals -> bf16 subnormals
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.3895314e38, 3.4e38, 0.0, -0.0,
                  2 ** -133, 1.5 * 2 ** -133, 2 ** -134], np.float32),
    ])
    ref_bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_bits = O.round_bf16(vals.astype(np.float64))
    assert np.array_equal(got_bits, ref_bits), "bf16 rounding vs torch"


def pin_act_quant_golden():
    for name, x, q, s in golden_act_quant():
        for dt, xin in (("f32", x), ("bf16", (x.view(np.uint32) >> 16).astype(np.uint16))):
            q2, s2 = O.quantize_act_absmax_int8(xin, dt)
            assert np.array_equal(q2, q), "act quant %s %s: %s" % (name, dt, q2)
            assert s2.view(np.uint32)[0] == s.view(np.uint32)[0], "act quant scale %s %s" % (name, dt)


def pin_act_quant_bound():
    """Reconstruction error under 1% of the row maximum ("binary-gemm",
    "Correctness"); here |q*s - x| <= s/2 (+ one rounding) and max|q| = 127."""
    g = np.random.Generator(np.random.PCG64(37))
    x = (g.standard_normal((16, 1000)) * g.uniform(0.01, 100, (16, 1))).astype(np.float32)
    q, s = O.quantize_act_absmax_int8(x, "f32")
    rec = q.astype(np.float64) * s[:, None]
    amax = np.abs(x).max(1)
    err = np.abs(rec - x).max(1)
    assert (err < 0.01 * amax).all(), "act quant 1% bound"
    assert (err <= s * 0.5 * (1 + 1e-5) + amax * 2 ** -23).all(), "act quant half-step bound"
    assert (np.abs(q).max(1) == 127).all(), "act quant uses the full range"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
