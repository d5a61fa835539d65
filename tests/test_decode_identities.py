"""CPU checks of the hand-typed constants in the kernels' decode steps.

Each test restates, with numpy, one bit-level identity that a kernel relies on
and checks it exhaustively over its input domain against the plain decode
(code tables of the formats, int8 values).  The GPU parity tests check the
compiled kernels; these check that the identities and constants themselves
are exact, so that a wrong constant shows up here and not only as a parity
failure on some inputs.  fp16 arithmetic is emulated exactly: each fp16
operation is computed in float64 (exact for these operands) and rounded once.
"""
import numpy as np


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def rn16(v):
    """Round float64 values to fp16 (nearest even), as fp16 bit patterns."""
    return np.asarray(v, np.float64).astype(np.float16).view(np.uint16)


def lo_hi(u32):
    u32 = np.asarray(u32, np.uint64)
    return (u32 & 0xFFFF).astype(np.uint16), ((u32 >> 16) & 0xFFFF).astype(np.uint16)


I8 = np.arange(-128, 128)


def test_int8_to_fp16_magic():
    """int8 q -> fp16: the byte q ^ 0x80 under the exponent byte 0x64 reads
    1024 + (q + 128); one fp16 FMA with (scale, -1152 * scale) gives
    q * scale exactly for the power-of-two scales of the i2_s prefill
    (2^(2t-6)), the W1A8 path (1) and the TQ2_0 path (1/4^k)."""
    half = (0x64 << 8) | ((I8 + 256) % 256 ^ 0x80)
    assert np.array_equal(f16(half), 1024.0 + I8 + 128)
    for sc in [2.0 ** (2 * t - 6) for t in range(4)] + [1.0, 0.25, 1 / 16, 1 / 64]:
        bias = float(f16(rn16(-1152.0 * sc)))
        assert bias == -1152.0 * sc                      # the constant itself is exact
        out = f16(rn16(f16(half) * sc + bias))           # one rounding of a*b + c
        assert np.array_equal(out, I8 * sc)
    # the TQ2_0 kernel's packed constants: scales (1, 1/4), (1/16, 1/64), biases -1152 S^-1
    assert list(f16([0x3C00, 0x3400, 0x2C00, 0x2400])) == [1.0, 0.25, 1 / 16, 1 / 64]
    assert list(f16([0xE480, 0xDC80, 0xD480, 0xCC80])) == [-1152.0, -288.0, -72.0, -18.0]


def test_i2s_class_decode():
    """i2_s B operand: code byte p (element 32t + j at bits (7-2t):(6-2t)),
    masked with 3 << (6-2t) under the exponent of 1024, minus 1024 + 2^(6-2t),
    is w * 2^(6-2t) with w = code - 1 (codes 00 -> -1, 01 -> 0, 10 -> +1)."""
    p = np.arange(256)
    for t in range(4):
        sh = 6 - 2 * t
        code = (p >> sh) & 3
        b = f16((p & (3 << sh)) | 0x6400)
        off = float(f16(0x6400 | (1 << sh)))
        assert off == 1024 + 2 ** sh
        w = f16(rn16(b - off))
        ok = code < 3
        assert np.array_equal(w[ok], (code[ok] - 1) * 2.0 ** sh)
    # the product with the activation of the same class is exactly q * w
    for t in range(4):
        a = I8 * 2.0 ** (2 * t - 6)
        for w in (-1, 0, 1):
            assert np.array_equal(a * (w * 2.0 ** (6 - 2 * t)), I8 * w)


def test_prefill_accumulator_bound():
    """Every partial sum of acc = sum_k q w is an integer of magnitude at most
    128 K; at K = 131072 that is 2^24, so the fp32 accumulator holds each one
    exactly, while 128 more columns of q = -128 reach odd sums above 2^24."""
    assert 128 * 131072 == 2 ** 24 and float(np.float32(2 ** 24)) == 2 ** 24
    odd = 128 * (131072 + 128) - 127          # e.g. one q = -127 among the -128s
    assert odd > 2 ** 24 and odd % 2 == 1 and int(np.float32(odd)) != odd


def test_w1_sign_decode():
    """W1A8 tensor-core B operand: for byte b of a bit word and pair k, the
    product b * (2^(15-2k) + 2^(30-2k)) mod 2^32 holds bit 2k of b at bit 15
    and bit 2k+1 at bit 31 (the two copies never overlap), so
    (~x & 0x80008000) ^ (ws, ws) is the fp16 pair (+-ws) with + for a set bit."""
    b = np.arange(256, dtype=np.uint64)
    ws = np.array([0x2A3C, 0xAA3C, 0x0001, 0x7BFF], np.uint64)  # positive, negative, subnormal, max
    for k in range(4):
        x = (b * ((1 << (15 - 2 * k)) + (1 << (30 - 2 * k)))) & 0xFFFFFFFF
        assert np.array_equal((x >> 15) & 1, (b >> (2 * k)) & 1)
        assert np.array_equal((x >> 31) & 1, (b >> (2 * k + 1)) & 1)
        for s in ws:
            o = (~x & 0x80008000) ^ (s | (s << 16))
            lo, hi = lo_hi(o)
            sign = lambda bit: np.where(bit == 1, 1.0, -1.0)
            assert np.array_equal(f16(lo), sign((b >> (2 * k)) & 1) * f16(s)[()])
            assert np.array_equal(f16(hi), sign((b >> (2 * k + 1)) & 1) * f16(s)[()])


def test_tq2_0_in_place_decode():
    """TQ2_0 tensor-core B operand: the 8 codes of a 16-bit word c (element e
    at bits 2e, 2e+1; 00 -> 0, 01 -> +1, 11 -> -1), copied into both halves,
    masked per pair and XOR-ed with 0x64086402 / 0x64806420 give
    1024 + f * S (f = w + 2, S = 4^(e % 4)); minus the same constant's value
    1024 + 2S, times d, is w * d * S exactly for |d| < 1024."""
    table = {0: 0, 1: 1, 3: -1}
    words = [c for c in range(1 << 16) if all(((c >> (2 * e)) & 3) != 2 for e in range(8))]
    c = np.array(words, np.uint64)
    w = c * 0x00010001
    w8 = w >> 8
    pairs = [((w & 0x000C0003) ^ 0x64086402, 0x64086402, (0, 1)), ((w & 0x00C00030) ^ 0x64806420, 0x64806420, (2, 3)),
             ((w8 & 0x000C0003) ^ 0x64086402, 0x64086402, (4, 5)), ((w8 & 0x00C00030) ^ 0x64806420, 0x64806420, (6, 7))]
    ds = f16(np.array([0x3C00, 0x63FF, 0x8001, 0xE3FF, 0x2E66], np.uint16))  # 1, 1023.5, -2^-24, -1023.5, 0.1
    for p, kconst, (e0, e1) in pairs:
        plo, phi = lo_hi(p)
        klo, khi = lo_hi(np.uint64(kconst))
        for half, kk, e in ((plo, klo, e0), (phi, khi, e1)):
            S = 4.0 ** (e % 4)
            assert f16(kk)[()] == 1024 + 2 * S
            wS = f16(rn16(f16(half) - f16(kk)[()]))
            wv = np.array([table[int(v)] for v in (c >> (2 * e)) & 3], np.float64)
            assert np.array_equal(wS, wv * S)
            for d in ds:
                assert np.array_equal(f16(rn16(wS * d)), wv * d * S)
    # 0x6400 is the smallest |d| the kernel flags (BL_DEVERR_RANGE): 1024
    assert f16(0x6400)[()] == 1024.0 and f16(0x63FF)[()] * 64 == 65504.0


def test_tq2_0_gemv_xor_map():
    """TQ2_0 GEMV: XOR with 0b01 maps the codes to t = 1 - w in {1, 0, 2}
    (00 -> 01, 01 -> 00, 11 -> 10), so the i2_s mask/dp4a decode applies with
    sum w X = sum X - sum t X."""
    for code, w in ((0b00, 0), (0b01, 1), (0b11, -1)):
        assert (code ^ 0b01) == 1 - w


def test_gemv_digit_decomposition():
    """i2_s / TQ2_0 GEMV activations: an integer X with |X| < 2^(8D-1) is the
    sum of its D two's-complement bytes, the low ones unsigned and the top
    one signed, each times 256^d; per-digit dp4a sums then recombine
    exactly."""
    g = np.random.Generator(np.random.PCG64(47))
    for D in (2, 3, 4):
        lim = 2 ** (8 * D - 1) - 1
        X = np.concatenate([g.integers(-lim, lim + 1, 4096), [lim, -lim, 0, 1, -1]]).astype(np.int64)
        u = X.astype(np.int64) & ((1 << (8 * D)) - 1)
        digits = [(u >> (8 * d)) & 0xFF for d in range(D)]
        top = np.where(digits[-1] >= 128, digits[-1] - 256, digits[-1])
        rec = sum(digits[d] * 256 ** d for d in range(D - 1)) + top * 256 ** (D - 1)
        assert np.array_equal(rec, X)
        codes = g.integers(0, 3, X.size)                     # c = w + 1
        dots = sum((codes * digits[d]).sum() * 256 ** d for d in range(D - 1)) + (codes * top).sum() * 256 ** (D - 1)
        assert dots - X.sum() == ((codes - 1) * X).sum()


def test_gemv_fixed_point_exact_range():
    """The GEMV fixed point: with the group maximum m in [2^(e-1), 2^e) and
    F = (8D - 1) - e, x * 2^F is an integer of magnitude < 2^(8D-1) for every
    |x| <= m whose binade is at most (8D - 1) - p below m's (p: significand
    bits, 24 for fp32 and 8 for bf16): 7, 15 and 7 binades for
    (fp32, D=4), (bf16, D=3) and (bf16, D=2); one binade lower it is not."""
    for p, D, span in ((24, 4, 7), (8, 3, 15), (8, 2, 7)):
        e = 1                                            # m in [1, 2)
        F = (8 * D - 1) - e
        top = (2 ** p - 1) / 2 ** (p - 1)                # largest significand, the group maximum
        assert top * 2.0 ** F < 2 ** (8 * D - 1)
        odd = 1 + 2.0 ** (1 - p)                         # significand with its lowest bit set
        assert float(odd * 2.0 ** (-span) * 2.0 ** F).is_integer()
        assert not float(odd * 2.0 ** (-span - 1) * 2.0 ** F).is_integer()


def test_i2s_gemv_shift_class_masks():
    """i2_s GEMV decode: in a 32-bit word holding bytes p..p+3 of a group, the
    four masks w & 0x03030303, (w >> 2) & 0x03030303, w & 0x30303030 and
    (w >> 2) & 0x30303030 hold, byte by byte, the codes of elements 96+p,
    64+p (times 1) and 32+p, p (times 16): shift 0, 2, 4, 6 of each byte."""
    g = np.random.Generator(np.random.PCG64(53))
    words = g.integers(0, 2 ** 32, 2000, dtype=np.uint64)
    for w in words:
        w = int(w)
        byts = [(w >> (8 * b)) & 0xFF for b in range(4)]
        masks = [w & 0x03030303, (w >> 2) & 0x03030303, w & 0x30303030, (w >> 2) & 0x30303030]
        scale = [1, 1, 16, 16]
        shift = [0, 2, 4, 6]
        for mk, sc, sh in zip(masks, scale, shift):
            for b in range(4):
                assert ((mk >> (8 * b)) & 0xFF) == sc * ((byts[b] >> sh) & 3)


def test_w1_bit_class_masks():
    """W1A8 rows decode: word & (0x01010101 << j) holds, in byte b, bit j of
    byte b times 2^j, i.e. element 8b + j of the 32-element word; so the eight
    class sums acc_j = 2^j S_j recombine as sum_j acc_j >> j."""
    g = np.random.Generator(np.random.PCG64(59))
    for w in g.integers(0, 2 ** 32, 500, dtype=np.uint64):
        w = int(w)
        a = g.integers(-128, 128, 32)
        S = 0
        for j in range(8):
            m = w & (0x01010101 << j)
            acc = sum(((m >> (8 * b)) & 0xFF) * a[8 * b + j] for b in range(4))
            assert acc % (1 << j) == 0
            S += acc >> j
        bits = [(w >> k) & 1 for k in range(32)]
        assert S == sum(int(a[k]) for k in range(32) if bits[k])


def test_block_scales_include_subnormals():
    """The |N(0, 0.02)| fp16 block and group scales of the workloads include
    fp16 subnormals (about 0.24% of them), so the exact subnormal decode of
    every scale path is exercised by the parity inputs."""
    from gemm_bl_gemv_gb300 import synth
    d = synth.block_scale_matrix(3, 2048, 20)
    sub = np.mean((d & 0x7C00) == 0)
    assert 0.001 < sub < 0.005
