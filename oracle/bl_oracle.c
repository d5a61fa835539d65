/*
 * bl_oracle.c -- plain, slow CPU oracle for the packed BitLinear product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; both sides see only the seeded synthetic inputs.
 *
 * Every function computes the plain definition of the operation:
 *   1. read each weight out of its packed container one element at a time,
 *      by the format's own element formula and code table;
 *   2. form the dot products in exact int64 (integer paths) or fp64;
 *   3. leave rounding to the output type to the caller (y is returned in
 *      fp64; bf16 rounding is offered by orc_round_bf16()).
 * Accumulation order is the natural k = 0..K-1 order; there is no blocking,
 * fusion or reordering.  OpenMP, when compiled in, only spreads independent
 * output rows over threads.
 *
 * Sources (page title, section):
 *   "Hesper/Layers/BitLinear": "i2_s Packing Format" (code table, the four
 *       shift positions 6/4/2/0 over a 32-byte group of 128, the single F32
 *       scale stored after the tensor data), "BitLinear Mathematics"
 *       (y[i] = scale * sum_j w[i,j] x[j]).
 *   "Hesper/Quantization/TQ2_0": "TQ2_0 Format" (256-element blocks, 64
 *       packed bytes then an FP16 scale, 66 bytes per block, codes
 *       00 -> 0, 01 -> +1, 11 -> -1).
 *   "binary-gemm" card: "API" (pack_weights: {-1,+1} int8 [N,K] -> int32
 *       [N,K/32]; quantize_activation: per-token int8 + fp32 scale;
 *       binary_gemm: packed product with fp16 group scales, optional bias),
 *       "Method" (stored bit b = (w+1)/2), "Correctness" (zeros pack as -1,
 *       per-token absmax activation quantization).
 * Readings where the pages are silent (element order inside a TQ2_0 block,
 * bit order inside a W1 word, the exact absmax formula) are stated next to
 * the code that takes them.
 *
 * Parity pins: every function here is pinned by the CPU test suite to hand
 * derived byte values, identities from the pages, closed forms, library
 * routines (numpy matmul, numpy float16, torch bfloat16) and brute force.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_SHAPE (-1)
#define ORC_ERR_VALUE (-2)

static int g_threads = 1;

int orc_set_threads(int n) {
  g_threads = n < 1 ? 1 : n;
#ifdef _OPENMP
  return g_threads;
#else
  g_threads = 1;
  return 1;
#endif
}

int orc_has_openmp(void) {
#ifdef _OPENMP
  return 1;
#else
  return 0;
#endif
}

/* ------------------------------------------------------------------ */
/* Scalar format helpers, written from the IEEE 754 definitions.       */
/* ------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_fp16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double orc_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 255;
  int m = b & 127;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133);                /* subnormal: m * 2^-133 */
  } else if (e == 255) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(128 + m), e - 134);     /* (1 + m/128) * 2^(e-127) */
  }
  return sign ? -v : v;
}

/* Round an fp64 value to the nearest bfloat16, ties to even. */
uint16_t orc_round_bf16(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7FC0;
  if (isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int e;
  double f = frexp(a, &e);                     /* a = f * 2^e, f in [0.5, 1) */
  /* normal bf16 value = (r / 128) * 2^(e-1) with r in [128, 256) */
  int biased = (e - 1) + 127;
  if (biased <= 0) {
    /* subnormal range: value = m * 2^-133, m in [0, 128] */
    double m = nearbyint(ldexp(a, 133));       /* default mode: ties to even */
    return sign | (uint16_t)m;                 /* m == 128 encodes 2^-126 */
  }
  double r = nearbyint(ldexp(f, 8));           /* in [128, 256] */
  if (r == 256.0) { r = 128.0; biased += 1; }
  if (biased >= 255) return sign | 0x7F80;
  return sign | (uint16_t)(biased << 7) | (uint16_t)((int)r - 128);
}

void orc_bf16_array_to_double(const uint16_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_double(b[i]);
}

void orc_fp16_array_to_double(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp16_to_double(h[i]);
}

void orc_round_bf16_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(x[i]);
}

static float read_f32_le(const uint8_t* p) {
  uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static void write_f32_le(uint8_t* p, float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  p[0] = u & 0xFF; p[1] = (u >> 8) & 0xFF; p[2] = (u >> 16) & 0xFF; p[3] = (u >> 24) & 0xFF;
}

/* ------------------------------------------------------------------ */
/* i2_s ("Hesper/Layers/BitLinear", "i2_s Packing Format")             */
/*   code table: -1 -> 0b00, 0 -> 0b01, +1 -> 0b10 (0b11 never used)  */
/*   group of 128 elements in 32 bytes; element j of the group sits in */
/*   byte (j mod 32) at shift 6, 4, 2, 0 for j in [0,32), [32,64),     */
/*   [64,96), [96,128); rows of K/4 bytes follow each other; one F32   */
/*   scale follows the last row (little-endian).                       */
/* ------------------------------------------------------------------ */

static int i2s_code_of(int w) {      /* ternary -> code, -1 on bad value */
  if (w == -1) return 0;
  if (w == 0) return 1;
  if (w == 1) return 2;
  return -1;
}

static int i2s_value_of(int code) {  /* code -> ternary, 99 on code 3 */
  static const int table[4] = {-1, 0, 1, 99};
  return table[code & 3];
}

/* byte offset and shift of element e of row n */
static int64_t i2s_byte_index(int64_t n, int64_t K, int64_t e) {
  return n * (K / 4) + (e / 128) * 32 + (e % 32);
}
static int i2s_shift(int64_t e) {
  return 6 - 2 * (int)((e % 128) / 32);
}

static int i2s_weight(const uint8_t* packed, int64_t K, int64_t n, int64_t e) {
  int code = (packed[i2s_byte_index(n, K, e)] >> i2s_shift(e)) & 3;
  return i2s_value_of(code);
}

int64_t orc_i2s_packed_bytes(int64_t N, int64_t K) { return N * (K / 4) + 4; }

int orc_pack_i2s(const int8_t* w, float scale, int64_t N, int64_t K, uint8_t* out) {
  if (N < 0 || K < 0 || K % 128 != 0) return ORC_ERR_SHAPE;
  memset(out, 0, (size_t)(N * (K / 4)));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t e = 0; e < K; ++e) {
      int code = i2s_code_of(w[n * K + e]);
      if (code < 0) return ORC_ERR_VALUE;
      out[i2s_byte_index(n, K, e)] |= (uint8_t)(code << i2s_shift(e));
    }
  }
  write_f32_le(out + N * (K / 4), scale);
  return ORC_OK;
}

int orc_unpack_i2s(const uint8_t* packed, int64_t N, int64_t K, int8_t* w, float* scale) {
  if (N < 0 || K < 0 || K % 128 != 0) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t e = 0; e < K; ++e) {
      int v = i2s_weight(packed, K, n, e);
      if (v == 99) return ORC_ERR_VALUE;
      w[n * K + e] = (int8_t)v;
    }
  }
  *scale = read_f32_le(packed + N * (K / 4));
  return ORC_OK;
}

/*
 * y[r] = scale * sum_e w[n,e] x[e]  ("BitLinear Mathematics"), n = rows[r]
 * (or r when rows is NULL).  cond[r] = |scale| * sum_e |w[n,e]| |x[e]|.
 */
int orc_gemv_i2s(const uint8_t* packed, const double* x, int64_t N, int64_t K,
                 const int64_t* rows, int64_t nrows, double* y, double* cond) {
  if (N < 0 || K < 0 || K % 128 != 0) return ORC_ERR_SHAPE;
  const double s = (double)read_f32_le(packed + N * (K / 4));
  int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static) reduction(| : bad)
#endif
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t n = rows ? rows[r] : r;
    if (n < 0 || n >= N) { bad |= 1; continue; }
    double acc = 0.0, c = 0.0;
    for (int64_t e = 0; e < K; ++e) {
      const int w = i2s_weight(packed, K, n, e);
      if (w == 99) { bad |= 2; break; }
      acc += (double)w * x[e];
      c += fabs((double)w) * fabs(x[e]);
    }
    y[r] = s * acc;
    if (cond) cond[r] = fabs(s) * c;
  }
  return bad ? (bad & 1 ? ORC_ERR_SHAPE : ORC_ERR_VALUE) : ORC_OK;
}

/*
 * Fused gate + up + ReLU^2 x mul for one token ("Hesper/Layers/BitLinear",
 * "Fused Gate+Up+ReLU²×Mul M=1 Kernel"): with the two i2_s tensors' own
 * scales,
 *   g[n] = s_g * sum_e wg[n,e] x[e],   u[n] = s_u * sum_e wu[n,e] x[e],
 *   h[n] = max(0, g[n])^2 * u[n]                     (fp64 throughout).
 * cond[r] = 2 max(0,g) |u| cond_g + max(0,g)^2 cond_u: the first-order bound
 * of h's error when g and u are each off by at most their own cond.
 */
int orc_gemv_i2s_gate_up(const uint8_t* packed_gate, const uint8_t* packed_up, const double* x, int64_t N,
                         int64_t K, const int64_t* rows, int64_t nrows, double* h, double* cond) {
  if (nrows < 0) return ORC_ERR_SHAPE;
  double* buf = (double*)malloc(sizeof(double) * 4 * (size_t)(nrows > 0 ? nrows : 1));
  if (!buf) return ORC_ERR_SHAPE;
  double *g = buf, *cg = buf + nrows, *u = buf + 2 * nrows, *cu = buf + 3 * nrows;
  int st = orc_gemv_i2s(packed_gate, x, N, K, rows, nrows, g, cg);
  if (st == ORC_OK) st = orc_gemv_i2s(packed_up, x, N, K, rows, nrows, u, cu);
  if (st == ORC_OK) {
    for (int64_t r = 0; r < nrows; ++r) {
      const double a = g[r] > 0.0 ? g[r] : 0.0;
      h[r] = a * a * u[r];
      if (cond) cond[r] = 2.0 * a * fabs(u[r]) * cg[r] + a * a * cu[r];
    }
  }
  free(buf);
  return st;
}

/*
 * Fused RMSNorm + BitLinear + residual for one token ("Hesper/Layers/BitLinear",
 * "Fused RMSNorm + BitLinear + Residual Add M=1 Kernel" and the M=1 kernel
 * with fused residual add), fp64 throughout:
 *   rmsInv = 1 / sqrt(sum_e x[e]^2 / K + eps)      (when rms_w is given)
 *   x'[e]  = x[e] * rmsInv * rms_w[e]               (else x' = x)
 *   y[r]   = residual[n] + s * sum_e w[n,e] x'[e]   (residual may be NULL: 0)
 * cond[r] = |s| * sum_e |w[n,e]| |x'[e]| (the rounding of the residual sum is
 * covered by the |y| term of the tolerance).
 */
int orc_gemv_i2s_norm_residual(const uint8_t* packed, const double* x, const double* rms_w, double eps,
                               const double* residual, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                               double* y, double* cond) {
  if (N < 0 || K <= 0 || K % 128 != 0 || nrows < 0) return ORC_ERR_SHAPE;
  double* xn = (double*)malloc(sizeof(double) * (size_t)K);
  if (!xn) return ORC_ERR_SHAPE;
  double inv = 1.0;
  if (rms_w) {
    double ss = 0.0;
    for (int64_t e = 0; e < K; ++e) ss += x[e] * x[e];
    inv = 1.0 / sqrt(ss / (double)K + eps);
  }
  for (int64_t e = 0; e < K; ++e) xn[e] = rms_w ? x[e] * inv * rms_w[e] : x[e];
  int st = orc_gemv_i2s(packed, xn, N, K, rows, nrows, y, cond);
  if (st == ORC_OK && residual) {
    for (int64_t r = 0; r < nrows; ++r) y[r] += residual[rows ? rows[r] : r];
  }
  free(xn);
  return st;
}

/*
 * Large-M product with int8 activations:
 *   acc[m,r] = sum_k q[m,k] w[n,k]   (exact, int64)
 *   y[m,r]   = acc[m,r] * s_act[m] * s_w   (fp64)
 * cond[m,r] = |s_act[m] s_w| * sum_k |q[m,k]| |w[n,k]|.
 */
int orc_gemm_i2s_int8(const int8_t* q, const float* s_act, const uint8_t* packed,
                      int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                      int64_t* acc_out, double* y, double* cond) {
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return ORC_ERR_SHAPE;
  const double sw = (double)read_f32_le(packed + N * (K / 4));
  int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static) reduction(| : bad)
#endif
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t n = rows ? rows[r] : r;
    if (n < 0 || n >= N) { bad |= 1; continue; }
    for (int64_t m = 0; m < M; ++m) {
      int64_t acc = 0, c = 0;
      for (int64_t k = 0; k < K; ++k) {
        const int w = i2s_weight(packed, K, n, k);
        if (w == 99) { bad |= 2; break; }
        acc += (int64_t)q[m * K + k] * w;
        c += (int64_t)abs(q[m * K + k]) * abs(w);
      }
      const double sm = (double)s_act[m];
      if (acc_out) acc_out[m * nrows + r] = acc;
      y[m * nrows + r] = (double)acc * sm * sw;
      if (cond) cond[m * nrows + r] = fabs(sm * sw) * (double)c;
    }
  }
  return bad ? (bad & 1 ? ORC_ERR_SHAPE : ORC_ERR_VALUE) : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* TQ2_0 ("Hesper/Quantization/TQ2_0", "TQ2_0 Format")                 */
/*   block of 256 elements = 64 code bytes then an FP16 scale (LE),    */
/*   66 bytes; blocks in K order, rows contiguous.                     */
/*   codes: 00 -> 0, 01 -> +1, 11 -> -1 (10 never used).              */
/*   Reading (order inside a block is not printed): element e of the   */
/*   block sits in byte e/4 at shift 2*(e%4), i.e. the 2*idx shift of  */
/*   the page's unpack helper, lowest bits first.                      */
/* ------------------------------------------------------------------ */

static int tq2_code_of(int w) {
  if (w == 0) return 0;
  if (w == 1) return 1;
  if (w == -1) return 3;
  return -1;
}

static int tq2_value_of(int code) {
  static const int table[4] = {0, 1, 99, -1};
  return table[code & 3];
}

int64_t orc_tq2_0_packed_bytes(int64_t N, int64_t K) { return N * (K / 256) * 66; }

static const uint8_t* tq2_block(const uint8_t* packed, int64_t K, int64_t n, int64_t b) {
  return packed + (n * (K / 256) + b) * 66;
}

static int tq2_weight(const uint8_t* packed, int64_t K, int64_t n, int64_t e) {
  const uint8_t* blk = tq2_block(packed, K, n, e / 256);
  const int64_t j = e % 256;
  return tq2_value_of((blk[j / 4] >> (2 * (j % 4))) & 3);
}

static uint16_t tq2_scale_bits(const uint8_t* packed, int64_t K, int64_t n, int64_t b) {
  const uint8_t* blk = tq2_block(packed, K, n, b);
  return (uint16_t)(blk[64] | (blk[65] << 8));
}

int orc_pack_tq2_0(const int8_t* w, const uint16_t* d, int64_t N, int64_t K, uint8_t* out) {
  if (N < 0 || K < 0 || K % 256 != 0) return ORC_ERR_SHAPE;
  const int64_t nb = K / 256;
  memset(out, 0, (size_t)(N * nb * 66));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t* blk = out + (n * nb + b) * 66;
      for (int64_t j = 0; j < 256; ++j) {
        int code = tq2_code_of(w[n * K + b * 256 + j]);
        if (code < 0) return ORC_ERR_VALUE;
        blk[j / 4] |= (uint8_t)(code << (2 * (j % 4)));
      }
      blk[64] = d[n * nb + b] & 0xFF;
      blk[65] = (d[n * nb + b] >> 8) & 0xFF;
    }
  }
  return ORC_OK;
}

int orc_unpack_tq2_0(const uint8_t* packed, int64_t N, int64_t K, int8_t* w, uint16_t* d) {
  if (N < 0 || K < 0 || K % 256 != 0) return ORC_ERR_SHAPE;
  const int64_t nb = K / 256;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t e = 0; e < K; ++e) {
      int v = tq2_weight(packed, K, n, e);
      if (v == 99) return ORC_ERR_VALUE;
      w[n * K + e] = (int8_t)v;
    }
    for (int64_t b = 0; b < nb; ++b) d[n * nb + b] = tq2_scale_bits(packed, K, n, b);
  }
  return ORC_OK;
}

/*
 * y[r] = sum_b d[n,b] * sum_{j<256} w[n,256b+j] x[256b+j]
 * cond[r] = sum_b |d[n,b]| * sum_j |w| |x|.
 */
int orc_gemv_tq2_0(const uint8_t* packed, const double* x, int64_t N, int64_t K,
                   const int64_t* rows, int64_t nrows, double* y, double* cond) {
  if (N < 0 || K < 0 || K % 256 != 0) return ORC_ERR_SHAPE;
  const int64_t nb = K / 256;
  int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static) reduction(| : bad)
#endif
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t n = rows ? rows[r] : r;
    if (n < 0 || n >= N) { bad |= 1; continue; }
    double total = 0.0, c = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
      const double d = orc_fp16_to_double(tq2_scale_bits(packed, K, n, b));
      double blk = 0.0, blk_abs = 0.0;
      for (int64_t j = 0; j < 256; ++j) {
        const int64_t e = b * 256 + j;
        const int w = tq2_weight(packed, K, n, e);
        if (w == 99) { bad |= 2; break; }
        blk += (double)w * x[e];
        blk_abs += fabs((double)w) * fabs(x[e]);
      }
      total += d * blk;
      c += fabs(d) * blk_abs;
    }
    y[r] = total;
    if (cond) cond[r] = c;
  }
  return bad ? (bad & 1 ? ORC_ERR_SHAPE : ORC_ERR_VALUE) : ORC_OK;
}

/*
 * TQ2_0 weights against int8 activations (large batches).  The TQ2_0 page
 * defines the container and the per-block value d_b * w; the activations
 * are the per-token int8 codes and fp32 scales of the "binary-gemm" card's
 * quantize_activation.  Reading: the product is the definition with x
 * replaced by its quantized form s_m * q[m,:]:
 *   dot[m,n,b] = sum_{j<256} w[n,256b+j] q[m,256b+j]          (exact int64)
 *   y[m,r]     = s_m * sum_b d[n,b] * dot[m,n,b]               (fp64)
 *   cond[m,r]  = |s_m| * sum_b |d[n,b]| * sum_j |w| |q|.
 */
int orc_gemm_tq2_0_int8(const int8_t* q, const float* s_act, const uint8_t* packed,
                        int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                        double* y, double* cond) {
  if (M < 0 || N < 0 || K < 0 || K % 256 != 0) return ORC_ERR_SHAPE;
  const int64_t nb = K / 256;
  int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static) reduction(| : bad)
#endif
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t n = rows ? rows[r] : r;
    if (n < 0 || n >= N) { bad |= 1; continue; }
    for (int64_t m = 0; m < M; ++m) {
      double total = 0.0, c = 0.0;
      for (int64_t b = 0; b < nb; ++b) {
        const double d = orc_fp16_to_double(tq2_scale_bits(packed, K, n, b));
        int64_t dot = 0, dot_abs = 0;
        for (int64_t j = 0; j < 256; ++j) {
          const int64_t e = b * 256 + j;
          const int w = tq2_weight(packed, K, n, e);
          if (w == 99) { bad |= 2; break; }
          dot += (int64_t)q[m * K + e] * w;
          dot_abs += (int64_t)abs(q[m * K + e]) * abs(w);
        }
        total += d * (double)dot;
        c += fabs(d) * (double)dot_abs;
      }
      const double sm = (double)s_act[m];
      y[m * nrows + r] = sm * total;
      if (cond) cond[m * nrows + r] = fabs(sm) * c;
    }
  }
  return bad ? (bad & 1 ? ORC_ERR_SHAPE : ORC_ERR_VALUE) : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* W1 sign bits ("binary-gemm": API, Method, Correctness)              */
/*   {-1,+1} int8 [N,K] -> int32 [N,K/32], stored bit b = (w+1)/2;     */
/*   zeros are stored as -1 (bit 0).                                   */
/*   Reading (bit order is not printed): element k sits at bit k%32 of */
/*   word k/32, lowest bit first.                                      */
/* ------------------------------------------------------------------ */

int orc_pack_w1(const int8_t* w, int64_t N, int64_t K, int32_t* out) {
  if (N < 0 || K < 0 || K % 32 != 0) return ORC_ERR_SHAPE;
  const int64_t words = K / 32;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < words; ++j) {
      uint32_t word = 0;
      for (int i = 0; i < 32; ++i) {
        const int v = w[n * K + j * 32 + i];
        if (v != -1 && v != 0 && v != 1) return ORC_ERR_VALUE;
        const uint32_t bit = (v == 1) ? 1u : 0u;   /* b = (w+1)/2, zero -> -1 */
        word |= bit << i;
      }
      out[n * words + j] = (int32_t)word;
    }
  }
  return ORC_OK;
}

static int w1_weight(const int32_t* wq, int64_t K, int64_t n, int64_t k) {
  const uint32_t word = (uint32_t)wq[n * (K / 32) + k / 32];
  return ((word >> (k % 32)) & 1u) ? 1 : -1;
}

int orc_unpack_w1(const int32_t* wq, int64_t N, int64_t K, int8_t* w) {
  if (N < 0 || K < 0 || K % 32 != 0) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) w[n * K + k] = (int8_t)w1_weight(wq, K, n, k);
  return ORC_OK;
}

/*
 * W1A8 product ("binary-gemm": API binary_gemm, Method):
 *   dot[m,r,g] = sum_{k in group g} w[n,k] q[m,k]              (exact)
 *   y[m,r]     = s_act[m] * sum_g ws[n,g] * dot[m,r,g] + bias[n]  (fp64)
 * ws are fp16 bit patterns [N, K/G]; bias bf16 bit patterns [N] or NULL.
 * cond[m,r] = |s_act[m]| * sum_g |ws| sum_k |q| + |bias|.
 */
int orc_gemm_w1a8(const int8_t* q, const float* s_act, const int32_t* wq, const uint16_t* ws,
                  const uint16_t* bias, int64_t M, int64_t N, int64_t K, int64_t G,
                  const int64_t* rows, int64_t nrows, int64_t* dots, double* y, double* cond) {
  if (M < 0 || N < 0 || K < 0 || G <= 0 || K % 32 != 0 || K % G != 0) return ORC_ERR_SHAPE;
  const int64_t ng = K / G;
  int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static) reduction(| : bad)
#endif
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t n = rows ? rows[r] : r;
    if (n < 0 || n >= N) { bad |= 1; continue; }
    const double b = bias ? orc_bf16_to_double(bias[n]) : 0.0;
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0, c = 0.0;
      for (int64_t g = 0; g < ng; ++g) {
        int64_t dot = 0, qa = 0;
        for (int64_t k = g * G; k < (g + 1) * G; ++k) {
          dot += (int64_t)w1_weight(wq, K, n, k) * q[m * K + k];
          qa += abs(q[m * K + k]);
        }
        const double wsg = orc_fp16_to_double(ws[n * ng + g]);
        if (dots) dots[(m * nrows + r) * ng + g] = dot;
        acc += wsg * (double)dot;
        c += fabs(wsg) * (double)qa;
      }
      const double sm = (double)s_act[m];
      y[m * nrows + r] = sm * acc + b;
      if (cond) cond[m * nrows + r] = fabs(sm) * c + fabs(b);
    }
  }
  return bad ? ORC_ERR_SHAPE : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Per-token absmax activation quantization ("binary-gemm": API        */
/* quantize_activation, Correctness).  The pages give only "per-token  */
/* absmax" and the < 1% reconstruction bound; the reading taken here,  */
/* in IEEE binary32 with round-to-nearest-even everywhere:             */
/*   amax = max_k |x[m,k]|                                             */
/*   amax == 0  ->  q = 0, s = 0                                       */
/*   inv  = 127 / amax                                                 */
/*   q    = clamp(rint(x * inv), -127, 127)   (rint: ties to even)     */
/*   s    = amax / 127                                                 */
/* Inputs are fp32 (x32) or bf16 bit patterns (x16); exactly one is    */
/* non-NULL.  Compiled with floating-point contraction off so that     */
/* x * inv is one rounded multiply.                                    */
/* ------------------------------------------------------------------ */

static float bf16_to_float(uint16_t b) {
  return (float)orc_bf16_to_double(b);          /* exact: bf16 is a subset of binary32 */
}

int orc_quantize_act_absmax_int8(const float* x32, const uint16_t* x16, int64_t M, int64_t K,
                                 int8_t* q, float* s) {
  if (M < 0 || K <= 0 || (x32 == NULL) == (x16 == NULL)) return ORC_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float v = x32 ? x32[m * K + k] : bf16_to_float(x16[m * K + k]);
      const float a = fabsf(v);
      if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
      for (int64_t k = 0; k < K; ++k) q[m * K + k] = 0;
      s[m] = 0.0f;
      continue;
    }
    volatile float inv = 127.0f / amax;
    for (int64_t k = 0; k < K; ++k) {
      const float v = x32 ? x32[m * K + k] : bf16_to_float(x16[m * K + k]);
      volatile float t = v * inv;
      float r = rintf(t);
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q[m * K + k] = (int8_t)r;
    }
    volatile float sv = amax / 127.0f;
    s[m] = sv;
  }
  return ORC_OK;
}
