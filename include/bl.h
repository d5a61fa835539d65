/*
 * bl.h -- C ABI of libbl, packed BitLinear products on NVIDIA GB300 (sm_103a).
 *
 * The library computes the BitLinear product y = scale * W x where W is
 * ternary {-1,0,+1} or binary {-1,+1} and stays packed in memory; weights are
 * decoded in registers inside the kernels and never written out.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory and keeps no per-call state.
 *  - Every call is asynchronous: it only enqueues kernels on `stream` (a
 *    cudaStream_t / CUstream handle passed as void*, NULL = legacy default
 *    stream) and returns.  Nothing inside a call synchronizes with the host.
 *  - Arguments are checked on the host BEFORE any launch; a failed check
 *    returns a status and launches nothing.  A shape that passes the checks
 *    but has no launch plan (a tile, the activation records or x do not fit
 *    in a CTA's shared memory, or a grid or tensor-map limit is exceeded)
 *    returns BL_ERR_UNSUPPORTED, also before any launch.  A launch failure
 *    returns BL_ERR_CUDA.  bl_last_error() gives a message for the calling
 *    thread.
 *  - Row-major layouts throughout.  bf16 and fp16 values are passed as their
 *    16-bit patterns (uint16_t); int32 words and fp32 scales are
 *    little-endian as in device memory.
 *  - Results are deterministic: repeated calls with the same inputs give
 *    bitwise identical outputs (fixed reduction order, no atomics on data).
 *  - Kernels never spin without bound.  A pipeline wait that exceeds its
 *    time limit (about one second) makes the kernel record a flag in the
 *    library's device error word and return; bl_device_error() reads it.
 *
 * Passages referred to below (page title, section):
 *  [BL]  "Hesper/Layers/BitLinear": "i2_s Packing Format", "BitLinear
 *        Mathematics", "High-Level API".
 *  [TQ]  "Hesper/Quantization/TQ2_0": "TQ2_0 Format", "Memory Layout Example".
 *  [BG]  "binary-gemm" card: "API", "Method", "Correctness",
 *        "Requirements and limits".
 */
#ifndef BL_H
#define BL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BL_OK = 0,
  BL_ERR_NULL = 1,         /* a required pointer is NULL                      */
  BL_ERR_SHAPE = 2,        /* a size is negative, zero where not allowed, or
                              not a multiple the format requires              */
  BL_ERR_ALIGN = 3,        /* a pointer is not aligned as documented          */
  BL_ERR_DTYPE = 4,        /* an unsupported bl_dtype value                   */
  BL_ERR_UNSUPPORTED = 5,  /* valid request outside what the library supports */
  BL_ERR_CUDA = 6          /* the CUDA runtime reported an error              */
} bl_status;

typedef enum {
  BL_F32 = 0,              /* IEEE binary32                                   */
  BL_BF16 = 1              /* bfloat16, passed as uint16_t bit patterns        */
} bl_dtype;

typedef void* bl_stream_t; /* a cudaStream_t / CUstream handle                */

/* Human-readable name of a status code (static string). */
const char* bl_status_string(bl_status s);

/* Message describing the last failed call on the calling host thread. */
const char* bl_last_error(void);

/*
 * Read the library's device error word (synchronizes the device).
 * *flags receives the OR of BL_DEVERR_* bits recorded since the last clear;
 * clear != 0 resets it to zero.  Returns BL_ERR_NULL if flags is NULL and
 * BL_ERR_CUDA if the read fails.
 */
#define BL_DEVERR_WAIT_TIMEOUT 0x1u   /* a pipeline wait exceeded its limit */
#define BL_DEVERR_RANGE 0x2u          /* an input value outside a kernel's stated range (see the entry point) */
bl_status bl_device_error(uint32_t* flags, int clear);

/*
 * Test aid for the failure path (no counterpart on the pages): the weight
 * waits of the i2_s GEMV kernels (bl_gemv_i2s, bl_gemv_i2s_residual,
 * bl_gemv_i2s_rmsnorm and bl_gemv_i2s_gate_up, in their one-CTA-per-SM
 * resident plan) launched afterwards give up after `ns` nanoseconds of
 * %globaltimer instead of the default second (ns = 0 restores the default;
 * the setting is process-wide and read at each launch).  With a test limit
 * the wait polls without the hardware's suspension, so a copy still in
 * flight runs the limit out.  A wait that gives up records
 * BL_DEVERR_WAIT_TIMEOUT, the kernel skips the rest of its work and its
 * outputs are unspecified; the waits that let a CTA's own copies land before
 * it exits keep the full second, so the kernel still returns cleanly.  Other
 * kernels keep the default limit.  Always returns BL_OK.
 */
bl_status bl_set_wait_limit(uint64_t ns);

/*
 * Allow back-to-back launches to overlap (programmatic dependent launch).
 * When enabled, the GEMV/GEMM kernels launched afterwards on any stream may
 * start while the previous kernel on the same stream is still running: they
 * fetch their PACKED WEIGHTS before waiting for that kernel, and wait for it
 * before reading activations or writing outputs.  Enable it only when no
 * kernel writes the weight buffers right before a product that reads them
 * (weights written by bl_pack_* must be followed by a stream-ordered event
 * or any other kernel first).  Default: disabled.  Process-wide setting.
 */
void bl_set_overlap(int enable);
int bl_get_overlap(void);

/* ------------------------------------------------------------------------ */
/* Packing (load time).                                                       */
/* ------------------------------------------------------------------------ */

/*
 * i2_s packing [BL "i2_s Packing Format"].
 *   w     : int8 [N, K] ternary values, row-major.  Values > 0 store +1,
 *           < 0 store -1, 0 stores 0 (code 0b11 is never produced).
 *   scale : the tensor's fp32 scale, stored after the codes.
 *   out   : uint8 [N*K/4 + 4].  Row n occupies bytes [n*K/4, (n+1)*K/4);
 *           element e of a row sits in byte (e/128)*32 + e%32 at bits
 *           (7-2t):(6-2t) with t = (e%128)/32; codes -1 -> 0b00, 0 -> 0b01,
 *           +1 -> 0b10.  The 4 bytes after the last row hold `scale`
 *           (little-endian).
 * Requires K % 128 == 0, N >= 1; `out` 16-byte aligned.
 */
bl_status bl_pack_i2s(const int8_t* w, float scale, int64_t N, int64_t K, uint8_t* out, bl_stream_t stream);

/*
 * TQ2_0 packing [TQ "TQ2_0 Format", "Memory Layout Example"].
 *   w      : int8 [N, K] ternary values (sign taken as for i2_s).
 *   d_fp16 : fp16 bit patterns [N, K/256], one scale per 256-element block.
 *   out    : uint8 [N * (K/256) * 66].  Blocks follow each other in K order
 *            within a row, rows follow each other.  A block is 64 code bytes
 *            then its fp16 scale (low byte first).  Element j of a block sits
 *            in byte j/4 at bits (2*(j%4)+1):(2*(j%4)), codes 0 -> 0b00,
 *            +1 -> 0b01, -1 -> 0b11 (0b10 is never produced).  The in-byte
 *            order is this library's reading of the page, which prints the
 *            code table and the 2*idx shift of its unpack helper but not the
 *            element order.
 * Requires K % 256 == 0, N >= 1; `out` and `d_fp16` 2-byte aligned.
 */
bl_status bl_pack_tq2_0(const int8_t* w, const uint16_t* d_fp16, int64_t N, int64_t K, uint8_t* out,
                        bl_stream_t stream);

/*
 * W1 sign-bit packing [BG "API" pack_weights, "Method", "Correctness"].
 *   w   : int8 [N, K]; values > 0 store bit 1 (+1), all others bit 0 (-1):
 *         zeros pack as -1, as the card states.
 *   out : int32 [N, K/32]; element k of a row sits at bit k%32 of word k/32
 *         (lowest bit first; the bit order is this library's reading).
 * Requires K % 32 == 0, N >= 1; `out` 4-byte aligned.
 */
bl_status bl_pack_w1(const int8_t* w, int64_t N, int64_t K, int32_t* out, bl_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Activation quantization.                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Per-token absmax int8 quantization [BG "API" quantize_activation,
 * "Correctness"].  For every row m of x [M, K] (fp32 or bf16), in binary32
 * with round-to-nearest-even:
 *   amax = max_k |x[m,k]|;  if amax == 0: q[m,:] = 0, s[m] = 0;
 *   otherwise inv = 127/amax, q[m,k] = clamp(rint(x[m,k]*inv), -127, 127),
 *   s[m] = amax/127.
 * (The card states only "per-token absmax" with under 1% reconstruction
 * error; this formula is the library's reading and meets that bound.)
 *   q : int8 [M, K];  s : fp32 [M].
 * Requires M >= 1, K >= 1.  x must be aligned to its element size, s to 4
 * bytes.
 * Non-finite inputs give unspecified q and s.
 */
bl_status bl_quantize_act_absmax_int8(const void* x, bl_dtype xt, int64_t M, int64_t K, int8_t* q, float* s,
                                      bl_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Products.                                                                  */
/* ------------------------------------------------------------------------ */

/*
 * i2_s GEMV, one token [BL "BitLinear Mathematics": y[i] = scale *
 * sum_j w[i,j] x[j]].
 *   packed : the i2_s tensor as written by bl_pack_i2s (codes + trailing
 *            fp32 scale, which the kernel reads from device memory).
 *   x      : [K] fp32 (xt = BL_F32) or bf16 (xt = BL_BF16).
 *   y      : [N] fp32 or bf16 (yt).  bf16 output is rounded to nearest even.
 * Accuracy: within each 128-element group x is carried as a fixed-point
 * integer of 22 bits below the group maximum's leading bit (fp32 input, or
 * bf16 input with fp32 output) or 14 bits (bf16 input and output); shapes
 * the tiled fallback kernel takes (a CTA's rows, records and partials do
 * not fit its shared memory, or x is not 16-byte aligned) carry fp32 input
 * in 30 bits.  bf16 values within 15 (22 bits) or 7 (14 bits) binades of the
 * group maximum are carried exactly; every other value, fp32 values
 * included, with an absolute error of at most 2^-23, 2^-15 (or, 30 bits,
 * 2^-31) times the group maximum.  Products and sums inside a group are exact
 * integers; the partial sums are converted to fp32 once each and added in
 * fp32, then rounded to bf16 if asked.  The error of y[i] is at most
 * rho |y[i]| + 1e-5 |scale| sum_j |w[i,j]| |x[j]| (rho = 1e-5 for fp32 output,
 * 2^-7 for bf16 output: twice its rounding), plus, for activations outside
 * the exact range, |scale| sum_g E max|x_g| sum_{j in g} |w[i,j]| with
 * E = 2^-23, 2^-15 or 2^-31 as above.
 * Requires K % 128 == 0, K <= 32768, N >= 1; `packed` 16-byte aligned; x
 * and y aligned to their element size.  Non-finite x gives unspecified y.
 */
bl_status bl_gemv_i2s(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N, int64_t K,
                      bl_stream_t stream);

/*
 * i2_s GEMV with the residual added [BL "M=1 warp-cooperative kernel with
 * fused residual add"]:  y[n] = residual[n] + scale * sum_j w[n,j] x[j].
 *   residual : [N] in y's dtype (yt); may alias y.
 * Otherwise as bl_gemv_i2s (the sum is formed in fp32, then rounded).
 */
bl_status bl_gemv_i2s_residual(const uint8_t* packed, const void* x, bl_dtype xt, const void* residual, void* y,
                               bl_dtype yt, int64_t N, int64_t K, bl_stream_t stream);

/*
 * Fused RMSNorm + i2_s GEMV + residual [BL "Fused RMSNorm + BitLinear +
 * Residual Add M=1 Kernel"]:
 *   rmsInv = 1 / sqrt(sum_j x[j]^2 / K + eps)
 *   y[n]   = residual[n] + scale * sum_j w[n,j] * (x[j] * rmsInv * rms_weight[j])
 *   rms_weight : [K] in x's dtype (xt).   residual : [N] in yt, or NULL (0).
 * rmsInv is computed in fp32 (fixed summation order, IEEE sqrt and
 * division); the normalized activations are fp32 and go through the same
 * per-group fixed-point path as bl_gemv_i2s.  Requirements as for
 * bl_gemv_i2s; rms_weight aligned to its element size.
 */
bl_status bl_gemv_i2s_rmsnorm(const uint8_t* packed, const void* x, bl_dtype xt, const void* rms_weight, float eps,
                              const void* residual, void* y, bl_dtype yt, int64_t N, int64_t K, bl_stream_t stream);

/*
 * Fused gate + up + ReLU^2 x mul of the MLP, one token [BL "Fused
 * Gate+Up+ReLU²×Mul M=1 Kernel"]:
 *   g[n] = scale_g * sum_j wg[n,j] x[j],   u[n] = scale_u * sum_j wu[n,j] x[j]
 *   h[n] = max(0, g[n])^2 * u[n]
 *   packed_gate, packed_up : two i2_s tensors of the same shape [N, K] as
 *            written by bl_pack_i2s (each with its own trailing scale).
 *   x : [K] fp32 or bf16 (xt).   h : [N] fp32 or bf16 (ht).
 * x is read once for both products.  Accuracy: g and u as bl_gemv_i2s
 * computes them with an fp32 result; h is formed in fp32 and rounded to bf16
 * if asked.  Requirements as for bl_gemv_i2s; both tensors 16-byte aligned.
 */
bl_status bl_gemv_i2s_gate_up(const uint8_t* packed_gate, const uint8_t* packed_up, const void* x, bl_dtype xt,
                              void* h, bl_dtype ht, int64_t N, int64_t K, bl_stream_t stream);

/*
 * TQ2_0 GEMV, one token [TQ "TQ2_0 Format"]:
 *   y[n] = sum_b d[n,b] * sum_{j<256} w[n,256b+j] x[256b+j].
 *   packed : as written by bl_pack_tq2_0.  x : [K] fp32 or bf16.  y : fp32 [N].
 * Accuracy as for bl_gemv_i2s (fp32 output), with one fixed-point exponent
 * per 256-element block.
 * Requires K % 256 == 0, N >= 1; `packed` 16-byte aligned, x and y aligned
 * to their element size.  An 8-row tile, the activation records and x share
 * a CTA's shared memory, which bounds K: with 227 KB per CTA (GB300), K <=
 * 32000 for bf16 x and K <= 22528 for fp32 x; longer rows (and any K above
 * 262144) return BL_ERR_UNSUPPORTED.
 */
bl_status bl_gemv_tq2_0(const uint8_t* packed, const void* x, bl_dtype xt, float* y, int64_t N, int64_t K,
                        bl_stream_t stream);

/*
 * W1A8 product [BG "API" binary_gemm, "Method"]:
 *   dot[m,n,g] = sum_{k in group g} w[n,k] q[m,k]              (exact int32)
 *   y[m,n]     = bf16( s[m] * sum_g f32(ws[n,g]) * dot[m,n,g] + bias[n] )
 *   q        : int8 [M, K] activations; s : fp32 [M] per-token scales.
 *   wq       : int32 [N, K/32] as written by bl_pack_w1.
 *   ws_fp16  : fp16 bit patterns [N, K/group].
 *   bias_bf16: bf16 bit patterns [N], or NULL for no bias.
 *   y_bf16   : bf16 bit patterns [M, N].
 *   group_dots: int32 [M, N, K/group] or NULL; when given, the exact group
 *              dot products are written too (a separate, slower kernel
 *              variant meant for verification).
 * The fp32 sum over groups runs in an order of the library's choosing.
 * M <= 8 runs a CUDA-core kernel (exact int32 group dots, dp4a): for one
 * token with group = 128 (K / 128 <= 512, N * K / 128 a multiple of 8) an
 * activation-stationary kernel whose threads keep a group of the token in
 * registers while the rows stream past, otherwise a row-tiled one; M > 8 runs
 * on the tensor cores with B = +-ws (exact fp16), every product exact and
 * the sum over K in fp32 (group_dots must then be NULL, and K % 128 == 0).
 * Requires M >= 1, K % 32 == 0, group % 32 == 0, K % group == 0, N >= 1;
 * at most 1024 groups per row, and for M > 8 K <= 132096 (BL_ERR_UNSUPPORTED
 * otherwise); q, wq, ws 16-byte aligned, the other pointers aligned to
 * their element size.  For M <= 8 the tokens' activation records sit in
 * shared memory, which bounds K further (at M = 8 about 12-16 K depending on
 * the group size, at M = 1 from 32 K to about 100 K); longer rows return
 * BL_ERR_UNSUPPORTED.
 */
bl_status bl_gemm_w1a8(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws_fp16,
                       const uint16_t* bias_bf16, int64_t M, int64_t N, int64_t K, int group, uint16_t* y_bf16,
                       int32_t* group_dots, bl_stream_t stream);

/*
 * W1A8 product with the activation quantization fused in
 * [BG "API" quantize_activation and binary_gemm, "Method"]:
 *   the same y as bl_quantize_act_absmax_int8(x) followed by bl_gemm_w1a8,
 *   bit for bit, in one launch: every CTA quantizes the M tokens itself.
 *   x : [M, K] fp32 or bf16 (xt), unquantized activations.
 *   wq, ws_fp16, bias_bf16, y_bf16 : as for bl_gemm_w1a8.
 * Decode sizes only: 1 <= M <= 8 (BL_ERR_UNSUPPORTED above; larger batches
 * take the two calls).  Otherwise the requirements of bl_gemm_w1a8 for
 * M <= 8: K % 32 == 0, group % 32 == 0, K % group == 0, at most 1024 groups
 * per row.  x, wq, ws 16-byte aligned.
 */
bl_status bl_gemm_w1a8_act(const void* x, bl_dtype xt, const int32_t* wq, const uint16_t* ws_fp16,
                           const uint16_t* bias_bf16, int64_t M, int64_t N, int64_t K, int group, uint16_t* y_bf16,
                           bl_stream_t stream);

/*
 * TQ2_0 product with int8 activations (large M) [TQ "TQ2_0 Format";
 * activations as BG "quantize_activation"]:
 *   y[m,n] = s[m] * sum_b f32(d[n,b]) * sum_{j<256} w[n,256b+j] q[m,256b+j]
 *   q : int8 [M, K];  s : fp32 [M];  packed : TQ2_0 tensor (bl_pack_tq2_0).
 *   y : fp32 [M, N].
 * Runs on the tensor cores with exact fp16 operands (q scaled by 4^-(k%4),
 * w*d by 4^(k%4)): every product is exactly q*w*d and the sum over K is
 * fp32 in an order of the library's choosing.  Block scales must satisfy
 * |d| < 1024 (fp16 subnormals included); a larger one sets BL_DEVERR_RANGE
 * in the device error word and its rows of y are undefined.  Tiles are 128
 * tokens: meant for M in the tens and above (one token is bl_gemv_tq2_0's
 * job).
 * Requires M, N >= 1, K % 256 == 0, K <= 2^24, a packed tensor under 2 GiB;
 * q, packed and y 16-byte aligned, s 4-byte aligned.
 */
bl_status bl_gemm_tq2_0_int8(const int8_t* q, const float* s, const uint8_t* packed, int64_t M, int64_t N, int64_t K,
                             float* y, bl_stream_t stream);

/*
 * i2_s product with int8 activations (prefill, large M)
 * [BL "BitLinear Mathematics"; activations as BG "quantize_activation"]:
 *   acc[m,n] = sum_k q[m,k] w[n,k]          (exact int32)
 *   y[m,n]   = f32(acc[m,n]) * s[m] * scale  (scale: the i2_s tensor scale)
 *   q : int8 [M, K];  s : fp32 [M];  packed : i2_s tensor (bl_pack_i2s).
 *   y : fp32 [M, N];  acc : int32 [M, N] or NULL (when given, also written).
 * Requires M >= 1, N >= 1, K % 128 == 0, K <= 131072 (then |acc| <= 128 K
 * <= 2^24 for any int8 q, so every partial sum stays exactly representable
 * in the fp32 tensor-core accumulator); all pointers 16-byte aligned.
 */
bl_status bl_gemm_i2s_int8(const int8_t* q, const float* s, const uint8_t* packed, int64_t M, int64_t N, int64_t K,
                           float* y, int32_t* acc, bl_stream_t stream);

/*
 * The i2_s prefill from unquantized activations, in one call
 * [BG "API" binary_linear = quantize_activation + the product;
 * BL "BitLinear Mathematics"]: bl_quantize_act_absmax_int8 then
 * bl_gemm_i2s_int8.
 *   x : [M, K] fp32 (xt = BL_F32) or bf16 (BL_BF16);  packed, y as for
 *   bl_gemm_i2s_int8.  The codes, scales and y are bit for bit those of the
 *   two calls.
 *   workspace : device memory of at least bl_gemm_i2s_int8_act_workspace(M,
 *   K) bytes, 256-byte aligned, zero-filled before its first use; owned by
 *   the caller.  It receives the int8 codes [M, K] at byte 256 and the
 *   scales (fp32 [M]) at the next 256-byte boundary after them; its first 8
 *   bytes are grid-barrier words that every call leaves as it found them.
 *   Calls that share a workspace must not overlap on the GPU.
 *   fuse : 0 runs the two launches through the workspace (the faster form on
 *   GB300: 22.1 us for 512 x 2560 bf16 tokens against 6912 rows); 1 fuses the
 *   quantization into the product's launch when M >= 64, K % 8 == 0, x's
 *   rows are 16-byte aligned and the product's CTAs (one per 128 x 192 tile)
 *   fit on the GPU at once: the CTAs quantize their share of the tokens, meet
 *   at a grid barrier (bounded: a timeout sets BL_DEVERR_WAIT_TIMEOUT) and
 *   run the product (23.3 us for the same shape); otherwise the two launches.
 * Requires what bl_gemm_i2s_int8 requires of M, N, K, packed and y; x
 * aligned to its element size.
 */
size_t bl_gemm_i2s_int8_act_workspace(int64_t M, int64_t K);
bl_status bl_gemm_i2s_int8_act(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N, int64_t K,
                               float* y, void* workspace, size_t workspace_bytes, int fuse, bl_stream_t stream);

/*
 * bl_gemm_i2s_int8_act without a workspace argument, for callers that
 * cannot allocate device memory: code handed only its input and output
 * pointers by a host program that owns all device memory (a plugin, an
 * inference server's callback), or a loop that must not call cudaMalloc
 * (it can synchronize the device and fail under memory pressure).  The pages
 * have no counterpart; this is an interface convenience.
 * The workspace is a static device array of
 * BL_GEMM_I2S_INT8_ACT_NOALLOC_WORKSPACE bytes inside the library, which
 * every GPU that loads the library holds until the process exits; nothing is
 * allocated at call time.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current): make that
 * first call before any stream capture.  All calls share the one array,
 * which keeps the last call's contents (the codes and scales of the last
 * call; each call rewrites them, and the single-launch form clears its
 * barrier words on the stream first), so calls that overlap on the GPU race
 * and give wrong results: issue them on one stream, or order them.
 * Arguments, results and fuse as for bl_gemm_i2s_int8_act.  Returns
 * BL_ERR_UNSUPPORTED, before any launch, when
 * bl_gemm_i2s_int8_act_workspace(M, K) exceeds the array (8 MiB: M * K up
 * to about 8.3 million, e.g. 2048 tokens with K = 3968).
 */
#define BL_GEMM_I2S_INT8_ACT_NOALLOC_WORKSPACE (8u << 20)
bl_status bl_gemm_i2s_int8_act_noalloc(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N,
                                       int64_t K, float* y, int fuse, bl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BL_H */
