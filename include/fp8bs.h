/*
 * fp8bs — fine-grained FP8 quantisation and block-scaled FP8 GEMM for
 * NVIDIA GB300 (sm_103a).  C ABI.
 *
 * The method is DeepSeek-V3's FP8 training scheme ("Infrastructure" §3.3):
 *   - §3.3.2 "fine-grained quantization": activations are scaled per 1x128
 *     tile (one token, 128 channels), weights per 128x128 block, and the
 *     scales vary along the GEMM's inner dimension;
 *   - §3.3.2 "online quantization": the max absolute value of each tile or
 *     block is computed when the tensor is used;
 *   - §3.3.2 "mantissa over exponents": every tensor is E4M3;
 *   - §3.3.2 "increasing accumulation precision" (Figure 7b): every
 *     N_C = 128 elements of K the tensor-core partial sum is promoted to
 *     FP32, multiplied by the two scales and accumulated;
 *   - the explicit formulas are the Figure 7 explainer's ("DeepSeek-V3 FP8
 *     动态量化", "Fine-grained quantization"): s = absmax / F_max,
 *     FP8(x) = round(x / s), out += MMA(FP8(x), FP8(w)) * s_x * s_w.
 * Precise readings used here: F_max = 448 (largest finite E4M3, OCP "FN"
 * encoding); round = nearest-even with saturation to +-448; x / s is an IEEE
 * float32 division; the stored scale is s as float32; a group whose absmax
 * is 0 gets s = 0 and all-zero codes.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates no device memory and never synchronises, except
 *     fp8bs_get_device_status().  Every call is asynchronous on `stream`
 *     (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Matrices are row-major.  BF16 is IEEE bfloat16 (uint16 bit patterns),
 *     E4M3 codes are bytes, scales are float32.
 *   - "kb-major" scale layout: the scale of row r and 128-column group kb
 *     is stored at s[kb * rows + r] (the rows of one group are contiguous).
 *   - Argument errors are returned before anything is launched.  All device
 *     pointers must be 16-byte aligned, every leading dimension in bytes a
 *     multiple of 16.  The current device must have compute capability
 *     10.3 (FP8BS_ERR_UNSUPPORTED_ARCH otherwise).
 *   - Every wait inside a kernel is bounded in time; a wait that expires, or
 *     a device-side argument check that fails, records a status that
 *     fp8bs_get_device_status() returns.
 *   - Inputs holding NaN or Inf are outside the contract.
 */
#ifndef FP8BS_H_
#define FP8BS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8BS_OK = 0,
  FP8BS_ERR_INVALID_ARG = 1,      /* NULL pointer, negative size, unknown enum value */
  FP8BS_ERR_SHAPE = 2,            /* a size breaks a multiple-of-128 rule */
  FP8BS_ERR_ALIGNMENT = 3,        /* pointer or leading dimension not 16-byte aligned */
  FP8BS_ERR_UNSUPPORTED_ARCH = 4, /* current device is not sm_103 */
  FP8BS_ERR_CUDA = 5,             /* a CUDA runtime or driver call failed */
  FP8BS_ERR_TIMEOUT = 6,          /* a bounded device wait expired */
  FP8BS_ERR_DEVICE_ARG = 7        /* a device-resident argument (group offsets) was invalid */
} fp8bs_status;

typedef enum { FP8BS_OUT_F32 = 0, FP8BS_OUT_BF16 = 1 } fp8bs_out_dtype;

typedef enum {
  /* B's scale is per 128x128 block: sb[(n / 128) * (K / 128) + kb], i.e. a
   * row-major [ceil(N/128)][K/128] array (weights, §3.3.2 (2)). */
  FP8BS_SCALE_BLOCK128x128 = 0,
  /* B's scale is per row and 1x128 group, kb-major: sb[kb * N + n] (both
   * operands are activations, as in the Wgrad GEMM, §3.3.1 / Figure 6). */
  FP8BS_SCALE_ROW1x128 = 1
} fp8bs_b_scale_kind;

typedef enum {
  /* s = fl32(absmax / 448), the Figure 7 explainer's s = absmax / F_max. */
  FP8BS_SCALE_ABSMAX = 0,
  /* Power-of-two ("rounded") scale, §3.3.3 "low-precision activations" (1)
   * and "low-precision communication": s = 2^k, the smallest power of two
   * with absmax / s <= 448 (k >= -149).  Used for activations that are later
   * re-tiled from 1x128 to 128x1, where it makes the re-tiling lossless. */
  FP8BS_SCALE_POW2 = 1
} fp8bs_scale_mode;

/*
 * Activation quantisation, 1x128 tiles (§3.3.2 "fine-grained quantization"
 * (1) and "online quantization"), optionally also 128x1 tiles of the same
 * input (§3.3.3 "low-precision activations" (1): the backward pass needs the
 * activations grouped along tokens; here they are quantised directly from
 * BF16 in the same pass).
 *
 *   x     [M][ldx] BF16, K columns used.                       (in)
 *   xq    [M][K]   E4M3 codes of the 1x128 tiles.              (out)
 *   sx    [K/128][M] float32, kb-major: sx[kb*M + m].          (out)
 *   xq_t  [K][M]   E4M3 codes of X^T grouped 1x128 along M,    (out, optional)
 *                  i.e. of the 128x1 tiles of X.
 *   sx_t  [M/128][K] float32, kb-major: sx_t[tb*K + k] is the   (out, optional)
 *                  scale of column k, rows 128*tb .. 128*tb+127.
 * Rules: K % 128 == 0; M >= 0 arbitrary, but M % 128 == 0 when xq_t/sx_t
 * are given (both or neither).  ldx >= K, ldx*2 % 16 == 0.
 * Codes and scales are bit-exact with the rule: s = fl32(absmax / 448),
 * code = E4M3_rne_satfinite(fl32(x / s)), s == 0 -> codes 0.
 */
int fp8bs_quantize_act(const void* x, int64_t M, int64_t K, int64_t ldx,
                       uint8_t* xq, float* sx, uint8_t* xq_t, float* sx_t,
                       void* stream);

/* fp8bs_quantize_act with a choice of scale (fp8bs_scale_mode): with
 * FP8BS_SCALE_POW2 every group's scale is a power of two and each code is
 * E4M3_rne_satfinite(x / s) (the quotient is exact).  Same arguments, rules
 * and errors otherwise; an unknown scale_mode is FP8BS_ERR_INVALID_ARG. */
int fp8bs_quantize_act_ex(const void* x, int64_t M, int64_t K, int64_t ldx,
                          uint8_t* xq, float* sx, uint8_t* xq_t, float* sx_t,
                          int scale_mode, void* stream);

/*
 * Weight quantisation, 128x128 blocks (§3.3.2 "fine-grained quantization"
 * (2); weights are quantised online too, "online quantization").
 *
 *   w     [N][ldw] BF16, K columns used.                        (in)
 *   wq    [N][K]   E4M3 codes.                                  (out)
 *   sw    [N/128][K/128] float32, row-major.                    (out)
 *   wq_t  [K][N]   the same codes transposed (optional): B operand of a  (out)
 *                  GEMM that uses the weight transposed (Dgrad, Figure 6).
 *   sw_t  [K/128][N/128] the scales transposed (optional, with wq_t).     (out)
 * Rules: N % 128 == 0, K % 128 == 0, ldw >= K, ldw*2 % 16 == 0.
 */
int fp8bs_quantize_weight(const void* w, int64_t N, int64_t K, int64_t ldw,
                          uint8_t* wq, float* sw, uint8_t* wq_t, float* sw_t,
                          void* stream);

/* fp8bs_quantize_weight with a choice of scale (fp8bs_scale_mode). */
int fp8bs_quantize_weight_ex(const void* w, int64_t N, int64_t K, int64_t ldw,
                             uint8_t* wq, float* sw, uint8_t* wq_t, float* sw_t,
                             int scale_mode, void* stream);

/*
 * Both operands of an FP8 Linear (Figure 6, the online quantisation of
 * §3.3.2) in one launch: X in 1x128 groups exactly as fp8bs_quantize_act_ex
 * without the transposed output, and W in 128x128 blocks exactly as
 * fp8bs_quantize_weight_ex without the transposed copy, with one
 * scale_mode for both.  Codes and scales are bit-identical to the two
 * separate calls; one persistent grid walks X's tiles, then W's.
 *
 *   x  [M][ldx] BF16, K columns;  xq [M][K];  sx [K/128][M] (kb-major).
 *   w  [N][ldw] BF16, Kw columns; wq [N][Kw]; sw [N/128][Kw/128].
 * Rules: the union of the two calls' rules (K, N, Kw multiples of 128,
 * 16-byte aligned pointers and leading dimensions); M == 0 or N == 0 leaves
 * that operand out; errors as those calls.
 */
int fp8bs_quantize_act_weight(const void* x, int64_t M, int64_t K, int64_t ldx,
                              uint8_t* xq, float* sx,
                              const void* w, int64_t N, int64_t Kw, int64_t ldw,
                              uint8_t* wq, float* sw, int scale_mode, void* stream);

/*
 * Backward re-tiling from FP8 (§3.5.2 "support for transposed GEMM
 * operations": read the 1x128-quantised activations, dequantise, transpose,
 * requantise in 128x1 tiles; §3.3.3 "low-precision activations" (1): with
 * power-of-two scales this adds no quantisation error):
 *
 *   v[m][k]       = fl32(dec(xq[m][k]) * sx[kb*M + m])        (kb = k / 128)
 *   group (k, tb) = v[128*tb .. 128*tb+127][k]
 *   sx_t[tb*K + k] = scale of the group (scale_mode), xq_t[k][m] = its codes.
 *
 *   xq    [M][K] E4M3, 1x128 groups.  sx [K/128][M] float32, kb-major.   (in)
 *   xq_t  [K][M] E4M3, 128x1 groups.  sx_t [M/128][K] float32.           (out)
 * The outputs have the layout of fp8bs_quantize_act's xq_t / sx_t, so they
 * feed the Wgrad GEMM (FP8BS_SCALE_ROW1x128) directly.
 * Rules: M % 128 == 0, K % 128 == 0; all pointers 16-byte aligned.
 */
int fp8bs_requant_1x128_to_128x1(const uint8_t* xq, const float* sx, int64_t M, int64_t K,
                                 uint8_t* xq_t, float* sx_t, int scale_mode, void* stream);

/*
 * Fused SwiGLU and 1x128 quantisation: the input of the MoE down projection
 * (§3.3.3 "low-precision activations" (2): the SwiGLU output feeds the
 * down-projection FP8 GEMM; doing the cast in the producer avoids writing and
 * re-reading the BF16 activation, the cost §3.5.2 names):
 *
 *   v[m][i] = BF16_rne( silu(h[m][i]) * h[m][I + i] ),  silu(g) = g / (1 + e^-g)
 *   (xq, sx) = the 1x128 quantisation of v, as fp8bs_quantize_act(_ex).
 *
 *   h   [M][ldh] BF16: the gate/up projection output, gate in columns [0, I),
 *       up in columns [I, 2I).                                        (in)
 *   q   [M][I] E4M3 codes.  s [I/128][M] float32, kb-major.            (out)
 * silu(gate) * up is evaluated in FP32 with a relative error below 2^-16 for
 * every gate (gates below -64 take an overflow-free form g * up * e^g),
 * so a value within that distance of a BF16 rounding boundary may round either
 * way; codes and scales are otherwise those of quantising the rounded v.
 * Rules: I % 128 == 0, ldh >= 2*I, ldh*2 % 16 == 0; pointers 16-byte aligned.
 */
int fp8bs_swiglu_quantize(const void* h, int64_t M, int64_t I, int64_t ldh,
                          uint8_t* q, float* s, int scale_mode, void* stream);

/*
 * Block-scaled FP8 GEMM, D = A * B^T with per-128-K-block dequantisation
 * (§3.3.2 "increasing accumulation precision", Figure 7b; Figure 7 explainer
 * formula out += MMA(FP8(x), FP8(w)) * s_x * s_w):
 *
 *   D[m][n] (+)= sum_kb  P_kb[m][n] * sa[kb*M + m] * s_b(n, kb),
 *   P_kb[m][n]  = sum_{k in 128*kb .. 128*kb+127} A[m][k] * B[n][k]
 * with P_kb computed on the tensor cores and the scaled sum in FP32.
 *
 *   a   [M][K] E4M3, K-major.   sa [K/128][M] float32, kb-major.
 *   b   [N][K] E4M3, K-major.   sb per sb_kind (see fp8bs_b_scale_kind).
 *   d   [M][N] FP32 or BF16 (round-to-nearest-even from FP32).
 *   accumulate: FP32 output only; non-zero -> D += result (Wgrad
 *   accumulation), zero -> D = result.
 * Rules: K % 128 == 0, K > 0; N % 128 == 0; M >= 0 arbitrary.
 */
int fp8bs_gemm(const uint8_t* a, const float* sa,
               const uint8_t* b, const float* sb, int sb_kind,
               void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
               int accumulate, void* stream);

/*
 * Grouped block-scaled FP8 GEMM for MoE experts (the expert GEMMs consume
 * FP8 activations dispatched per expert, §3.3.3 "low-precision
 * communication").  Rows [offsets[g], offsets[g+1]) of A belong to expert
 * g and are multiplied by expert g's weight:
 *
 *   D[r][n] = sum_kb P_kb[r][n] * sa[kb*M_total + r] * sb[g][n/128][kb]
 *
 *   a        [M_total][K] E4M3.  sa [K/128][M_total] float32, kb-major.
 *   offsets  DEVICE int32 [num_groups + 1]: non-decreasing, offsets[0] >= 0,
 *            every offset a multiple of 128, offsets[G] <= M_total.  Checked
 *            on the device: a violation skips the launch's work and records
 *            FP8BS_ERR_DEVICE_ARG.
 *   b        [num_groups][N][K] E4M3.  sb [num_groups][N/128][K/128].
 *   d        [M_total][N] FP32 or BF16; rows outside every group are not written.
 * Rules: K % 128 == 0, N % 128 == 0, 1 <= num_groups <= 512.
 */
int fp8bs_grouped_gemm(const uint8_t* a, const float* sa, int64_t M_total,
                       const int32_t* offsets, int num_groups,
                       const uint8_t* b, const float* sb,
                       void* d, int d_dtype, int64_t N, int64_t K, void* stream);

/*
 * The block-scaled FP8 GEMM for power-of-two scales, with the scales applied
 * by the tensor core: §3.5.2 (compute hardware) asks for tensor cores that
 * take the group scaling factors themselves, so that partial sums need not
 * be promoted to the CUDA cores for dequantisation; §3.3.2 notes the
 * microscaling formats of the Blackwell generation.  Here the MMA is
 * tcgen05.mma.kind::mxf8f6f4.block_scale: each group scale becomes an UE8M0
 * scale (an 8-bit biased exponent) repeated over the group's four
 * 32-element blocks of K, and all of K accumulates in FP32 in tensor memory.
 *
 *   D[m][n] (+)= sum_kb P_kb[m][n] * sa[kb*M + m] * s_b(n, kb)
 *
 * Same arguments, layouts, rules and errors as fp8bs_gemm, and the same
 * result up to FP32 summation order, for operands whose scales are all
 * powers of two: quantised with FP8BS_SCALE_POW2 (fp8bs_quantize_act_ex,
 * fp8bs_quantize_weight_ex, fp8bs_requant_1x128_to_128x1).  Every scale of
 * a row or column inside the output must be 0 (a group of zero codes) or a
 * power of two in [2^-127, 2^127]; any other value is detected on the device
 * and records FP8BS_ERR_DEVICE_ARG for fp8bs_get_device_status(), and D is
 * then undefined.  The quantisers produce scales below 2^-127 only for
 * groups whose absmax is below 448 * 2^-127; such operands need fp8bs_gemm.
 */
int fp8bs_gemm_pow2(const uint8_t* a, const float* sa,
                    const uint8_t* b, const float* sb, int sb_kind,
                    void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                    int accumulate, void* stream);

/*
 * Grouped (MoE) form of fp8bs_gemm_pow2: arguments, layouts, rules and
 * errors of fp8bs_grouped_gemm, scales as fp8bs_gemm_pow2.  The activations
 * dispatched to the experts carry power-of-two scales (§3.3.3
 * "low-precision communication"); the expert weights must be quantised with
 * FP8BS_SCALE_POW2 as well.
 */
int fp8bs_grouped_gemm_pow2(const uint8_t* a, const float* sa, int64_t M_total,
                            const int32_t* offsets, int num_groups,
                            const uint8_t* b, const float* sb,
                            void* d, int d_dtype, int64_t N, int64_t K, void* stream);

/* Layout of the float32 scales of a matrix of E4M3 codes [rows][H] (1x128
 * groups) in fp8bs_gather_q_rows. */
typedef enum {
  FP8BS_SCALES_KB_MAJOR = 0,  /* s[kb * rows + r]: the layout every GEMM reads */
  FP8BS_SCALES_ROW_MAJOR = 1  /* s[r * (H/128) + kb]: one contiguous record per row */
} fp8bs_scale_layout;

/*
 * Row gather of FP8 codes with their 1x128 scales, the data movement of the
 * MoE dispatch (§3.3.3 "low-precision communication": the activations are
 * quantised to FP8, with power-of-two scales, before they are dispatched to
 * the experts, so the FP8 bytes and scales are what moves; the expert GEMMs
 * consume them directly):
 *
 *   q_out[i][:] = q[idx[i]][:],  scales of out row i = scales of row idx[i];
 *   idx[i] < 0 (or >= rows_in): a row of zero codes with zero scales (the
 *   padding of an expert's segment to a multiple of 128 rows).
 *
 *   q      [rows_in][H] E4M3 codes.  s: float32 scales in s_in_layout.   (in)
 *   idx    DEVICE int32 [rows_out].                                       (in)
 *   q_out  [rows_out][H] E4M3.  s_out: float32 scales in s_out_layout.   (out)
 * Packing the rows a rank sends into one buffer per destination (row-major
 * scales: one record per row travels with it) and unpacking received rows
 * into the experts' padded segments (kb-major scales, as the grouped GEMM
 * reads them) are both this call.
 * Rules: H % 128 == 0; q, q_out 16-byte aligned; the layouts are
 * fp8bs_scale_layout values (FP8BS_ERR_INVALID_ARG otherwise).
 */
int fp8bs_gather_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, int s_in_layout,
                        const int32_t* idx, int64_t rows_out, uint8_t* q_out, float* s_out, int s_out_layout,
                        void* stream);

/*
 * Row scatter of FP8 codes with their 1x128 scales: the dispatch written from
 * the sender's side, each token row read once and written to each of its k
 * destinations (§3.3.3 "low-precision communication", as fp8bs_gather_q_rows):
 *
 *   for r < rows_in, j < k:  if 0 <= pos[r*k + j] < rows_out, out row
 *     pos[r*k + j] = q[r][:] with the scales of row r;
 *   for i < n_zero:  if 0 <= zero_rows[i] < rows_out, out row zero_rows[i] =
 *     zero codes with zero scales (the padding of an expert's segment).
 *
 *   q      [rows_in][H] E4M3 codes.  s: float32 scales in s_in_layout.   (in)
 *   pos    DEVICE int32 [rows_in][k]; zero_rows DEVICE int32 [n_zero]
 *          (NULL allowed when n_zero == 0).                               (in)
 *   q_out  [rows_out][H] E4M3.  s_out: float32 scales in s_out_layout.   (out)
 * Out rows named by neither list are left as they are; a row named more than
 * once gets one of its writes, which one is unspecified.
 * Rules: H % 128 == 0; 1 <= k <= 64; n_zero >= 0; q, q_out 16-byte aligned;
 * the layouts are fp8bs_scale_layout values (FP8BS_ERR_INVALID_ARG otherwise).
 */
int fp8bs_scatter_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, int s_in_layout,
                         const int32_t* pos, int k, const int32_t* zero_rows, int64_t n_zero, int64_t rows_out,
                         uint8_t* q_out, float* s_out, int s_out_layout, void* stream);

/*
 * Row gather of a BF16 matrix (the expert outputs put back in send order for
 * the combine, which §3.3.3 keeps in BF16):
 *   out[i][:] = y[idx[i]][:], zeros where idx[i] < 0 or >= rows_in.
 *   y [rows_in][N] BF16; idx DEVICE int32 [rows_out]; out [rows_out][N] BF16.
 * Rules: N % 8 == 0; y, out 16-byte aligned.
 */
int fp8bs_gather_bf16_rows(const void* y, int64_t rows_in, int64_t N, const int32_t* idx, int64_t rows_out,
                           void* out, void* stream);

/*
 * The MoE combine in BF16 (§3.3.3: the combine components stay in BF16):
 *   out[t][n] = BF16_rne( sum_{j<k} w[t][j] * y[idx[t][j]][n] ),
 * the products and the sum in FP32 (fused multiply-adds, j ascending) and one
 * rounding to BF16; idx[t][j] < 0 (or >= rows_y) contributes nothing.
 *   y    [rows_y][N] BF16: the expert outputs, one row per (token, expert).
 *   idx  DEVICE int32 [T][k]: the row of y holding token t's j-th expert output.
 *   w    DEVICE float32 [T][k]: the gate weights.
 *   out  [T][N] BF16.
 * Rules: N % 8 == 0; 1 <= k <= 64; y, out 16-byte aligned.
 */
int fp8bs_moe_combine(const void* y, int64_t rows_y, int64_t N, const int32_t* idx, const float* w, int64_t T, int k,
                      void* out, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status of the
 * current device: FP8BS_OK, FP8BS_ERR_TIMEOUT, FP8BS_ERR_DEVICE_ARG, or
 * FP8BS_ERR_CUDA if the synchronisation itself failed.
 */
int fp8bs_get_device_status(void* stream);

/* Diagnostic of the failure path: launches a kernel that waits, through the
 * same bounded mbarrier wait every kernel here uses, on a barrier nothing
 * arrives on.  After `timeout_us` microseconds (1 .. 10^7) the wait gives up,
 * the kernel records FP8BS_ERR_TIMEOUT and returns normally, so the next
 * fp8bs_get_device_status() reports FP8BS_ERR_TIMEOUT and the CUDA context
 * stays usable.  Returns FP8BS_OK once the kernel is launched. */
int fp8bs_selftest_wait_timeout(int64_t timeout_us, void* stream);

/*
 * Diagnostic, not part of the hot path: D = A B^T with the FP8 products of
 * all of K accumulated by the tensor core alone (no promotion to FP32
 * registers every 128 K, no scales), the configuration whose accumulation
 * precision DeepSeek-V3 §3.3.2 "Increasing accumulation precision" measures
 * (a maximum relative error near 2% for K = 4096 on H800).  Comparing its
 * result with the exact sum gives the same measurement on this GPU.
 *
 *   a  [M][K] E4M3, K-major;  b  [N][K] E4M3, K-major;  d  [M][N] float32.
 * Rules: M % 128 == 0, N % 256 == 0, K % 128 == 0, K > 0 (FP8BS_ERR_SHAPE);
 * pointers 16-byte aligned (FP8BS_ERR_ALIGNMENT).  Asynchronous on
 * `stream`; a bounded wait that expires records FP8BS_ERR_TIMEOUT for
 * fp8bs_get_device_status() and leaves d unwritten.  Caller owns all
 * buffers.
 */
int fp8bs_diag_gemm_unpromoted(const uint8_t* a, const uint8_t* b, float* d, int64_t M, int64_t N, int64_t K,
                               void* stream);

/* Sets the limit of every bounded device wait, in milliseconds (default
 * 2000; 0 restores the default).  Applies to launches made after the call. */
int fp8bs_set_wait_timeout_ms(int64_t ms);

/* Static, NUL-terminated description of a status code. */
const char* fp8bs_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H_ */
