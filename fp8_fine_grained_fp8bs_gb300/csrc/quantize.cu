// Online absmax quantisation BF16 -> E4M3 + float32 scales.
//
// DeepSeek-V3 "Infrastructure" §3.3.2, "fine-grained quantization" and
// "online quantization"; formulas of the Figure 7 explainer: for each group
// s = absmax / 448 and code = round(x / s).  Exactly as the C ABI states:
// s = fl32(absmax / 448) and code = E4M3_rne_satfinite(fl32(x / s)), both
// quotients IEEE round-to-nearest; a group with s == 0 gets all-zero codes.
// Each quotient is the correctly rounded x / s, obtained from the
// reciprocal by Markstein's fused multiply-add correction (quant_pair
// below), so every byte is read once and written once and no element needs
// a division.
//
// Also here: the power-of-two scale mode (§3.3.3 "low-precision
// activations" (1)), the one-launch quantisation of both operands of an FP8
// Linear (X in 1x128 groups, then W in 128x128 blocks, by one persistent
// tile grid), the FP8 re-tiling 1x128 -> 128x1 of the backward pass
// (§3.5.2 "support for transposed GEMM operations"), and the fused SwiGLU ->
// 1x128 quantisation of the MoE down projection's input (§3.3.3 (2)).
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8bs {
namespace {

// Two float32 -> two E4M3 codes (RNE, saturating to +-448); a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Per-group divisor: s and y = RN(1/s).  Quotients use Markstein's
// correctly rounded division by a fused multiply-add correction (P.
// Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990):
//   q0 = RN(x * y),  r = x - s * q0 (exact by one FMA),  q1 = RN(q0 + r * y),
// which gives q1 = RN(x / s) when y = RN(1/s) and r does not underflow.  For
// every quotient that can give a non-zero E4M3 code (|x / s| >= 2^-10) r is
// exact once s >= 2^-93, and smaller quotients encode to a signed zero
// either way; groups with s < 2^-93 (and s == 0) take IEEE divisions.  An
// input of -0 yields q1 = +0, so the sign of x is ORed back into its code
// (a no-op for every other input, whose code already has x's sign).
struct Divisor {
  float s;
  float y;    // RN(1/s)
  bool fast;  // s >= 2^-93: Markstein path; otherwise IEEE divisions
};

constexpr float kMinFastScale = 1.0097419586828951e-28f;  // 2^-93

__device__ __forceinline__ Divisor make_divisor(float absmax) {
  Divisor d;
  d.s = __fdiv_rn(absmax, kE4M3Max);  // s = fl32(absmax / 448)
  d.fast = d.s >= kMinFastScale;      // false for s == 0
  d.y = __frcp_rn(d.fast ? d.s : 1.0f);
  return d;
}

// Table-driven divisor.  For a normal BF16 absmax a = (1 + f/128) * 2^e the
// scale is s = fl32(a / 448) = fl32((1 + f/128) / 448) * 2^e exactly, and
// RN(1/s) scales by 2^-e in the same way (scaling by a power of two
// commutes with rounding while everything stays normal).  So the 128
// values fl32((1 + f/128) / 448) and their reciprocals are computed once
// per block with the IEEE intrinsics and the per-group work is an exponent
// add.  Absmax values outside the range where s >= 2^-93 and 1/s is normal
// take make_divisor.
struct DivTable {
  uint32_t s[128];  // bits of fl32((1 + f/128) / 448)
  uint32_t y[128];  // bits of RN(1 / s)
};

__device__ __forceinline__ void div_table_init(DivTable& t) {
  for (int f = threadIdx.x; f < 128; f += blockDim.x) {
    const float sf = __fdiv_rn(1.0f + static_cast<float>(f) * (1.0f / 128.0f), kE4M3Max);
    t.s[f] = __float_as_uint(sf);
    t.y[f] = __float_as_uint(__frcp_rn(sf));
  }
}

// absmax given as BF16 bits (non-negative).
__device__ __forceinline__ Divisor table_divisor(const DivTable& t, uint32_t a16) {
  const uint32_t e = a16 >> 7;  // biased exponent of the absmax
  // biased exponents 43..254 give s >= 2^-93 with a normal reciprocal
  if (e < 43 || e > 254) return make_divisor(__uint_as_float(a16 << 16));
  const uint32_t f = a16 & 0x7Fu;
  const int sh = static_cast<int>(e) - 127;
  Divisor d;
  d.s = __uint_as_float(t.s[f] + (static_cast<uint32_t>(sh) << 23));
  d.y = __uint_as_float(t.y[f] - (static_cast<uint32_t>(sh) << 23));
  d.fast = true;
  return d;
}

// Power-of-two ("rounded") scale, §3.3.3 "low-precision activations" (1):
// s = 2^k, the smallest power of two with absmax / s <= 448, k >= -149 (the
// smallest positive float32).  y = 2^-k is then exact and so is x * y (the
// correction term vanishes); the same s >= 2^-93 bound as for any divisor
// selects the fast path.
__device__ __forceinline__ Divisor pow2_from_exp(int k) {
  k = max(k, -149);
  Divisor d;
  d.s = k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23) : __uint_as_float(1u << (k + 149));
  d.fast = k >= -93 && k <= 126;
  d.y = d.fast ? __uint_as_float(static_cast<uint32_t>(127 - k) << 23) : 1.0f;
  return d;
}

// absmax a = m * 2^e with m in [1, 2): a / 448 = (m / 1.75) * 2^(e - 8) and
// m / 1.75 lies in (0.5, 1.143), so k = e - 8, plus 1 when m > 1.75.
__device__ __forceinline__ Divisor pow2_divisor_f32(float a) {
  if (!(a > 0.0f)) {
    Divisor d;
    d.s = 0.0f;
    d.y = 1.0f;
    d.fast = false;
    return d;
  }
  uint32_t b = __float_as_uint(a);
  int bias = 0;
  if ((b >> 23) == 0) {  // subnormal: scale up by 2^64 (exact) and take it back from the exponent
    b = __float_as_uint(a * 18446744073709551616.0f);
    bias = 64;
  }
  const int e = static_cast<int>(b >> 23) - 127 - bias;
  return pow2_from_exp(e - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0));
}

// The same from BF16 absmax bits (1.75 = 1 + 96/128 in BF16's 7-bit fraction).
__device__ __forceinline__ Divisor pow2_divisor_bits(uint32_t a16) {
  const uint32_t e = a16 >> 7;
  if (e == 0) return pow2_divisor_f32(__uint_as_float(a16 << 16));
  return pow2_from_exp(static_cast<int>(e) - 127 - 8 + ((a16 & 0x7Fu) > 96u ? 1 : 0));
}

// Divisor of a group from its BF16 absmax bits, in the requested scale mode.
__device__ __forceinline__ Divisor group_divisor(const DivTable& t, uint32_t a16, bool pow2) {
  return pow2 ? pow2_divisor_bits(a16) : table_divisor(t, a16);
}

// Largest |x| of BF16 values: for non-negative floats the integer order of
// the bit patterns is the numeric order, so the magnitudes are compared as
// unsigned 16-bit pairs (two per instruction).
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Running |x| maximum of BF16 pairs, one instruction per word: the
// magnitude of max.xorsign.abs is max(|a|, |b|); its sign bit is junk that
// abs_bits clears once at the end.
__device__ __forceinline__ uint32_t absmax_step(uint32_t m, uint32_t w) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(m), "r"(w));
  return d;
}

__device__ __forceinline__ uint32_t abs_bits(uint32_t m) { return m & 0x7FFF7FFFu; }

__device__ __forceinline__ uint32_t absmax8_bits(uint4 v) {
  return abs_bits(absmax_step(absmax_step(v.x, v.y), absmax_step(v.z, v.w)));
}

// Codes of the BF16 pair w (low half first) in bits 0..15, by the
// Markstein quotient (see Divisor); ns2 = (-s, -s), y2 = (y, y).  The sign of
// a -0 input is restored by the caller (signs4).
__device__ __forceinline__ uint32_t quant_pair(uint32_t w, float2 y2, float2 ns2) {
  const float2 a = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  const float2 q0 = __fmul2_rn(a, y2);
  const float2 r = __ffma2_rn(q0, ns2, a);
  const float2 q1 = __ffma2_rn(r, y2, q0);
  return e4m3x2(q1.x, q1.y);
}

// Sign bits of the four BF16 values in words w0, w1 at bit 7 of the code
// bytes they map to (byte i = value i).
__device__ __forceinline__ uint32_t signs4(uint32_t w0, uint32_t w1) {
  return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// Codes of one value pair through IEEE divisions (x / s, then E4M3, sign
// from the quotient): groups whose scale is below 2^-93 or zero.
__device__ __forceinline__ uint32_t quant2_exact(uint32_t w, float s) {
  if (s == 0.0f) return 0u;
  return e4m3x2(__fdiv_rn(__uint_as_float(w << 16), s), __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), s));
}

// The BF16 pair w (low half first) widened to float32 and negated: -x is
// what quot_pair_nx takes.
__device__ __forceinline__ float2 neg_widen(uint32_t w) {
  return make_float2(__uint_as_float((w << 16) ^ 0x80000000u), __uint_as_float((w & 0xFFFF0000u) ^ 0x80000000u));
}

// Quotients x / s of a value pair given as nx = -x, with a divisor per half:
// s2 the scales, ny2 = -RN(1/s).  The same Markstein quotient as quant_pair
// with the signs moved: q0 = RN(nx * ny), r = RN(s q0 + nx) = -(x - s q0)
// (exact), q1 = RN(q0 + r * ny).  In this form a zero input keeps its sign
// (x = -0: q0 = -0, r = +0, q1 = -0 + -0 = -0), so no sign restoration
// follows; every other input gives the same q1 as quant_pair.
__device__ __forceinline__ float2 quot_pair_nx(float2 nx, float2 ny2, float2 s2) {
  const float2 q0 = __fmul2_rn(nx, ny2);
  const float2 r = __ffma2_rn(q0, s2, nx);
  return __ffma2_rn(r, ny2, q0);
}

// Quotients of the BF16 pair w through IEEE divisions, a scale per half (a
// zero scale gives +0, hence a zero code).
__device__ __forceinline__ float2 quot2_exact(uint32_t w, float s0, float s1) {
  return make_float2(s0 == 0.0f ? 0.0f : __fdiv_rn(__uint_as_float(w << 16), s0),
                     s1 == 0.0f ? 0.0f : __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), s1));
}

// Four float32 -> four E4M3 codes (RNE, saturating) packed in one word, a
// in the low byte: two conversions written into the two halves of the word.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n}\n"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Eight consecutive values of one group -> eight codes (byte i = value i).
__device__ __forceinline__ uint2 quant8m(uint4 v, const Divisor& d) {
  if (!d.fast)
    return make_uint2(quant2_exact(v.x, d.s) | (quant2_exact(v.y, d.s) << 16),
                      quant2_exact(v.z, d.s) | (quant2_exact(v.w, d.s) << 16));
  const float2 y2 = make_float2(d.y, d.y), ns2 = make_float2(-d.s, -d.s);
  const uint32_t c0 = quant_pair(v.x, y2, ns2), c1 = quant_pair(v.y, y2, ns2);
  const uint32_t c2 = quant_pair(v.z, y2, ns2), c3 = quant_pair(v.w, y2, ns2);
  return make_uint2(__byte_perm(c0, c1, 0x5410) | signs4(v.x, v.y), __byte_perm(c2, c3, 0x5410) | signs4(v.z, v.w));
}

// Word k (0..3) of a 16-byte vector.
__device__ __forceinline__ uint32_t word_of(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// ---------------------------------------------------------------------------
// Tile pipeline.  The BF16 input is cut into 128x128 tiles (128 rows of one
// 128-column block).  A producer warp (in the block-layout kernels: compute
// thread 0) streams the tiles with TMA into a ring of shared-memory stages;
// eight compute warps quantise each tile out of shared memory and store codes
// and scales with coalesced writes.  Loads are thereby decoupled from the
// arithmetic: several tiles per SM are in flight while the warps compute,
// which a load-then-compute kernel cannot sustain.
//
// Two thread layouts:
//  - row layout (1x128 groups, and weights without the transposed copy):
//    thread t owns the 64 values of half t%2 of tile row t/2, so a row's
//    absmax is one shuffle away and each thread derives one divisor per
//    tile.  TMA stores the two 64-column halves of the tile as separate
//    boxes with 128-byte swizzling (chunk i of a 128-byte row r lands at
//    chunk i ^ (r % 8)), and the thread's i-th load reads logical chunk
//    (i + 4 * half) % 8: the eight lanes of a quarter-warp then read eight
//    different bank groups.
//  - block layout (128x1 groups, transposed codes): thread t owns rows
//    8*(t/16) .. +7 of the 8-column chunk t%16 (an 8x8 sub-block whose
//    column codes are packed straight from the quotients, no transposes);
//    the tile is stored unswizzled and a quarter-warp reads 128 consecutive
//    bytes of a row.
enum TileMode : int {
  kModeAct = 0,      // 1x128 groups, row layout
  kModeWeight = 1,   // one 128x128 group per tile, row layout
  kModeWeightT = 2,  // one 128x128 group per tile plus the transposed codes, block layout
  kModeDual = 3,     // 1x128 and 128x1 groups, block layout
  kModeActWeight = 4 // one launch over the tiles of X (1x128 groups) then of W (128x128), row layout
};

template <int kMode>
struct QCfg {
  static constexpr bool kRowLayout = kMode == kModeAct || kMode == kModeWeight || kMode == kModeActWeight;
  // block layouts also stage the transposed codes of a tile (16 KB) in
  // shared memory; two input stages keep two CTAs per SM
  static constexpr int kStages = kRowLayout ? 3 : 2;
  static constexpr int kStageOutBytes = kRowLayout ? 0 : kGroup * kGroup;
  static constexpr int kMinBlocks = 2;  // CTAs per SM the registers and shared memory are budgeted for
};

constexpr int kQComputeThreads = 256;
constexpr int kQThreads = kQComputeThreads + 32;  // + the producer warp
// Threads of a launch.  The block-layout kernels (dual, weight with the
// transposed copy) have no producer warp: their thread 0 issues the loads,
// so two CTAs of 8 warps (16 per SM, 4 per scheduler) leave each thread 128
// registers, which the quotients of a sub-block's two layouts need; 18 warps
// would leave 96.
template <int kMode>
constexpr bool q_inline_loads() { return kMode == kModeDual || kMode == kModeWeightT; }
template <int kMode>
constexpr int q_threads() { return q_inline_loads<kMode>() ? kQComputeThreads : kQThreads; }
constexpr int kTileBytes = kGroup * kGroup * 2;    // 32 KB of BF16
constexpr int kTileRowBytes = kGroup * 2;
constexpr int kQMaxStages = 3;

struct TileParams {
  int64_t rows;     // rows of the input (M, or N for a weight)
  int64_t nrb;      // row blocks, ceil(rows / 128)
  int nkb;          // column blocks, K / 128
  uint8_t* q;       // [rows][K] codes (1x128 groups, or the weight's blocks)
  float* s;         // act, dual: [nkb][rows]; weight: [nrb][nkb]
  uint8_t* q_t;     // dual: [K][rows] codes of the 128x1 groups; weight: transposed codes; or null
  float* s_t;       // dual: [nrb][K]; weight: [nkb][nrb]; or null
  uint64_t timeout_ns;
  int pow2;         // power-of-two scales instead of absmax / 448
};

struct QShared {
  uint64_t full[kQMaxStages];
  uint64_t empty[kQMaxStages];
  DivTable tab;
  uint32_t red[2][kQComputeThreads / 32];              // weight: per-warp maxima, by tile parity
  uint32_t colred[kQComputeThreads / 32][kGroup / 2];  // dual: per-warp column maxima, two per word
  float2 rowdiv[kGroup];                               // dual: per row (s, -RN(1/s))
  alignas(16) float col_s[kGroup];                     // dual: per column s (read as float4)
  alignas(16) float col_ny[kGroup];                    // dual: per column -RN(1/s) (read as float4)
};

template <int kMode>
constexpr int q_smem_bytes() {
  return QCfg<kMode>::kStages * kTileBytes + QCfg<kMode>::kStageOutBytes + static_cast<int>(sizeof(QShared)) + 1024;
}

__device__ int g_quant_status;

// Barrier over the 256 compute threads (named barrier 1; the producer warp
// never takes part) returning the AND of `v` over them.
__device__ __forceinline__ bool compute_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void compute_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// |x| maxima of the two halves of a packed BF16 pair, in both halves.
__device__ __forceinline__ uint32_t umax_halves(uint32_t m) { return umax16x2(m, __byte_perm(m, 0u, 0x1032)); }

// Row layout: quantises the thread's 64 values (32 words in load order) with
// one divisor and stores the 64 codes as four 16-byte writes.
__device__ __forceinline__ void quant_row64(const uint32_t (&w)[32], const Divisor& d, int h, uint8_t* out) {
  uint2 cc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) cc[i] = quant8m(make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]), d);
  // load order -> column order: the upper half started at chunk 4
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint2 a = cc[i], b = cc[i + 4];
    cc[i] = h ? b : a;
    cc[i + 4] = h ? a : b;
  }
#pragma unroll
  for (int p = 0; p < 4; ++p)
    *reinterpret_cast<uint4*>(out + 16 * p) = make_uint4(cc[2 * p].x, cc[2 * p].y, cc[2 * p + 1].x, cc[2 * p + 1].y);
}

// Tiles [0, p.nrb * p.nkb) are p's tensor (read through tmx); with
// kModeActWeight they are followed by pw's tensor (through tmw), quantised
// in 128x128 groups.  Other modes ignore tmw and pw.
template <int kMode>
__global__ void __launch_bounds__(q_threads<kMode>(), QCfg<kMode>::kMinBlocks)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                      const TileParams p, const TileParams pw) {
  using Q = QCfg<kMode>;
  griddep_launch_dependents();  // a GEMM launched behind this kernel may start its set-up
  extern __shared__ uint8_t qsmem_raw[];
  // 1024-byte aligned base, offset from the shared array itself so that the
  // compiler keeps the shared address space (shared loads and stores rather
  // than generic ones)
  uint8_t* tiles = qsmem_raw + ((1024u - (smem_u32(qsmem_raw) & 1023u)) & 1023u);
  // transposed codes of the current tile (block layouts): row R of the
  // tile's X^T part as 16 units of 8 codes, unit u stored at u ^ (R / 8)
  uint2 (*stg)[kGroup / 8] = reinterpret_cast<uint2 (*)[kGroup / 8]>(tiles + Q::kStages * kTileBytes);
  QShared& S = *reinterpret_cast<QShared*>(tiles + Q::kStages * kTileBytes + Q::kStageOutBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t ntiles_x = p.nrb * p.nkb;
  const int64_t ntiles = ntiles_x + (kMode == kModeActWeight ? pw.nrb * pw.nkb : 0);
  const int64_t K = static_cast<int64_t>(p.nkb) * kGroup;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Q::kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kQComputeThreads / 32);  // one arrival per compute warp
    }
    fence_barrier_init();
  }
  div_table_init(S.tab);
  __syncthreads();
  // Block-layout kernels' loads: thread 0 fills the ring here and refills a
  // stage once every thread has passed the tile's first barrier (all have
  // read the stage by then); it counts the loads it issued and the tiles it
  // saw land, so that after a timeout it waits for the copies still in flight.
  constexpr bool kInline = q_inline_loads<kMode>();
  int issued_inline = 0, consumed_inline = 0;
  if (kInline && threadIdx.x == 0) {
    prefetch_tmap(&tmx);
    for (int i = 0; i < Q::kStages; ++i) {
      const int64_t tile = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
      if (tile >= ntiles) break;
      const int64_t rb0 = tile / p.nkb;
      const int kb0 = static_cast<int>(tile - rb0 * p.nkb);
      mbar_arrive_expect_tx(&S.full[i], kTileBytes);
      tma_load_2d(tiles + i * kTileBytes, &tmx, &S.full[i], kb0 * kGroup, static_cast<int>(rb0 * kGroup));
      ++issued_inline;
    }
  }

  if (warp == kQComputeThreads / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmx);
      if (kMode == kModeActWeight) prefetch_tmap(&tmw);
    }
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    bool live = true;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      if (!__shfl_sync(0xffffffffu, mbar_wait(&S.empty[s], ph ^ 1u, p.timeout_ns), 0)) {
        live = false;
        break;
      }
      if (lane == 0) {
        const bool second = kMode == kModeActWeight && tile >= ntiles_x;
        const int64_t lt = second ? tile - ntiles_x : tile;
        const int nkb = second ? pw.nkb : p.nkb;
        const CUtensorMap* map = second ? &tmw : &tmx;
        const int64_t rb = lt / nkb;
        const int kb = static_cast<int>(lt - rb * nkb);
        uint8_t* dst = tiles + s * kTileBytes;
        mbar_arrive_expect_tx(&S.full[s], kTileBytes);
        if (Q::kRowLayout) {
          tma_load_2d(dst, map, &S.full[s], kb * kGroup, static_cast<int>(rb * kGroup));
          tma_load_2d(dst + kTileBytes / 2, map, &S.full[s], kb * kGroup + kGroup / 2, static_cast<int>(rb * kGroup));
        } else {
          tma_load_2d(dst, &tmx, &S.full[s], kb * kGroup, static_cast<int>(rb * kGroup));
        }
      }
      __syncwarp();
      ++issued;
      if (++s == Q::kStages) { s = 0; ph ^= 1u; }
    }
    if (!live) {
      if (lane == 0) atomicCAS(&g_quant_status, 0, kStatusTimeout);
      // the copies already issued land before the CTA may exit
      for (int i = 0; i < Q::kStages && i < issued; ++i) {
        int st = s - 1 - i;
        uint32_t q = ph;
        if (st < 0) { st += Q::kStages; q ^= 1u; }
        (void)mbar_wait(&S.full[st], q, p.timeout_ns);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- compute
  const int t = threadIdx.x;
  int s = 0;
  uint32_t ph = 0, par = 0;
  // (row block, column block) of the tile, advanced by the grid stride
  // without a division per tile
  const int64_t step_rb = static_cast<int64_t>(gridDim.x) / p.nkb;
  const int step_kb = static_cast<int>(gridDim.x - step_rb * p.nkb);
  int64_t rb = static_cast<int64_t>(blockIdx.x) / p.nkb;
  int kb = static_cast<int>(blockIdx.x - rb * p.nkb);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, par ^= 1u) {
    bool second = false;  // kModeActWeight: a tile of W
    if (kMode == kModeActWeight) {
      second = tile >= ntiles_x;
      const int64_t lt = second ? tile - ntiles_x : tile;
      const int nkb = second ? pw.nkb : p.nkb;
      rb = lt / nkb;
      kb = static_cast<int>(lt - rb * nkb);
    } else if (tile != blockIdx.x) {
      rb += step_rb;
      kb += step_kb;
      if (kb >= p.nkb) { kb -= p.nkb; ++rb; }
    }
    const bool ok = mbar_wait(&S.full[s], ph, p.timeout_ns);
    if (kInline && threadIdx.x == 0 && ok) ++consumed_inline;
    const int cur_s = s;
    const uint8_t* stage = tiles + s * kTileBytes;

    if (Q::kRowLayout) {
      const int r = t >> 1, h = t & 1, rsw = r & 7;  // 128-byte swizzle: chunk i of row r at i ^ (r % 8)
      const uint8_t* rowp = stage + h * (kTileBytes / 2) + r * 128;
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = (i + 4 * h) & 7;
        const uint4 v = ok ? *reinterpret_cast<const uint4*>(rowp + ((j ^ rsw) << 4)) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
      // the tile is in registers: hand the stage back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
      if (++s == Q::kStages) { s = 0; ph ^= 1u; }
      uint32_t m = w[0];
#pragma unroll
      for (int k = 1; k < 32; ++k) m = absmax_step(m, w[k]);
      m = umax_halves(abs_bits(m));
      m = umax16x2(m, __shfl_xor_sync(0xffffffffu, m, 1));  // the other half of the row
      const int64_t row = rb * kGroup + r;
      // the tensor this tile belongs to
      const int64_t rows = second ? pw.rows : p.rows;
      uint8_t* const q = second ? pw.q : p.q;
      float* const sc = second ? pw.s : p.s;
      const int64_t ld = second ? static_cast<int64_t>(pw.nkb) * kGroup : K;
      Divisor d;
      if (kMode == kModeWeight || second) {
#pragma unroll
        for (int o = 2; o <= 16; o <<= 1) m = umax16x2(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) S.red[par][warp] = m & 0xFFFFu;
        if (!compute_bar_and(ok)) {
          if (t == 0) atomicCAS(&g_quant_status, 0, kStatusTimeout);
          break;
        }
        uint32_t a = S.red[par][0];
#pragma unroll
        for (int i = 1; i < kQComputeThreads / 32; ++i) a = max(a, S.red[par][i]);
        d = group_divisor(S.tab, a, p.pow2 != 0);
        if (t == 0) sc[rb * (ld / kGroup) + kb] = d.s;
      } else {
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) atomicCAS(&g_quant_status, 0, kStatusTimeout);
          break;
        }
        d = group_divisor(S.tab, m & 0xFFFFu, p.pow2 != 0);
        if (h == 0 && row < rows) sc[static_cast<int64_t>(kb) * rows + row] = d.s;
      }
      if (row < rows) quant_row64(w, d, h, q + row * ld + static_cast<int64_t>(kb) * kGroup + 64 * h);
      continue;
    }

    // block layout
    const int g = t >> 4;  // row group: rows 8g .. 8g+7 of the tile
    const int c = t & 15;  // column chunk: columns 8c .. 8c+7 of the tile
    const uint8_t* src = stage + (8 * g) * kTileRowBytes + 16 * c;
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[j] = ok ? *reinterpret_cast<const uint4*>(src + j * kTileRowBytes) : make_uint4(0u, 0u, 0u, 0u);
    const int64_t r0 = rb * kGroup + 8 * g;                        // this thread's first row
    const int64_t c0 = static_cast<int64_t>(kb) * kGroup + 8 * c;  // and first column
    // the tile is in registers; its stage is refilled once every thread has
    // passed the tile's first barrier (refill below)
    static_assert(Q::kRowLayout || kInline, "the block layouts load in-kernel");
    if (++s == Q::kStages) { s = 0; ph ^= 1u; }

    // thread 0 of a block-layout kernel: load the CTA's tile kStages ahead
    // into the stage this tile came from
    auto refill = [&]() {
      if (kInline && t == 0) {
        const int64_t next = tile + static_cast<int64_t>(Q::kStages) * gridDim.x;
        if (next < ntiles) {
          const int64_t rbn = next / p.nkb;
          const int kbn = static_cast<int>(next - rbn * p.nkb);
          mbar_arrive_expect_tx(&S.full[cur_s], kTileBytes);
          tma_load_2d(tiles + cur_s * kTileBytes, &tmx, &S.full[cur_s], kbn * kGroup,
                      static_cast<int>(rbn * kGroup));
          ++issued_inline;
        }
      }
    };
    if (kMode == kModeWeightT) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = umax16x2(m, absmax8_bits(v[j]));
      m = umax_halves(m) & 0xFFFFu;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) S.red[par][warp] = m;
      if (!compute_bar_and(ok)) {
        if (t == 0) atomicCAS(&g_quant_status, 0, kStatusTimeout);
        break;
      }
      refill();
      uint32_t a = S.red[par][0];
#pragma unroll
      for (int i = 1; i < kQComputeThreads / 32; ++i) a = max(a, S.red[par][i]);
      const Divisor d = group_divisor(S.tab, a, p.pow2 != 0);
      if (t == 0) {
        p.s[rb * p.nkb + kb] = d.s;
        p.s_t[static_cast<int64_t>(kb) * p.nrb + rb] = d.s;
      }
      // one scale for the block: the codes of W^T are the same quotients,
      // packed by column
      const float2 ny2 = make_float2(-d.y, -d.y), s2 = make_float2(d.s, d.s);
      float2 q[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w = word_of(v[j], k);
          q[j][k] = d.fast ? quot_pair_nx(neg_widen(w), ny2, s2) : quot2_exact(w, d.s, d.s);
        }
        *reinterpret_cast<uint2*>(p.q + (r0 + j) * K + c0) = make_uint2(
            e4m3x4(q[j][0].x, q[j][0].y, q[j][1].x, q[j][1].y), e4m3x4(q[j][2].x, q[j][2].y, q[j][3].x, q[j][3].y));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        stg[8 * c + 2 * k][g ^ c] = make_uint2(e4m3x4(q[0][k].x, q[1][k].x, q[2][k].x, q[3][k].x),
                                               e4m3x4(q[4][k].x, q[5][k].x, q[6][k].x, q[7][k].x));
        stg[8 * c + 2 * k + 1][g ^ c] = make_uint2(e4m3x4(q[0][k].y, q[1][k].y, q[2][k].y, q[3][k].y),
                                                   e4m3x4(q[4][k].y, q[5][k].y, q[6][k].y, q[7][k].y));
      }
    } else {
      // dual: 1x128 groups, row 8g+j reducing over the 16 threads of a
      // half-warp (the maxima of rows 2i and 2i+1 travel packed in one word)
      uint32_t am[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        am[i] = __byte_perm(umax_halves(absmax8_bits(v[2 * i])), umax_halves(absmax8_bits(v[2 * i + 1])), 0x5410);
#pragma unroll
        for (int o = 1; o <= 8; o <<= 1) am[i] = umax16x2(am[i], __shfl_xor_sync(0xffffffffu, am[i], o));
      }
      // one divisor per row, computed by one thread of the row's half-warp
      // and shared through shared memory with the other fifteen
      bool fast = true;  // this thread's row or column divisor takes the quotient path
      if (c < 8) {
        uint32_t a16 = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j == c) a16 = (j & 1) ? (am[j >> 1] >> 16) : (am[j >> 1] & 0xFFFFu);
        const Divisor d = group_divisor(S.tab, a16, p.pow2 != 0);
        S.rowdiv[8 * g + c] = make_float2(d.s, -d.y);
        fast = d.fast;
        p.s[static_cast<int64_t>(kb) * p.rows + r0 + c] = d.s;
      }
      // 128x1 groups: word k of the thread's eight rows holds columns
      // 8c+2k and 8c+2k+1, so the column maxima over the sub-block are
      // running maxima over the rows; the two row groups of a warp meet by
      // one shuffle and the 16 warps' partial maxima in shared memory.
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t m = word_of(v[0], k);
#pragma unroll
        for (int j = 1; j < 8; ++j) m = absmax_step(m, word_of(v[j], k));
        m = abs_bits(m);
        m = umax16x2(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (lane < 16) S.colred[warp][4 * c + k] = m;
      }
      if (!compute_bar_and(ok)) {
        if (t == 0) atomicCAS(&g_quant_status, 0, kStatusTimeout);
        break;
      }
      refill();  // every thread has read this tile's stage
      if (t < kGroup) {  // one divisor per column
        uint32_t m = S.colred[0][t >> 1];
#pragma unroll
        for (int w = 1; w < kQComputeThreads / 32; ++w) m = umax16x2(m, S.colred[w][t >> 1]);
        const Divisor d = group_divisor(S.tab, (t & 1) ? (m >> 16) : (m & 0xFFFFu), p.pow2 != 0);
        S.col_s[t] = d.s;
        S.col_ny[t] = -d.y;
        fast = fast && d.fast;
        p.s_t[rb * K + static_cast<int64_t>(kb) * kGroup + t] = d.s;
      }
      // every row and column divisor of the tile on the quotient path, or
      // IEEE divisions for the whole tile
      const bool all_fast = compute_bar_and(fast);
      // Both layouts from one widening per value pair: the row quotients
      // with the row's divisor, the column quotients with the two columns'
      // divisors.  A row's codes are its quotients in order; the codes of
      // column 8c+2k for rows 8g+4jg .. +3 are the low halves of those rows'
      // column quotients of word k (the high halves: column 8c+2k+1), four
      // conversions packed into one word, so no byte transposes follow.
      const float4 cs_a = *reinterpret_cast<const float4*>(&S.col_s[8 * c]);
      const float4 cs_b = *reinterpret_cast<const float4*>(&S.col_s[8 * c + 4]);
      const float4 cy_a = *reinterpret_cast<const float4*>(&S.col_ny[8 * c]);
      const float4 cy_b = *reinterpret_cast<const float4*>(&S.col_ny[8 * c + 4]);
      const float2 cs2[4] = {make_float2(cs_a.x, cs_a.y), make_float2(cs_a.z, cs_a.w), make_float2(cs_b.x, cs_b.y),
                             make_float2(cs_b.z, cs_b.w)};
      const float2 cy2[4] = {make_float2(cy_a.x, cy_a.y), make_float2(cy_a.z, cy_a.w), make_float2(cy_b.x, cy_b.y),
                             make_float2(cy_b.z, cy_b.w)};
#pragma unroll
      for (int jg = 0; jg < 2; ++jg) {  // rows 8g+4jg .. 8g+4jg+3
        float2 cq[4][4];                // column quotients [row][word]
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * jg + jj;
          const float2 rd = S.rowdiv[8 * g + j];
          float2 rq[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t w = word_of(v[j], k);
            if (all_fast) {
              const float2 nx = neg_widen(w);
              rq[k] = quot_pair_nx(nx, make_float2(rd.y, rd.y), make_float2(rd.x, rd.x));
              cq[jj][k] = quot_pair_nx(nx, cy2[k], cs2[k]);
            } else {
              rq[k] = quot2_exact(w, rd.x, rd.x);
              cq[jj][k] = quot2_exact(w, cs2[k].x, cs2[k].y);
            }
          }
          *reinterpret_cast<uint2*>(p.q + (r0 + j) * K + c0) =
              make_uint2(e4m3x4(rq[0].x, rq[0].y, rq[1].x, rq[1].y), e4m3x4(rq[2].x, rq[2].y, rq[3].x, rq[3].y));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          reinterpret_cast<uint32_t*>(&stg[8 * c + 2 * k][g ^ c])[jg] =
              e4m3x4(cq[0][k].x, cq[1][k].x, cq[2][k].x, cq[3][k].x);
          reinterpret_cast<uint32_t*>(&stg[8 * c + 2 * k + 1][g ^ c])[jg] =
              e4m3x4(cq[0][k].y, cq[1][k].y, cq[2][k].y, cq[3][k].y);
        }
      }
    }
    // write the staged transposed codes: 8 threads per 128-byte row
    compute_bar();
#pragma unroll
    for (int it = 0; it < (Q::kRowLayout ? 0 : kGroup * kGroup / 16 / kQComputeThreads); ++it) {
      const int idx = it * kQComputeThreads + t;
      const int R = idx >> 3, k = idx & 7, cr = R >> 3;
      uint4 w = *reinterpret_cast<const uint4*>(&stg[R][2 * k]);
      if (cr & 1) w = make_uint4(w.z, w.w, w.x, w.y);
      const int kl = k ^ (cr >> 1);  // logical 16-byte chunk of the row
      *reinterpret_cast<uint4*>(p.q_t + (static_cast<int64_t>(kb) * kGroup + R) * p.rows + rb * kGroup + 16 * kl) = w;
    }
  }
  if (kInline && threadIdx.x == 0) {
    for (int i = consumed_inline; i < issued_inline; ++i)
      (void)mbar_wait(&S.full[i % Q::kStages], (i / Q::kStages) & 1u, p.timeout_ns);
  }
}

// Tensor map of a BF16 matrix [rows][ld] (cols used): 128x128 boxes, or for
// the row layout 128-row x 64-column boxes with 128-byte swizzling.
bool encode_bf16_tiles(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t cols, int64_t ld,
                       bool row_layout) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_layout ? kGroup / 2 : kGroup), static_cast<cuuint32_t>(kGroup)};
  cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), gdim, gstride, box,
                         estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         row_layout ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One persistent launch over p's tiles (and, for kModeActWeight, then over
// pw's tiles of the BF16 matrix w with leading dimension ldw).
template <int kMode>
cudaError_t launch_tiles(const uint16_t* x, int64_t ld, const TileParams& p, int sm_count, cudaStream_t stream,
                         const uint16_t* w = nullptr, int64_t ldw = 0, const TileParams* pw = nullptr) {
  const int64_t ntiles = p.nrb * p.nkb + (pw != nullptr ? pw->nrb * pw->nkb : 0);
  if (ntiles <= 0) return cudaSuccess;
  CUtensorMap map{}, map_w{};
  if (p.nrb > 0 &&
      !encode_bf16_tiles(&map, x, p.rows, static_cast<int64_t>(p.nkb) * kGroup, ld, QCfg<kMode>::kRowLayout))
    return cudaErrorInvalidValue;
  if (pw != nullptr && pw->nrb > 0 &&
      !encode_bf16_tiles(&map_w, w, pw->rows, static_cast<int64_t>(pw->nkb) * kGroup, ldw, QCfg<kMode>::kRowLayout))
    return cudaErrorInvalidValue;
  if (p.nrb <= 0) map = map_w;  // never read: p has no tiles
  if (pw == nullptr || pw->nrb <= 0) map_w = map;
  auto kern = quant_tile_kernel<kMode>;
  constexpr int smem = q_smem_bytes<kMode>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  static std::atomic<int> per_sm_cache[kMaxCachedDevices];  // co-resident CTAs per SM, per device
  int per_sm = 0;
  e = cached_per_device(
      per_sm_cache,
      [&](int* n) { return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, q_threads<kMode>(), smem); },
      &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t slots = static_cast<int64_t>(sm_count) * per_sm;
  const int grid = static_cast<int>(ntiles < slots ? ntiles : slots);
  TileParams none = p;
  none.nrb = 0;
  kern<<<grid, q_threads<kMode>(), smem, stream>>>(map, map_w, p, pw != nullptr ? *pw : none);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Re-tiling from FP8 (§3.5.2 "support for transposed GEMM operations": the
// backward pass reads the 1x128-quantised activations, dequantises them,
// transposes and requantises them in 128x1 groups; with power-of-two scales,
// §3.3.3 (1), this adds no quantisation error).  One 128x128 tile per step:
// thread t holds rows 8*(t/16) .. +7 of the 8-column chunk t%16 of the tile
// (eight 8-byte code rows, read coalesced straight from global memory, the
// next tile's already in flight), dequantises them with their row scales,
// reduces the column maxima (shuffle, then shared memory across the eight
// warps), and quantises each column's 8 values into 8 consecutive bytes of
// X^T.
constexpr int kRqThreads = 256;

struct RequantParams {
  const uint8_t* xq;  // [M][K] codes of the 1x128 groups
  const float* sx;    // [K/128][M] their scales, kb-major
  int64_t M, K;
  int nkb;
  int64_t ntiles;
  uint8_t* xq_t;      // [K][M] codes of the 128x1 groups
  float* sx_t;        // [M/128][K]
  int pow2;
};

// Eight float32 values, given negated (nv = -x), -> eight codes with one
// divisor: s and ny = -RN(1/s).  Markstein quotients in the sign-keeping form
// of quot_pair_nx (a zero input keeps its sign), IEEE divisions for a slow
// divisor.  With a power-of-two divisor on the fast path 1/s is exact, so
// RN(nv * ny) already is the correctly rounded quotient: one multiply.
__device__ __forceinline__ uint2 quant8f_nx(const float (&nv)[8], float s, float ny, bool fast, bool pow2) {
  float q[8];
  if (!fast) {
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = s == 0.0f ? 0.0f : __fdiv_rn(-nv[j], s);
  } else if (pow2) {
    const float2 ny2 = make_float2(ny, ny);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 r = __fmul2_rn(make_float2(nv[2 * j], nv[2 * j + 1]), ny2);
      q[2 * j] = r.x;
      q[2 * j + 1] = r.y;
    }
  } else {
    const float2 ny2 = make_float2(ny, ny), s2 = make_float2(s, s);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 r = quot_pair_nx(make_float2(nv[2 * j], nv[2 * j + 1]), ny2, s2);
      q[2 * j] = r.x;
      q[2 * j + 1] = r.y;
    }
  }
  return make_uint2(e4m3x4(q[0], q[1], q[2], q[3]), e4m3x4(q[4], q[5], q[6], q[7]));
}

__device__ __forceinline__ Divisor divisor_f32(float a, bool pow2) {
  return pow2 ? pow2_divisor_f32(a) : make_divisor(a);
}

__global__ void __launch_bounds__(kRqThreads, 2) requant_kernel(const RequantParams p) {
  griddep_launch_dependents();
  __shared__ float colred[kRqThreads / 32][kGroup];     // per-warp column maxima of |v|
  __shared__ float2 coldiv[kGroup];                     // per column: (s, -RN(1/s)); +1 in place of -RN(1/s): IEEE path
  // Output tile: row R of X^T's tile (tile column R) as 16 units of 8 codes;
  // unit u of row R is stored at u ^ (R / 8), so the 8-byte writes of a warp
  // (16 rows R = 8c+i, one unit each) hit 16 different bank pairs.
  __shared__ __align__(16) uint2 stg[kGroup][kGroup / 8];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int g = t >> 4, c = t & 15;
  uint2 nq[8];
  float4 ns[2];
  auto load = [&](int64_t tile, uint2 (&q)[8], float4 (&sc)[2]) {
    if (tile >= p.ntiles) return;
    const int64_t rb = tile / p.nkb;
    const int kb = static_cast<int>(tile - rb * p.nkb);
    const uint8_t* src = p.xq + (rb * kGroup + 8 * g) * p.K + static_cast<int64_t>(kb) * kGroup + 8 * c;
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = __ldg(reinterpret_cast<const uint2*>(src + j * p.K));
    const float4* sp = reinterpret_cast<const float4*>(p.sx + static_cast<int64_t>(kb) * p.M + rb * kGroup + 8 * g);
    sc[0] = __ldg(sp);
    sc[1] = __ldg(sp + 1);
  };
  load(blockIdx.x, nq, ns);
  for (int64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
    // dequantise, negated: v[i][j] = -x of column i, row j of the thread's
    // 8x8 sub-block (x = code * s_row, so -x = code * -s_row exactly)
    float v[8][8];
    {
      const float sr[8] = {-ns[0].x, -ns[0].y, -ns[0].z, -ns[0].w, -ns[1].x, -ns[1].y, -ns[1].z, -ns[1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w2[2] = {nq[j].x, nq[j].y};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
              static_cast<__nv_fp8x2_storage_t>((w2[h >> 1] >> (16 * (h & 1))) & 0xFFFFu), __NV_E4M3);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
          v[2 * h][j] = __fmul_rn(f.x, sr[j]);
          v[2 * h + 1][j] = __fmul_rn(f.y, sr[j]);
        }
      }
    }
    load(tile + gridDim.x, nq, ns);  // the next tile's codes and scales are in flight meanwhile
    const int64_t rb = tile / p.nkb;
    const int kb = static_cast<int>(tile - rb * p.nkb);
    // column maxima of |v|
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(v[i][j]));
      m[i] = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));  // the other row group of this warp
    }
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 8; ++i) colred[warp][8 * c + i] = m[i];
    }
    __syncthreads();
    if (t < kGroup) {
      // one divisor per column, shared with the 16 threads that quantise it
      float amax = colred[0][t];
#pragma unroll
      for (int w = 1; w < kRqThreads / 32; ++w) amax = fmaxf(amax, colred[w][t]);
      const Divisor d = divisor_f32(amax, p.pow2 != 0);
      coldiv[t] = make_float2(d.s, d.fast ? -d.y : 1.0f);
      p.sx_t[rb * p.K + static_cast<int64_t>(kb) * kGroup + t] = d.s;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 sd = coldiv[8 * c + i];
      stg[8 * c + i][g ^ c] = quant8f_nx(v[i], sd.x, sd.y, sd.y < 0.0f, p.pow2 != 0);
    }
    __syncthreads();
    // write the tile out: 8 threads per 128-byte row of X^T
#pragma unroll
    for (int it = 0; it < kGroup * kGroup / 16 / kRqThreads; ++it) {
      const int idx = it * kRqThreads + t;
      const int R = idx >> 3, k = idx & 7, cr = R >> 3;
      uint4 w = *reinterpret_cast<const uint4*>(&stg[R][2 * k]);
      if (cr & 1) w = make_uint4(w.z, w.w, w.x, w.y);
      const int kl = k ^ (cr >> 1);  // logical 16-byte chunk of the row
      *reinterpret_cast<uint4*>(p.xq_t + (static_cast<int64_t>(kb) * kGroup + R) * p.M + rb * kGroup + 16 * kl) = w;
    }
  }
}

// ---------------------------------------------------------------------------
// Fused SwiGLU -> 1x128 quantisation: the input of the MoE down projection
// (§3.3.3 "low-precision activations" (2): the SwiGLU input is cached and
// its output recomputed; the output feeds the FP8 down-projection GEMM).
// Fusing the cast into the producer removes the BF16 write and re-read of
// the SwiGLU output (the read-write-reread cost §3.5.2 names).  h [M][ldh]
// BF16 holds the gate projection in columns [0, I) and the up projection in
// [I, 2I).  Thread = 8 consecutive outputs of one row (16-byte loads of gate
// and up, the next ones in flight); the 16 lanes of a half-warp are one
// 1x128 group.  v = BF16_rne(silu(g) * u), silu(g) = g / (1 + exp(-g)) in
// FP32 (hardware base-2 exponential and reciprocal: relative error below
// 2^-16 for every gate), then the group is quantised exactly as
// fp8bs_quantize_act does with a BF16 input.
constexpr int kSgThreads = 256;

struct SwigluParams {
  const uint16_t* h;
  int64_t ldh, M, I;
  uint8_t* q;     // [M][I]
  float* s;       // [I/128][M], kb-major
  int64_t units;  // M * I / 8 (zero: nothing to do)
  int pow2;
};

// Hardware base-2 exponential and reciprocal, one instruction each
// (subnormal inputs and results flushed to zero).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Gates below -64 are redone by swiglu_far_negative when the fast form
// flushed: there 1 + e^-g exceeds 2^92 and, from about -87.3 on, its
// one-instruction reciprocal flushes to zero although silu(g) * u is still a
// normal number.  As BF16 bit patterns these gates are exactly the patterns
// above 0xC280 (-64.0; NaNs are outside the contract).
constexpr uint32_t kFarNegativeBits = 0xC280u;

// silu(g) * u for g < -64, where silu(g) = g e^g / (1 + e^g) and e^g < 2^-92,
// so silu(g) * u = g u e^g to well within 2^-24.  Evaluated without overflow
// or flushing: with g = mg 2^eg and u = mu 2^eu (frexp, exact),
// g log2(e) = n + f split by a two-part constant (log2 e = kHi + kLo, kHi with
// 15 significant bits so that g * kHi is exact for a BF16 g, n = rint of it,
// f in about [-0.5, 0.5]), the result is ldexp(mg mu 2^f, eg + eu + n): one
// rounding in mg mu 2^f (mg mu is exact), ex2's error, and ldexp's exact
// scaling (or its one rounding into the subnormal range).  Relative error
// about 2^-21.  Below g = -200 the value is under 2^-152 for every finite
// BF16 u, so it is a signed zero.
__device__ __forceinline__ float swiglu_far_negative(float g, float u) {
  constexpr float kLog2eHi = 1.44268798828125f;   // 23637 / 16384
  constexpr float kLog2eLo = 7.0526077e-06f;      // log2(e) - kLog2eHi, rounded to float32
  if (g < -200.0f) return -copysignf(0.0f, u);    // the sign of g * u (g < 0)
  int eg, eu;
  const float mg = frexpf(g, &eg);
  const float mu = frexpf(u, &eu);
  const float th = g * kLog2eHi;                   // exact
  const float n = rintf(th);
  const float f = __fadd_rn(th - n, g * kLog2eLo); // th - n exact
  return ldexpf(mg * mu * ex2_ftz(f), eg + eu + static_cast<int>(n));
}

// Two outputs v = BF16(silu(g) * u), silu(g) = g / (1 + e^-g) with
// e^-g = 2^(-g log2 e); the multiplies and the add run as packed FP32x2
// operations.  Relative error below 2^-16 wherever the reciprocal does not
// flush (the rounding of -g log2 e dominates: |g| log2(e) 2^-24 in the
// exponent); the smallest reciprocal is kept in *rmin, and a zero there
// means a gate below about -87.3 whose output swiglu8 redoes.  Flushing
// subnormals in ex2 and rcp changes nothing else: a subnormal e^-g only adds
// to 1, a subnormal g gives 2^0 = 1.
__device__ __forceinline__ uint32_t swiglu_pair(uint32_t gw, uint32_t uw, float& rmin) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float2 g = make_float2(__uint_as_float(gw << 16), __uint_as_float(gw & 0xFFFF0000u));
  const float2 u = make_float2(__uint_as_float(uw << 16), __uint_as_float(uw & 0xFFFF0000u));
  const float2 t = __fmul2_rn(g, make_float2(-kLog2e, -kLog2e));
  const float2 d = __fadd2_rn(make_float2(ex2_ftz(t.x), ex2_ftz(t.y)), make_float2(1.0f, 1.0f));
  const float2 r = make_float2(rcp_ftz(d.x), rcp_ftz(d.y));
  rmin = fminf(rmin, fminf(r.x, r.y));
  const float2 v = __fmul2_rn(__fmul2_rn(g, r), u);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);  // v.x in the low half
  return *reinterpret_cast<const uint32_t*>(&b);
}

// The outputs of the gates below -64 among 8 (g, up) pairs, redone with
// swiglu_far_negative; the others are kept from v.  Runs only for groups of
// 8 in which a reciprocal flushed, so it is kept out of line.
__device__ __noinline__ uint4 swiglu8_far_negative(const uint4 g, const uint4 up, uint4 v) {
  uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {up.x, up.y, up.z, up.w}, vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll 1
  for (int i = 0; i < 8; ++i) {
    const uint32_t sh = (i & 1) * 16;
    const uint32_t gb = (gw[i >> 1] >> sh) & 0xFFFFu;
    if (gb > kFarNegativeBits) {
      const float r = swiglu_far_negative(__uint_as_float(gb << 16), __uint_as_float(((uw[i >> 1] >> sh) & 0xFFFFu) << 16));
      const uint32_t rb = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(r)));
      vw[i >> 1] = (vw[i >> 1] & ~(0xFFFFu << sh)) | (rb << sh);
    }
  }
  return make_uint4(vw[0], vw[1], vw[2], vw[3]);
}

// Eight outputs (BF16 words of v) for the 8 gates in g and up values in up.
__device__ __forceinline__ uint4 swiglu8(const uint4& g, const uint4& up) {
  float rmin = 1.0f;
  uint4 v;
  v.x = swiglu_pair(g.x, up.x, rmin);
  v.y = swiglu_pair(g.y, up.y, rmin);
  v.z = swiglu_pair(g.z, up.z, rmin);
  v.w = swiglu_pair(g.w, up.w, rmin);
  if (rmin == 0.0f) v = swiglu8_far_negative(g, up, v);
  return v;
}

__global__ void __launch_bounds__(kSgThreads) swiglu_quant_kernel(const SwigluParams p) {
  griddep_launch_dependents();
  __shared__ DivTable tab;
  div_table_init(tab);
  __syncthreads();
  // Thread -> (row of a block of R rows, unit of that row); the units of a
  // row come in whole groups of 16, so every half-warp is one 1x128 group and
  // is entirely active or idle: shuffles use half-warp masks.  Rows with more
  // than 256 units are walked in steps of 256.  No per-element integer
  // division: the mapping is set up once.
  const int t = threadIdx.x;
  const int upr = static_cast<int>(p.I / 8);              // units (8 outputs) per row, a multiple of 16
  const int R = upr <= kSgThreads ? kSgThreads / upr : 1;  // rows per block iteration
  const int sub = upr <= kSgThreads ? t / upr : 0;
  const int u0 = upr <= kSgThreads ? t - sub * upr : t;
  if (sub >= R) return;                                    // idle half-warps (R * upr < 256)
  const uint32_t hmask = 0xFFFFu << (t & 16);
  const int64_t rstep = static_cast<int64_t>(gridDim.x) * R;
  auto process = [&](int64_t row, int u, const uint4& g, const uint4& up) {
    const uint4 v = swiglu8(g, up);
    uint32_t m = umax_halves(absmax8_bits(v)) & 0xFFFFu;
#pragma unroll
    for (int o = 1; o <= 8; o <<= 1) m = max(m, __shfl_xor_sync(hmask, m, o));  // the 16 lanes of a group
    const Divisor d = group_divisor(tab, m, p.pow2 != 0);
    *reinterpret_cast<uint2*>(p.q + row * p.I + u * 8) = quant8m(v, d);
    if ((u & 15) == 0) p.s[static_cast<int64_t>(u >> 4) * p.M + row] = d.s;
  };
  auto load = [&](int64_t row, int u, uint4& g, uint4& up) {
    const uint16_t* hrow = p.h + row * p.ldh + u * 8;
    g = __ldg(reinterpret_cast<const uint4*>(hrow));
    up = __ldg(reinterpret_cast<const uint4*>(hrow + p.I));
  };
  if (upr <= kSgThreads) {
    // one unit per row: the next row's loads are issued before this row is processed
    int64_t row = static_cast<int64_t>(blockIdx.x) * R + sub;
    uint4 ng = make_uint4(0u, 0u, 0u, 0u), nu = ng;
    if (row < p.M) load(row, u0, ng, nu);
    for (; row < p.M; row += rstep) {                      // uniform per half-warp
      const uint4 g = ng, up = nu;
      if (row + rstep < p.M) load(row + rstep, u0, ng, nu);
      process(row, u0, g, up);
    }
  } else {
    for (int64_t row = blockIdx.x; row < p.M; row += rstep) {
      for (int u = u0; u < upr; u += kSgThreads) {         // uniform per half-warp
        uint4 g, up;
        load(row, u, g, up);
        process(row, u, g, up);
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                      float* sx, bool pow2, int sm_count, uint64_t timeout_ns, cudaStream_t stream) {
  const TileParams p{M,       (M + kGroup - 1) / kGroup, static_cast<int>(K / kGroup), xq, sx, nullptr, nullptr,
                     timeout_ns, pow2 ? 1 : 0};
  return launch_tiles<kModeAct>(x, ldx, p, sm_count, stream);
}

cudaError_t launch_quantize_act_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                     float* sx, uint8_t* xq_t, float* sx_t, bool pow2, int sm_count,
                                     uint64_t timeout_ns, cudaStream_t stream) {
  const TileParams p{M, M / kGroup, static_cast<int>(K / kGroup), xq, sx, xq_t, sx_t, timeout_ns, pow2 ? 1 : 0};
  return launch_tiles<kModeDual>(x, ldx, p, sm_count, stream);
}

cudaError_t launch_quantize_weight(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* wq,
                                   float* sw, uint8_t* wq_t, float* sw_t, bool pow2, int sm_count,
                                   uint64_t timeout_ns, cudaStream_t stream) {
  const TileParams p{N, N / kGroup, static_cast<int>(K / kGroup), wq, sw, wq_t, sw_t, timeout_ns, pow2 ? 1 : 0};
  if (wq_t != nullptr) return launch_tiles<kModeWeightT>(w, ldw, p, sm_count, stream);
  return launch_tiles<kModeWeight>(w, ldw, p, sm_count, stream);
}

cudaError_t launch_quantize_act_weight(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, float* sx,
                                       const uint16_t* w, int64_t N, int64_t Kw, int64_t ldw, uint8_t* wq, float* sw,
                                       bool pow2, int sm_count, uint64_t timeout_ns, cudaStream_t stream) {
  const TileParams p{M,       (M + kGroup - 1) / kGroup, static_cast<int>(K / kGroup), xq, sx, nullptr, nullptr,
                     timeout_ns, pow2 ? 1 : 0};
  const TileParams pw{N, N / kGroup, static_cast<int>(Kw / kGroup), wq, sw, nullptr, nullptr, timeout_ns,
                      pow2 ? 1 : 0};
  return launch_tiles<kModeActWeight>(x, ldx, p, sm_count, stream, w, ldw, &pw);
}

cudaError_t launch_requant_1x128_to_128x1(const uint8_t* xq, const float* sx, int64_t M, int64_t K, uint8_t* xq_t,
                                          float* sx_t, bool pow2, int sm_count, cudaStream_t stream) {
  RequantParams p;
  p.xq = xq;
  p.sx = sx;
  p.M = M;
  p.K = K;
  p.nkb = static_cast<int>(K / kGroup);
  p.ntiles = (M / kGroup) * p.nkb;
  p.xq_t = xq_t;
  p.sx_t = sx_t;
  p.pow2 = pow2 ? 1 : 0;
  if (p.ntiles <= 0) return cudaSuccess;
  static std::atomic<int> per_sm_cache[kMaxCachedDevices];
  int per_sm = 0;
  const cudaError_t e = cached_per_device(
      per_sm_cache, [](int* n) { return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, requant_kernel, kRqThreads, 0); },
      &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t slots = static_cast<int64_t>(sm_count) * per_sm;
  requant_kernel<<<static_cast<int>(p.ntiles < slots ? p.ntiles : slots), kRqThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_quantize(const uint16_t* h, int64_t M, int64_t I, int64_t ldh, uint8_t* q, float* s,
                                   bool pow2, int sm_count, cudaStream_t stream) {
  SwigluParams p;
  p.h = h;
  p.ldh = ldh;
  p.M = M;
  p.I = I;
  p.q = q;
  p.s = s;
  p.units = M * (I / 8);
  p.pow2 = pow2 ? 1 : 0;
  if (p.units <= 0) return cudaSuccess;
  static std::atomic<int> per_sm_cache[kMaxCachedDevices];
  int per_sm = 0;
  const cudaError_t e = cached_per_device(
      per_sm_cache,
      [](int* n) { return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, swiglu_quant_kernel, kSgThreads, 0); },
      &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t upr = I / 8;
  const int64_t rows_per_block = upr <= kSgThreads ? kSgThreads / upr : 1;
  const int64_t need = (M + rows_per_block - 1) / rows_per_block;
  const int64_t slots = static_cast<int64_t>(sm_count) * per_sm;
  swiglu_quant_kernel<<<static_cast<int>(need < slots ? need : slots), kSgThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t quant_take_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_quant_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(int));
  }
  *status = v;
  return e;
}

}  // namespace fp8bs
