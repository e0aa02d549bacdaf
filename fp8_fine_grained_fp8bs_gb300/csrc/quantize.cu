// Online absmax quantisation BF16 -> E4M3 + float32 scales.
//
// DeepSeek-V3 "Infrastructure" §3.3.2, "fine-grained quantization" and
// "online quantization"; formulas of the Figure 7 explainer: for each group
// s = absmax / 448 and code = round(x / s).  Exactly as the C ABI states:
// s = fl32(absmax / 448) and code = E4M3_rne_satfinite(fl32(x / s)), both
// quotients IEEE round-to-nearest; a group with s == 0 gets all-zero codes.
// The per-element quotient is decided from a two-sided bracket of x * (1/s)
// (quant2 below), so the kernels stay HBM-bound streaming kernels: every
// byte is read once and written once, with coalesced 16-byte loads.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8bs {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two float32 -> two E4M3 codes (RNE, saturating to +-448); a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Per-group divisor s and a bracket [r_lo, r_hi] of 1/s (both float32).
struct Divisor {
  float s;
  float r_lo, r_hi;
  uint64_t r_lo2, r_hi2;  // {r_lo, r_lo} and {r_hi, r_hi} for packed FP32x2 multiplies
  bool fast;  // s is a normal float32; s == 0 and subnormal s take the exact path
};

__device__ __forceinline__ Divisor make_divisor(float absmax) {
  Divisor d;
  d.s = __fdiv_rn(absmax, kE4M3Max);  // s = fl32(absmax / 448)
  d.fast = d.s >= 1.17549435e-38f;    // FLT_MIN: 1/s is then a finite normal float
  const float s = d.fast ? d.s : 1.0f;
  d.r_lo = __frcp_rd(s);              // r_lo <= 1/s
  // r_hi >= 1/s: r_lo itself when 1/s is exact (r_lo * s == 1, tested
  // exactly by one fused multiply-add), else the next float up.
  d.r_hi = (fmaf(d.r_lo, s, -1.0f) == 0.0f) ? d.r_lo : __uint_as_float(__float_as_uint(d.r_lo) + 1u);
  asm("mov.b64 %0, {%1, %1};" : "=l"(d.r_lo2) : "f"(d.r_lo));
  asm("mov.b64 %0, {%1, %1};" : "=l"(d.r_hi2) : "f"(d.r_hi));
  return d;
}

// Table-driven divisor.  For a normal BF16 absmax a = (1 + f/128) * 2^e the
// scale is s = fl32(a / 448) = fl32((1 + f/128) / 448) * 2^e exactly, and
// the reciprocal brackets scale by 2^-e in the same way (scaling by a power
// of two commutes with rounding while everything stays normal).  So the
// 128 values fl32((1 + f/128) / 448), their RD reciprocals and the RU
// reciprocals are computed once per block with the IEEE intrinsics and the
// per-group work is an exponent add.  Zero, subnormal or huge absmax values
// take make_divisor.
struct DivTable {
  uint32_t s[128];     // bits of fl32((1 + f/128) / 448)
  uint32_t rlo[128];   // bits of RD(1 / s)
  uint32_t rhi[128];   // bits of RU(1 / s)
};

__device__ __forceinline__ void div_table_init(DivTable& t) {
  for (int f = threadIdx.x; f < 128; f += blockDim.x) {
    const float sf = __fdiv_rn(1.0f + static_cast<float>(f) * (1.0f / 128.0f), kE4M3Max);
    const float lo = __frcp_rd(sf);
    const float hi = (fmaf(lo, sf, -1.0f) == 0.0f) ? lo : __uint_as_float(__float_as_uint(lo) + 1u);
    t.s[f] = __float_as_uint(sf);
    t.rlo[f] = __float_as_uint(lo);
    t.rhi[f] = __float_as_uint(hi);
  }
}

// absmax given as BF16 bits (non-negative).
__device__ __forceinline__ Divisor table_divisor(const DivTable& t, uint32_t a16) {
  const uint32_t e = a16 >> 7;  // biased exponent of the absmax
  // the scale (about 2^(e-127) / 448) and the reciprocals stay normal for
  // biased exponents 10..254 of the absmax
  if (e < 10 || e > 254) return make_divisor(__uint_as_float(a16 << 16));
  const uint32_t f = a16 & 0x7Fu;
  const int sh = static_cast<int>(e) - 127;
  Divisor d;
  d.s = __uint_as_float(t.s[f] + (static_cast<uint32_t>(sh) << 23));
  d.r_lo = __uint_as_float(t.rlo[f] - (static_cast<uint32_t>(sh) << 23));
  d.r_hi = __uint_as_float(t.rhi[f] - (static_cast<uint32_t>(sh) << 23));
  d.fast = true;
  asm("mov.b64 %0, {%1, %1};" : "=l"(d.r_lo2) : "f"(d.r_lo));
  asm("mov.b64 %0, {%1, %1};" : "=l"(d.r_hi2) : "f"(d.r_hi));
  return d;
}

// E4M3 codes of fl32(x0 / s) and fl32(x1 / s) for the two BF16 values of
// `w` (x0 in the low half), without a division per element:
//   lo = RD(|x| * r_lo) <= |x| / s <= RU(|x| * r_hi) = hi,
// so the correctly rounded quotient fl32(|x| / s) lies in [lo, hi] too.
// Rounding to E4M3 (RNE, saturating) is monotonic, hence when lo and hi
// round to the same codes, so does fl32(|x| / s).  When an E4M3 rounding
// boundary falls inside the 2-3 ulp wide bracket (rare), or s is not a
// normal float, `bad` is set and the caller redoes the chunk with IEEE
// divisions (quant8_exact).  The sign is applied last: the quotient has
// x's sign, also for -0 and for results that round to zero.
__device__ __forceinline__ uint32_t quant2(uint32_t w, const Divisor& d, bool& bad) {
  const uint32_t aw = w & 0x7FFF7FFFu;
  const float2 a = make_float2(__uint_as_float(aw << 16), __uint_as_float(aw & 0xFFFF0000u));
  const float2 l = __fmul2_rd(a, make_float2(d.r_lo, d.r_lo));
  const float2 h = __fmul2_ru(a, make_float2(d.r_hi, d.r_hi));
  const uint32_t c = e4m3x2(l.x, l.y);
  bad |= (c != e4m3x2(h.x, h.y));
  return c | (__byte_perm(w, 0u, 0x4431) & 0x8080u);
}

// Largest |x| of BF16 values: for non-negative floats the integer order of
// the bit patterns is the numeric order, so the magnitudes are compared as
// unsigned 16-bit pairs (two per instruction).
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t absmax8_bits(uint4 v) {
  const uint32_t k = 0x7FFF7FFFu;
  return umax16x2(umax16x2(v.x & k, v.y & k), umax16x2(v.z & k, v.w & k));
}

// Packed |bf16| maximum -> float32.
__device__ __forceinline__ float absmax_to_f32(uint32_t m) {
  return __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
}

__device__ __forceinline__ float absmax8(uint4 v) { return absmax_to_f32(absmax8_bits(v)); }

// Eight consecutive values -> eight codes (byte i = value i).  The code
// pairs of both brackets are packed and compared; the sign bits of the
// inputs are gathered with one byte permute per word pair.  Bit j of
// `badmask` is set when pair j (values 2j, 2j+1) needs the exact path.
__device__ __forceinline__ uint2 quant8m(uint4 v, const Divisor& d, uint32_t& badmask) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const float2 rlo = make_float2(d.r_lo, d.r_lo), rhi = make_float2(d.r_hi, d.r_hi);
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // |x| of both halves as float32, times the brackets with rounding down
    // and up (packed FP32x2 multiplies)
    const uint32_t aw = w[j] & 0x7FFF7FFFu;
    const float2 a = make_float2(__uint_as_float(aw << 16), __uint_as_float(aw & 0xFFFF0000u));
    const float2 l = __fmul2_rd(a, rlo);
    const float2 h = __fmul2_ru(a, rhi);
    lo[j] = e4m3x2(l.x, l.y);
    hi[j] = e4m3x2(h.x, h.y);
    badmask |= (lo[j] != hi[j] || !d.fast) ? (1u << j) : 0u;
  }
  const uint32_t s0 = __byte_perm(w[0], w[1], 0x7531) & 0x80808080u;
  const uint32_t s1 = __byte_perm(w[2], w[3], 0x7531) & 0x80808080u;
  const uint32_t c0 = __byte_perm(lo[0], lo[1], 0x5410), c1 = __byte_perm(lo[2], lo[3], 0x5410);
  return d.s == 0.0f ? make_uint2(0u, 0u) : make_uint2(c0 | s0, c1 | s1);
}

__device__ __forceinline__ uint2 quant8(uint4 v, const Divisor& d, bool& bad) {
  uint32_t m = 0;
  const uint2 q = quant8m(v, d, m);
  bad |= m != 0u;
  return q;
}

// Codes of one value pair through IEEE divisions (x / s, then E4M3, sign
// from the quotient): the exact path for a pair whose bracket straddles an
// E4M3 rounding boundary.  Quotients of BF16 values close to such a
// boundary are common (about 0.4% of the values of normal data), so the
// fix-up is done per pair.
__device__ __forceinline__ uint32_t quant2_exact(uint32_t w, float s) {
  if (s == 0.0f) return 0u;
  return e4m3x2(__fdiv_rn(__uint_as_float(w << 16), s), __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), s));
}

// Patches the pairs flagged in `badmask` of an 8-code chunk.
__device__ __forceinline__ uint2 fix8(uint2 q, uint4 v, float s, uint32_t badmask) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[2] = {q.x, q.y};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (badmask & (1u << j)) {
      const uint32_t e = quant2_exact(w[j], s);
      const int sh = 16 * (j & 1);
      c[j >> 1] = (c[j >> 1] & ~(0xFFFFu << sh)) | (e << sh);
    }
  }
  return make_uint2(c[0], c[1]);
}

// The same codes through IEEE divisions, x / s then E4M3 (the fix-up path).
__device__ __forceinline__ uint32_t quant1_exact(uint32_t h, float s) {
  if (s == 0.0f) return 0u;
  const float q = __fdiv_rn(__uint_as_float(h << 16), s);
  return e4m3x2(q, 0.0f) & 0xFFu;
}

__device__ __forceinline__ uint2 quant8_exact(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = quant1_exact((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu), s);
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// 1x128 tiles.  A flat grid-stride stream over 16-value chunks: lane i of
// the grid owns values 16i..16i+15 of the row-major group enumeration (two
// 16-byte loads, one 16-byte store of codes), so eight consecutive lanes
// form one 128-value group and a warp covers four contiguous groups.  The
// (row, k-block) of a group comes from a multiply-high division by the
// number of k-blocks.  Each lane loads its next chunk before quantising the
// current one.
__device__ __forceinline__ void group_rc(uint32_t g, uint64_t magic, int nkb, uint32_t& m, uint32_t& kb) {
  // m = g / nkb with magic = ceil(2^40 / nkb): exact for g < 2^31, nkb < 512.
  m = magic ? static_cast<uint32_t>((static_cast<uint64_t>(g) * magic) >> 40) : g / static_cast<uint32_t>(nkb);
  kb = g - m * static_cast<uint32_t>(nkb);
}

struct Chunk16 {
  uint4 a, b;
};

__device__ __forceinline__ void chunk_load(Chunk16& c, const uint16_t* __restrict__ x, int64_t i, int64_t n16,
                                           uint64_t magic, int nkb, int64_t ldx) {
  if (i < n16) {
    uint32_t m, kb;
    group_rc(static_cast<uint32_t>(i >> 3), magic, nkb, m, kb);
    const uint16_t* p = x + static_cast<int64_t>(m) * ldx + static_cast<int64_t>(kb) * kGroup + (i & 7) * 16;
    c.a = ld_stream_16(p);
    c.b = ld_stream_16(p + 8);
  } else {
    c.a = make_uint4(0, 0, 0, 0);
    c.b = make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(256) quant_act_1x128_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                               int nkb, int64_t ldx, uint64_t magic,
                                                               uint8_t* __restrict__ xq, float* __restrict__ sx) {
  __shared__ DivTable tab;
  div_table_init(tab);
  __syncthreads();
  const int64_t n16 = M * nkb * 8;  // 16-value chunks
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t K = static_cast<int64_t>(nkb) * kGroup;
  // Warp-uniform trip count: every lane of a warp runs the same number of
  // steps (out-of-range chunks are zeros and are not stored), so the group
  // shuffles always see all 32 lanes.
  const int64_t warp_first = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  Chunk16 cur;
  chunk_load(cur, x, i, n16, magic, nkb, ldx);
  for (int64_t w0 = warp_first; w0 < n16; w0 += nthreads, i += nthreads) {
    Chunk16 nxt;
    chunk_load(nxt, x, i + nthreads, n16, magic, nkb, ldx);
    uint32_t am = umax16x2(absmax8_bits(cur.a), absmax8_bits(cur.b));
    am = umax16x2(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = umax16x2(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = umax16x2(am, __shfl_xor_sync(0xffffffffu, am, 4));
    const Divisor d = table_divisor(tab, max(am & 0xFFFFu, am >> 16));
    uint32_t bad_a = 0, bad_b = 0;
    uint2 qa = quant8m(cur.a, d, bad_a);
    uint2 qb = quant8m(cur.b, d, bad_b);
    if (bad_a) qa = fix8(qa, cur.a, d.s, bad_a);
    if (bad_b) qb = fix8(qb, cur.b, d.s, bad_b);
    if (i < n16) {
      uint32_t m, kb;
      group_rc(static_cast<uint32_t>(i >> 3), magic, nkb, m, kb);
      *reinterpret_cast<uint4*>(xq + static_cast<int64_t>(m) * K + static_cast<int64_t>(kb) * kGroup + (i & 7) * 16) =
          make_uint4(qa.x, qa.y, qb.x, qb.y);
      if ((i & 7) == 0) sx[static_cast<int64_t>(kb) * M + m] = d.s;
    }
    cur = nxt;
  }
}

// BF16 bits of column i (0..7) of an 8-value row chunk.
__device__ __forceinline__ uint32_t col16(const uint4& v, int i) {
  const uint32_t w = (i < 2) ? v.x : (i < 4) ? v.y : (i < 6) ? v.z : v.w;
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Codes of column i of rows 0..7 (one byte per row, row 0 lowest).
__device__ __forceinline__ uint2 quant_col8(const uint4 (&v)[8], int i, const Divisor& d, bool& bad) {
  bad |= !d.fast;
  uint32_t p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) p[j] = quant2(col16(v[2 * j], i) | (col16(v[2 * j + 1], i) << 16), d, bad);
  return d.s == 0.0f ? make_uint2(0u, 0u) : make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// Column i (0..7) of an 8x8 byte tile held as 8 rows of 8 bytes: byte j of
// the result is byte i of row j.
__device__ __forceinline__ uint2 byte_column(const uint2 (&q)[8], int i) {
  const int wsel = i >> 2;
  const uint32_t b = static_cast<uint32_t>(i & 3);
  const uint32_t sel = b | ((b + 4) << 4);  // byte b of the first word, byte b of the second
  uint32_t p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x0 = wsel ? q[2 * j].y : q[2 * j].x;
    const uint32_t x1 = wsel ? q[2 * j + 1].y : q[2 * j + 1].x;
    p[j] = __byte_perm(x0, x1, sel);
  }
  return make_uint2(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410));
}

// Exact fix-up of one 8-row column chunk, re-reading the BF16 inputs.
__device__ __noinline__ uint2 quant_col8_exact(const uint16_t* x, int64_t ld, float s) {
  uint32_t b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = quant1_exact(x[j * ld], s);
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// Exact fix-up of one 8-value row chunk, re-reading the BF16 inputs.
__device__ __noinline__ uint2 quant_row8_exact(const uint16_t* x, float s) {
  return quant8_exact(*reinterpret_cast<const uint4*>(x), s);
}

// ---------------------------------------------------------------------------
// 128x128 tile of X, written both as 1x128 groups (rows) and as 128x1
// groups (columns, stored transposed).  Thread t owns 8 consecutive rows
// (8*(t/16) ..) of one 8-column chunk (t%16), loaded as 8 coalesced 16-byte
// vectors; rows reduce across the 16 threads of a half-warp, columns across
// the 16 row groups (shuffle, then shared memory).
__global__ void __launch_bounds__(256) quant_act_dual_kernel(const uint16_t* __restrict__ x, int64_t M, int nkb,
                                                              int64_t ldx, uint8_t* __restrict__ xq,
                                                              float* __restrict__ sx, uint8_t* __restrict__ xq_t,
                                                              float* __restrict__ sx_t) {
  __shared__ float red[8][kGroup];
  __shared__ float scol[kGroup];
  const int t = threadIdx.x;
  const int c = t & 15;
  const int g = t >> 4;
  const int warp = t >> 5;
  const int64_t K = static_cast<int64_t>(nkb) * kGroup;
  const int64_t rb = blockIdx.x / nkb;
  const int64_t kb = blockIdx.x - rb * nkb;
  const int64_t r0 = rb * kGroup + 8 * g;
  const int64_t c0 = kb * kGroup + 8 * c;

  uint4 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = ld_stream_16(x + (r0 + j) * ldx + c0);

  // 1x128 groups: one per row.
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = absmax8(v[j]);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const Divisor d = make_divisor(a);
    bool bad = false;
    const uint2 q = quant8(v[j], d, bad);
    uint8_t* o = xq + (r0 + j) * K + c0;
    *reinterpret_cast<uint2*>(o) = q;
    if (bad) *reinterpret_cast<uint2*>(o) = quant_row8_exact(x + (r0 + j) * ldx + c0, d.s);
    if (c == 0) sx[kb * M + r0 + j] = d.s;
  }

  // 128x1 groups: one per column.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) a = fmaxf(a, __uint_as_float((col16(v[j], i) & 0x7FFFu) << 16));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
    if ((t & 16) == 0) red[warp][8 * c + i] = a;
  }
  __syncthreads();
  if (t < kGroup) {
    float a = red[0][t];
#pragma unroll
    for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][t]);
    scol[t] = a;
    sx_t[rb * K + kb * kGroup + t] = __fdiv_rn(a, kE4M3Max);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const Divisor d = make_divisor(scol[8 * c + i]);
    bool bad = false;
    const uint2 q = quant_col8(v, i, d, bad);
    uint8_t* o = xq_t + (c0 + i) * M + r0;
    *reinterpret_cast<uint2*>(o) = q;
    if (bad) *reinterpret_cast<uint2*>(o) = quant_col8_exact(x + r0 * ldx + c0 + i, ldx, d.s);
  }
}

// ---------------------------------------------------------------------------
// One 128x128 weight block per CTA: the block's absmax is reduced over all
// 256 threads, then every element is quantised with the one block scale.
// Optionally also writes the transposed codes (Dgrad uses W transposed).
__global__ void __launch_bounds__(256) quant_weight_kernel(const uint16_t* __restrict__ w, int nnb, int nkb,
                                                            int64_t ldw, uint8_t* __restrict__ wq,
                                                            float* __restrict__ sw, uint8_t* __restrict__ wq_t,
                                                            float* __restrict__ sw_t) {
  __shared__ float red[8];
  const int t = threadIdx.x;
  const int c = t & 15;
  const int g = t >> 4;
  const int64_t N = static_cast<int64_t>(nnb) * kGroup;
  const int64_t K = static_cast<int64_t>(nkb) * kGroup;
  const int64_t nb = blockIdx.x / nkb;
  const int64_t kb = blockIdx.x - nb * nkb;
  const int64_t r0 = nb * kGroup + 8 * g;
  const int64_t c0 = kb * kGroup + 8 * c;

  uint4 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = ld_stream_16(w + (r0 + j) * ldw + c0);
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) a = fmaxf(a, absmax8(v[j]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((t & 31) == 0) red[t >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  const Divisor d = make_divisor(a);
  if (t == 0) {
    sw[nb * nkb + kb] = d.s;
    if (sw_t != nullptr) sw_t[kb * nnb + nb] = d.s;
  }
  uint2 q[8];
  uint32_t bad_rows = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bool bad = false;
    q[j] = quant8(v[j], d, bad);
    bad_rows |= bad ? (1u << j) : 0u;
  }
  if (bad_rows) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (bad_rows & (1u << j)) q[j] = quant_row8_exact(w + (r0 + j) * ldw + c0, d.s);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) *reinterpret_cast<uint2*>(wq + (r0 + j) * K + c0) = q[j];
  if (wq_t != nullptr) {
    // One scale for the whole block, so the codes of W^T are the transposed
    // codes of W: transpose this thread's 8x8 byte tile in registers.
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(wq_t + (c0 + i) * N + r0) = byte_column(q, i);
  }
}

}  // namespace

cudaError_t launch_quantize_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                      float* sx, int sm_count, cudaStream_t stream) {
  const int nkb = static_cast<int>(K / kGroup);
  const int64_t n16 = M * nkb * 8;
  if (n16 >= (int64_t(1) << 34)) return cudaErrorInvalidValue;  // group index must fit 31 bits
  // ceil(2^40 / nkb): the multiply-high division is exact for nkb < 512
  const uint64_t magic = nkb < 512 ? ((uint64_t(1) << 40) + nkb - 1) / nkb : 0;
  static int per_sm = 0;  // resident 256-thread blocks per SM
  if (per_sm == 0) {
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_act_1x128_kernel, 256, 0);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
  }
  const int64_t blocks_needed = (n16 + 255) / 256;
  const int64_t max_blocks = static_cast<int64_t>(sm_count) * per_sm;
  const int blocks = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  if (blocks <= 0) return cudaSuccess;
  quant_act_1x128_kernel<<<blocks, 256, 0, stream>>>(x, M, nkb, ldx, magic, xq, sx);
  return cudaGetLastError();
}

cudaError_t launch_quantize_act_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                     float* sx, uint8_t* xq_t, float* sx_t, cudaStream_t stream) {
  const int nkb = static_cast<int>(K / kGroup);
  const int64_t tiles = (M / kGroup) * nkb;
  if (tiles <= 0) return cudaSuccess;
  quant_act_dual_kernel<<<static_cast<unsigned>(tiles), 256, 0, stream>>>(x, M, nkb, ldx, xq, sx, xq_t, sx_t);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weight(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* wq,
                                   float* sw, uint8_t* wq_t, float* sw_t, cudaStream_t stream) {
  const int nnb = static_cast<int>(N / kGroup);
  const int nkb = static_cast<int>(K / kGroup);
  const int64_t tiles = static_cast<int64_t>(nnb) * nkb;
  if (tiles <= 0) return cudaSuccess;
  quant_weight_kernel<<<static_cast<unsigned>(tiles), 256, 0, stream>>>(w, nnb, nkb, ldw, wq, sw, wq_t, sw_t);
  return cudaGetLastError();
}

}  // namespace fp8bs
