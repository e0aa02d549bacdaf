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
  const float a0 = fabsf(bf16_lo(w)), a1 = fabsf(bf16_hi(w));
  const uint32_t c = e4m3x2(__fmul_rd(a0, d.r_lo), __fmul_rd(a1, d.r_lo));
  const uint32_t c_hi = e4m3x2(__fmul_ru(a0, d.r_hi), __fmul_ru(a1, d.r_hi));
  bad |= (c != c_hi);
  return d.s == 0.0f ? 0u : (c | ((w >> 8) & 0x80u) | ((w >> 16) & 0x8000u));
}

__device__ __forceinline__ float absmax8(uint4 v) {
  const float m0 = fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x)));
  const float m1 = fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)));
  const float m2 = fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z)));
  const float m3 = fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)));
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// Eight consecutive values -> eight codes (byte i = value i).
__device__ __forceinline__ uint2 quant8(uint4 v, const Divisor& d, bool& bad) {
  bad |= !d.fast;
  return make_uint2(quant2(v.x, d, bad) | (quant2(v.y, d, bad) << 16),
                    quant2(v.z, d, bad) | (quant2(v.w, d, bad) << 16));
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
// 1x128 tiles.  Eight lanes own one group: lane l holds elements 8l..8l+7
// and 64+8l..64+8l+7 (two 16-byte loads, each warp-wide load instruction
// covering four contiguous 128-byte segments); a warp owns four consecutive
// groups of the row-major (row, kb) enumeration, so consecutive warps stream
// consecutive memory.  Each thread keeps 2*kUnroll 16-byte loads in flight.
template <int kUnroll>
__global__ void __launch_bounds__(256) quant_act_1x128_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                               int nkb, int64_t ldx, uint8_t* __restrict__ xq,
                                                               float* __restrict__ sx) {
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;
  const int gl = lane & 7;
  const int64_t K = static_cast<int64_t>(nkb) * kGroup;
  const int64_t units = M * nkb;
  const int64_t quads = (units + 3) >> 2;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t q0 = warp0; q0 < quads; q0 += nwarps * kUnroll) {
    uint4 v0[kUnroll], v1[kUnroll];
    int64_t m[kUnroll], kb[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const int64_t u = 4 * (q0 + i * nwarps) + sub;
      ok[i] = u < units;
      m[i] = ok[i] ? u / nkb : 0;
      kb[i] = ok[i] ? u - m[i] * nkb : 0;
      const uint16_t* p = x + m[i] * ldx + kb[i] * kGroup + gl * 8;
      v0[i] = ok[i] ? ld_stream_16(p) : make_uint4(0, 0, 0, 0);
      v1[i] = ok[i] ? ld_stream_16(p + 64) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      float a = fmaxf(absmax8(v0[i]), absmax8(v1[i]));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
      const Divisor d = make_divisor(a);
      bool bad0 = false, bad1 = false;
      uint2 q0v = quant8(v0[i], d, bad0);
      uint2 q1v = quant8(v1[i], d, bad1);
      if (bad0) q0v = quant8_exact(v0[i], d.s);
      if (bad1) q1v = quant8_exact(v1[i], d.s);
      if (ok[i]) {
        uint8_t* o = xq + m[i] * K + kb[i] * kGroup + gl * 8;
        *reinterpret_cast<uint2*>(o) = q0v;
        *reinterpret_cast<uint2*>(o + 64) = q1v;
        if (gl == 0) sx[kb[i] * M + m[i]] = d.s;
      }
    }
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
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
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
  constexpr int kUnroll = 2;
  const int nkb = static_cast<int>(K / kGroup);
  const int64_t quads = (M * nkb + 3) / 4;
  const int64_t warps_needed = (quads + kUnroll - 1) / kUnroll;
  const int64_t blocks_needed = (warps_needed + 7) / 8;
  const int64_t max_blocks = static_cast<int64_t>(sm_count) * 8;  // 8 x 256 threads per SM
  const int blocks = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  if (blocks <= 0) return cudaSuccess;
  quant_act_1x128_kernel<kUnroll><<<blocks, 256, 0, stream>>>(x, M, nkb, ldx, xq, sx);
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
