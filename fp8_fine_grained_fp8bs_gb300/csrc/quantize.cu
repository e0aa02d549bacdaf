// Online absmax quantisation BF16 -> E4M3 + float32 scales.
//
// DeepSeek-V3 "Infrastructure" §3.3.2, "fine-grained quantization" and
// "online quantization"; formulas of the Figure 7 explainer: for each group
// s = absmax / 448 and code = round(x / s).  Exactly as the C ABI states:
// s = fl32(absmax / 448) and code = E4M3_rne_satfinite(fl32(x / s)), both
// divisions IEEE round-to-nearest (__fdiv_rn); a group with s == 0 gets
// all-zero codes.  The kernels are HBM-bound streaming kernels: every byte
// is read once and written once, with coalesced 16-byte loads.
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

// Quotient x / s rounded once to float32, then to E4M3; s == 0 gives code 0.
__device__ __forceinline__ uint32_t quant2(float a, float b, float s) {
  if (s == 0.0f) return 0u;
  return e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// 1x128 tiles.  A half-warp owns one group (16 lanes x 8 BF16 = 128 values,
// 256 contiguous bytes); a warp owns two consecutive groups of the
// row-major (row, kb) enumeration, so consecutive warps stream consecutive
// memory.  Each thread keeps kUnroll independent 16-byte loads in flight.
template <int kUnroll>
__global__ void __launch_bounds__(256) quant_act_1x128_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                               int nkb, int64_t ldx, uint8_t* __restrict__ xq,
                                                               float* __restrict__ sx) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int hl = lane & 15;
  const int64_t K = static_cast<int64_t>(nkb) * kGroup;
  const int64_t units = M * nkb;
  const int64_t pairs = (units + 1) >> 1;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t p0 = warp0; p0 < pairs; p0 += nwarps * kUnroll) {
    uint4 v[kUnroll];
    int64_t m[kUnroll], kb[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const int64_t u = 2 * (p0 + i * nwarps) + half;
      ok[i] = u < units;
      m[i] = ok[i] ? u / nkb : 0;
      kb[i] = ok[i] ? u - m[i] * nkb : 0;
      v[i] = ok[i] ? ld_stream_16(x + m[i] * ldx + kb[i] * kGroup + hl * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const float f0 = bf16_lo(v[i].x), f1 = bf16_hi(v[i].x), f2 = bf16_lo(v[i].y), f3 = bf16_hi(v[i].y);
      const float f4 = bf16_lo(v[i].z), f5 = bf16_hi(v[i].z), f6 = bf16_lo(v[i].w), f7 = bf16_hi(v[i].w);
      float a = fmaxf(fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))),
                      fmaxf(fmaxf(fabsf(f4), fabsf(f5)), fmaxf(fabsf(f6), fabsf(f7))));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
      const float s = __fdiv_rn(a, kE4M3Max);
      uint2 q;
      q.x = quant2(f0, f1, s) | (quant2(f2, f3, s) << 16);
      q.y = quant2(f4, f5, s) | (quant2(f6, f7, s) << 16);
      if (ok[i]) {
        *reinterpret_cast<uint2*>(xq + m[i] * K + kb[i] * kGroup + hl * 8) = q;
        if (hl == 0) sx[kb[i] * M + m[i]] = s;
      }
    }
  }
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

  float f[8][8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 v = ld_stream_16(x + (r0 + j) * ldx + c0);
    f[j][0] = bf16_lo(v.x); f[j][1] = bf16_hi(v.x); f[j][2] = bf16_lo(v.y); f[j][3] = bf16_hi(v.y);
    f[j][4] = bf16_lo(v.z); f[j][5] = bf16_hi(v.z); f[j][6] = bf16_lo(v.w); f[j][7] = bf16_hi(v.w);
  }

  // 1x128 groups: one per row.
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[j][i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const float s = __fdiv_rn(a, kE4M3Max);
    uint2 q;
    q.x = quant2(f[j][0], f[j][1], s) | (quant2(f[j][2], f[j][3], s) << 16);
    q.y = quant2(f[j][4], f[j][5], s) | (quant2(f[j][6], f[j][7], s) << 16);
    *reinterpret_cast<uint2*>(xq + (r0 + j) * K + c0) = q;
    if (c == 0) sx[kb * M + r0 + j] = s;
  }

  // 128x1 groups: one per column.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j][i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
    if ((t & 16) == 0) red[warp][8 * c + i] = a;
  }
  __syncthreads();
  if (t < kGroup) {
    float a = red[0][t];
#pragma unroll
    for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][t]);
    const float s = __fdiv_rn(a, kE4M3Max);
    scol[t] = s;
    sx_t[rb * K + kb * kGroup + t] = s;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float s = scol[8 * c + i];
    uint2 q;
    q.x = quant2(f[0][i], f[1][i], s) | (quant2(f[2][i], f[3][i], s) << 16);
    q.y = quant2(f[4][i], f[5][i], s) | (quant2(f[6][i], f[7][i], s) << 16);
    *reinterpret_cast<uint2*>(xq_t + (c0 + i) * M + r0) = q;
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

  float f[8][8];
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 v = ld_stream_16(w + (r0 + j) * ldw + c0);
    f[j][0] = bf16_lo(v.x); f[j][1] = bf16_hi(v.x); f[j][2] = bf16_lo(v.y); f[j][3] = bf16_hi(v.y);
    f[j][4] = bf16_lo(v.z); f[j][5] = bf16_hi(v.z); f[j][6] = bf16_lo(v.w); f[j][7] = bf16_hi(v.w);
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[j][i]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((t & 31) == 0) red[t >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  const float s = __fdiv_rn(a, kE4M3Max);
  if (t == 0) {
    sw[nb * nkb + kb] = s;
    if (sw_t != nullptr) sw_t[kb * nnb + nb] = s;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint2 q;
    q.x = quant2(f[j][0], f[j][1], s) | (quant2(f[j][2], f[j][3], s) << 16);
    q.y = quant2(f[j][4], f[j][5], s) | (quant2(f[j][6], f[j][7], s) << 16);
    *reinterpret_cast<uint2*>(wq + (r0 + j) * K + c0) = q;
  }
  if (wq_t != nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint2 q;
      q.x = quant2(f[0][i], f[1][i], s) | (quant2(f[2][i], f[3][i], s) << 16);
      q.y = quant2(f[4][i], f[5][i], s) | (quant2(f[6][i], f[7][i], s) << 16);
      *reinterpret_cast<uint2*>(wq_t + (c0 + i) * N + r0) = q;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                      float* sx, int sm_count, cudaStream_t stream) {
  constexpr int kUnroll = 4;
  const int nkb = static_cast<int>(K / kGroup);
  const int64_t pairs = (M * nkb + 1) / 2;
  const int64_t warps_needed = (pairs + kUnroll - 1) / kUnroll;
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
