// Row movement of the MoE layer around the expert GEMMs: the FP8 dispatch
// and the BF16 combine (DeepSeek-V3 "Infrastructure" §3.3.3, low-precision
// communication: the activations before the MoE up-projection are quantised
// to FP8 with power-of-two scales before the dispatch, which the FP8 expert
// GEMMs then consume directly; the combine is kept in BF16).
//
//   * gather_q_rows: out row i = in row idx[i] of E4M3 codes [rows][H] and
//     its H/128 float32 scales, each side's scales in either layout
//     (kb-major [H/128][rows], as the GEMMs read them, or row-major
//     [rows][H/128], one contiguous record per row for an exchange);
//     idx[i] < 0 gives a zero row with zero scales (the padding of an
//     expert's segment to a multiple of 128 rows).
//   * scatter_q_rows: the same movement from the sender's side: in row r
//     goes to out rows pos[r][0..k), each read once and written k times
//     (the gather form reads a row k times, from L2 at best); a second list
//     names out rows to fill with zero codes and scales (padding).
//   * gather_bf16_rows: out row i = in row idx[i] of a BF16 matrix (zeros
//     for idx[i] < 0): the expert outputs put back in send order.
//   * moe_combine: out[t] = BF16(sum_j w[t][j] * y[idx[t][j]]) with the
//     products and the sum in FP32 (j ascending, one rounding to BF16);
//     idx[t][j] < 0 contributes nothing.
// All three are memory-bound copies: one warp per row, 16-byte accesses.
#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8bs {
namespace {

constexpr int kMoeThreads = 256;
constexpr int kMoeWarps = kMoeThreads / 32;
constexpr int kRowBatch = 4;  // 16-byte pieces per lane loaded before they are stored

__global__ void __launch_bounds__(kMoeThreads) gather_q_rows_kernel(const uint8_t* __restrict__ q,
                                                                     const float* __restrict__ s, int64_t rows_in,
                                                                     int64_t H, int s_in_kb_major,
                                                                     const int32_t* __restrict__ idx, int64_t rows_out,
                                                                     uint8_t* __restrict__ q_out,
                                                                     float* __restrict__ s_out, int s_out_kb_major) {
  griddep_launch_dependents();  // the grouped GEMM on the gathered rows may start its set-up
  const int lane = threadIdx.x & 31;
  const int64_t nkb = H / kGroup;
  const int64_t vec = H / 16;  // 16-byte pieces of a row of codes
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMoeWarps + (threadIdx.x >> 5); i < rows_out;
       i += static_cast<int64_t>(gridDim.x) * kMoeWarps) {
    const int32_t src = idx[i];
    const bool valid = src >= 0 && src < rows_in;
    const uint4* qi = reinterpret_cast<const uint4*>(q + (valid ? static_cast<int64_t>(src) : 0) * H);
    uint4* qo = reinterpret_cast<uint4*>(q_out + i * H);
    for (int64_t v0 = lane; v0 < vec; v0 += 32 * kRowBatch) {
      uint4 d[kRowBatch];  // the batch's loads in flight together
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u) {
        const int64_t v = v0 + 32 * u;
        d[u] = valid && v < vec ? __ldg(qi + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u)
        if (v0 + 32 * u < vec) qo[v0 + 32 * u] = d[u];
    }
    for (int64_t kb = lane; kb < nkb; kb += 32) {
      float sv = 0.0f;
      if (valid) sv = __ldg(s + (s_in_kb_major ? kb * rows_in + src : static_cast<int64_t>(src) * nkb + kb));
      s_out[s_out_kb_major ? kb * rows_out + i : i * nkb + kb] = sv;
    }
  }
}

__global__ void __launch_bounds__(kMoeThreads) scatter_q_rows_kernel(
    const uint8_t* __restrict__ q, const float* __restrict__ s, int64_t rows_in, int64_t H, int s_in_kb_major,
    const int32_t* __restrict__ pos, int k, const int32_t* __restrict__ zero_rows, int64_t n_zero, int64_t rows_out,
    uint8_t* __restrict__ q_out, float* __restrict__ s_out, int s_out_kb_major) {
  griddep_launch_dependents();  // the grouped GEMM on the scattered rows may start its set-up
  const int lane = threadIdx.x & 31;
  const int64_t nkb = H / kGroup;
  const int64_t vec = H / 16;
  const int64_t items = rows_in + n_zero;  // source rows, then padding rows
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMoeWarps + (threadIdx.x >> 5); i < items;
       i += static_cast<int64_t>(gridDim.x) * kMoeWarps) {
    if (i >= rows_in) {
      const int32_t dst = zero_rows[i - rows_in];
      if (dst < 0 || dst >= rows_out) continue;
      uint4* qo = reinterpret_cast<uint4*>(q_out + static_cast<int64_t>(dst) * H);
      for (int64_t v = lane; v < vec; v += 32) qo[v] = make_uint4(0u, 0u, 0u, 0u);
      for (int64_t kb = lane; kb < nkb; kb += 32)
        s_out[s_out_kb_major ? kb * rows_out + dst : static_cast<int64_t>(dst) * nkb + kb] = 0.0f;
      continue;
    }
    const int32_t* pr = pos + i * k;  // this row's destinations (the same address for every lane)
    const uint4* qi = reinterpret_cast<const uint4*>(q + i * H);
    for (int64_t v0 = lane; v0 < vec; v0 += 32 * kRowBatch) {
      uint4 d[kRowBatch];
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u) {
        const int64_t v = v0 + 32 * u;
        d[u] = v < vec ? __ldg(qi + v) : make_uint4(0u, 0u, 0u, 0u);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t dst = __ldg(pr + j);
        if (dst < 0 || dst >= rows_out) continue;
        uint4* qo = reinterpret_cast<uint4*>(q_out + static_cast<int64_t>(dst) * H);
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u)
          if (v0 + 32 * u < vec) qo[v0 + 32 * u] = d[u];
      }
    }
    for (int64_t kb = lane; kb < nkb; kb += 32) {
      const float sv = __ldg(s + (s_in_kb_major ? kb * rows_in + i : i * nkb + kb));
      for (int j = 0; j < k; ++j) {
        const int32_t dst = __ldg(pr + j);
        if (dst < 0 || dst >= rows_out) continue;
        s_out[s_out_kb_major ? kb * rows_out + dst : static_cast<int64_t>(dst) * nkb + kb] = sv;
      }
    }
  }
}

__global__ void __launch_bounds__(kMoeThreads) gather_bf16_rows_kernel(const uint16_t* __restrict__ y,
                                                                        int64_t rows_in, int64_t N,
                                                                        const int32_t* __restrict__ idx,
                                                                        int64_t rows_out, uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t vec = N / 8;  // 16-byte pieces of a row
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMoeWarps + (threadIdx.x >> 5); i < rows_out;
       i += static_cast<int64_t>(gridDim.x) * kMoeWarps) {
    const int32_t src = idx[i];
    const bool valid = src >= 0 && src < rows_in;
    const uint4* yi = reinterpret_cast<const uint4*>(y + (valid ? static_cast<int64_t>(src) : 0) * N);
    uint4* o = reinterpret_cast<uint4*>(out + i * N);
    for (int64_t v = lane; v < vec; v += 32) o[v] = valid ? __ldg(yi + v) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Eight BF16 values (a 16-byte piece) into FP32, added with weight w.
__device__ __forceinline__ void axpy8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(w, __uint_as_float(words[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, __uint_as_float(words[i] & 0xFFFF0000u), acc[2 * i + 1]);
  }
}

__global__ void __launch_bounds__(kMoeThreads) moe_combine_kernel(const uint16_t* __restrict__ y, int64_t rows_y,
                                                                   int64_t N, const int32_t* __restrict__ idx,
                                                                   const float* __restrict__ w, int64_t T, int k,
                                                                   uint16_t* __restrict__ out) {
  constexpr int kBatch = 8;  // expert rows whose loads are in flight together
  const int lane = threadIdx.x & 31;
  const int64_t vec = N / 8;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kMoeWarps + (threadIdx.x >> 5); t < T;
       t += static_cast<int64_t>(gridDim.x) * kMoeWarps) {
    const int32_t* it = idx + t * k;
    const float* wt = w + t * k;
    for (int64_t v = lane; v < vec; v += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int j0 = 0; j0 < k; j0 += kBatch) {
        // all of the batch's loads first, then the multiply-adds in j order
        uint4 val[kBatch];
        float wj[kBatch];
        bool okj[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u;
          const int32_t src = j < k ? it[j] : -1;
          const bool ok = src >= 0 && src < rows_y;
          okj[u] = ok;
          wj[u] = ok ? wt[j] : 0.0f;
          val[u] = ok ? __ldg(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(src) * N) + v)
                      : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (okj[u]) axpy8(acc, wj[u], val[u]);
      }
      uint4 r;
      uint32_t* rw = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        rw[i] = *reinterpret_cast<const uint32_t*>(&b);
      }
      reinterpret_cast<uint4*>(out + t * N)[v] = r;
    }
  }
}

// Grid: enough warps for every row, at most 8 CTAs of 256 threads per SM.
int grid_for_rows(int64_t rows, int sm_count) {
  const int64_t blocks = (rows + kMoeWarps - 1) / kMoeWarps;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  return static_cast<int>(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_gather_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, bool s_in_kb_major,
                                 const int32_t* idx, int64_t rows_out, uint8_t* q_out, float* s_out,
                                 bool s_out_kb_major, int sm_count, cudaStream_t stream) {
  if (rows_out <= 0) return cudaSuccess;
  gather_q_rows_kernel<<<grid_for_rows(rows_out, sm_count), kMoeThreads, 0, stream>>>(
      q, s, rows_in, H, s_in_kb_major ? 1 : 0, idx, rows_out, q_out, s_out, s_out_kb_major ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_scatter_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, bool s_in_kb_major,
                                  const int32_t* pos, int k, const int32_t* zero_rows, int64_t n_zero,
                                  int64_t rows_out, uint8_t* q_out, float* s_out, bool s_out_kb_major, int sm_count,
                                  cudaStream_t stream) {
  const int64_t items = rows_in + n_zero;
  if (items <= 0 || rows_out <= 0) return cudaSuccess;
  scatter_q_rows_kernel<<<grid_for_rows(items, sm_count), kMoeThreads, 0, stream>>>(
      q, s, rows_in, H, s_in_kb_major ? 1 : 0, pos, k, zero_rows, n_zero, rows_out, q_out, s_out,
      s_out_kb_major ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_gather_bf16_rows(const uint16_t* y, int64_t rows_in, int64_t N, const int32_t* idx,
                                    int64_t rows_out, uint16_t* out, int sm_count, cudaStream_t stream) {
  if (rows_out <= 0) return cudaSuccess;
  gather_bf16_rows_kernel<<<grid_for_rows(rows_out, sm_count), kMoeThreads, 0, stream>>>(y, rows_in, N, idx,
                                                                                          rows_out, out);
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const uint16_t* y, int64_t rows_y, int64_t N, const int32_t* idx, const float* w,
                               int64_t T, int k, uint16_t* out, int sm_count, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  moe_combine_kernel<<<grid_for_rows(T, sm_count), kMoeThreads, 0, stream>>>(y, rows_y, N, idx, w, T, k, out);
  return cudaGetLastError();
}

}  // namespace fp8bs
