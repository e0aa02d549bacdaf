// Diagnostic GEMM without promotion: D = A B^T over all of K accumulated in
// tensor memory by the tensor core alone, with no per-128-K hand-off to
// FP32 registers and no scales.  This is the configuration whose limited
// accumulation precision motivates DeepSeek-V3 §3.3.2 "Increasing
// accumulation precision" (on H800, about 14 bits kept, a maximum relative
// error near 2% for K = 4096); it measures what the same experiment gives on
// this chip.  Not part of the hot path and not tuned: one CTA per 128x256
// tile, operands copied into shared memory by plain loads, one k-block at a
// time.
#include "common.cuh"
#include "kernels.h"

namespace fp8bs {
namespace {

__device__ int g_diag_status;

constexpr int kDiagThreads = 128;
constexpr int kDiagM = 128;
constexpr int kDiagN = 256;
constexpr int kDiagK = 128;  // bytes of one k-block of a K-major E4M3 row
// Operand tiles (48 KB), the barrier and the TMEM slot, 1024-byte alignment
// slack; the request is padded to 100 KB so that at most two CTAs share an
// SM and their two 256-column TMEM allocations always fit.
constexpr int kDiagSmemUsed = (kDiagM + kDiagN) * kDiagK + 64 + 1024;
constexpr int kDiagSmem = 100 * 1024;
static_assert(kDiagSmemUsed <= kDiagSmem, "diagnostic shared memory");

// rows x 128 bytes of k-block kb of a K-major E4M3 matrix into shared memory,
// 16-byte chunk c of row r at chunk position c ^ (r % 8) (the 128-byte
// swizzle the MMA's shared-memory descriptor names).
__device__ __forceinline__ void copy_tile(uint8_t* dst, const uint8_t* src, int rows, int64_t K, int kb) {
  for (int i = threadIdx.x; i < rows * 8; i += kDiagThreads) {
    const int r = i >> 3, c = i & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(r) * K + kb * kDiagK + c * 16);
    *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
}

__global__ void __launch_bounds__(kDiagThreads, 1)
    unpromoted_gemm_kernel(const uint8_t* A, const uint8_t* B, float* D, int64_t N, int64_t K, uint64_t timeout_ns) {
  extern __shared__ uint8_t diag_raw[];
  uint8_t* smem = diag_raw + ((1024u - (smem_u32(diag_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kDiagM * kDiagK;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (kDiagM + kDiagN) * kDiagK);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kDiagM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kDiagN;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(slot, kDiagN);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *slot;
  constexpr uint32_t idesc = idesc_e4m3_f32(kDiagM, kDiagN);
  const int nkb = static_cast<int>(K / kDiagK);
  bool ok = true;
  for (int kb = 0; kb < nkb && ok; ++kb) {
    copy_tile(sA, A + m0 * K, kDiagM, K, kb);
    copy_tile(sB, B + n0 * K, kDiagN, K, kb);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (threadIdx.x == 0) {
      const uint64_t ad = sw128_kmajor_desc(smem_u32(sA));
      const uint64_t bd = sw128_kmajor_desc(smem_u32(sB));
#pragma unroll
      for (int k = 0; k < kDiagK / 32; ++k)  // K = 32 bytes per MMA; only the very first overwrites D
        mma_e4m3(tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      mma_commit(bar);
    }
    __syncwarp();
    // the MMAs have read the tiles once the commit lands: the next copy may
    // overwrite them
    ok = __syncthreads_and(mbar_wait(bar, static_cast<uint32_t>(kb) & 1u, timeout_ns)) != 0;
    tc_fence_after_sync();
  }
  if (ok) {
    const uint32_t t = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // TMEM lane = row of the tile
    float* drow = D + (m0 + warp * 32 + lane) * N + n0;
    for (int c = 0; c < kDiagN; c += 32) {
      uint32_t r[32];
      tmem_ld32(t + c, r);
      tmem_wait_ld(r);
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(drow + c + j) = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                               __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    }
  } else if (threadIdx.x == 0) {
    atomicCAS(&g_diag_status, 0, kStatusTimeout);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, kDiagN);
}

}  // namespace

cudaError_t launch_unpromoted_gemm(const uint8_t* a, const uint8_t* b, float* d, int64_t M, int64_t N, int64_t K,
                                   uint64_t timeout_ns, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(unpromoted_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDiagSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(M / kDiagM), static_cast<unsigned>(N / kDiagN), 1);
  unpromoted_gemm_kernel<<<grid, kDiagThreads, kDiagSmem, stream>>>(a, b, d, N, K, timeout_ns);
  return cudaGetLastError();
}

cudaError_t diag_take_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_diag_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_diag_status, &zero, sizeof(int));
  }
  *status = v;
  return e;
}

}  // namespace fp8bs
