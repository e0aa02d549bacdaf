// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8bs {

// ---- quantize.cu
// Every quantiser streams 128x128 BF16 tiles through shared memory with
// TMA; its waits are bounded by timeout_ns and a wait that expires records
// FP8BS_ERR_TIMEOUT in the status word that quant_take_status reads.
// pow2: power-of-two scales instead of fl32(absmax / 448).
cudaError_t launch_quantize_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                      float* sx, bool pow2, int sm_count, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_quantize_act_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                     float* sx, uint8_t* xq_t, float* sx_t, bool pow2, int sm_count,
                                     uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_quantize_weight(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* wq,
                                   float* sw, uint8_t* wq_t, float* sw_t, bool pow2, int sm_count,
                                   uint64_t timeout_ns, cudaStream_t stream);
// One launch quantising X [M][K] in 1x128 groups and W [N][Kw] in 128x128
// blocks (the two operands of an FP8 Linear); either may be empty (M or N 0).
cudaError_t launch_quantize_act_weight(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, float* sx,
                                       const uint16_t* w, int64_t N, int64_t Kw, int64_t ldw, uint8_t* wq, float* sw,
                                       bool pow2, int sm_count, uint64_t timeout_ns, cudaStream_t stream);
// FP8 -> FP8 re-tiling 1x128 -> 128x1 (dequantise, transpose, requantise);
// plain loads, no waits.
cudaError_t launch_requant_1x128_to_128x1(const uint8_t* xq, const float* sx, int64_t M, int64_t K, uint8_t* xq_t,
                                          float* sx_t, bool pow2, int sm_count, cudaStream_t stream);
// Fused SwiGLU (gate columns [0, I), up columns [I, 2I) of h) and 1x128
// quantisation of the BF16-rounded result; plain loads, no waits.
cudaError_t launch_swiglu_quantize(const uint16_t* h, int64_t M, int64_t I, int64_t ldh, uint8_t* q, float* s,
                                   bool pow2, int sm_count, cudaStream_t stream);
// Reads and clears the quantisers' device status word (synchronous copy on
// the current device).
cudaError_t quant_take_status(int* status);

// ---- gemm.cu
struct GemmArgs {
  const uint8_t* a;        // [M][K] E4M3, K-major
  const float* sa;         // [K/128][M] kb-major
  const uint8_t* b;        // [G][N][K] E4M3 (G = 1 for the dense GEMM)
  const float* sb;         // block: [G][N/128][K/128]; row: [K/128][N]
  void* d;                 // [M][N]
  const int32_t* offsets;  // grouped only: device [G+1]
  int64_t M;               // rows of A (M_total for the grouped GEMM)
  int64_t N, K;
  int num_groups;          // 1 for the dense GEMM
  bool grouped;
  bool sb_row;             // FP8BS_SCALE_ROW1x128
  bool out_bf16;
  bool accumulate;
  uint64_t timeout_ns;
};

// Returns cudaSuccess, or an error; *tmap_failed is set when a tensor map
// could not be encoded, *reg_check_failed when the compiled kernel's
// register count does not match the warp-specialised register split.
cudaError_t launch_gemm(const GemmArgs& args, int sm_count, cudaStream_t stream, bool* tmap_failed,
                        bool* reg_check_failed);

// Reads and clears the device status word of the GEMM kernels; synchronous
// copy on the current device.
cudaError_t gemm_take_status(int* status);

// ---- gemm_mx.cu
// The same GEMM for power-of-two scales, with the scales applied by the
// tensor core (tcgen05.mma.kind::mxf8f6f4.block_scale, UE8M0) and all of K
// accumulated in tensor memory.  A scale that is not zero or a power of two
// in [2^-127, 2^127] records FP8BS_ERR_DEVICE_ARG in its status word.
cudaError_t launch_gemm_pow2(const GemmArgs& args, int sm_count, cudaStream_t stream, bool* tmap_failed,
                             bool* reg_check_failed);
cudaError_t gemm_mx_take_status(int* status);

// ---- moe.cu (row movement of the MoE dispatch and combine; no waits)
cudaError_t launch_gather_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, bool s_in_kb_major,
                                 const int32_t* idx, int64_t rows_out, uint8_t* q_out, float* s_out,
                                 bool s_out_kb_major, int sm_count, cudaStream_t stream);
cudaError_t launch_scatter_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, bool s_in_kb_major,
                                  const int32_t* pos, int k, const int32_t* zero_rows, int64_t n_zero,
                                  int64_t rows_out, uint8_t* q_out, float* s_out, bool s_out_kb_major, int sm_count,
                                  cudaStream_t stream);
cudaError_t launch_gather_bf16_rows(const uint16_t* y, int64_t rows_in, int64_t N, const int32_t* idx,
                                    int64_t rows_out, uint16_t* out, int sm_count, cudaStream_t stream);
cudaError_t launch_moe_combine(const uint16_t* y, int64_t rows_y, int64_t N, const int32_t* idx, const float* w,
                               int64_t T, int k, uint16_t* out, int sm_count, cudaStream_t stream);

// Diagnostic: a kernel whose bounded wait runs out (nothing ever arrives on
// its barrier) and records FP8BS_ERR_TIMEOUT in the GEMM status word.
cudaError_t launch_wait_timeout_selftest(uint64_t timeout_ns, cudaStream_t stream);

// Diagnostic GEMM without promotion (diag.cu): D[M][N] = A[M][K] B[N][K]^T
// in FP32, accumulated over all of K in tensor memory; M % 128 == 0,
// N % 256 == 0, K % 128 == 0.
cudaError_t launch_unpromoted_gemm(const uint8_t* a, const uint8_t* b, float* d, int64_t M, int64_t N, int64_t K,
                                   uint64_t timeout_ns, cudaStream_t stream);

// Reads and clears the diagnostic kernel's device status word.
cudaError_t diag_take_status(int* status);

}  // namespace fp8bs
