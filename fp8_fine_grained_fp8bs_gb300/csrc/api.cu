// The C ABI of fp8bs (declared in include/fp8bs.h): argument checks, the
// architecture check, and dispatch to the kernels on the caller's stream.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "fp8bs.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000ull * 1000ull * 1000ull;

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 supported, -1 unsupported
  int sm_count = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// FP8BS_OK with the SM count of the current device, or an error status.
int current_device(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8BS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& info = g_dev[dev];
  if (info.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    info.checked = (major == 10 && minor == 3) ? 1 : -1;
    info.sm_count = sms;
  }
  if (info.checked < 0) return FP8BS_ERR_UNSUPPORTED_ARCH;
  *sm_count = info.sm_count;
  return FP8BS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA; }

}  // namespace

extern "C" {

int fp8bs_quantize_act_ex(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, float* sx, uint8_t* xq_t,
                          float* sx_t, int scale_mode, void* stream) {
  if (M < 0 || K < 0 || ldx < K) return FP8BS_ERR_INVALID_ARG;
  if (scale_mode != FP8BS_SCALE_ABSMAX && scale_mode != FP8BS_SCALE_POW2) return FP8BS_ERR_INVALID_ARG;
  if ((xq_t == nullptr) != (sx_t == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (M > 0 && K > 0 && (x == nullptr || xq == nullptr || sx == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0) return FP8BS_ERR_SHAPE;
  if (xq_t != nullptr && M % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M > (int64_t(1) << 31) || K > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(xq_t) || (ldx * 2) % 16 != 0) return FP8BS_ERR_ALIGNMENT;
  if (!aligned16(sx) || !aligned16(sx_t)) return FP8BS_ERR_ALIGNMENT;
  if (M == 0 || K == 0) return FP8BS_OK;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  const auto* xb = static_cast<const uint16_t*>(x);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t tmo = g_timeout_ns.load();
  const bool pow2 = scale_mode == FP8BS_SCALE_POW2;
  if (xq_t != nullptr)
    return from_cuda(fp8bs::launch_quantize_act_dual(xb, M, K, ldx, xq, sx, xq_t, sx_t, pow2, sms, tmo, s));
  return from_cuda(fp8bs::launch_quantize_act_1x128(xb, M, K, ldx, xq, sx, pow2, sms, tmo, s));
}

int fp8bs_quantize_act(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, float* sx, uint8_t* xq_t,
                       float* sx_t, void* stream) {
  return fp8bs_quantize_act_ex(x, M, K, ldx, xq, sx, xq_t, sx_t, FP8BS_SCALE_ABSMAX, stream);
}

int fp8bs_quantize_weight_ex(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* wq, float* sw,
                             uint8_t* wq_t, float* sw_t, int scale_mode, void* stream) {
  if (N < 0 || K < 0 || ldw < K) return FP8BS_ERR_INVALID_ARG;
  if (scale_mode != FP8BS_SCALE_ABSMAX && scale_mode != FP8BS_SCALE_POW2) return FP8BS_ERR_INVALID_ARG;
  if ((wq_t == nullptr) != (sw_t == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (N > 0 && K > 0 && (w == nullptr || wq == nullptr || sw == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BS_ERR_SHAPE;
  if (N > (int64_t(1) << 24) || K > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(wq) || !aligned16(wq_t) || (ldw * 2) % 16 != 0) return FP8BS_ERR_ALIGNMENT;
  if (N == 0 || K == 0) return FP8BS_OK;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_quantize_weight(static_cast<const uint16_t*>(w), N, K, ldw, wq, sw, wq_t, sw_t,
                                                 scale_mode == FP8BS_SCALE_POW2, sms, g_timeout_ns.load(),
                                                 static_cast<cudaStream_t>(stream)));
}

int fp8bs_quantize_act_weight(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, float* sx,
                              const void* w, int64_t N, int64_t Kw, int64_t ldw, uint8_t* wq, float* sw,
                              int scale_mode, void* stream) {
  if (M < 0 || K < 0 || ldx < K || N < 0 || Kw < 0 || ldw < Kw) return FP8BS_ERR_INVALID_ARG;
  if (scale_mode != FP8BS_SCALE_ABSMAX && scale_mode != FP8BS_SCALE_POW2) return FP8BS_ERR_INVALID_ARG;
  const bool x_empty = M == 0 || K == 0, w_empty = N == 0 || Kw == 0;
  if (!x_empty && (x == nullptr || xq == nullptr || sx == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (!w_empty && (w == nullptr || wq == nullptr || sw == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0 || Kw % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M > (int64_t(1) << 31) || K > (int64_t(1) << 24) || N > (int64_t(1) << 24) || Kw > (int64_t(1) << 24))
    return FP8BS_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(sx) || (ldx * 2) % 16 != 0) return FP8BS_ERR_ALIGNMENT;
  if (!aligned16(w) || !aligned16(wq) || (ldw * 2) % 16 != 0) return FP8BS_ERR_ALIGNMENT;
  if (x_empty && w_empty) return FP8BS_OK;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_quantize_act_weight(
      static_cast<const uint16_t*>(x), x_empty ? 0 : M, K, ldx, xq, sx, static_cast<const uint16_t*>(w),
      w_empty ? 0 : N, Kw, ldw, wq, sw, scale_mode == FP8BS_SCALE_POW2, sms, g_timeout_ns.load(),
      static_cast<cudaStream_t>(stream)));
}

int fp8bs_quantize_weight(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* wq, float* sw, uint8_t* wq_t,
                          float* sw_t, void* stream) {
  return fp8bs_quantize_weight_ex(w, N, K, ldw, wq, sw, wq_t, sw_t, FP8BS_SCALE_ABSMAX, stream);
}

int fp8bs_requant_1x128_to_128x1(const uint8_t* xq, const float* sx, int64_t M, int64_t K, uint8_t* xq_t,
                                 float* sx_t, int scale_mode, void* stream) {
  if (M < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (scale_mode != FP8BS_SCALE_ABSMAX && scale_mode != FP8BS_SCALE_POW2) return FP8BS_ERR_INVALID_ARG;
  if (M % 128 != 0 || K % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M > (int64_t(1) << 31) || K > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (xq == nullptr || sx == nullptr || xq_t == nullptr || sx_t == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(sx) || !aligned16(xq_t) || !aligned16(sx_t)) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_requant_1x128_to_128x1(xq, sx, M, K, xq_t, sx_t, scale_mode == FP8BS_SCALE_POW2, sms,
                                                        static_cast<cudaStream_t>(stream)));
}

int fp8bs_swiglu_quantize(const void* h, int64_t M, int64_t I, int64_t ldh, uint8_t* q, float* s, int scale_mode,
                          void* stream) {
  if (M < 0 || I < 0 || ldh < 2 * I) return FP8BS_ERR_INVALID_ARG;
  if (scale_mode != FP8BS_SCALE_ABSMAX && scale_mode != FP8BS_SCALE_POW2) return FP8BS_ERR_INVALID_ARG;
  if (I % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M > (int64_t(1) << 31) || I > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (M == 0 || I == 0) return FP8BS_OK;
  if (h == nullptr || q == nullptr || s == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(q) || !aligned16(s) || (ldh * 2) % 16 != 0) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_swiglu_quantize(static_cast<const uint16_t*>(h), M, I, ldh, q, s,
                                                 scale_mode == FP8BS_SCALE_POW2, sms,
                                                 static_cast<cudaStream_t>(stream)));
}

static int run_gemm(const fp8bs::GemmArgs& args, bool pow2, void* stream) {
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  bool tmap_failed = false, reg_failed = false;
  const cudaError_t e = pow2 ? fp8bs::launch_gemm_pow2(args, sms, static_cast<cudaStream_t>(stream), &tmap_failed,
                                                       &reg_failed)
                             : fp8bs::launch_gemm(args, sms, static_cast<cudaStream_t>(stream), &tmap_failed,
                                                  &reg_failed);
  if (tmap_failed) return FP8BS_ERR_ALIGNMENT;
  return from_cuda(e);
}

// Argument checks of fp8bs_gemm(_pow2); FP8BS_OK with *g filled, or an
// error; *nothing is set when the call has no work (M or N zero).
static int gemm_args(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int sb_kind, void* d,
                     int d_dtype, int64_t M, int64_t N, int64_t K, int accumulate, fp8bs::GemmArgs* g,
                     bool* nothing) {
  *nothing = false;
  if (M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (sb_kind != FP8BS_SCALE_BLOCK128x128 && sb_kind != FP8BS_SCALE_ROW1x128) return FP8BS_ERR_INVALID_ARG;
  if (d_dtype != FP8BS_OUT_F32 && d_dtype != FP8BS_OUT_BF16) return FP8BS_ERR_INVALID_ARG;
  if (accumulate && d_dtype != FP8BS_OUT_F32) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 24) || K > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (M == 0 || N == 0) {
    *nothing = true;
    return FP8BS_OK;
  }
  if (K == 0) return FP8BS_ERR_SHAPE;
  if (a == nullptr || sa == nullptr || b == nullptr || sb == nullptr || d == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8BS_ERR_ALIGNMENT;
  if (sb_kind == FP8BS_SCALE_ROW1x128 && !aligned16(sb)) return FP8BS_ERR_ALIGNMENT;
  *g = fp8bs::GemmArgs{};
  g->a = a; g->sa = sa; g->b = b; g->sb = sb; g->d = d; g->offsets = nullptr;
  g->M = M; g->N = N; g->K = K; g->num_groups = 1; g->grouped = false;
  g->sb_row = sb_kind == FP8BS_SCALE_ROW1x128;
  g->out_bf16 = d_dtype == FP8BS_OUT_BF16;
  g->accumulate = accumulate != 0;
  g->timeout_ns = g_timeout_ns.load();
  return FP8BS_OK;
}

// Argument checks of fp8bs_grouped_gemm(_pow2), as gemm_args.
static int grouped_args(const uint8_t* a, const float* sa, int64_t M_total, const int32_t* offsets, int num_groups,
                        const uint8_t* b, const float* sb, void* d, int d_dtype, int64_t N, int64_t K,
                        fp8bs::GemmArgs* g, bool* nothing) {
  *nothing = false;
  if (M_total < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (num_groups < 1 || num_groups > 512) return FP8BS_ERR_INVALID_ARG;
  if (d_dtype != FP8BS_OUT_F32 && d_dtype != FP8BS_OUT_BF16) return FP8BS_ERR_INVALID_ARG;
  if (offsets == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M_total > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 24) || K > (int64_t(1) << 24))
    return FP8BS_ERR_SHAPE;
  if (M_total == 0 || N == 0) {
    *nothing = true;
    return FP8BS_OK;
  }
  if (K == 0) return FP8BS_ERR_SHAPE;
  if (a == nullptr || sa == nullptr || b == nullptr || sb == nullptr || d == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8BS_ERR_ALIGNMENT;
  *g = fp8bs::GemmArgs{};
  g->a = a; g->sa = sa; g->b = b; g->sb = sb; g->d = d; g->offsets = offsets;
  g->M = M_total; g->N = N; g->K = K; g->num_groups = num_groups; g->grouped = true;
  g->sb_row = false;
  g->out_bf16 = d_dtype == FP8BS_OUT_BF16;
  g->accumulate = false;
  g->timeout_ns = g_timeout_ns.load();
  return FP8BS_OK;
}

int fp8bs_gemm(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int sb_kind, void* d,
               int d_dtype, int64_t M, int64_t N, int64_t K, int accumulate, void* stream) {
  fp8bs::GemmArgs g;
  bool nothing = false;
  const int st = gemm_args(a, sa, b, sb, sb_kind, d, d_dtype, M, N, K, accumulate, &g, &nothing);
  if (st != FP8BS_OK || nothing) return st;
  return run_gemm(g, false, stream);
}

int fp8bs_gemm_pow2(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int sb_kind, void* d,
                    int d_dtype, int64_t M, int64_t N, int64_t K, int accumulate, void* stream) {
  fp8bs::GemmArgs g;
  bool nothing = false;
  const int st = gemm_args(a, sa, b, sb, sb_kind, d, d_dtype, M, N, K, accumulate, &g, &nothing);
  if (st != FP8BS_OK || nothing) return st;
  return run_gemm(g, true, stream);
}

int fp8bs_grouped_gemm(const uint8_t* a, const float* sa, int64_t M_total, const int32_t* offsets, int num_groups,
                       const uint8_t* b, const float* sb, void* d, int d_dtype, int64_t N, int64_t K, void* stream) {
  fp8bs::GemmArgs g;
  bool nothing = false;
  const int st = grouped_args(a, sa, M_total, offsets, num_groups, b, sb, d, d_dtype, N, K, &g, &nothing);
  if (st != FP8BS_OK || nothing) return st;
  return run_gemm(g, false, stream);
}

int fp8bs_grouped_gemm_pow2(const uint8_t* a, const float* sa, int64_t M_total, const int32_t* offsets,
                            int num_groups, const uint8_t* b, const float* sb, void* d, int d_dtype, int64_t N,
                            int64_t K, void* stream) {
  fp8bs::GemmArgs g;
  bool nothing = false;
  const int st = grouped_args(a, sa, M_total, offsets, num_groups, b, sb, d, d_dtype, N, K, &g, &nothing);
  if (st != FP8BS_OK || nothing) return st;
  return run_gemm(g, true, stream);
}

int fp8bs_gather_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, int s_in_layout,
                        const int32_t* idx, int64_t rows_out, uint8_t* q_out, float* s_out, int s_out_layout,
                        void* stream) {
  if (rows_in < 0 || rows_out < 0 || H < 0) return FP8BS_ERR_INVALID_ARG;
  if ((s_in_layout != FP8BS_SCALES_KB_MAJOR && s_in_layout != FP8BS_SCALES_ROW_MAJOR) ||
      (s_out_layout != FP8BS_SCALES_KB_MAJOR && s_out_layout != FP8BS_SCALES_ROW_MAJOR))
    return FP8BS_ERR_INVALID_ARG;
  if (H % 128 != 0) return FP8BS_ERR_SHAPE;
  if (rows_in > (int64_t(1) << 31) - 1 || rows_out > (int64_t(1) << 31) || H > (int64_t(1) << 24))
    return FP8BS_ERR_SHAPE;
  if (rows_out == 0 || H == 0) return FP8BS_OK;
  if (idx == nullptr || q_out == nullptr || s_out == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (rows_in > 0 && (q == nullptr || s == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(q_out)) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_gather_q_rows(q, s, rows_in, H, s_in_layout == FP8BS_SCALES_KB_MAJOR, idx, rows_out,
                                               q_out, s_out, s_out_layout == FP8BS_SCALES_KB_MAJOR, sms,
                                               static_cast<cudaStream_t>(stream)));
}

int fp8bs_scatter_q_rows(const uint8_t* q, const float* s, int64_t rows_in, int64_t H, int s_in_layout,
                         const int32_t* pos, int k, const int32_t* zero_rows, int64_t n_zero, int64_t rows_out,
                         uint8_t* q_out, float* s_out, int s_out_layout, void* stream) {
  if (rows_in < 0 || rows_out < 0 || H < 0 || n_zero < 0) return FP8BS_ERR_INVALID_ARG;
  if (k < 1 || k > 64) return FP8BS_ERR_INVALID_ARG;
  if ((s_in_layout != FP8BS_SCALES_KB_MAJOR && s_in_layout != FP8BS_SCALES_ROW_MAJOR) ||
      (s_out_layout != FP8BS_SCALES_KB_MAJOR && s_out_layout != FP8BS_SCALES_ROW_MAJOR))
    return FP8BS_ERR_INVALID_ARG;
  if (H % 128 != 0) return FP8BS_ERR_SHAPE;
  if (rows_in > ((int64_t(1) << 31) - 1) / k || rows_out > (int64_t(1) << 31) || n_zero > (int64_t(1) << 31) ||
      H > (int64_t(1) << 24))
    return FP8BS_ERR_SHAPE;
  if (rows_out == 0 || H == 0 || (rows_in == 0 && n_zero == 0)) return FP8BS_OK;
  if (q_out == nullptr || s_out == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (rows_in > 0 && (q == nullptr || s == nullptr || pos == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (n_zero > 0 && zero_rows == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(q_out)) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_scatter_q_rows(q, s, rows_in, H, s_in_layout == FP8BS_SCALES_KB_MAJOR, pos, k,
                                                zero_rows, n_zero, rows_out, q_out, s_out,
                                                s_out_layout == FP8BS_SCALES_KB_MAJOR, sms,
                                                static_cast<cudaStream_t>(stream)));
}

int fp8bs_gather_bf16_rows(const void* y, int64_t rows_in, int64_t N, const int32_t* idx, int64_t rows_out,
                           void* out, void* stream) {
  if (rows_in < 0 || rows_out < 0 || N < 0) return FP8BS_ERR_INVALID_ARG;
  if (N % 8 != 0) return FP8BS_ERR_SHAPE;
  if (rows_in > (int64_t(1) << 31) - 1 || rows_out > (int64_t(1) << 31) || N > (int64_t(1) << 24))
    return FP8BS_ERR_SHAPE;
  if (rows_out == 0 || N == 0) return FP8BS_OK;
  if (idx == nullptr || out == nullptr || (rows_in > 0 && y == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_gather_bf16_rows(static_cast<const uint16_t*>(y), rows_in, N, idx, rows_out,
                                                  static_cast<uint16_t*>(out), sms, static_cast<cudaStream_t>(stream)));
}

int fp8bs_moe_combine(const void* y, int64_t rows_y, int64_t N, const int32_t* idx, const float* w, int64_t T, int k,
                      void* out, void* stream) {
  if (rows_y < 0 || N < 0 || T < 0 || k < 1 || k > 64) return FP8BS_ERR_INVALID_ARG;
  if (N % 8 != 0) return FP8BS_ERR_SHAPE;
  if (rows_y > (int64_t(1) << 31) - 1 || T > (int64_t(1) << 31) / 64 || N > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (T == 0 || N == 0) return FP8BS_OK;
  if (idx == nullptr || w == nullptr || out == nullptr || (rows_y > 0 && y == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_moe_combine(static_cast<const uint16_t*>(y), rows_y, N, idx, w, T, k,
                                             static_cast<uint16_t*>(out), sms, static_cast<cudaStream_t>(stream)));
}

int fp8bs_selftest_wait_timeout(int64_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return FP8BS_ERR_INVALID_ARG;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_wait_timeout_selftest(static_cast<uint64_t>(timeout_us) * 1000ull,
                                                       static_cast<cudaStream_t>(stream)));
}

int fp8bs_diag_gemm_unpromoted(const uint8_t* a, const uint8_t* b, float* d, int64_t M, int64_t N, int64_t K,
                               void* stream) {
  if (M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (M % 128 != 0 || N % 256 != 0 || K % 128 != 0) return FP8BS_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 256 || N > (int64_t(1) << 24) || K > (int64_t(1) << 24)) return FP8BS_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8BS_OK;
  if (K == 0) return FP8BS_ERR_SHAPE;
  if (a == nullptr || b == nullptr || d == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8BS_ERR_ALIGNMENT;
  int sms = 0;
  const int st = current_device(&sms);
  if (st != FP8BS_OK) return st;
  return from_cuda(fp8bs::launch_unpromoted_gemm(a, b, d, M, N, K, g_timeout_ns.load(),
                                                 static_cast<cudaStream_t>(stream)));
}

int fp8bs_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
  int v = 0, mx = 0, q = 0, dg = 0;
  if (fp8bs::gemm_take_status(&v) != cudaSuccess) return FP8BS_ERR_CUDA;
  if (fp8bs::gemm_mx_take_status(&mx) != cudaSuccess) return FP8BS_ERR_CUDA;
  if (fp8bs::quant_take_status(&q) != cudaSuccess) return FP8BS_ERR_CUDA;
  if (fp8bs::diag_take_status(&dg) != cudaSuccess) return FP8BS_ERR_CUDA;
  return v != FP8BS_OK ? v : mx != FP8BS_OK ? mx : q != FP8BS_OK ? q : dg;
}

int fp8bs_set_wait_timeout_ms(int64_t ms) {
  if (ms < 0) return FP8BS_ERR_INVALID_ARG;
  g_timeout_ns.store(ms == 0 ? kDefaultTimeoutNs : static_cast<uint64_t>(ms) * 1000000ull);
  return FP8BS_OK;
}

const char* fp8bs_status_string(int status) {
  switch (status) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_INVALID_ARG: return "invalid argument";
    case FP8BS_ERR_SHAPE: return "shape breaks a multiple-of-128 rule";
    case FP8BS_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
    case FP8BS_ERR_UNSUPPORTED_ARCH: return "current device is not sm_103";
    case FP8BS_ERR_CUDA: return "CUDA call failed";
    case FP8BS_ERR_TIMEOUT: return "a bounded device wait expired";
    case FP8BS_ERR_DEVICE_ARG: return "invalid device-resident argument (group offsets)";
    default: return "unknown status";
  }
}

}  // extern "C"
