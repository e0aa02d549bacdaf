// Pieces shared by the two block-scaled GEMM kernels (gemm.cu: per-block
// promotion on the CUDA cores; gemm_mx.cu: hardware block scaling for
// power-of-two scales): tile geometry, kernel parameters, the epilogue's
// staged TMA store, the work-unit walk, and the host-side tensor maps.
#pragma once

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "tmap.h"

namespace fp8bs {
namespace {

constexpr int kBlockM = 128;
constexpr int kBlockK = 128;         // = N_C
constexpr int kUmmaK = 32;           // K of one kind::f8f6f4 / mxf8f6f4 MMA (bytes of E4M3)
constexpr int kMaxGroups = 512;

// Output staging: each epilogue warp writes its 32 rows x BN/2 columns
// through kOutSlots boxes of 32 rows x 128 bytes in shared memory (128-byte
// swizzled, the layout TMA expects), each stored by one TMA copy.
constexpr int kOutRows = 32;
constexpr int kOutBoxBytes = kOutRows * 128;
constexpr int kOutSlots = 2;
constexpr int kSmemBudget = 227 * 1024;

struct KParams {
  const float* sa;
  const float* sb;
  void* d;
  const int32_t* offsets;
  int64_t M;
  int N;
  int nkb;
  int num_groups;
  int out_bf16;
  int accumulate;
  uint64_t timeout_ns;
};

// Two float32 -> BF16x2 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Stores one thread's row segment, kCols FP32 accumulators starting at
// column x0 of row y0 + lane, for the 32 rows of its warp: per 128-byte
// column block the warp writes its rows into a staging box (16-byte chunk c
// of row r at chunk position c ^ (r % 8), the 128-byte swizzle), and lane 0
// stores the box with TMA (or adds it into D).  Boxes rotate over kOutSlots
// staging slots; a slot is rewritten only once the store that last used it
// has read it out.  `seq` counts the warp's boxes over the kernel (one bulk
// group each).  kSlots staging boxes per warp (kOutSlots by default).
template <int kCols, bool kBf16, int kSlots = kOutSlots>
__device__ __forceinline__ void store_segment(const float* acc, uint8_t* slots, uint32_t& seq, int lane,
                                              const CUtensorMap* tmD, int x0, int y0, bool add) {
  constexpr int kPerChunk = kBf16 ? 8 : 4;   // columns in 16 bytes
  constexpr int kBoxCols = 8 * kPerChunk;    // columns in 128 bytes
  static_assert(kCols % kBoxCols == 0, "segment of whole boxes");
#pragma unroll
  for (int b = 0; b < kCols / kBoxCols; ++b, ++seq) {
    uint8_t* box = slots + (seq % kSlots) * kOutBoxBytes;
    if (lane == 0) bulk_wait_read<kSlots - 1>();
    __syncwarp();
    uint8_t* row = box + lane * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float* v = acc + b * kBoxCols + c * kPerChunk;
      uint4 w;
      if (kBf16) {
        w.x = pack_bf16x2(v[0], v[1]);
        w.y = pack_bf16x2(v[2], v[3]);
        w.z = pack_bf16x2(v[4], v[5]);
        w.w = pack_bf16x2(v[6], v[7]);
      } else {
        w = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
      }
      *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = w;
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      if (add)
        tma_reduce_add_2d(tmD, box, x0 + b * kBoxCols, y0);
      else
        tma_store_2d(tmD, box, x0 + b * kBoxCols, y0);
      bulk_commit();
    }
  }
}

// The same store for a warp whose accumulators are in the fragment layout
// of tcgen05.ld.16x256b (the fold with per-column scales):
// acc2[((h * (kCols / 32) + c) * 4 + g) * 2 + j] holds columns
// x0 + 32c + 8g + 2(lane % 4) + {0, 1} of row y0 + 16h + 8j + lane / 4.
// Same staging boxes, swizzle and TMA stores as store_segment.
template <int kCols, bool kBf16, int kSlots = kOutSlots>
__device__ __forceinline__ void store_segment_frag(const float2* acc2, uint8_t* slots, uint32_t& seq, int lane,
                                                   const CUtensorMap* tmD, int x0, int y0, bool add) {
  constexpr int kChunks = kCols / 32;
  constexpr int kBoxCols = kBf16 ? 64 : 32;  // columns in 128 bytes
  constexpr int kChunksPerBox = kBoxCols / 32;
  static_assert(kCols % kBoxCols == 0, "segment of whole boxes");
  const int q4 = lane & 3;
#pragma unroll
  for (int b = 0; b < kCols / kBoxCols; ++b, ++seq) {
    uint8_t* box = slots + (seq % kSlots) * kOutBoxBytes;
    if (lane == 0) bulk_wait_read<kSlots - 1>();
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int row = 16 * h + 8 * j + (lane >> 2);
        uint8_t* rowp = box + row * 128;
#pragma unroll
        for (int cc = 0; cc < kChunksPerBox; ++cc) {
          const int c = b * kChunksPerBox + cc;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float2 v = acc2[((h * kChunks + c) * 4 + g) * 2 + j];
            if (kBf16) {  // bytes 64cc + 16g + 4(lane % 4) of the row
              *reinterpret_cast<uint32_t*>(rowp + (((4 * cc + g) ^ (row & 7)) << 4) + 4 * q4) =
                  pack_bf16x2(v.x, v.y);
            } else {      // bytes 32g + 8(lane % 4) of the row
              *reinterpret_cast<float2*>(rowp + (((2 * g + (q4 >> 1)) ^ (row & 7)) << 4) + 8 * (q4 & 1)) = v;
            }
          }
        }
      }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      if (add)
        tma_reduce_add_2d(tmD, box, x0 + b * kBoxCols, y0);
      else
        tma_store_2d(tmD, box, x0 + b * kBoxCols, y0);
      bulk_commit();
    }
  }
}

// A bounded mbarrier wait made by a whole warp, with lane 0's outcome.  The
// producer and MMA-issuer warps run their loops converged (lane 0 issues
// the copies and MMAs): a warp whose lane 0 loops alone while its other
// lanes wait at the final CTA barrier slowed the epilogue warps sharing its
// SM sub-partition.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  return __shfl_sync(0xffffffffu, mbar_wait(bar, parity, timeout_ns), 0);
}

// Work unit t -> (first row, first column, group, end of the rows the
// unit may write); g carries the group of the caller's previous unit in.  Units run m-tile-major with the BN-wide n-tiles of one
// m-tile consecutive, so concurrently running CTAs share A rows.
//
// With CTA pairs (a cluster of two running one 2-SM MMA over a 256-row
// tile), unit t names an (m-tile pair, n-tile) and the CTA of rank r takes
// the pair's m-tile r.  In the grouped GEMM the pairs are formed within
// each group's segment (s_cum counts units per group); a group with an odd
// number of m-tiles ends in a pair whose second m-tile lies past the
// segment: that CTA still loads its half of B and joins the MMA, and stores
// nothing (row0 >= row_end).
//
// Every role walks the k-blocks of a unit in order, so the CTAs that share
// an A or B tile read its k-slices at about the same time and the second
// reader finds them in L2 (when A and B together exceed L2, as in Wgrad,
// starting each unit at its own k-block cost 9% with the scales in the MMA).
template <int BN, bool kPair>
__device__ __forceinline__ void tile_coords(int t, int ntn, bool grouped, const int* s_off, const int* s_cum,
                                            int num_groups, uint32_t rank, int64_t M, int& row0, int& n0, int& g,
                                            int64_t& row_end) {
  const int mu = t / ntn;  // m-tile, or m-tile pair
  n0 = (t - mu * ntn) * BN;
  if (!grouped) {
    g = 0;
    row0 = (kPair ? 2 * mu + static_cast<int>(rank) : mu) * kBlockM;
    row_end = M;
    return;
  }
  // last g with cum[g] <= mu.  A CTA's units only move forward, so the
  // search resumes from the group of its previous unit (g on entry, 0 for
  // the first): usually no step, a few shared loads at most.
  while (g + 1 < num_groups && s_cum[g + 1] <= mu) ++g;
  const int local = kPair ? 2 * (mu - s_cum[g]) + static_cast<int>(rank) : mu - s_cum[g];
  row0 = s_off[g] + local * kBlockM;
  row_end = s_off[g + 1];
}

// ----------------------------------------------------------- host side
// K-major E4M3 operand [outer...][inner=K] with a 128 x box_rows box and
// 128-byte swizzling (one 128-byte row of K per box row).
bool encode_operand(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                    uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t gdim[3];
  cuuint64_t gstride[2];
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), box_rows, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
  for (int i = 0; i < rank - 1; ++i) gstride[i] = strides[i];
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim, gstride,
          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output D [rows][N] (BF16 or FP32, row-major) with a 128-byte x box_rows
// box and 128-byte swizzling, for the epilogue's TMA stores.
bool encode_output(CUtensorMap* map, void* base, int64_t rows, int64_t N, bool bf16, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const uint64_t elt = bf16 ? 2 : 4;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(N) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt), box_rows};
  cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base,
                         gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Launches a persistent GEMM grid: one CTA per SM, or with kPair one
// cluster of two CTAs per SM pair (as many clusters as can be co-resident),
// or fewer when there are fewer work units.  The launch allows programmatic
// stream serialisation: the kernel's set-up (barriers, tensor memory, tensor
// map prefetch) overlaps the tail of the kernel before it on the stream, and
// the kernel calls griddep_wait() before it touches memory.
template <bool kPair, typename Kern, typename... Args>
cudaError_t launch_persistent(Kern kern, int64_t units, int sm_count, int threads, int smem_bytes,
                              cudaStream_t stream, std::atomic<int> (&cluster_cache)[kMaxCachedDevices],
                              Args... args) {
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  if (!kPair) {
    cfg.attrs = attrs + 1;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(units, sm_count)), 1, 1);
  } else {
    cfg.attrs = attrs;
    cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (sm_count / 2)), 1, 1);
    int max_clusters = 0;
    const cudaError_t e = cached_per_device(
        cluster_cache, [&](int* n) { return cudaOccupancyMaxActiveClusters(n, kern, &cfg); }, &max_clusters);
    if (e != cudaSuccess) return e;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(2 * static_cast<unsigned>(std::min<int64_t>(units, max_clusters)), 1, 1);
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace
}  // namespace fp8bs
