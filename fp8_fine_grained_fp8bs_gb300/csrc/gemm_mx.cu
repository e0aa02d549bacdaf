// Block-scaled FP8 GEMM with the scales applied by the tensor core, for
// power-of-two scales.
//
// DeepSeek-V3 "Infrastructure" §3.5.2 (compute hardware) asks for tensor
// cores that take the group scaling factors themselves, so that the partial
// sums need not be moved to the CUDA cores for dequantisation; §3.3.2 notes
// the microscaling formats of the Blackwell generation.  On sm_103a that is
// tcgen05.mma.kind::mxf8f6f4.block_scale: every 32 elements of K of a row of
// A (and of a row of B) carry an UE8M0 scale, an 8-bit biased exponent, so
// the instruction computes sum_k A[m][k] B[n][k] 2^ea(m, k/32) 2^eb(n, k/32)
// with FP32 accumulation.  A 1x128 or 128x128 group scale that is a power
// of two (the "rounded" scales of §3.3.3 (1), FP8BS_SCALE_POW2) is exactly
// such a scale repeated over the group's four 32-element blocks, so
//
//   D[m][n] = sum_kb P_kb[m][n] * s_a[m][kb] * s_b(n, kb)
//
// is computed with no CUDA-core fold: all of K accumulates in one TMEM
// accumulator per tile.  The result is the block-scaled GEMM's, up to the
// FP32 summation order.
//
// Layout of the scale factors in tensor memory (as this GPU reads them):
// for the D rows of lane quarter q (TMEM lanes 32q .. 32q+31, one CTA), the
// scale of A row 32q + i is in lane 32q + i, column sfa + q; the scale of B
// row (output column) n is in lane 32q + n % 32, column sfb + n / 32.  Each
// 32-bit column holds four scales, one per byte, and the MMA's scale-factor
// id (instruction descriptor bits 29-30 for A, 4-5 for B) selects the byte.
// With the 2-SM MMA each CTA holds the scales of its own 128 rows of A and
// all of the tile's B columns, in the same layout.
//
// Structure (persistent, warp-specialised, CTA pairs as in gemm.cu):
//   * warp 0: TMA producer of A and B tiles into a shared-memory ring;
//   * warp 1 (leader CTA): the single MMA issuer: per scale slot (four
//     128-K blocks) it copies the slot's UE8M0 scales from shared memory into
//     tensor memory with tcgen05.cp (in order with its MMAs, so no other
//     warp touches tensor memory while the MMAs run), then per k-block four
//     mxf8f6f4 MMAs of K = 32 into the tile's accumulator, the scale-factor
//     id the k-block's byte in the slot;
//   * warp 2: copies each k-block's float32 scales (128 rows of A, the
//     tile's B scales) into a shared-memory scale ring with cp.async;
//   * warp 3: converts the float32 scales of four k-blocks at a time to
//     UE8M0 bytes in the shared-memory layout tcgen05.cp.32x128b.warpx4
//     takes (32 rows of 16 bytes, row i landing in lane 32q + i of every
//     lane quarter q, bytes 4c..4c+3 in column c); a scale that is neither
//     zero nor a power of two in [2^-127, 2^127] records
//     FP8BS_ERR_DEVICE_ARG;
//   * warps 4-11: the epilogue: after a tile's last MMA, read the
//     accumulator out of TMEM (each thread one row, half of the columns),
//     hand it back to the MMA, and store through shared memory with TMA.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8bs {
namespace {

__device__ int g_gemm_mx_status;

constexpr int kMxThreads = 384;       // 12 warps
constexpr int kMxEpiWarp0 = 4;        // warps 4..11: epilogue
constexpr int kMxEpiThreads = 256;
constexpr int kMxScaleChunks = 2;
constexpr uint32_t kMxTmemCols = 512;
constexpr int kSfSlotCols = 32;       // one scale slot: A scales at +0..3, B scales at +16..+16+BN/32
constexpr int kSfbOffset = 16;
constexpr int kStepsPerSlot = 4;      // k-blocks per slot: one byte each
// Shared-memory scale slot: A scales (32 rows x 16 bytes: row i holds rows
// i, 32+i, 64+i, 96+i of the tile, four k-block bytes each), then B scales,
// one 512-byte block per 128 columns (row i: columns i, 32+i, 64+i, 96+i).
constexpr int kSfRowsBytes = 512;
// Register split: warps 0-3 (producer, MMA, scale loader, converter) at
// MxCfg::kRegsProducer, warps 4-11 at MxCfg::kRegsEpilogue (128
// accumulators and the store); 4 x 32 x 72 + 8 x 32 x 216 or 4 x 32 x 88 +
// 8 x 32 x 208 = 384 x 168, the CTA's allocation at launch.  The converter
// of row-scaled B (eight B scales per lane and k-block) gets the larger
// share: every spill is local-memory traffic through the same on-chip
// memory that feeds the tensor core, and a late scale slot holds back the
// operand loads.
constexpr uint32_t kMxLaunchRegs = 168;
// One staging box per epilogue warp: the accumulator is handed back before
// the stores, so a store waiting for the previous box's copy delays no MMA;
// the shared memory goes to one more operand stage.
constexpr int kMxOutSlots = 1;

template <int BN, bool kPair, bool kRowScale>
struct MxCfg {
  static constexpr int kABytes = kBlockM * kBlockK;
  static constexpr int kBBytes = (kPair ? BN / 2 : BN) * kBlockK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // accumulators: two for 128-wide tiles, one for 256-wide tiles (the rest
  // of TMEM holds the scale slots)
  static constexpr int kAccBufs = BN == 256 ? 1 : 2;
  static constexpr int kSfBase = kAccBufs * BN;
  static constexpr int kSfSlots = (static_cast<int>(kMxTmemCols) - kSfBase) / kSfSlotCols;
  static constexpr int kSfbCols = BN / 32;
  static constexpr uint32_t kRegsProducer = kRowScale ? 88 : 72;
  static constexpr uint32_t kRegsEpilogue = kRowScale ? 208 : 216;
  static_assert(kRegsProducer * 128 + kRegsEpilogue * kMxEpiThreads == kMxLaunchRegs * kMxThreads, "register split");
  static_assert(kSfSlots >= 4, "scale slots");
  static_assert(kSfbOffset + kSfbCols <= kSfSlotCols, "scale slot width");
  static constexpr int kSfSmemBytes = kSfRowsBytes * (1 + BN / 128);   // one shared-memory scale slot
  static constexpr int kSlotFloats = kBlockM + (kRowScale ? BN : 4);
  static constexpr int kScaleChunk = 8;
  static constexpr int kScaleSlots = kScaleChunk * kMxScaleChunks;
  static constexpr int kColsPerThread = BN / 2;
  static constexpr int kOutBytes = (kMxEpiThreads / 32) * kMxOutSlots * kOutBoxBytes;
  static constexpr int kMaxStages = 6;
  static constexpr int kNumBarsMax = 2 * kMaxStages + 2 * kMxScaleChunks + 2 * 8 + 2 * 2 + 1;
  static constexpr int kFixedBytes = kOutBytes + kSfSlots * kSfSmemBytes + kScaleSlots * kSlotFloats * 4 +
                                     kNumBarsMax * 8 + 16 + 2 * (kMaxGroups + 1) * 4 + 1024;
  static constexpr int kFit = (kSmemBudget - kFixedBytes) / kStageBytes;
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static_assert(kStages >= 3, "operand ring too shallow");
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffOut = kOffB + kStages * kBBytes;
  static constexpr int kOffSf = kOffOut + kOutBytes;                     // 1024-aligned
  static constexpr int kOffScale = kOffSf + kSfSlots * kSfSmemBytes;
  static constexpr int kOffBar = kOffScale + kScaleSlots * kSlotFloats * 4;
  static constexpr int kNumBars = 2 * kStages + 2 * kMxScaleChunks + 2 * kSfSlots + 2 * kAccBufs + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffGroups = kOffMisc + 16;
  static constexpr int kSmemBytes = kOffGroups + 2 * (kMaxGroups + 1) * 4 + 1024;
  static_assert(kNumBars <= kNumBarsMax, "barrier budget");
  static_assert(kOffOut % 1024 == 0, "staging boxes need 1024-byte alignment for the 128-byte swizzle");
  static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
};

__device__ __forceinline__ void record_mx_status(int code) { atomicCAS(&g_gemm_mx_status, 0, code); }

// Instruction descriptor of kind::mxf8f6f4 with UE8M0 scales: B scale id in
// bits 4-5, A and B E4M3 (bits 7-9, 10-12 = 0), both K-major, N >> 3 in bits
// 17-22, scale type UE8M0 (bit 23), M >> 4 in bits 24-28, A scale id in
// bits 29-30.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n, uint32_t sf_id) {
  return (sf_id << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mx_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t tmem_sfa, uint32_t tmem_sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tmem_sfa), "r"(tmem_sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mx_e4m3_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t tmem_sfa, uint32_t tmem_sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tmem_sfa), "r"(tmem_sfb), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor of 32 rows x 16 bytes stored contiguously
// without swizzling (8-row core matrices 128 bytes apart), the source of
// tcgen05.cp.32x128b: start address, leading- and stride-dimension offsets
// (both 128 bytes), descriptor version 1 (bits 46-48), no swizzle.
__device__ __forceinline__ uint64_t sf_rows_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Copies 32 rows x 16 bytes from shared memory into four TMEM columns of
// every lane quarter: row i to lane 32q + i, bytes 4c..4c+3 to column c.
// Ordered with the issuing thread's MMAs (the same asynchronous pipe).
__device__ __forceinline__ void tmem_cp_rows(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// The same in both CTAs of a pair, each from its own shared memory into its
// own tensor memory (issued by the leader).
__device__ __forceinline__ void tmem_cp_rows_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// UE8M0 byte of a float32 scale, without branches (the loads of a whole
// slot stay in flight together): the biased exponent of a normal power of
// two; 2^-127 (a float32 subnormal) is byte 0; zero (the scale of an
// all-zero group, whose codes are all zero) is taken as byte 0 too.  Any
// other value sets a bit in *bad.
__device__ __forceinline__ uint32_t ue8m0_of(float s, uint32_t& bad) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t e = b >> 23;  // sign bit included: negative scales are invalid
  const bool pow2 = (b & 0x7FFFFFu) == 0u && e - 1u < 254u;
  const bool tiny = b == 0u || b == 0x00400000u;
  bad |= (pow2 || tiny) ? 0u : 1u;
  return pow2 ? e : 0u;
}

template <int BN, bool kRowScale, bool kGrouped, bool kPair>
__global__ void __launch_bounds__(kMxThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const KParams p) {
  using C = MxCfg<BN, kPair, kRowScale>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::kOffA;
  uint8_t* sB = smem + C::kOffB;
  float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
  uint8_t* sSf = smem + C::kOffSf;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;                                // [kStages] TMA -> MMA
  uint64_t* empty = full + C::kStages;                  // [kStages] MMA -> TMA
  uint64_t* sc_full = empty + C::kStages;               // [2] float scales landed in shared memory
  uint64_t* sc_empty = sc_full + kMxScaleChunks;        // [2] converter done with them
  uint64_t* sf_full = sc_empty + kMxScaleChunks;        // [kSfSlots] UE8M0 slot written to shared memory
  uint64_t* sf_empty = sf_full + C::kSfSlots;           // [kSfSlots] copy and MMAs that read the slot done
  uint64_t* acc_full = sf_empty + C::kSfSlots;          // [kAccBufs] tile accumulated
  uint64_t* acc_empty = acc_full + C::kAccBufs;         // [kAccBufs] accumulator read out
  uint64_t* teardown = acc_empty + C::kAccBufs;         // [1]
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* s_off = reinterpret_cast<int*>(smem + C::kOffGroups);
  int* s_cum = s_off + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ntn = (p.N + BN - 1) / BN;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int unit0 = kPair ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int nunits = kPair ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int nnb = (p.N + kGroup - 1) / kGroup;
  const int nsl = (p.nkb + kStepsPerSlot - 1) / kStepsPerSlot;  // scale slots per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kMxScaleChunks; ++s) {
      mbar_init(&sc_full[s], 32);                   // one cp.async arrival per loader lane
      mbar_init(&sc_empty[s], 1);                   // the converter warp
    }
    for (int s = 0; s < C::kSfSlots; ++s) {
      mbar_init(&sf_full[s], kPair ? 2 : 1);        // the converters of both CTAs, on the leader (producer waits)
      mbar_init(&sf_empty[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], (kPair ? 2 : 1) * kMxEpiThreads / 32);
    }
    mbar_init(&teardown[0], 1);
    fence_barrier_init();
    griddep_wait();  // the group table below may come from the preceding kernel
    int total_mt = 0;
    bool ok = true;
    if (kGrouped) {
      int prev = 0;
      for (int g = 0; g <= p.num_groups; ++g) {
        const int o = p.offsets[g];
        ok = ok && (o >= prev || g == 0) && o >= 0 && (o % kBlockM) == 0 && o <= p.M;
        s_off[g] = o;
        prev = o;
      }
      if (ok) {
        for (int g = 0; g < p.num_groups; ++g) {
          s_cum[g] = total_mt;
          const int mt = (s_off[g + 1] - s_off[g]) / kBlockM;
          total_mt += kPair ? (mt + 1) / 2 : mt;
        }
        s_cum[p.num_groups] = total_mt;
      } else {
        record_mx_status(kStatusDeviceArg);
        total_mt = 0;
      }
    } else {
      total_mt = static_cast<int>((p.M + kBlockM - 1) / kBlockM);
      if (kPair) total_mt = (total_mt + 1) / 2;
    }
    misc[1] = 0;
    misc[2] = static_cast<uint32_t>(total_mt * ntn);
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(&misc[0], kMxTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&misc[0], kMxTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (kPair) cluster_sync();
  // Launched behind another kernel (programmatic dependent launch), the
  // set-up above overlaps that kernel's tail; operands, scales and D are
  // touched only after it has completed.
  griddep_wait();
  const uint32_t tmem_base = misc[0];
  const int total_tiles = static_cast<int>(misc[2]);
  volatile uint32_t* abort_flag = &misc[1];

  if (warp < kMxEpiWarp0) {
    setmaxnreg_dec<C::kRegsProducer>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      bool live = true;
      int issued = 0;
      int g = 0;
      uint32_t gs = 0;   // scale slots (the leader waits for each before loading its first k-block)
      for (int t = unit0; t < total_tiles && live; t += nunits) {
        int row0, n0;
        int64_t row_end;
        tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!warp_wait(&empty[stage], phase ^ 1, p.timeout_ns)) { live = false; break; }
          // The slot's scales are in shared memory (both CTAs') before its
          // first stage is loaded: a full stage then implies ready scales,
          // and the MMA thread waits on the stage alone.
          if (rank == 0 && kb % kStepsPerSlot == 0) {
            const bool ok = __shfl_sync(0xffffffffu,
                                        mbar_wait_cluster(&sf_full[gs % C::kSfSlots], (gs / C::kSfSlots) & 1u,
                                                          p.timeout_ns), 0);
            ++gs;
            if (!ok) { live = false; break; }
          } else if (kb % kStepsPerSlot == 0) {
            ++gs;
          }
          if (lane == 0) {
            if (kPair) {
              if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (C::kABytes + C::kBBytes));
              const uint32_t leader_full = mapa_shared(&full[stage], 0);
              tma_load_2d_pair(sA + stage * C::kABytes, &tmA, leader_full, kb * kBlockK, row0);
              if (kGrouped)
                tma_load_3d_pair(sB + stage * C::kBBytes, &tmB, leader_full, kb * kBlockK,
                                 n0 + static_cast<int>(rank) * (BN / 2), g);
              else
                tma_load_2d_pair(sB + stage * C::kBBytes, &tmB, leader_full, kb * kBlockK,
                                 n0 + static_cast<int>(rank) * (BN / 2));
            } else {
              mbar_arrive_expect_tx(&full[stage], C::kABytes + C::kBBytes);
              tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], kb * kBlockK, row0);
              if (kGrouped)
                tma_load_3d(sB + stage * C::kBBytes, &tmB, &full[stage], kb * kBlockK, n0, g);
              else
                tma_load_2d(sB + stage * C::kBBytes, &tmB, &full[stage], kb * kBlockK, n0);
            }
          }
          __syncwarp();
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!live) {
        record_mx_status(kStatusTimeout);
        *abort_flag = 1;
        for (int s = 0; s < C::kStages && s < issued && (!kPair || rank == 0); ++s) {
          int st = stage - 1 - s;
          uint32_t ph = phase;
          if (st < 0) { st += C::kStages; ph ^= 1; }
          (void)mbar_wait(&full[st], ph, p.timeout_ns);
        }
      }
    } else if (warp == 1 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t gs = 0;           // scale slots used so far (ring position and phase)
      uint32_t tiles_done = 0;
      bool live = true;
      for (int t = unit0; t < total_tiles && live; t += nunits, ++tiles_done) {
        const uint32_t abuf = tiles_done % C::kAccBufs;
        const uint32_t aphase = (tiles_done / C::kAccBufs) & 1u;
        if (!warp_wait(&acc_empty[abuf], aphase ^ 1u, p.timeout_ns)) { live = false; break; }
        const uint32_t dtmem = tmem_base + abuf * BN;
        for (int kk = 0; kk < p.nkb; ++kk) {
          const uint32_t ring = gs % C::kSfSlots;
          // a full stage implies its slot's scales are in shared memory (the
          // producer waited for them before loading the slot's first stage)
          if (!warp_wait(&full[stage], phase, p.timeout_ns)) { live = false; break; }
          tc_fence_after_sync();
          if (lane == 0) {
            const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::kABytes));
            const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::kBBytes));
            const uint32_t sfa = tmem_base + C::kSfBase + ring * kSfSlotCols;
            if (kk % kStepsPerSlot == 0) {
              // the slot's scales: A rows into columns sfa .. sfa+3, B
              // columns into sfb + 4j .. sfb + 4j + 3 for each 128 of them
              const uint32_t src = smem_u32(sSf + ring * C::kSfSmemBytes);
#pragma unroll
              for (int j = 0; j <= BN / 128; ++j) {
                const uint32_t dst = j == 0 ? sfa : sfa + kSfbOffset + 4 * (j - 1);
                if (kPair)
                  tmem_cp_rows_pair(dst, sf_rows_desc(src + j * kSfRowsBytes));
                else
                  tmem_cp_rows(dst, sf_rows_desc(src + j * kSfRowsBytes));
              }
            }
            const uint32_t idesc = idesc_mx_e4m3(kPair ? 2 * kBlockM : kBlockM, BN,
                                                 static_cast<uint32_t>(kk % kStepsPerSlot));
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k) {
              const uint32_t acc = (kk > 0 || k > 0) ? 1u : 0u;
              if (kPair)
                mma_mx_e4m3_pair(dtmem, adesc + 2 * k, bdesc + 2 * k, idesc, sfa, sfa + kSfbOffset, acc);
              else
                mma_mx_e4m3(dtmem, adesc + 2 * k, bdesc + 2 * k, idesc, sfa, sfa + kSfbOffset, acc);
            }
            if (kPair) {
              mma_commit_pair(&empty[stage], 0x3);
            } else {
              mma_commit(&empty[stage]);
            }
            if (kk % kStepsPerSlot == kStepsPerSlot - 1 || kk + 1 == p.nkb) {
              if (kPair)
                mma_commit_pair(&sf_empty[ring], 0x3);
              else
                mma_commit(&sf_empty[ring]);
            }
            if (kk + 1 == p.nkb) {
              if (kPair)
                mma_commit_pair(&acc_full[abuf], 0x3);
              else
                mma_commit(&acc_full[abuf]);
            }
          }
          __syncwarp();
          if (kk % kStepsPerSlot == kStepsPerSlot - 1 || kk + 1 == p.nkb) ++gs;
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!live) {
        record_mx_status(kStatusTimeout);
        *abort_flag = 1;
      }
      // every MMA issued must have completed before TMEM is released
      if (lane == 0) {
        if (kPair)
          mma_commit_pair(&teardown[0], 0x1);
        else
          mma_commit(&teardown[0]);
      }
      __syncwarp();
      (void)mbar_wait(&teardown[0], 0, p.timeout_ns);
    } else if (warp == 2) {
      // ----------------------------------------------------- scale loader
      uint32_t step = 0;
      bool live = true;
      int g = 0;
      for (int t = unit0; t < total_tiles && live; t += nunits) {
        int row0, n0;
        int64_t row_end;
        tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
        const bool last_tile = t + nunits >= total_tiles;
        for (int kb = 0; kb < p.nkb; ++kb, ++step) {
          const uint32_t chunk = (step / C::kScaleChunk) % kMxScaleChunks;
          if (step % C::kScaleChunk == 0 &&
              !mbar_wait(&sc_empty[chunk], ((step / C::kScaleSlots) & 1u) ^ 1u, p.timeout_ns)) {
            live = false;
            break;
          }
          float* dst = sScale + (step % C::kScaleSlots) * C::kSlotFloats;
          const float* sa_kb = p.sa + static_cast<int64_t>(kb) * p.M;
#pragma unroll
          for (int i = 0; i < kBlockM / 32; ++i) {
            const int64_t r = static_cast<int64_t>(row0) + lane + 32 * i;
            if (r < p.M) cp_async_4(dst + lane + 32 * i, sa_kb + r);
          }
          if (kRowScale) {
#pragma unroll
            for (int i = 0; i < BN / 128; ++i) {
              const int c = 4 * (lane + 32 * i);
              if (n0 + c < p.N)
                cp_async_16(dst + kBlockM + c, p.sb + static_cast<int64_t>(kb) * p.N + n0 + c);
            }
          } else if (lane < BN / 128 && n0 + 128 * lane < p.N) {
            const int64_t nb = static_cast<int64_t>(g) * nnb + n0 / 128 + lane;
            cp_async_4(dst + kBlockM + lane, p.sb + nb * p.nkb + kb);
          }
          if (step % C::kScaleChunk == C::kScaleChunk - 1 || (last_tile && kb + 1 == p.nkb))
            cp_async_mbar_arrive(&sc_full[chunk]);
        }
      }
      if (!live) {
        record_mx_status(kStatusTimeout);
        *abort_flag = 1;
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == 3) {
      // -------------------------------------------------------- converter
      // Per scale slot (four k-blocks of a tile), lane i builds the rows i of
      // the slot's 512-byte blocks: A rows row0 + 32j + i (j = 0..3) and B
      // columns n0 + 32c + i, one byte per k-block, reading the float32 scale
      // ring kBatch k-blocks at a time (loads in flight together), and stores
      // them with 16-byte writes.  Block-scaled B has one scale per 128
      // columns, so a lane converts BN/128 B scales per k-block.
      constexpr int kBVals = kRowScale ? C::kSfbCols : BN / 128;
      constexpr int kBatch = kRowScale ? 2 : 4;
      uint32_t step = 0;
      uint32_t gs = 0;
      uint32_t bad = 0;
      bool live = true;
      int g = 0;
      for (int t = unit0; t < total_tiles && live; t += nunits) {
        int row0, n0;
        int64_t row_end;
        tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
        // scales outside the rows and columns the tile writes are not read
        // (their bytes are 127, 2^0) and not checked
        uint32_t a_ok = 0, b_ok = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t r = static_cast<int64_t>(row0) + 32 * j + lane;
          a_ok |= (r < row_end && r < p.M) ? 1u << j : 0u;
        }
#pragma unroll
        for (int v = 0; v < kBVals; ++v)
          b_ok |= (n0 + (kRowScale ? 32 * v + lane : 128 * v) < p.N) ? 1u << v : 0u;
        for (int sl = 0; sl < nsl && live; ++sl, ++gs) {
          const int nsteps = min(kStepsPerSlot, p.nkb - sl * kStepsPerSlot);
          uint32_t wa[4] = {0u, 0u, 0u, 0u};
          uint32_t wb[kBVals];
#pragma unroll
          for (int v = 0; v < kBVals; ++v) wb[v] = 0u;
#pragma unroll
          for (int b0 = 0; b0 < kStepsPerSlot; b0 += kBatch) {
            float va[kBatch][4];
            float vb[kBatch][kBVals];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              if (b0 + b < nsteps) {
                const uint32_t st = step + b0 + b;
                const uint32_t chunk = (st / C::kScaleChunk) % kMxScaleChunks;
                if (st % C::kScaleChunk == 0 &&
                    !mbar_wait(&sc_full[chunk], (st / C::kScaleSlots) & 1u, p.timeout_ns))
                  live = false;
                const float* scs = sScale + (st % C::kScaleSlots) * C::kSlotFloats;
#pragma unroll
                for (int j = 0; j < 4; ++j) va[b][j] = scs[32 * j + lane];
#pragma unroll
                for (int v = 0; v < kBVals; ++v) vb[b][v] = scs[kBlockM + (kRowScale ? 32 * v + lane : v)];
              }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              if (b0 + b < nsteps) {
                const uint32_t sh = 8u * static_cast<uint32_t>(b0 + b);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t e_bad = 0;
                  wa[j] |= ue8m0_of(va[b][j], e_bad) << sh;
                  bad |= (a_ok >> j) & e_bad;
                }
#pragma unroll
                for (int v = 0; v < kBVals; ++v) {
                  uint32_t e_bad = 0;
                  wb[v] |= ue8m0_of(vb[b][v], e_bad) << sh;
                  bad |= (b_ok >> v) & e_bad;
                }
                const uint32_t st = step + b0 + b;
                if (st % C::kScaleChunk == C::kScaleChunk - 1) {   // the chunk is read: hand it back
                  __syncwarp();
                  if (lane == 0) mbar_arrive(&sc_empty[(st / C::kScaleChunk) % kMxScaleChunks]);
                }
              }
            }
          }
          if (!live) break;
          step += nsteps;
#pragma unroll
          for (int j = 0; j < 4; ++j) wa[j] = (a_ok >> j) & 1u ? wa[j] : 0x7F7F7F7Fu;
#pragma unroll
          for (int v = 0; v < kBVals; ++v) wb[v] = (b_ok >> v) & 1u ? wb[v] : 0x7F7F7F7Fu;
          const uint32_t ring = gs % C::kSfSlots;
          if (!warp_wait(&sf_empty[ring], ((gs / C::kSfSlots) & 1u) ^ 1u, p.timeout_ns)) {
            live = false;
            break;
          }
          uint8_t* slot = sSf + ring * C::kSfSmemBytes;
          *reinterpret_cast<uint4*>(slot + 16 * lane) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
#pragma unroll
          for (int q = 0; q < BN / 128; ++q) {
            const uint4 w = kRowScale ? make_uint4(wb[4 * q % kBVals], wb[(4 * q + 1) % kBVals], wb[(4 * q + 2) % kBVals],
                                                   wb[(4 * q + 3) % kBVals])
                                      : make_uint4(wb[q % kBVals], wb[q % kBVals], wb[q % kBVals], wb[q % kBVals]);
            *reinterpret_cast<uint4*>(slot + kSfRowsBytes * (1 + q) + 16 * lane) = w;
          }
          fence_proxy_async_shared();   // visible to tcgen05.cp (async proxy)
          __syncwarp();
          if (lane == 0)
            mbar_arrive_cluster_release(kPair ? mapa_shared(&sf_full[ring], 0) : smem_u32(&sf_full[ring]));
        }
      }
      if (__any_sync(0xffffffffu, bad != 0u) && lane == 0) record_mx_status(kStatusDeviceArg);
      if (!live) {
        record_mx_status(kStatusTimeout);
        *abort_flag = 1;
      }
    }
  } else {
    setmaxnreg_inc<C::kRegsEpilogue>();
    const int e = warp - kMxEpiWarp0;    // 0..7
    const int quarter = warp & 3;        // TMEM lanes 32*quarter .. +31
    const int colhalf = e >> 2;          // which BN/2 columns this warp stores
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint8_t* s_out = smem + C::kOffOut + e * kMxOutSlots * kOutBoxBytes;
    uint32_t out_seq = 0;
    if (lane == 0 && e == 0) prefetch_tmap(&tmD);
    bool live = true;
    uint32_t epi_tiles = 0;   // tiles drained

    // Drains one tile's accumulator: read this thread's row (BN/2 columns)
    // out of TMEM, hand the accumulator back, store through shared memory.
    auto drain = [&](int row0, int n0, int64_t row_end) {
      const uint32_t abuf = epi_tiles % C::kAccBufs;
      const uint32_t aphase = (epi_tiles / C::kAccBufs) & 1u;
      ++epi_tiles;
      if (!mbar_wait(&acc_full[abuf], aphase, p.timeout_ns)) {
        live = false;
        return;
      }
      tc_fence_after_sync();
      uint32_t acc[C::kColsPerThread / 32][32];
      const uint32_t taddr = tmem_base + lane_base + abuf * BN + colhalf * C::kColsPerThread;
#pragma unroll
      for (int ch = 0; ch < C::kColsPerThread / 32; ++ch) tmem_ld32(taddr + ch * 32, acc[ch]);
#pragma unroll
      for (int ch = 0; ch < C::kColsPerThread / 32; ++ch) tmem_wait_ld(acc[ch]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (kPair)
          mbar_arrive_cluster(mapa_shared(&acc_empty[abuf], 0));
        else
          mbar_arrive(&acc_empty[abuf]);
      }
      const int ncol0 = n0 + colhalf * C::kColsPerThread;
      const int y0 = row0 + quarter * 32;
      if (y0 < row_end && ncol0 < p.N) {
        const float* v = reinterpret_cast<const float*>(&acc[0][0]);
        if (p.out_bf16)
          store_segment<C::kColsPerThread, true, kMxOutSlots>(v, s_out, out_seq, lane, &tmD, ncol0, y0, false);
        else
          store_segment<C::kColsPerThread, false, kMxOutSlots>(v, s_out, out_seq, lane, &tmD, ncol0, y0,
                                                               p.accumulate != 0);
      }
    };

    int g = 0;
    for (int t = unit0; t < total_tiles && live; t += nunits) {
      int row0, n0;
      int64_t row_end;
      tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
      drain(row0, n0, row_end);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (!live) {
      record_mx_status(kStatusTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (kPair) cluster_sync();
  if (warp == 1) {
    if (kPair)
      tmem_dealloc_pair(tmem_base, kMxTmemCols);
    else
      tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

template <int BN, bool kRowScale, bool kGrouped, bool kPair>
cudaError_t run_mx(const GemmArgs& a, int sm_count, cudaStream_t stream, bool* tmap_failed, bool* reg_check_failed) {
  using C = MxCfg<BN, kPair, kRowScale>;
  auto kern = gemm_mx_kernel<BN, kRowScale, kGrouped, kPair>;
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, kern);
  if (err != cudaSuccess) return err;
  if (static_cast<int64_t>(attr.numRegs) * kMxThreads <
      static_cast<int64_t>(C::kRegsProducer) * 128 + static_cast<int64_t>(C::kRegsEpilogue) * kMxEpiThreads) {
    *reg_check_failed = true;
    return cudaErrorInvalidConfiguration;
  }
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;

  CUtensorMap tmA, tmB, tmD;
  const uint64_t dA[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
  const uint64_t sA[1] = {static_cast<uint64_t>(a.K)};
  if (!encode_operand(&tmA, a.a, 2, dA, sA, kBlockM)) { *tmap_failed = true; return cudaErrorInvalidValue; }
  const uint32_t b_rows = kPair ? BN / 2 : BN;
  if (kGrouped) {
    const uint64_t dB[3] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.N),
                            static_cast<uint64_t>(a.num_groups)};
    const uint64_t sB[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.K) * a.N};
    if (!encode_operand(&tmB, a.b, 3, dB, sB, b_rows)) { *tmap_failed = true; return cudaErrorInvalidValue; }
  } else {
    const uint64_t dB[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.N)};
    const uint64_t sB[1] = {static_cast<uint64_t>(a.K)};
    if (!encode_operand(&tmB, a.b, 2, dB, sB, b_rows)) { *tmap_failed = true; return cudaErrorInvalidValue; }
  }
  if (!encode_output(&tmD, a.d, a.M, a.N, a.out_bf16, kOutRows)) { *tmap_failed = true; return cudaErrorInvalidValue; }

  KParams kp;
  kp.sa = a.sa;
  kp.sb = a.sb;
  kp.d = a.d;
  kp.offsets = a.offsets;
  kp.M = a.M;
  kp.N = static_cast<int>(a.N);
  kp.nkb = static_cast<int>(a.K / kBlockK);
  kp.num_groups = a.num_groups;
  kp.out_bf16 = a.out_bf16 ? 1 : 0;
  kp.accumulate = a.accumulate ? 1 : 0;
  kp.timeout_ns = a.timeout_ns;

  const int64_t ntn = (a.N + BN - 1) / BN;
  int64_t mt_bound = kGrouped ? (a.M / kBlockM + a.num_groups) : (a.M + kBlockM - 1) / kBlockM;
  if (kPair) mt_bound = (mt_bound + 1) / 2;
  const int64_t units = mt_bound * ntn;
  if (units <= 0) return cudaSuccess;
  static std::atomic<int> cluster_cache[kMaxCachedDevices];  // co-resident clusters, per device
  return launch_persistent<kPair>(kern, units, sm_count, kMxThreads, C::kSmemBytes, stream, cluster_cache, tmA, tmB,
                                  tmD, kp);
}

}  // namespace

cudaError_t launch_gemm_pow2(const GemmArgs& a, int sm_count, cudaStream_t stream, bool* tmap_failed,
                             bool* reg_check_failed) {
  *tmap_failed = false;
  *reg_check_failed = false;
  const int64_t mt = (a.M + kBlockM - 1) / kBlockM;
  const bool narrow = a.N <= 128 || (!a.grouped && mt * ((a.N + 255) / 256) < sm_count);
  if (a.grouped) {
    if (a.sb_row) return cudaErrorInvalidValue;
    return narrow ? run_mx<128, false, true, false>(a, sm_count, stream, tmap_failed, reg_check_failed)
                  : run_mx<256, false, true, true>(a, sm_count, stream, tmap_failed, reg_check_failed);
  }
  if (a.sb_row)
    return narrow ? run_mx<128, true, false, false>(a, sm_count, stream, tmap_failed, reg_check_failed)
                  : run_mx<256, true, false, true>(a, sm_count, stream, tmap_failed, reg_check_failed);
  return narrow ? run_mx<128, false, false, false>(a, sm_count, stream, tmap_failed, reg_check_failed)
                : run_mx<256, false, false, true>(a, sm_count, stream, tmap_failed, reg_check_failed);
}

cudaError_t gemm_mx_take_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_mx_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_mx_status, &zero, sizeof(int));
  }
  *status = v;
  return e;
}

}  // namespace fp8bs
