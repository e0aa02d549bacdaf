// Block-scaled FP8 GEMM on the 5th-generation tensor cores (tcgen05).
//
// D[m][n] = sum_kb P_kb[m][n] * s_a[m][kb] * s_b(n, kb), where P_kb is the
// E4M3 x E4M3 product over one 128-wide block of K.  This is the
// "increasing accumulation precision" scheme of DeepSeek-V3 §3.3.2 / Figure
// 7b (every N_C = 128 elements the tensor-core partial is promoted to FP32,
// multiplied by the two scales and accumulated; §3.5.2 names the cost of
// that data movement), mapped onto Blackwell:
//
//   * a persistent, warp-specialised CTA per SM (or per SM of a CTA pair
//     running the 2-SM MMA over 256-row tiles): warp 0 issues TMA loads of
//     128x128 A and B tiles into a shared-memory ring; warps 1 and 3 issue
//     the MMAs of alternate k-blocks (4 x tcgen05.mma K=32 per 128-K block)
//     into one of two TMEM partial buffers, the first of the four
//     overwriting the buffer; warp 2 copies each k-block's scales (128 row
//     scales of A, the B scales of the tile's columns) into a shared-memory
//     scale ring with cp.async; warps 4-11 (two warpgroups) fold each
//     finished partial into FP32 registers with the block's scales
//     (acc += P_kb * s_a * s_b) while the tensor core computes the next
//     block into the other buffer;
//   * the running FP32 accumulator never leaves the registers; each thread
//     owns one output row (its TMEM lane) and BN/2 columns.  A TMEM buffer
//     is released as soon as its last columns are in registers, before the
//     last multiply-adds.  At the end of a tile each warp stages its rows in
//     shared memory and TMA stores them, so the write drains while the warp
//     folds the next tile;
//   * mbarrier pipelines (operand ring, scale ring, TMEM buffers) with
//     bounded waits; a timeout records a status and unwinds.
//
// The same kernel serves the dense GEMM (one group) and the grouped MoE
// GEMM (per-expert row segments whose offsets are multiples of 128, read
// from device memory; CTA pairs are formed inside each segment; the expert
// index selects B's slice through a 3-D tensor map).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8bs {
namespace {

__device__ int g_gemm_status;

constexpr int kThreads = 384;        // 12 warps
constexpr int kEpiWarp0 = 4;         // warps 4..11 fold and store
constexpr int kEpiThreads = 256;
// Scale ring: Cfg::kScaleSlots k-blocks of scales, handed between the
// loader and the epilogue in kScaleChunks chunks of Cfg::kScaleChunk slots.
// Every mbarrier operation costs the epilogue warps a shared-memory round
// trip of some 170 cycles while TMA and the tensor core keep shared memory
// busy, and each epilogue warp handles every k-block, so the hand-off is
// per chunk rather than per k-block: 16 k-blocks per chunk where the slots
// are small (block-scaled B), 8 for row-scaled B, whose per-column slots
// would otherwise crowd out operand stages.
constexpr int kScaleChunks = 2;
constexpr uint32_t kTmemCols = 512;  // all of TMEM: 512 / BN partial buffers
// Register split (setmaxnreg): the four producer/issuer warps shrink to
// kRegsProducer, the eight epilogue warps grow to kRegsEpilogue, which holds
// the 128 FP32 accumulators, two 32-column TMEM reads in flight and the
// loop state without spilling; 4 x 32 x 40 + 8 x 32 x 232 = 384 x 168, the
// CTA's allocation at launch.
constexpr uint32_t kRegsProducer = 40;
constexpr uint32_t kRegsEpilogue = 232;


// BN is the tile width of one CTA's output; with kPair (2-SM MMA) each CTA
// holds only half of the B tile's rows in its shared memory.
template <int BN, bool kPair, bool kRowScale>
struct Cfg {
  static constexpr int kABytes = kBlockM * kBlockK;                   // 16 KB
  static constexpr int kBBytes = (kPair ? BN / 2 : BN) * kBlockK;     // 16 or 32 KB per CTA
  static constexpr int kStageBytes = kABytes + kBBytes;
  // TMEM partial buffers: the MMA of k-block j+kBufs may start only once
  // the epilogue has read k-block j out, so more buffers hide more of that
  // hand-off (commit, TMEM read-out, release) behind tensor-core work.
  static constexpr int kBufs = static_cast<int>(kTmemCols) / BN;
  // scale slot: A row scales, then B scales (per column, or one per
  // 128-column block padded to 16 bytes)
  static constexpr int kSlotFloats = kBlockM + (kRowScale ? BN : 4);
  static constexpr int kScaleChunk = kRowScale ? 8 : 16;
  static constexpr int kScaleSlots = kScaleChunk * kScaleChunks;
  static constexpr int kColsPerThread = BN / 2;
  static constexpr int kChunks = kColsPerThread / 32;
  static constexpr int kOutBytes = (kEpiThreads / 32) * kOutSlots * kOutBoxBytes;
  static constexpr int kMaxStages = 6;
  static constexpr int kNumBarsMax = 2 * kMaxStages + 2 * kScaleChunks + 2 * kBufs + 2;
  static constexpr int kFixedBytes =
      kOutBytes + kScaleSlots * kSlotFloats * 4 + kNumBarsMax * 8 + 16 + 2 * (kMaxGroups + 1) * 4 + 1024;
  // Operand ring: as many stages as the rest leaves room for, rounded down
  // to an even count.  The two MMA-issuing warps take alternate k-block
  // steps, so with an even ring each stage is only ever consumed by the
  // same warp, which therefore never waits on a stage more than one phase
  // ahead of its barrier.
  static constexpr int kFit = (kSmemBudget - kFixedBytes) / kStageBytes;
  static constexpr int kStages = (kFit < kMaxStages ? kFit : kMaxStages) & ~1;
  static_assert(kStages >= 4, "operand ring too shallow");
  // dynamic shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffOut = kOffB + kStages * kBBytes;             // 1024-aligned
  static constexpr int kOffScale = kOffOut + kOutBytes;
  static constexpr int kOffBar = kOffScale + kScaleSlots * kSlotFloats * 4;
  static constexpr int kNumBars = 2 * kStages + 2 * kScaleChunks + 2 * kBufs + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;       // tmem slot, abort flag, tile count
  static constexpr int kOffGroups = kOffMisc + 16;              // offsets[G+1], cum[G+1]
  static constexpr int kSmemBytes = kOffGroups + 2 * (kMaxGroups + 1) * 4 + 1024;  // + alignment slack
  static_assert(kOffOut % 1024 == 0, "staging boxes need 1024-byte alignment for the 128-byte swizzle");
  static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
};

// acc[j] += p[j] * s for 32 accumulators (16 pairs), one packed FP32x2
// FMA per pair.
__device__ __forceinline__ void fold_block(float2* acc, const uint32_t (&p)[32], float s) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    acc[j] = __ffma2_rn(make_float2(__uint_as_float(p[2 * j]), __uint_as_float(p[2 * j + 1])), s2, acc[j]);
}

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_gemm_status, 0, code); }

template <int BN, bool kRowScale, bool kGrouped, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmD, const KParams p) {
  using C = Cfg<BN, kPair, kRowScale>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::kOffA;
  uint8_t* sB = smem + C::kOffB;
  float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;                               // [kStages] TMA -> MMA
  uint64_t* empty = bars + C::kStages;                 // [kStages] MMA -> TMA
  uint64_t* sc_full = bars + 2 * C::kStages;           // [kScaleChunks] scales landed
  uint64_t* sc_empty = sc_full + kScaleChunks;         // [kScaleChunks] epilogue done with them
  uint64_t* t_full = sc_empty + kScaleChunks;          // [kBufs] partial ready in TMEM
  uint64_t* t_empty = t_full + C::kBufs;               // [kBufs] partial read out of TMEM
  uint64_t* teardown = t_empty + C::kBufs;             // [2] one per MMA issuer
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* s_off = reinterpret_cast<int*>(smem + C::kOffGroups);
  int* s_cum = s_off + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ntn = (p.N + BN - 1) / BN;
  // work units are tiles, or tile pairs handled by the two CTAs of a cluster
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int unit0 = kPair ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int nunits = kPair ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int nnb = (p.N + kGroup - 1) / kGroup;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kScaleChunks; ++s) {
      mbar_init(&sc_full[s], 32);                      // one cp.async arrival per loader lane
      mbar_init(&sc_empty[s], kEpiThreads / 32);       // one arrival per epilogue warp
    }
    for (int b = 0; b < C::kBufs; ++b) {
      mbar_init(&t_full[b], 1);
      mbar_init(&t_empty[b], (kPair ? 2 : 1) * kEpiThreads / 32);  // with pairs: both CTAs' epilogue warps
    }
    mbar_init(&teardown[0], 1);
    mbar_init(&teardown[1], 1);
    fence_barrier_init();
    griddep_wait();  // the group table below may come from the preceding kernel
    // tile count (and, for the grouped GEMM, the validated group table)
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
        for (int g = 0; g < p.num_groups; ++g) {  // work units (m-tiles or m-tile pairs) per group
          s_cum[g] = total_mt;
          const int mt = (s_off[g + 1] - s_off[g]) / kBlockM;
          total_mt += kPair ? (mt + 1) / 2 : mt;
        }
        s_cum[p.num_groups] = total_mt;
      } else {
        record_status(kStatusDeviceArg);
        total_mt = 0;
      }
    } else {
      total_mt = static_cast<int>((p.M + kBlockM - 1) / kBlockM);
      if (kPair) total_mt = (total_mt + 1) / 2;
    }
    misc[1] = 0;  // abort flag
    misc[2] = static_cast<uint32_t>(total_mt * ntn);
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(&misc[0], kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&misc[0], kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (kPair) cluster_sync();  // the peer's barriers exist before anything signals them
  // Launched behind another kernel (programmatic dependent launch), the
  // set-up above overlaps that kernel's tail; operands, scales and D are
  // touched only after it has completed.
  griddep_wait();
  const uint32_t tmem_base = misc[0];
  const int total_tiles = static_cast<int>(misc[2]);
  volatile uint32_t* abort_flag = &misc[1];

  if (warp < kEpiWarp0) {
    setmaxnreg_dec<kRegsProducer>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      bool live = true;
      int issued = 0;
      int g = 0;
      for (int t = unit0; t < total_tiles && live; t += nunits) {
        int row0, n0;
        int64_t row_end;
        tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!warp_wait(&empty[stage], phase ^ 1, p.timeout_ns)) { live = false; break; }
          if (lane == 0) {
            if (kPair) {
              // Both CTAs' tiles complete on the leader's barrier, which the
              // leader arms for the pair's bytes; each CTA loads its A rows
              // and its half of the B tile into its own shared memory.
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
        record_status(kStatusTimeout);
        *abort_flag = 1;
        // let the copies already issued land before the CTA can exit
        for (int s = 0; s < C::kStages && s < issued && (!kPair || rank == 0); ++s) {
          int st = stage - 1 - s;
          uint32_t ph = phase;
          if (st < 0) { st += C::kStages; ph ^= 1; }
          (void)mbar_wait(&full[st], ph, p.timeout_ns);
        }
      }
    } else if ((warp == 1 || warp == 3) && rank == 0) {
      // --------------------------------------------------------- MMA issuers
      // Two issuing warps take alternate k-block steps (warp 1 the even
      // ones, warp 3 the odd ones; lane 0 issues): issuing a k-block's MMAs
      // blocks the issuing thread for about as long as the tensor core
      // takes to accept them, so one warp can prepare the next step while
      // the other's MMAs drain.  Step s uses TMEM buffer s % kBufs.  With pairs
      // only the leader CTA issues: one M=256 MMA covers both CTAs.
      constexpr uint32_t idesc = idesc_e4m3_f32(kPair ? 2 * kBlockM : kBlockM, BN);
      const uint32_t parity = warp == 1 ? 0u : 1u;
      uint32_t step = 0;
      bool live = true;
      for (int t = unit0; t < total_tiles && live; t += nunits) {
        for (int kk = 0; kk < p.nkb; ++kk, ++step) {
          if ((step & 1u) != parity) continue;
          const int stage = static_cast<int>(step % C::kStages);
          const uint32_t phase = (step / C::kStages) & 1u;
          const uint32_t buf = step % C::kBufs;
          const uint32_t tphase = (step / C::kBufs) & 1u;
          if (!warp_wait(&full[stage], phase, p.timeout_ns)) { live = false; break; }
          if (!warp_wait(&t_empty[buf], tphase ^ 1, p.timeout_ns)) { live = false; break; }
          tc_fence_after_sync();
          if (lane == 0) {
            const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::kABytes));
            const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::kBBytes));
            const uint32_t dtmem = tmem_base + buf * BN;
            if (kPair) {
#pragma unroll
              for (int k = 0; k < kBlockK / kUmmaK; ++k)
                mma_e4m3_pair(dtmem, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
              mma_commit_pair(&empty[stage], 0x3);
              mma_commit_pair(&t_full[buf], 0x3);
            } else {
#pragma unroll
              for (int k = 0; k < kBlockK / kUmmaK; ++k)
                mma_e4m3(dtmem, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
              mma_commit(&empty[stage]);
              mma_commit(&t_full[buf]);
            }
          }
          __syncwarp();
        }
      }
      if (!live) {
        record_status(kStatusTimeout);
        *abort_flag = 1;
      }
      // wait for every MMA this warp issued before TMEM can be released
      if (lane == 0) {
        if (kPair)
          mma_commit_pair(&teardown[parity], 0x1);
        else
          mma_commit(&teardown[parity]);
      }
      __syncwarp();
      (void)mbar_wait(&teardown[parity], 0, p.timeout_ns);
    } else if (warp == 2) {
      // ----------------------------------------------------- scale loader
      // Slot layout: [0,128) row scales of A for the tile's 128 rows,
      // [128, 128+BN) B scales: per column (row kind) or, for 128x128
      // block scales, one per 128-column block of the tile.  Step s (the
      // CTA's s-th k-block over all its tiles) uses slot s % kScaleSlots;
      // a chunk is announced once its last slot is issued (or at the CTA's
      // final step).
      uint32_t step = 0;
      bool live = true;
      int g = 0;
      for (int t = unit0; t < total_tiles && live; t += nunits) {
        int row0, n0;
        int64_t row_end;
        tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
        const bool last_tile = t + nunits >= total_tiles;
        for (int kb = 0; kb < p.nkb; ++kb, ++step) {
          const uint32_t chunk = (step / C::kScaleChunk) % kScaleChunks;
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
        record_status(kStatusTimeout);
        *abort_flag = 1;
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else {
    setmaxnreg_inc<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;      // 0..7
    const int quarter = warp & 3;        // TMEM lanes 32*quarter .. +31
    const int colhalf = e >> 2;          // which BN/2 columns
    const int row_in_tile = quarter * 32 + lane;
    uint8_t* s_out = smem + C::kOffOut + e * kOutSlots * kOutBoxBytes;
    uint32_t out_seq = 0;
    if (lane == 0 && e == 0) prefetch_tmap(&tmD);
    uint32_t buf = 0, tphase = 0;
    uint32_t step = 0;
    bool live = true;
    int g = 0;
    for (int t = unit0; t < total_tiles && live; t += nunits) {
      int row0, n0;
      int64_t row_end;
      tile_coords<BN, kPair>(t, ntn, kGrouped, s_off, s_cum, p.num_groups, rank, p.M, row0, n0, g, row_end);
      const int ncol0 = n0 + colhalf * C::kColsPerThread;
      const int bsel = (colhalf * C::kColsPerThread) / 128;   // which 128-column block of the tile
      float2 acc2[C::kColsPerThread / 2];
#pragma unroll
      for (int j = 0; j < C::kColsPerThread / 2; ++j) acc2[j] = make_float2(0.0f, 0.0f);
      for (int kk = 0; kk < p.nkb; ++kk, ++step) {
        const uint32_t chunk = (step / C::kScaleChunk) % kScaleChunks;
        if (step % C::kScaleChunk == 0 &&
            !mbar_wait(&sc_full[chunk], (step / C::kScaleSlots) & 1u, p.timeout_ns)) {
          live = false;
          break;
        }
        const float* scs = sScale + (step % C::kScaleSlots) * C::kSlotFloats;
        if constexpr (kRowScale) {
          // Per-column scales: the partial is read in the fragment layout of
          // tcgen05.ld.16x256b, where a thread holds 8 of every 32 columns
          // (of 4 rows), so it needs a quarter of the column scales a
          // row-per-thread layout needs: per 64-column chunk 8 pairs, loaded
          // one chunk ahead (the first chunk's and the 4 row scales before
          // the wait for the partial).  Pieces of 16 lanes x 64 columns (32
          // registers) take half the loads of 32-column ones (3% faster).
          float sa4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) sa4[i] = scs[quarter * 32 + 8 * i + (lane >> 2)];
          const float* scol = scs + kBlockM + colhalf * C::kColsPerThread + 2 * (lane & 3);
          float2 sbc[2][8];
#pragma unroll
          for (int i = 0; i < 8; ++i) sbc[0][i] = *reinterpret_cast<const float2*>(scol + 8 * i);
          if (!mbar_wait(&t_full[buf], tphase, p.timeout_ns)) { live = false; break; }
          tc_fence_after_sync();
          const uint32_t tcol = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN +
                                colhalf * C::kColsPerThread;
          // pieces (64-column chunk c, 16-lane half h), chunk-major, the next
          // piece's load in flight while the current one is folded
          constexpr int kC64 = C::kChunks / 2;
          constexpr int kFrag = 2 * kC64;
          uint32_t fr[2][32];
          tmem_ld16x256b_x8(tcol, fr[0]);
          tmem_wait_ld(fr[0]);
#pragma unroll
          for (int f = 0; f < kFrag; ++f) {
            const int h = f & 1, c = f >> 1;
            if (h == 0 && c + 1 < kC64) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                sbc[(c + 1) & 1][i] = *reinterpret_cast<const float2*>(scol + 64 * (c + 1) + 8 * i);
            }
            if (f + 1 < kFrag) {
              const int nh = (f + 1) & 1, nc = (f + 1) >> 1;
              tmem_ld16x256b_x8(tcol + (static_cast<uint32_t>(16 * nh) << 16) + 64 * nc, fr[(f + 1) & 1]);
            } else {
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) {
                if (kPair)
                  mbar_arrive_cluster(mapa_shared(&t_empty[buf], 0));  // the leader's MMA waits on it
                else
                  mbar_arrive(&t_empty[buf]);
              }
            }
            {
              const uint32_t (&pp)[32] = fr[f & 1];
              const float2 a0 = make_float2(sa4[2 * h], sa4[2 * h]);
              const float2 a1 = make_float2(sa4[2 * h + 1], sa4[2 * h + 1]);
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                const int cc = 2 * c + (g >> 2), gg = g & 3;
                float2* ac = acc2 + ((h * C::kChunks + cc) * 4 + gg) * 2;
                ac[0] = __ffma2_rn(make_float2(__uint_as_float(pp[4 * g]), __uint_as_float(pp[4 * g + 1])),
                                   __fmul2_rn(a0, sbc[c & 1][g]), ac[0]);
                ac[1] = __ffma2_rn(make_float2(__uint_as_float(pp[4 * g + 2]), __uint_as_float(pp[4 * g + 3])),
                                   __fmul2_rn(a1, sbc[c & 1][g]), ac[1]);
              }
            }
            if (f + 1 < kFrag) tmem_wait_ld(fr[(f + 1) & 1]);
          }
        } else {
          if (!mbar_wait(&t_full[buf], tphase, p.timeout_ns)) { live = false; break; }
          tc_fence_after_sync();
          const float sa = scs[row_in_tile];
          const float s_ab = sa * scs[kBlockM + bsel];
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN +
                                 colhalf * C::kColsPerThread;
          // TMEM -> registers 32 columns at a time, the next chunk's load in
          // flight while the current one is folded; the buffer is handed back
          // to the MMA as soon as the last chunk has landed.
          uint32_t rr[2][32];
          tmem_ld32(taddr, rr[0]);
          tmem_wait_ld(rr[0]);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch) {
            if (ch + 1 < C::kChunks) {
              tmem_ld32(taddr + (ch + 1) * 32, rr[(ch + 1) & 1]);
            } else {
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) {
                if (kPair)
                  mbar_arrive_cluster(mapa_shared(&t_empty[buf], 0));  // the leader's MMA waits on it
                else
                  mbar_arrive(&t_empty[buf]);
              }
            }
            fold_block(acc2 + ch * 16, rr[ch & 1], s_ab);
            if (ch + 1 < C::kChunks) tmem_wait_ld(rr[(ch + 1) & 1]);
          }
        }
        if (step % C::kScaleChunk == C::kScaleChunk - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sc_empty[chunk]);
        }
        if (++buf == C::kBufs) { buf = 0; tphase ^= 1; }
      }
      if (!live) break;
      // ---- store the warp's 32 rows x BN/2 columns through shared memory
      // and TMA; rows past M are clipped by the tensor map
      const float* acc = reinterpret_cast<const float*>(acc2);
      const int y0 = row0 + quarter * 32;
      if (y0 < row_end && ncol0 < p.N) {
        if constexpr (kRowScale) {
          if (p.out_bf16)
            store_segment_frag<C::kColsPerThread, true>(acc2, s_out, out_seq, lane, &tmD, ncol0, y0, false);
          else
            store_segment_frag<C::kColsPerThread, false>(acc2, s_out, out_seq, lane, &tmD, ncol0, y0,
                                                         p.accumulate != 0);
        } else {
          if (p.out_bf16)
            store_segment<C::kColsPerThread, true>(acc, s_out, out_seq, lane, &tmD, ncol0, y0, false);
          else
            store_segment<C::kColsPerThread, false>(acc, s_out, out_seq, lane, &tmD, ncol0, y0, p.accumulate != 0);
        }
      }
    }
    // the staging boxes stay in use until the last stores have completed
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (!live) {
      record_status(kStatusTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (kPair) cluster_sync();  // no CTA leaves while its peer may still signal or use it
  if (warp == 1) {
    if (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BN, bool kRowScale, bool kGrouped, bool kPair>
cudaError_t run(const GemmArgs& a, int sm_count, cudaStream_t stream, bool* tmap_failed, bool* reg_check_failed) {
  using C = Cfg<BN, kPair, kRowScale>;
  auto kern = gemm_kernel<BN, kRowScale, kGrouped, kPair>;
  // The register split (warps 0-3 shrink to kRegsProducer, warps 4-11 grow
  // to kRegsEpilogue) must fit in what the CTA is launched with.
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, kern);
  if (err != cudaSuccess) return err;
  if (static_cast<int64_t>(attr.numRegs) * kThreads <
      static_cast<int64_t>(kRegsProducer) * 128 + static_cast<int64_t>(kRegsEpilogue) * kEpiThreads) {
    *reg_check_failed = true;
    return cudaErrorInvalidConfiguration;
  }
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;

  CUtensorMap tmA, tmB;
  const uint64_t dA[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
  const uint64_t sA[1] = {static_cast<uint64_t>(a.K)};
  if (!encode_operand(&tmA, a.a, 2, dA, sA, kBlockM)) { *tmap_failed = true; return cudaErrorInvalidValue; }
  const uint32_t b_rows = kPair ? BN / 2 : BN;  // with pairs each CTA fetches half of the B tile
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

  CUtensorMap tmD;
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

  // Persistent grid: one CTA per SM (one cluster per SM pair), or fewer
  // when there are fewer work units.  (The grouped tile count lives on the
  // device; the grid covers its bound.)
  const int64_t ntn = (a.N + BN - 1) / BN;
  int64_t mt_bound = kGrouped ? (a.M / kBlockM + a.num_groups) : (a.M + kBlockM - 1) / kBlockM;
  if (kPair) mt_bound = (mt_bound + 1) / 2;
  const int64_t units = mt_bound * ntn;
  if (units <= 0) return cudaSuccess;
  static std::atomic<int> cluster_cache[kMaxCachedDevices];  // co-resident clusters, per device
  return launch_persistent<kPair>(kern, units, sm_count, kThreads, C::kSmemBytes, stream, cluster_cache, tmA, tmB,
                                  tmD, kp);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, int sm_count, cudaStream_t stream, bool* tmap_failed,
                        bool* reg_check_failed) {
  *tmap_failed = false;
  *reg_check_failed = false;
  // 128-wide n-tiles when 256-wide ones would leave most SMs idle.
  const int64_t mt = (a.M + kBlockM - 1) / kBlockM;
  const bool narrow = a.N <= 128 || (!a.grouped && mt * ((a.N + 255) / 256) < sm_count);
  if (a.grouped) {  // pairs formed within each expert's segment
    if (a.sb_row) return cudaErrorInvalidValue;
    return narrow ? run<128, false, true, false>(a, sm_count, stream, tmap_failed, reg_check_failed)
                  : run<256, false, true, true>(a, sm_count, stream, tmap_failed, reg_check_failed);
  }
  if (a.sb_row)
    return narrow ? run<128, true, false, false>(a, sm_count, stream, tmap_failed, reg_check_failed)
                  : run<256, true, false, true>(a, sm_count, stream, tmap_failed, reg_check_failed);
  return narrow ? run<128, false, false, false>(a, sm_count, stream, tmap_failed, reg_check_failed)
                : run<256, false, false, true>(a, sm_count, stream, tmap_failed, reg_check_failed);
}

// Diagnostic kernel: one thread waits, through the same bounded mbarrier
// wait every kernel here uses, on a barrier that nothing arrives on; when the
// wait gives up it records FP8BS_ERR_TIMEOUT in the GEMM status word and the
// kernel returns normally.  No copies or MMAs are in flight.
__global__ void wait_timeout_selftest_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait(&bar, 0, timeout_ns)) record_status(kStatusTimeout);
}

cudaError_t launch_wait_timeout_selftest(uint64_t timeout_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns);
  return cudaGetLastError();
}

cudaError_t gemm_take_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(int));
  }
  *status = v;
  return e;
}

}  // namespace fp8bs
