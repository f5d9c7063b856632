// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The grouped layer of the summary page of "Diagonal Batching Unlocks
// Parallelism in Recurrent Memory Transformers for Long Contexts" (section 三):
// every linear layer of the cells of one diagonal runs as one grouped matrix
// product over stacked per-layer weights, the outputs preallocated as one
// tensor and addressed per group.  Here a group is a layer l in
// [g_first, g_first + g_count); for each of them
//     out[l] = epilogue( A[l] (rows x K, bf16)  *  B[l]^T (B: N x K, bf16) )
// with fp32 accumulation.  A and B are read through 3-D TMA tensor maps
// {K, rows, layer} so that row tiles past the end of a cell are zero-filled.
//
// One persistent CTA per SM walks the tiles (layer-major, then N tile, then
// M tile, so CTAs running at the same time share the weight tile in L2):
//   warp 0      TMA producer: A tile 128 x 64 and B tile BN x 64 per stage,
//   warp 1      MMA issuer (one thread): 4 x tcgen05.mma (K = 16 each) per
//               stage into a 128 x BN fp32 accumulator in TMEM,
//   warps 2..    epilogue (4 or 8 warps): tcgen05.ld of their 32 TMEM lanes (= tile rows),
//               staged through shared memory so that the fused epilogue
//               reads and writes global memory row by row, lanes across
//               columns (epilogues_staged.cuh).
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1.  Every output element is reduced in the same fixed K order no matter
// how many groups a launch holds (no split-K, no atomics), so a cell gives
// bit-identical results in a one-cell launch and in a full diagonal.
#pragma once

#include "common.cuh"
#include "epilogues.cuh"
#include "epilogues_staged.cuh"

namespace armt {

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;  // one 128-byte swizzle row of bf16

// How a group index gi of a launch addresses its operands:
//   A rows  [r0, r0 + rows) of A slot gi + a_slot_off, with r0 = alt_row0
//           for gi in [alt_lo, alt_hi) and row0 otherwise (a cell whose
//           memory rows sit elsewhere, e.g. after a short last segment);
//   B       slot gi / b_div + b_slot_off (b_div = sequences per layer when
//           the groups are (layer, sequence) pairs sharing a layer's weights).
//   a_lo_slot > 0: A is split into a bf16 high part and a bf16 low part
//           (the rounding residual), the low part a_lo_slot slots after the
//           high one; b_lo_slot > 0: the same for B.  The K loop then runs
//           once per pair of parts (A high / low x B high / low, A fastest),
//           so the product sees split operands with about 16 significant
//           bits (split precision).
struct GemmGroupMap {
  int row0 = 0, a_slot_off = 0, b_slot_off = 0, b_div = 1;
  int alt_lo = 0, alt_hi = 0, alt_row0 = 0;
  int a_lo_slot = 0, b_lo_slot = 0;
  __host__ __device__ int a_parts() const { return a_lo_slot > 0 ? 2 : 1; }
  __host__ __device__ int passes() const { return a_parts() * (b_lo_slot > 0 ? 2 : 1); }
  __host__ __device__ int a_row0(int gi) const { return gi >= alt_lo && gi < alt_hi ? alt_row0 : row0; }
};

struct GemmTcShape {
  int rows;       // valid rows per group (M), counted from the group's first A row
  GemmGroupMap map;
  int N, K;
  int g_first, g_count;
  int m_tiles, n_tiles, k_blocks;
  int kb_split;   // k blocks of one pass when an operand is split (map.passes() > 1), else 0
  int* err;       // device error word
  WaitPolicy wp;  // wait limit and the test stall hook
};

// EPI_WG epilogue warpgroups (1 or 2); with 2, each takes half of the tile's
// columns (for GEMMs whose short K loop leaves the epilogue exposed) and the
// pipeline keeps one stage less to make room for their shared-memory stages.
template <int BN, int EPI_WG>
struct TcCfg {
  static constexpr int STAGES = BN >= 256 ? (EPI_WG == 2 ? 3 : 4) : 8;
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;
  static constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
  static constexpr int EPI_WARPS = 4 * EPI_WG;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr uint32_t EPI_STAGE_BYTES = EPI_WARPS * STAGED_FLOATS_PER_WARP * 4;
  static constexpr size_t SMEM = 1024 + STAGES * STAGE_BYTES + 256 + EPI_STAGE_BYTES;
  static_assert(SMEM <= 232448, "shared memory");
};

template <class Epi, int BN, int EPI_WG>
__global__ void __launch_bounds__(TcCfg<BN, EPI_WG>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmTcShape sh, const Epi epi) {
  using C = TcCfg<BN, EPI_WG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;  // completion of every MMA this CTA issued
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], C::EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tiles_per_g = sh.m_tiles * sh.n_tiles;
  const int num_tiles = sh.g_count * tiles_per_g;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;  // stage loads issued (full[] phases armed)
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        const int g = t / tiles_per_g, r = t - g * tiles_per_g;
        const int nt = r / sh.m_tiles, mt = r - nt * sh.m_tiles;
        const int layer = sh.g_first + g;
        const int a_row = sh.map.a_row0(layer) + mt * TC_BM;
        const int b_slot = layer / sh.map.b_div + sh.map.b_slot_off;
        // split operands: pass p (K blocks kpp p .. kpp (p + 1) - 1) reads A part
        // p % a_parts and B part p / a_parts (0 = high, 1 = low); tracked
        // incrementally, so the unsplit loop does no division
        const int kpp = sh.kb_split > 0 ? sh.kb_split : sh.k_blocks, two_a = sh.map.a_parts() == 2;
        int kk = 0, pass = 0;
        for (int kb = 0; kb < sh.k_blocks; ++kb) {
          if (issued == sh.wp.stall_after ||
              !mbar_wait_bounded(&empty[stage], phase ^ 1u, sh.err, DEV_TIMEOUT_EMPTY, sh.wp.limit_ns)) {
            ok = false;
            break;
          }
          const int kc = kk * TC_BK;
          const int ap = two_a ? (pass & 1) : 0, bp = two_a ? (pass >> 1) : pass;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_3d(sA + stage * C::A_BYTES, &tmA, kc, a_row,
                      layer + sh.map.a_slot_off + ap * sh.map.a_lo_slot, &full[stage]);
          tma_load_3d(sB + stage * C::B_BYTES, &tmB, kc, nt * BN, b_slot + bp * sh.map.b_lo_slot, &full[stage]);
          if (++kk == kpp) {
            kk = 0;
            ++pass;
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the loads of the last STAGES stages land before the CTA lets
      // go of its shared memory (the MMA thread may have stopped consuming
      // them).  Earlier stages were consumed, so they have landed already.
      for (int j = issued > C::STAGES ? issued - C::STAGES : 0; j < issued; ++j)
        mbar_wait_drain(&full[j % C::STAGES], (uint32_t)((j / C::STAGES) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // A last row tile with at most 16 valid rows (the memory rows that close
      // a 1040-row cell, or a 16-row write projection) runs as an M = 64 MMA:
      // half the tensor work of M = 128 for the same 16 rows, which land in
      // TMEM lanes 0..15 with either M -- the lanes the epilogue reads for them.
      constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
      constexpr uint32_t idesc64 = idesc_bf16_f32(64, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        const int mt = (t % tiles_per_g) % sh.m_tiles;
        const uint32_t id = sh.rows - mt * TC_BM <= 16 ? idesc64 : idesc;
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, sh.err, DEV_TIMEOUT_ACC_EMPTY, sh.wp.limit_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < sh.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, sh.err, DEV_TIMEOUT_FULL, sh.wp.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * C::A_BYTES));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k) {
            // advance 16 bf16 = 32 bytes along K inside the swizzled row
            tc_mma_bf16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), id,
                        (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);  // stage reusable once these MMAs finish
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);  // accumulator ready for the epilogue
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Drain: every MMA issued above has finished (and made its arrivals)
      // before TMEM is freed, also when the loop stopped early.
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int ew = warp - 2;       // epilogue warp index
    const int part = ew / 4;       // column part of the tile this warp handles
    float* stage = reinterpret_cast<float*>(base + C::STAGES * C::STAGE_BYTES + 256) +
                   ew * STAGED_FLOATS_PER_WARP;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const int g = t / tiles_per_g, r = t - g * tiles_per_g;
      const int nt = r / sh.m_tiles, mt = r - nt * sh.m_tiles;
      const bool got = mbar_wait_bounded(&acc_full[acc], acc_phase, sh.err, DEV_TIMEOUT_ACC_FULL, sh.wp.limit_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      staged_epilogue<BN, EPI_WG>(epi, sh.g_first + g, mt * TC_BM + quarter * 32, sh.rows, nt * BN,
                                  part, tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16),
                                  stage);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// Host side --------------------------------------------------------------

// Encodes a 3-D bf16 tensor map over [layers][rows][K] (K contiguous) with a
// box of {64, box_rows, 1} and 128-byte swizzling.  Returns false on error.
// Also used for fp16 data: a tile copy moves the 16-bit elements unchanged
// and its zero fill (all bits clear) is +0 in either type.
bool encode_tmap_bf16_3d(CUtensorMap* map, const void* base, int K, int rows, int layers,
                         int box_rows);

// Internal linkage: each translation unit configures and launches its own copy.
template <class Epi, int BN, int EPI_WG = 1>
static cudaError_t launch_gemm_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, int rows, int N, int K,
                           int g_first, int g_count, int* err, const Epi& epi, int num_sms,
                           cudaStream_t stream, const GemmGroupMap& map = GemmGroupMap(),
                           const WaitPolicy& wp = WaitPolicy()) {
  using C = TcCfg<BN, EPI_WG>;
  static std::atomic<bool> configured{false};  // once per translation unit (set-up is idempotent)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<Epi, BN, EPI_WG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  GemmTcShape sh;
  sh.rows = rows;
  sh.map = map;
  sh.N = N;
  sh.K = K;
  sh.g_first = g_first;
  sh.g_count = g_count;
  sh.m_tiles = (rows + TC_BM - 1) / TC_BM;
  sh.n_tiles = N / BN;
  sh.kb_split = map.passes() > 1 ? K / TC_BK : 0;
  sh.k_blocks = (K / TC_BK) * map.passes();
  sh.err = err;
  sh.wp = wp;
  const int tiles = g_count * sh.m_tiles * sh.n_tiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  gemm_tc_kernel<Epi, BN, EPI_WG><<<grid, C::THREADS, C::SMEM, stream>>>(tmA, tmB, sh, epi);
  return cudaGetLastError();
}

}  // namespace armt
