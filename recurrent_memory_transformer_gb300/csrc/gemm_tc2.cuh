// Grouped bf16 GEMM on CTA pairs (tcgen05 cta_group::2): 256 x 256 tiles.
//
// The same grouped layer as gemm_tc.cuh (summary page of "Diagonal Batching
// Unlocks Parallelism in Recurrent Memory Transformers for Long Contexts",
// section 三: one grouped product per linear layer over the cells of a
// diagonal, out[g] = epilogue(A[g] B[g]^T)), for the wide projections.
//
// Why pairs: with one CTA a 128 x 256 x 16 MMA reads 12 KB of operands from
// shared memory and TMA writes the same 12 KB into it, about 192 bytes per
// clock against the tensor core's rate -- more than shared memory delivers,
// so a single-CTA tile cannot keep the tensor core busy.  A CTA pair runs one
// 256 x 256 tile: each CTA loads its 128 rows of A and 128 of the 256 B rows
// and each SM reads only its own halves, 128 bytes per clock in all.
//
// Cluster of 2 CTAs (rank 0 = leader), persistent over pair tiles
// (group-major, then N tile, then 256-row M tile):
//   warp 0      TMA producer in both CTAs: A rows [m0 + 128 r, +128) and B rows
//               [n0 + 128 r, +128) of each 64-wide K block into its own
//               shared memory; completion counted on the LEADER's full barrier
//               (which expects both CTAs' bytes).
//   warp 1      leader only: one thread issues the pair MMAs (4 per K block)
//               into TMEM accumulator (acc) of both CTAs, commits the stage's
//               empty barrier and, per tile, the accumulator-full barrier of
//               both CTAs (multicast).
//   warps 2..   epilogue in both CTAs, as in gemm_tc.cuh, on the CTA's 128
//               rows x 256 columns; each warp then arrives on the leader's
//               accumulator-empty barrier (remote arrive).
// Every wait is bounded; an error word stops both CTAs, which then drain:
// the leader's MMA thread waits for its last pair commit, and once both
// producers have stopped (cluster barrier) the leader waits until every
// stage load either CTA issued has landed -- a stage whose phase one CTA
// armed or loaded and the other did not is balanced first (see the end of the
// kernel) -- before both CTAs meet at a second cluster barrier and free TMEM.
// Same fixed K order per element as gemm_tc.cuh.
#pragma once

#include "common.cuh"
#include "epilogues.cuh"
#include "epilogues_staged.cuh"
#include "gemm_tc.cuh"
#include "schedule.h"  // pair_tiles_pay_off

namespace armt {

template <int EPI_WG>
struct Tc2Cfg {
  static constexpr int BN = 256;                     // N per pair tile (each CTA loads BN/2 B rows)
  static constexpr int STAGES = EPI_WG == 2 ? 4 : 6;
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;        // 16 KB
  static constexpr uint32_t B_BYTES = (BN / 2) * TC_BK * 2;     // 16 KB
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;    // per CTA
  static constexpr uint32_t TMEM_COLS = 2 * BN;                 // two accumulators
  static constexpr int EPI_WARPS = 4 * EPI_WG;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr uint32_t EPI_STAGE_BYTES = EPI_WARPS * STAGED_FLOATS_PER_WARP * 4;
  static constexpr size_t SMEM = 1024 + STAGES * STAGE_BYTES + 256 + EPI_STAGE_BYTES;
  static_assert(SMEM <= 232448, "shared memory");
};

template <class Epi, int EPI_WG>
__global__ void __launch_bounds__(Tc2Cfg<EPI_WG>::THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmTcShape sh, const Epi epi) {
  using C = Tc2Cfg<EPI_WG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;  // completion of every pair MMA (multicast to both CTAs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* issued_slot = tmem_slot + 1;  // this CTA's stage-load count, read by the leader

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);   // the leader's producer arrival (+ both CTAs' bytes)
      mbar_init(&empty[s], 1);  // the pair commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);                  // the pair commit
      mbar_init(&acc_empty[a], 2 * C::EPI_WARPS);  // every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    *issued_slot = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int m_pairs = (sh.rows + 2 * TC_BM - 1) / (2 * TC_BM);
  const int tiles_per_g = m_pairs * sh.n_tiles;
  const int num_tiles = sh.g_count * tiles_per_g;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;  // stage loads issued (and, in the leader, full[] phases armed)
      for (int t = cid; ok && t < num_tiles; t += ncl) {
        const int g = t / tiles_per_g, r = t - g * tiles_per_g;
        const int nt = r / m_pairs, mp = r - nt * m_pairs;
        const int layer = sh.g_first + g;
        const int a_row = sh.map.a_row0(layer) + mp * 2 * TC_BM + (int)rank * TC_BM;
        const int b_row = nt * C::BN + (int)rank * (C::BN / 2);
        const int b_slot = layer / sh.map.b_div + sh.map.b_slot_off;
        // split operands: pass p (K blocks kpp p .. kpp (p + 1) - 1) reads A part
        // p % a_parts and B part p / a_parts (0 = high, 1 = low); tracked
        // incrementally, so the unsplit loop does no division
        const int kpp = sh.kb_split > 0 ? sh.kb_split : sh.k_blocks, two_a = sh.map.a_parts() == 2;
        int kk = 0, pass = 0;
        for (int kb = 0; kb < sh.k_blocks; ++kb) {
          if (issued == sh.wp.stall_after ||
              !mbar_wait_bounded_cluster(&empty[stage], phase ^ 1u, sh.err, DEV_TIMEOUT_EMPTY, sh.wp.limit_ns)) {
            ok = false;
            break;
          }
          const int kc = kk * TC_BK;
          const int ap = two_a ? (pass & 1) : 0, bp = two_a ? (pass >> 1) : pass;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
          tma_load_3d_pair(sA + stage * C::A_BYTES, &tmA, kc, a_row,
                           layer + sh.map.a_slot_off + ap * sh.map.a_lo_slot, fb);
          tma_load_3d_pair(sB + stage * C::B_BYTES, &tmB, kc, b_row, b_slot + bp * sh.map.b_lo_slot, fb);
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
      *issued_slot = (uint32_t)issued;
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * TC_BM, C::BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = cid; ok && t < num_tiles; t += ncl) {
        if (!mbar_wait_bounded_cluster(&acc_empty[acc], acc_phase ^ 1u, sh.err, DEV_TIMEOUT_ACC_EMPTY,
                                       sh.wp.limit_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::BN);
        for (int kb = 0; kb < sh.k_blocks; ++kb) {
          if (!mbar_wait_bounded_cluster(&full[stage], phase, sh.err, DEV_TIMEOUT_FULL, sh.wp.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * C::A_BYTES));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k)
            tc_mma_bf16_pair(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                             (kb | k) != 0 ? 1u : 0u);
          tc_commit_pair(&empty[stage]);  // the stage is free in both CTAs once these finish
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(&acc_full[acc]);  // both CTAs' accumulators ready
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Drain: every pair MMA issued above has finished (its arrivals made in
      // both CTAs) before either CTA frees TMEM, also after an early stop.
      tc_commit_pair(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    const int quarter = warp & 3;
    const int ew = warp - 2;
    const int part = ew / 4;
    float* stage = reinterpret_cast<float*>(base + C::STAGES * C::STAGE_BYTES + 256) +
                   ew * STAGED_FLOATS_PER_WARP;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cid; t < num_tiles; t += ncl) {
      const int g = t / tiles_per_g, r = t - g * tiles_per_g;
      const int nt = r / m_pairs, mp = r - nt * m_pairs;
      const bool got =
          mbar_wait_bounded_cluster(&acc_full[acc], acc_phase, sh.err, DEV_TIMEOUT_ACC_FULL, sh.wp.limit_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int row0 = mp * 2 * TC_BM + (int)rank * TC_BM + quarter * 32;
      staged_epilogue<C::BN, EPI_WG>(epi, sh.g_first + g, row0, sh.rows, nt * C::BN, part,
                                     tmem_base + (uint32_t)(acc * C::BN) + ((uint32_t)(quarter * 32) << 16),
                                     stage);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&acc_empty[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both producers have stopped issuing; the pair MMAs have finished
  // Every stage load of both CTAs completes on the leader's full[] barriers,
  // so the leader drains them for the pair.  With a and b the two CTAs' load
  // counts, iterations below min(a, b) were armed and loaded by both and
  // complete; at most one iteration per stage lies in [min, max) (a CTA runs
  // at most STAGES loads ahead of the MMA's consumption, which needs both
  // halves), and its phase lacks one share: the peer's bytes (balanced with
  // complete_tx) or the leader's arming (balanced with arrive.expect_tx for
  // the peer's bytes already in flight).  Its earlier phase is waited for
  // first, so the balancing lands in the right phase.
  if (leader && warp == 0 && lane == 0) {
    const int a = (int)*issued_slot;
    const int b = (int)ld_shared_cluster_u32(mapa_shared(smem_u32(issued_slot), 1));
    const int lo = a < b ? a : b, hi = a < b ? b : a;
    for (int s = 0; s < C::STAGES && s < hi; ++s) {
      const int j = s + ((hi - 1 - s) / C::STAGES) * C::STAGES;  // last iteration of stage s
      if (j >= lo) {
        if (j >= C::STAGES) mbar_wait_drain(&full[s], (uint32_t)(((j - C::STAGES) / C::STAGES) & 1));
        if (j < a)
          mbar_complete_tx(&full[s], C::STAGE_BYTES);
        else
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
      }
      mbar_wait_drain(&full[s], (uint32_t)((j / C::STAGES) & 1));
    }
  }
  // the leader's final pair commit also arrives here
  if (!leader && warp == 1 && lane == 0) mbar_wait_drain(drain, 0);
  __syncthreads();
  cluster_sync_all();  // no copy, remote arrival or pair MMA is still aimed at either CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

// Launch with clusters of two; the grid is the number of co-resident pairs
// (queried once per kernel), at most the number of pair tiles.
template <class Epi, int EPI_WG = 1>
static cudaError_t launch_gemm_tc2(const CUtensorMap& tmA, const CUtensorMap& tmB, int rows, int N, int K,
                            int g_first, int g_count, int* err, const Epi& epi, int num_sms,
                            cudaStream_t stream, const GemmGroupMap& map = GemmGroupMap(),
                            const WaitPolicy& wp = WaitPolicy()) {
  using C = Tc2Cfg<EPI_WG>;
  static std::atomic<int> max_clusters{0};  // once per translation unit (the query is idempotent)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc2_kernel<Epi, EPI_WG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel<Epi, EPI_WG>, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_clusters = n;
  }
  GemmTcShape sh;
  sh.rows = rows;
  sh.map = map;
  sh.N = N;
  sh.K = K;
  sh.g_first = g_first;
  sh.g_count = g_count;
  sh.m_tiles = (rows + TC_BM - 1) / TC_BM;
  sh.n_tiles = N / C::BN;
  sh.kb_split = map.passes() > 1 ? K / TC_BK : 0;
  sh.k_blocks = (K / TC_BK) * map.passes();
  sh.err = err;
  sh.wp = wp;
  const int tiles = g_count * ((rows + 2 * TC_BM - 1) / (2 * TC_BM)) * sh.n_tiles;
  const int mc = max_clusters.load();
  const int clusters = tiles < mc ? tiles : mc;
  if (clusters <= 0) return cudaSuccess;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<Epi, EPI_WG>, tmA, tmB, sh, epi);
}

}  // namespace armt
