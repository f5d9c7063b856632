// Segment-local causal grouped-query attention on tcgen05 tensor cores.
//
// The attention of every cell of a diagonal runs as one batched launch
// (summary page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
// Transformers for Long Contexts", section 三: attention is left as it is and
// run with the layers of a diagonal as the batch).  Inside a cell, rows
// 0..T-1 (segment tokens, then memory tokens) attend causally to rows <= their
// own; query head h reads kv head h / (Hq / Hkv).
//
// One CTA = (query head, layer, 128-row query tile m); it walks key tiles
// j = 0..m (causal block skipping):
//   warp 0      TMA: Q tile once; K_j and V_j tiles (single-buffered each),
//   warp 1      MMA issue: S_j = Q K_j^T (M=128, N=128) into TMEM buffer j%2,
//               O_j = P_j V_j (M=128, N=hd) into the first hd columns of the
//               same buffer once the softmax has read S_j,
//   warps 2..5  softmax, one thread per query row (= TMEM lane): a max pass
//               over S_j, then O_{j-1} folded into registers with the
//               running-max correction (which frees its buffer for S_{j+1}),
//               then an exp2 pass writing P_j as bf16 into shared memory in
//               the 128-byte-swizzled K-major layout the MMA reads.
// With two S buffers the MMA computes S_{j+1} while the softmax works on
// S_j; 256 TMEM columns per CTA keep two CTAs resident per SM.
// V comes pre-transposed (Vt[l][g][hd][T], written by the QKV epilogue) so
// that every MMA operand is K-major.  fp32 accumulation and softmax.
#pragma once

#include "common.cuh"

namespace armt {

template <int HD>
struct AttnCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int HD_ATOMS = HD / 64;
  static constexpr uint32_t Q_BYTES = BM * HD * 2;  // HD_ATOMS x [128 rows x 128 B]
  static constexpr uint32_t K_BYTES = BN * HD * 2;  // HD_ATOMS x [128 keys x 128 B]
  static constexpr uint32_t V_BYTES = HD * BN * 2;  // 2 x [HD rows x 128 B] (keys 0-63, 64-127)
  static constexpr uint32_t P_BYTES = BM * BN * 2;  // 2 x [128 rows x 128 B]
  static constexpr uint32_t TMEM_COLS = 256;        // two 128-column S/O buffers
  static constexpr size_t SMEM = 1024 + Q_BYTES + K_BYTES + V_BYTES + P_BYTES + 256;
  static constexpr int MIN_BLOCKS = HD == 64 ? 2 : 1;
};

struct AttnArgs {
  bf16* out;        // [L][T][Hq*HD]
  int T, Hq, Hkv;
  int g_first;
  int n_qtiles;
  float scale_log2;  // log2(e) / sqrt(HD)
  int* err;
};

// S_FULL/O_FULL/BUF_FREE come in pairs, one per TMEM buffer.
enum AttnBar {
  B_Q = 0, B_KF, B_KE, B_VF, B_VE, B_PF,
  B_SF0, B_SF1, B_OF0, B_OF1, B_FREE0, B_FREE1, B_COUNT
};

template <int HD>
__global__ void __launch_bounds__(192, AttnCfg<HD>::MIN_BLOCKS)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmV,
                   const AttnArgs a) {
  using C = AttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = base;
  uint8_t* sK = sQ + C::Q_BYTES;
  uint8_t* sV = sK + C::K_BYTES;
  uint8_t* sP = sV + C::V_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sP + C::P_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + B_COUNT);

  const int h = blockIdx.x;
  const int l = a.g_first + blockIdx.y;
  const int m = a.n_qtiles - 1 - (int)blockIdx.z;  // heavy tiles first
  const int g = h / (a.Hq / a.Hkv);
  const int nj = m + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    mbar_init(&bar[B_Q], 1);
    mbar_init(&bar[B_KF], 1);
    mbar_init(&bar[B_KE], 1);
    mbar_init(&bar[B_VF], 1);
    mbar_init(&bar[B_VE], 1);
    mbar_init(&bar[B_PF], 4);
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(&bar[B_SF0 + bb], 1);
      mbar_init(&bar[B_OF0 + bb], 1);
      mbar_init(&bar[B_FREE0 + bb], 4);
    }
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // buffer b at columns 128 b .. 128 b + 127

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[B_Q], C::Q_BYTES);
      for (int at = 0; at < C::HD_ATOMS; ++at)
        tma_load_3d(sQ + at * 16384, &tmQK, h * HD + 64 * at, m * 128, l, &bar[B_Q]);
      for (int j = 0; j < nj; ++j) {
        if (j > 0 && !mbar_wait_bounded(&bar[B_KE], (j - 1) & 1, a.err, DEV_TIMEOUT_EMPTY)) break;
        mbar_arrive_expect_tx(&bar[B_KF], C::K_BYTES);
        for (int at = 0; at < C::HD_ATOMS; ++at)
          tma_load_3d(sK + at * 16384, &tmQK, (a.Hq + g) * HD + 64 * at, j * 128, l, &bar[B_KF]);
        if (j > 0 && !mbar_wait_bounded(&bar[B_VE], (j - 1) & 1, a.err, DEV_TIMEOUT_EMPTY)) break;
        mbar_arrive_expect_tx(&bar[B_VF], C::V_BYTES);
        for (int at = 0; at < 2; ++at)
          tma_load_3d(sV + at * (HD * 128), &tmV, j * 128 + 64 * at, 0, l * a.Hkv + g, &bar[B_VF]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128);
      constexpr uint32_t idO = idesc_bf16_f32(128, HD);
      // S_j = Q K_j^T into buffer j % 2 (K_j must have arrived)
      auto issue_S = [&](int j) -> bool {
        if (!mbar_wait_bounded(&bar[B_KF], j & 1, a.err, DEV_TIMEOUT_FULL)) return false;
        tc_fence_after();
        const uint32_t d = tmem + 128u * (uint32_t)(j & 1);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const int at = ks >> 2, w = ks & 3;
          tc_mma_bf16(d, smem_desc_sw128(smem_u32(sQ + at * 16384)) + 2 * w,
                      smem_desc_sw128(smem_u32(sK + at * 16384)) + 2 * w, idS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bar[B_SF0 + (j & 1)]);
        tc_commit(&bar[B_KE]);
        return true;
      };
      bool ok = mbar_wait_bounded(&bar[B_Q], 0, a.err, DEV_TIMEOUT_FULL) && issue_S(0) &&
                (nj < 2 || issue_S(1));
      for (int j = 0; ok && j < nj; ++j) {
        // P_j written (the softmax has read S_j) and V_j loaded
        ok = mbar_wait_bounded(&bar[B_PF], j & 1, a.err, DEV_TIMEOUT_ACC_FULL) &&
             mbar_wait_bounded(&bar[B_VF], j & 1, a.err, DEV_TIMEOUT_FULL);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + 128u * (uint32_t)(j & 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int at = ks >> 2, w = ks & 3;
          tc_mma_bf16(d, smem_desc_sw128(smem_u32(sP + at * 16384)) + 2 * w,
                      smem_desc_sw128(smem_u32(sV + at * (HD * 128))) + 2 * w, idO,
                      ks > 0 ? 1u : 0u);
        }
        tc_commit(&bar[B_OF0 + (j & 1)]);
        tc_commit(&bar[B_VE]);
        if (j + 2 < nj) {
          // buffer j % 2 is reused once the softmax has taken O_j out of it
          ok = mbar_wait_bounded(&bar[B_FREE0 + (j & 1)], (j >> 1) & 1, a.err, DEV_TIMEOUT_ACC_EMPTY) &&
               issue_S(j + 2);
        }
      }
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;            // row within the tile = TMEM lane
    const int qi = m * 128 + r;                   // query index within the cell
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float o[HD];
#pragma unroll
    for (int i = 0; i < HD; ++i) o[i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f, corr_prev = 1.f;
    uint8_t* prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
    bool ok = true;
    // o = o * corr + O_t (O_t = P_t V_t, in buffer t % 2), then free the buffer
    auto fold = [&](int t, float corr) -> bool {
      const bool got = mbar_wait_bounded(&bar[B_OF0 + (t & 1)], (t >> 1) & 1, a.err, DEV_TIMEOUT_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after();
      const uint32_t tO = tmem + 128u * (uint32_t)(t & 1) + lane_off;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float ov[32];
        tmem_ld32(tO + 32 * c, ov);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[32 * c + i] = o[32 * c + i] * corr + ov[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_FREE0 + (t & 1)]);
      return true;
    };
    for (int j = 0; j < nj; ++j) {
      const bool got = mbar_wait_bounded(&bar[B_SF0 + (j & 1)], (j >> 1) & 1, a.err, DEV_TIMEOUT_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + 128u * (uint32_t)(j & 1) + lane_off;
      // Only the diagonal tile j == m is masked (key index > query index);
      // keys of earlier tiles are all visible.  lim = last visible key
      // column of this row within the tile.
      const bool diag = (j == m);
      const int lim = qi - j * 128;
      // pass 1: row max of the raw scores (the scale is positive)
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float sv[32];
        tmem_ld32(tS + 32 * c, sv);
        if (diag) {
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = (32 * c + i <= lim) ? fmaxf(mx, sv[i]) : mx;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, sv[i]);
        }
      }
      const float m_new = fmaxf(m_run, mx * a.scale_log2);
      const float corr = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // O_{j-1} (relative to the previous max) joins the running output; its
      // P.V has finished, so P may be overwritten below
      if (j > 0 && !fold(j - 1, corr_prev)) {
        ok = false;
        break;
      }
      // pass 2: p = 2^(s * scale - m), row sum, bf16 P into shared memory
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float sv[32];
        tmem_ld32(tS + 32 * c, sv);
        if (diag) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            sv[i] = (32 * c + i <= lim) ? fast_exp2(fmaf(sv[i], a.scale_log2, -m_use)) : 0.f;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[i] = fast_exp2(fmaf(sv[i], a.scale_log2, -m_use));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) rs += sv[i];
        uint8_t* atom = prow + (c >> 1) * 16384;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int chunk = 4 * (c & 1) + v;  // 16-byte chunk within the 128-byte row
          uint4 pk;
          pk.x = pack_bf16x2(sv[8 * v + 0], sv[8 * v + 1]);
          pk.y = pack_bf16x2(sv[8 * v + 2], sv[8 * v + 3]);
          pk.z = pack_bf16x2(sv[8 * v + 4], sv[8 * v + 5]);
          pk.w = pack_bf16x2(sv[8 * v + 6], sv[8 * v + 7]);
          *reinterpret_cast<uint4*>(atom + ((chunk ^ (r & 7)) << 4)) = pk;
        }
      }
      l_run = l_run * corr + rs;
      m_run = m_new;
      corr_prev = corr;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_PF]);
    }
    if (ok) ok = fold(nj - 1, corr_prev);
    if (ok && qi < a.T) {
      const float inv = 1.0f / l_run;
      bf16* dst = a.out + ((long long)l * a.T + qi) * (a.Hq * HD) + h * HD;
#pragma unroll
      for (int c = 0; c < HD; c += 8) {
        uint4 pk;
        pk.x = pack_bf16x2(o[c + 0] * inv, o[c + 1] * inv);
        pk.y = pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
        pk.z = pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
        pk.w = pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
        *reinterpret_cast<uint4*>(dst + c) = pk;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int HD>
cudaError_t launch_attn_tc(const CUtensorMap& tmQK, const CUtensorMap& tmV, const AttnArgs& a,
                           int g_count, cudaStream_t stream) {
  using C = AttnCfg<HD>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(a.Hq, g_count, a.n_qtiles);
  attn_tc_kernel<HD><<<grid, 192, C::SMEM, stream>>>(tmQK, tmV, a);
  return cudaGetLastError();
}

}  // namespace armt
