// Segment-local causal grouped-query attention on tcgen05 tensor cores.
//
// The attention of every cell of a diagonal runs as one batched launch
// (summary page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
// Transformers for Long Contexts", section 三: attention is left as it is and
// run with the layers of a diagonal as the batch).  Inside a cell, rows
// 0..T-1 (segment tokens, then memory tokens) attend causally to rows <= their
// own; query head h reads kv head h / (Hq / Hkv).
//
// Persistent CTAs (two per SM) take work items (query head, layer, 128-row
// query tile m) round-robin, heaviest tiles first; per item a CTA walks key
// tiles j = 0..m (causal block skipping):
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
// S_j; 256 TMEM columns per CTA keep two CTAs resident per SM.  TMEM and the
// barriers are set up once per CTA; a running tile count c (across items)
// gives every barrier's phase: per-tile barriers complete once per tile,
// buffer c % 2 holds tile c, and its barriers complete once every 2 tiles.
// V comes pre-transposed (Vt[l][g][hd][T], written by the QKV epilogue) so
// that every MMA operand is K-major.  fp32 accumulation and softmax.  The
// operands (q, k, v and the probabilities P) are 16-bit of type OpT: bf16
// for the stand-alone entry points, fp16 inside the bf16 model, whose
// attention operands are activations (10 mantissa bits instead of 7 at the
// same tensor-core rate; q and k come from RMS-normalised rows, P lies in
// [0, 1]).  The output is bf16, the operand type of the output projection.
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
  int g_first, g_count;
  int n_qtiles;
  float scale_log2;  // log2(e) / sqrt(HD)
  int* err;
  WaitPolicy wp;     // wait limit and the test stall hook (counted in K/V tile loads)
  long long out_lo_off = 0;  // split precision: bf16 low part of the output at out + out_lo_off
};

// Work item i (heaviest query tiles first): m = n_qtiles - 1 - i / (Hq * G),
// then cell, then head.
struct AttnItem {
  int h, l, m;
};
__device__ __forceinline__ AttnItem attn_item(const AttnArgs& a, int i) {
  const int per_m = a.Hq * a.g_count;
  const int mi = i / per_m, rem = i - mi * per_m;
  AttnItem it;
  it.m = a.n_qtiles - 1 - mi;
  it.l = a.g_first + rem / a.Hq;
  it.h = rem % a.Hq;
  return it;
}

// S_FULL/O_FULL/BUF_FREE come in pairs, one per TMEM buffer.
enum AttnBar {
  B_Q = 0, B_KF, B_KE, B_VF, B_VE, B_PF,
  B_SF0, B_SF1, B_OF0, B_OF1, B_FREE0, B_FREE1, B_DRAIN, B_COUNT
};

template <int HD, typename OpT>
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

  const int n_items = a.Hq * a.g_count * a.n_qtiles;
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
    mbar_init(&bar[B_DRAIN], 1);
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
      int c = 0;  // running tile count
      bool ok = true;
      // phases armed on the Q, K and V barriers; each is re-armed only after
      // its previous phase was consumed, so at most the last one is in flight
      int nq = 0, nk = 0, nv = 0;
      const uint64_t lim = a.wp.limit_ns;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const AttnItem it = attn_item(a, i);
        const int g = it.h / (a.Hq / a.Hkv);
        // Q is reused once every S of the previous item has run
        if (c > 0 && !mbar_wait_bounded(&bar[B_KE], (c - 1) & 1, a.err, DEV_TIMEOUT_EMPTY, lim)) break;
        mbar_arrive_expect_tx(&bar[B_Q], C::Q_BYTES);
        for (int at = 0; at < C::HD_ATOMS; ++at)
          tma_load_3d(sQ + at * 16384, &tmQK, it.h * HD + 64 * at, it.m * 128, it.l, &bar[B_Q]);
        ++nq;
        for (int j = 0; j <= it.m; ++j, ++c) {
          if (nk == a.wp.stall_after ||
              (j > 0 && !mbar_wait_bounded(&bar[B_KE], (c - 1) & 1, a.err, DEV_TIMEOUT_EMPTY, lim))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar[B_KF], C::K_BYTES);
          for (int at = 0; at < C::HD_ATOMS; ++at)
            tma_load_3d(sK + at * 16384, &tmQK, (a.Hq + g) * HD + 64 * at, j * 128, it.l, &bar[B_KF]);
          ++nk;
          if (c > 0 && !mbar_wait_bounded(&bar[B_VE], (c - 1) & 1, a.err, DEV_TIMEOUT_EMPTY, lim)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar[B_VF], C::V_BYTES);
          for (int at = 0; at < 2; ++at)
            tma_load_3d(sV + at * (HD * 128), &tmV, j * 128 + 64 * at, 0, it.l * a.Hkv + g, &bar[B_VF]);
          ++nv;
        }
      }
      // Drain: the last Q, K and V loads land before the CTA lets go of its
      // shared memory, also when a consumer stopped waiting for them.
      if (nq > 0) mbar_wait_drain(&bar[B_Q], (uint32_t)((nq - 1) & 1));
      if (nk > 0) mbar_wait_drain(&bar[B_KF], (uint32_t)((nk - 1) & 1));
      if (nv > 0) mbar_wait_drain(&bar[B_VF], (uint32_t)((nv - 1) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_16bit_f32<OpT>(128, 128);
      constexpr uint32_t idO = idesc_16bit_f32<OpT>(128, HD);
      // S for running tile cc = Q K^T into buffer cc % 2, once the buffer's
      // previous tile (cc - 2) has been folded by the softmax and K arrived
      auto issue_S = [&](int cc) -> bool {
        if (cc >= 2 && !mbar_wait_bounded(&bar[B_FREE0 + (cc & 1)], ((cc - 2) >> 1) & 1, a.err,
                                          DEV_TIMEOUT_ACC_EMPTY, a.wp.limit_ns))
          return false;
        if (!mbar_wait_bounded(&bar[B_KF], cc & 1, a.err, DEV_TIMEOUT_FULL, a.wp.limit_ns)) return false;
        tc_fence_after();
        const uint32_t d = tmem + 128u * (uint32_t)(cc & 1);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const int at = ks >> 2, w = ks & 3;
          tc_mma_bf16(d, smem_desc_sw128(smem_u32(sQ + at * 16384)) + 2 * w,
                      smem_desc_sw128(smem_u32(sK + at * 16384)) + 2 * w, idS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bar[B_SF0 + (cc & 1)]);
        tc_commit(&bar[B_KE]);
        return true;
      };
      int c = 0, k = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, ++k) {
        const AttnItem it = attn_item(a, i);
        const int nj = it.m + 1;
        ok = mbar_wait_bounded(&bar[B_Q], k & 1, a.err, DEV_TIMEOUT_FULL, a.wp.limit_ns) && issue_S(c) &&
             (nj < 2 || issue_S(c + 1));
        for (int j = 0; ok && j < nj; ++j) {
          const int cj = c + j;
          // P written (the softmax has read S) and V arrived
          ok = mbar_wait_bounded(&bar[B_PF], cj & 1, a.err, DEV_TIMEOUT_ACC_FULL, a.wp.limit_ns) &&
               mbar_wait_bounded(&bar[B_VF], cj & 1, a.err, DEV_TIMEOUT_FULL, a.wp.limit_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + 128u * (uint32_t)(cj & 1);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int at = ks >> 2, w = ks & 3;
            tc_mma_bf16(d, smem_desc_sw128(smem_u32(sP + at * 16384)) + 2 * w,
                        smem_desc_sw128(smem_u32(sV + at * (HD * 128))) + 2 * w, idO,
                        ks > 0 ? 1u : 0u);
          }
          tc_commit(&bar[B_OF0 + (cj & 1)]);
          tc_commit(&bar[B_VE]);
          if (j + 2 < nj) ok = issue_S(cj + 2);
        }
        c += nj;
      }
      // Drain: every MMA issued above has finished before TMEM is freed.
      tc_commit(&bar[B_DRAIN]);
      mbar_wait_drain(&bar[B_DRAIN], 0);
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;            // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t* prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
    float o[HD];
    // A warp whose 32 rows all lie at or past T (the short last query tile)
    // keeps the barrier protocol -- the same waits and arrivals in the same
    // order, so no arrival can run ahead into another tile's phase -- but
    // reads no TMEM and writes no P.  Its rows of P and O are never stored.
    bool idle = false;
    // o = o * corr + O_t (O_t = P_t V_t, in buffer t % 2), then free the buffer
    auto fold = [&](int t, float corr) -> bool {
      const bool got = mbar_wait_bounded(&bar[B_OF0 + (t & 1)], (t >> 1) & 1, a.err, DEV_TIMEOUT_ACC_FULL,
                                         a.wp.limit_ns);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after();
      if (!idle) {
        const uint32_t tO = tmem + 128u * (uint32_t)(t & 1) + lane_off;
        const float2 c2 = make_float2(corr, corr);
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          float ov[32];
          tmem_ld32(tO + 32 * cc, ov);
          if constexpr (HD == 64) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 r2 = __ffma2_rn(make_float2(o[32 * cc + i], o[32 * cc + i + 1]), c2,
                                           make_float2(ov[i], ov[i + 1]));
              o[32 * cc + i] = r2.x;
              o[32 * cc + i + 1] = r2.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[32 * cc + i] = o[32 * cc + i] * corr + ov[i];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_FREE0 + (t & 1)]);
      return true;
    };
    int c = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const AttnItem it = attn_item(a, item);
      const int m = it.m, nj = m + 1;
      const int qi = m * 128 + r;                 // query index within the cell
      idle = m * 128 + quarter * 32 >= a.T;
#pragma unroll
      for (int i = 0; i < HD; ++i) o[i] = 0.f;
      float m_run = -INFINITY, l_run = 0.f, corr_prev = 1.f;
      for (int j = 0; j < nj; ++j) {
        const int cj = c + j;
        const bool got = mbar_wait_bounded(&bar[B_SF0 + (cj & 1)], (cj >> 1) & 1, a.err, DEV_TIMEOUT_ACC_FULL,
                                           a.wp.limit_ns);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + 128u * (uint32_t)(cj & 1) + lane_off;
        // Only the diagonal tile j == m is masked (key index > query index);
        // keys of earlier tiles are all visible.  lim = last visible key
        // column of this row within the tile.
        const bool diag = (j == m);
        const int lim = qi - j * 128;
        // pass 1: row max of the raw scores (the scale is positive); NMX
        // independent partial maxima keep the dependency chains short
        constexpr int NMX = HD == 64 ? 8 : 4;  // fewer where o[] already fills the registers
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4 && !idle; ++cc) {
          float sv[32];
          tmem_ld32(tS + 32 * cc, sv);
          if (diag) {
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[i] = (32 * cc + i <= lim) ? sv[i] : -INFINITY;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) mx8[i % NMX] = fmaxf(mx8[i % NMX], sv[i]);
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_new = fmaxf(m_run, mx * a.scale_log2);
        const float corr = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        // O of the previous tile (relative to the previous max) joins the
        // running output; its P.V has finished, so P may be overwritten below
        if (j > 0 && !fold(cj - 1, corr_prev)) {
          ok = false;
          break;
        }
        // pass 2: p = 2^(s * scale - m) (masked keys: 2^-inf = 0), row sum
        // in four independent pairs, 16-bit P into shared memory
        float2 rs4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rs4[i] = make_float2(0.f, 0.f);
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(-m_use, -m_use);
#pragma unroll
        for (int cc = 0; cc < 4 && !idle; ++cc) {
          float sv[32];
          tmem_ld32(tS + 32 * cc, sv);
          if (diag) {
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[i] = (32 * cc + i <= lim) ? sv[i] : -INFINITY;
          }
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x2 = __ffma2_rn(make_float2(sv[i], sv[i + 1]), sc2, nm2);
            sv[i] = fast_exp2(x2.x);
            sv[i + 1] = fast_exp2(x2.y);
            rs4[(i >> 1) % (NMX / 2)] = __fadd2_rn(rs4[(i >> 1) % (NMX / 2)], make_float2(sv[i], sv[i + 1]));
          }
          uint8_t* atom = prow + (cc >> 1) * 16384;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int chunk = 4 * (cc & 1) + v;  // 16-byte chunk within the 128-byte row
            uint4 pk;
            pk.x = pack2<OpT>(sv[8 * v + 0], sv[8 * v + 1]);
            pk.y = pack2<OpT>(sv[8 * v + 2], sv[8 * v + 3]);
            pk.z = pack2<OpT>(sv[8 * v + 4], sv[8 * v + 5]);
            pk.w = pack2<OpT>(sv[8 * v + 6], sv[8 * v + 7]);
            *reinterpret_cast<uint4*>(atom + ((chunk ^ (r & 7)) << 4)) = pk;
          }
        }
        const float rs = ((rs4[0].x + rs4[0].y) + (rs4[1].x + rs4[1].y)) +
                         ((rs4[2].x + rs4[2].y) + (rs4[3].x + rs4[3].y));
        l_run = l_run * corr + rs;
        m_run = m_new;
        corr_prev = corr;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_PF]);
      }
      if (ok) ok = fold(c + nj - 1, corr_prev);
      if (ok && qi < a.T) {
        const float inv = 1.0f / l_run;
        bf16* dst = a.out + ((long long)it.l * a.T + qi) * (a.Hq * HD) + it.h * HD;
#pragma unroll
        for (int cc = 0; cc < HD; cc += 8) {
          uint4 pk;
          pk.x = pack_bf16x2(o[cc + 0] * inv, o[cc + 1] * inv);
          pk.y = pack_bf16x2(o[cc + 2] * inv, o[cc + 3] * inv);
          pk.z = pack_bf16x2(o[cc + 4] * inv, o[cc + 5] * inv);
          pk.w = pack_bf16x2(o[cc + 6] * inv, o[cc + 7] * inv);
          *reinterpret_cast<uint4*>(dst + cc) = pk;
        }
        if (a.out_lo_off != 0) {
#pragma unroll
          for (int cc = 0; cc < HD; cc += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(bf16_residual(o[cc + 0] * inv), bf16_residual(o[cc + 1] * inv));
            pk.y = pack_bf16x2(bf16_residual(o[cc + 2] * inv), bf16_residual(o[cc + 3] * inv));
            pk.z = pack_bf16x2(bf16_residual(o[cc + 4] * inv), bf16_residual(o[cc + 5] * inv));
            pk.w = pack_bf16x2(bf16_residual(o[cc + 6] * inv), bf16_residual(o[cc + 7] * inv));
            *reinterpret_cast<uint4*>(dst + a.out_lo_off + cc) = pk;
          }
        }
      }
      c += nj;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Internal linkage: every translation unit that launches the kernel configures
// (shared-memory opt-in) and launches its own copy of it.
template <int HD, typename OpT = bf16>
static cudaError_t launch_attn_tc(const CUtensorMap& tmQK, const CUtensorMap& tmV, const AttnArgs& a,
                           int g_count, int num_sms, cudaStream_t stream) {
  using C = AttnCfg<HD>;
  static std::atomic<bool> configured{false};  // once per translation unit (set-up is idempotent)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, OpT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  AttnArgs aa = a;
  aa.g_count = g_count;
  const int n_items = a.Hq * g_count * a.n_qtiles;
  const int grid = n_items < C::MIN_BLOCKS * num_sms ? n_items : C::MIN_BLOCKS * num_sms;
  attn_tc_kernel<HD, OpT><<<grid, 192, C::SMEM, stream>>>(tmQK, tmV, aa);
  return cudaGetLastError();
}

}  // namespace armt
