// Row-wise, associative-memory, attention and fp32 GEMM kernels of one
// diagonal step.  Every kernel takes a contiguous layer range
// [g_first, g_first + gridDim.{y|z}) -- the cells of one anti-diagonal, or a
// single cell in the sequential schedule -- and computes each cell with the
// same per-element operation order either way.
//
// Method: summary page of "Diagonal Batching Unlocks Parallelism in Recurrent
// Memory Transformers for Long Contexts".  Section 二: each layer owns an
// associative memory (A_l, z_l) read by every token and updated by the delta
// rule from that layer's memory-token outputs; section 三: the norms use
// stacked per-layer gains and every other operation runs batched over the
// cells of a diagonal.
#pragma once

#include "common.cuh"
#include "epilogues.cuh"

namespace armt {

// ------------------------------------------------------- layer-0 input --

// X[0] = [E[tokens of the segment]; memory embeddings] (fp32 residual stream)
// plus the activation-dtype copy Xa[0] (used as a GEMM operand; nullptr or
// equal to X when not needed).  Cell b (blockIdx.y) of the launch takes its
// tokens from tokens + b * tok_stride and fills rows [b * T, (b + 1) * T):
// n_seg token rows, then the M memory rows, then zero rows up to T (a short
// last segment; the zero rows come after every real row, so under the causal
// mask no real row ever sees them).  xa_lo_off != 0 (split precision): the
// bf16 low part of Xa at Xa + xa_lo_off.
template <typename WT>
__device__ __forceinline__ void embed_gather_kernel_block(const uint3 bid, const int32_t* tokens, long long tok_stride,
                                    const WT* embed, const WT* mem,
                                    float* X, WT* Xa, int T, int n_seg,
                                    int M, int d, int vocab, long long xa_lo_off) {
  const int t = bid.x, b = bid.y;
  const WT* src = nullptr;
  if (t < n_seg) {
    int id = tokens[b * tok_stride + t];
    id = id < 0 ? 0 : (id >= vocab ? vocab - 1 : id);
    src = embed + (long long)id * d;
  } else if (t < n_seg + M) {
    src = mem + (long long)(t - n_seg) * d;
  }
  const long long row = (long long)b * T + t;
  float* xo = X + row * d;
  WT* xa = Xa + row * d;
  const bool copy = Xa != nullptr && (void*)Xa != (void*)X;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = src != nullptr ? ld_as_f32(src + i) : 0.f;
    xo[i] = v;
    if (copy) {
      st_from_f32(xa + i, v);
      if (xa_lo_off != 0) st_from_f32(xa + xa_lo_off + i, bf16_residual(v));
    }
  }
}

template <typename WT>
__global__ void embed_gather_kernel(const int32_t* __restrict__ tokens, long long tok_stride,
                                    const WT* __restrict__ embed, const WT* __restrict__ mem,
                                    float* __restrict__ X, WT* __restrict__ Xa, int T, int n_seg,
                                    int M, int d, int vocab, long long xa_lo_off = 0) {
  embed_gather_kernel_block<WT>(blockIdx, tokens, tok_stride, embed, mem, X, Xa, T, n_seg, M, d, vocab, xa_lo_off);
}

// ------------------------------------------------------------- RMSNorm --

// out[l][row] = x[l][row] / sqrt(mean(x^2) + eps) * gain[l]  for the rows
// [0, rows) of layers g_first + blockIdx.y.  One block per row.
template <typename OutT>
__device__ __forceinline__ void rmsnorm_kernel_block(const uint3 bid, const float* x, long long x_gs, const float* gain,
                               long long gain_gs, OutT* out, long long out_gs, int d,
                               float eps, int g_first) {
  __shared__ float red[32];
  const int l = g_first + bid.y;
  const float* xr = x + l * x_gs + (long long)bid.x * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) ss += xr[i] * xr[i];
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  const float* g = gain + l * gain_gs;
  OutT* o = out + l * out_gs + (long long)bid.x * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) st_from_f32(o + i, xr[i] * inv * g[i]);
}

template <typename OutT>
__global__ void rmsnorm_kernel(const float* __restrict__ x, long long x_gs, const float* __restrict__ gain,
                               long long gain_gs, OutT* __restrict__ out, long long out_gs, int d,
                               float eps, int g_first) {
  rmsnorm_kernel_block<OutT>(blockIdx, x, x_gs, gain, gain_gs, out, out_gs, d, eps, g_first);
}

// ----------------------------------------------- associative read side --

// From q = Wq_a x (fp32 [rows][k] per layer): phi = DPFP_nu(q) (act dtype,
// [rows][P]) and den = z^T phi + eps.  One block per (row, layer).  A layer's
// rows are nb cells of cell_rows rows; cell b of layer l reads the
// normaliser z[l * nb + b].
template <typename PhiT>
__device__ __forceinline__ void assoc_phi_kernel_block(const uint3 bid, const float* q, const float* z,
                                 PhiT* phi, float* den, int rows, int k,
                                 int nu, float eps, int g_first, int cell_rows, int nb) {
  extern __shared__ float r[];  // 2k
  __shared__ float red[32];
  const int l = g_first + bid.y, row = bid.x;
  const int k2 = 2 * k, P = k2 * nu;
  const float* qr = q + ((long long)l * rows + row) * k;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const float v = qr[i];
    r[i] = v > 0.f ? v : 0.f;
    r[i + k] = v < 0.f ? -v : 0.f;
  }
  __syncthreads();
  const float* zl = z + ((long long)l * nb + row / cell_rows) * P;
  PhiT* pr = phi + ((long long)l * rows + row) * P;
  float acc = 0.f;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int j = p / k2 + 1, i = p - (j - 1) * k2;
    int src = i - j;
    src = src < 0 ? src + k2 : src;
    const float f = r[i] * r[src];
    st_from_f32(pr + p, f);
    acc += zl[p] * f;
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) den[(long long)l * rows + row] = acc + eps;
}

template <typename PhiT>
__global__ void assoc_phi_kernel(const float* __restrict__ q, const float* __restrict__ z,
                                 PhiT* __restrict__ phi, float* __restrict__ den, int rows, int k,
                                 int nu, float eps, int g_first, int cell_rows, int nb) {
  assoc_phi_kernel_block<PhiT>(blockIdx, q, z, phi, den, rows, k, nu, eps, g_first, cell_rows, nb);
}

// ---------------------------------------------- associative write side --

// Per layer (one block), memory tokens i = 0..M-1 in order:
//   phi_i = DPFP(k_i),  zphi_i = z_{i-1}^T phi_i,
//   gamma_i = clip(1 - zphi_i / (phi_i^T phi_i + eps), 0, 1),  z_i = z_{i-1} + gamma_i phi_i.
// The normaliser's recurrence does not involve A.  Expanding z_{i-1} gives
//   zphi_i = z_0^T phi_i + sum_{i' < i} gamma_i' (phi_i'^T phi_i),
// so the block computes every z_0^T phi_i and the Gram matrix G = Phi Phi^T
// in parallel, then one thread runs the 16-step scalar recurrence on shared
// memory, and finally z_M = z_0 + sum_i gamma_i phi_i.  Stores phiM[l][i][:]
// and coef[l][i] = {beta_i, 1 / (zphi_i + eps)} for the row update of A.
// vkb[l][i] = [v_i (d) | k_i (k) | beta logit | pad] (row stride nw), the
// output of the memory-row projection GEMM.  Index arithmetic uses no
// division: a warp takes one token, its lanes the feature columns.  M <= 32.
__device__ __forceinline__ void assoc_write_feat_kernel_block(const uint3 bid,
    const float* vkb, float* z, float* phiM,
    float* coef, int M, int k, int nu, float eps, int d, int nw, int g_first) {
  extern __shared__ float sm[];  // r: M * 2k, phi: M * (P + 1), z0: P
  __shared__ float G[32][33];
  __shared__ float z0phi[32], gam[32], logit[32];
  const int l = g_first + bid.x;
  const int k2 = 2 * k, P = k2 * nu, Pp = P + 1;
  float* r = sm;
  float* ph = sm + M * k2;
  float* zs = ph + M * Pp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  float* zl = z + (long long)l * P;
  for (int i = warp; i < M; i += nwarp) {
    const float* src = vkb + ((long long)l * M + i) * nw + d;
    for (int c = lane; c < k; c += 32) {
      const float v = src[c];
      r[i * k2 + c] = v > 0.f ? v : 0.f;
      r[i * k2 + c + k] = v < 0.f ? -v : 0.f;
    }
    if (lane == 0) logit[i] = src[k];
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x) zs[p] = zl[p];
  __syncthreads();
  for (int i = warp; i < M; i += nwarp) {
    const float* ri = r + i * k2;
    float* out = phiM + ((long long)l * M + i) * P;
    for (int j = 1; j <= nu; ++j)
      for (int c = lane; c < k2; c += 32) {
        const int src = c - j < 0 ? c - j + k2 : c - j;
        const float f = ri[c] * ri[src];
        ph[i * Pp + (j - 1) * k2 + c] = f;
        out[(j - 1) * k2 + c] = f;
      }
  }
  __syncthreads();
  // G[i][i2] (i <= i2) and z_0^T phi_i: one warp per dot product
  const int npairs = M * (M + 1) / 2;
  for (int t = warp; t < npairs + M; t += nwarp) {
    float acc = 0.f;
    if (t < npairs) {
      int i = 0, rem = t;
      while (rem >= M - i) {
        rem -= M - i;
        ++i;
      }
      const int i2 = i + rem;
      for (int p = lane; p < P; p += 32) acc += ph[i * Pp + p] * ph[i2 * Pp + p];
      acc = warp_sum(acc);
      if (lane == 0) {
        G[i][i2] = acc;
        G[i2][i] = acc;
      }
    } else {
      const int i = t - npairs;
      for (int p = lane; p < P; p += 32) acc += zs[p] * ph[i * Pp + p];
      acc = warp_sum(acc);
      if (lane == 0) z0phi[i] = acc;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < M; ++i) {
      float zp = z0phi[i];
      for (int i2 = 0; i2 < i; ++i2) zp += gam[i2] * G[i2][i];
      gam[i] = fminf(fmaxf(1.0f - zp / (G[i][i] + eps), 0.0f), 1.0f);  // keeps z >= 0
      z0phi[i] = zp;  // now z_{i-1}^T phi_i
    }
  }
  __syncthreads();
  if (threadIdx.x < M) {
    const int i = threadIdx.x;
    coef[((long long)l * M + i) * 2 + 0] = sigmoid_f(logit[i]);
    coef[((long long)l * M + i) * 2 + 1] = 1.0f / (z0phi[i] + eps);
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    float dz = 0.f;
    for (int i = 0; i < M; ++i) dz += gam[i] * ph[i * Pp + p];
    zl[p] = zs[p] + dz;
  }
}

__global__ void __launch_bounds__(256) assoc_write_feat_kernel(
    const float* __restrict__ vkb, float* __restrict__ z, float* __restrict__ phiM,
    float* __restrict__ coef, int M, int k, int nu, float eps, int d, int nw, int g_first) {
  assoc_write_feat_kernel_block(blockIdx, vkb, z, phiM, coef, M, k, nu, eps, d, nw, g_first);
}

// Delta-rule update of the rows of A_l, memory tokens applied in order.
// Row j of A only ever needs row j of the values, so each warp keeps rows of
// A in registers (lane owns entries lane + 32 t, t < NT = P / 32) and runs,
// for i = 0..M-1,
//   vbar = A[j] . phi_i * inv_den_i,     inv_den_i = 1 / (zphi_i + eps)
//   A[j] += beta_i (v_i[j] - vbar) phi_i,
// reading and writing each row of A once.  v_i[j] comes from the memory-row
// projection GEMM (vkb), phi_i and the coefficients from the feature kernel.
// Also refreshes the activation-dtype copy Aa of the state (the next read's
// GEMM operand) when Aa != A, and with aa_lo_off != 0 (split precision) its
// bf16 low part at Aa + aa_lo_off.  M <= 32.
// The rows [j0, j0 + rows_per_block) of A_l (one block's share), features ps
// [M][P] and coefficients cs [M][2] = {beta_i, 1 / (zphi_i + eps)} in shared
// memory.
template <typename AT, int NT>
__device__ __forceinline__ void assoc_write_rows(const float* ps, const float* cs, const float* vkb, int nw,
                                                 float* A, AT* Aa, int M, int d, int j0, int rows_per_block, int l,
                                                 long long aa_lo_off) {
  constexpr int P = 32 * NT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw_ = blockDim.x >> 5;
  float* Al = A + (long long)l * d * P;
  AT* Aal = Aa + (long long)l * d * P;
  const float* vl = vkb + (long long)l * M * nw;
  // Each warp runs RW rows side by side (independent dependency chains).
  constexpr int RW = 4;
  const int j_end = min(j0 + rows_per_block, d);
  for (int jb = j0 + warp * RW; jb < j_end; jb += nw_ * RW) {
    float vj[RW];
    float a[RW][NT];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int j = jb + r;
      const bool ok = j < j_end;
      vj[r] = (ok && lane < M) ? vl[(long long)lane * nw + j] : 0.f;  // lane i holds v_i[j]
#pragma unroll
      for (int t = 0; t < NT; ++t) a[r][t] = ok ? Al[(long long)j * P + lane + 32 * t] : 0.f;
    }
    for (int i = 0; i < M; ++i) {
      const float* pi = ps + i * P + lane;
      float phv[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) phv[t] = pi[32 * t];
      float dot[RW];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        dot[r] = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) dot[r] += a[r][t] * phv[t];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < RW; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
      const float beta = cs[2 * i], inv_den = cs[2 * i + 1];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const float vi = __shfl_sync(0xffffffffu, vj[r], i);
        const float c = beta * (vi - dot[r] * inv_den);
#pragma unroll
        for (int t = 0; t < NT; ++t) a[r][t] += c * phv[t];
      }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int j = jb + r;
      if (j < j_end) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          Al[(long long)j * P + lane + 32 * t] = a[r][t];
          if ((void*)Aal != (void*)Al) {
            st_from_f32(Aal + (long long)j * P + lane + 32 * t, a[r][t]);
            if (aa_lo_off != 0) st_from_f32(Aal + aa_lo_off + (long long)j * P + lane + 32 * t, bf16_residual(a[r][t]));
          }
        }
      }
    }
  }
}


template <typename AT, int NT>
__device__ __forceinline__ void assoc_write_update_kernel_block(const uint3 bid,
    const float* vkb, int nw, const float* phiM,
    const float* coef, float* A, AT* Aa, int M, int d,
    int rows_per_block, int g_first, long long aa_lo_off) {
  constexpr int P = 32 * NT;
  extern __shared__ float sm[];
  float* ps = sm;                 // [M][P]
  float* cs = ps + M * P;         // [M][2]
  const int l = g_first + bid.y;
  // stage the features 16 bytes at a time, four loads in flight per thread
  // (M * P is a multiple of 96 floats; the rows of phiM start 16-byte aligned)
  {
    const float4* src = reinterpret_cast<const float4*>(phiM + (long long)l * M * P);
    float4* dst = reinterpret_cast<float4*>(ps);
    const int n4 = M * P / 4;
#pragma unroll 4
    for (int t = threadIdx.x; t < n4; t += blockDim.x) dst[t] = src[t];
  }
  for (int t = threadIdx.x; t < 2 * M; t += blockDim.x) cs[t] = coef[(long long)l * M * 2 + t];
  __syncthreads();
  assoc_write_rows<AT, NT>(ps, cs, vkb, nw, A, Aa, M, d, bid.x * rows_per_block, rows_per_block, l, aa_lo_off);
}

template <typename AT, int NT>
__global__ void __launch_bounds__(128) assoc_write_update_kernel(
    const float* __restrict__ vkb, int nw, const float* __restrict__ phiM,
    const float* __restrict__ coef, float* __restrict__ A, AT* __restrict__ Aa, int M, int d,
    int rows_per_block, int g_first, long long aa_lo_off = 0) {
  assoc_write_update_kernel_block<AT, NT>(blockIdx, vkb, nw, phiM, coef, A, Aa, M, d, rows_per_block, g_first, aa_lo_off);
}

// State copy in the activation dtype: Aa = A (all layers); with lo_off != 0
// (split precision) also the bf16 low part at Aa + lo_off.
template <typename AT>
__global__ void convert_state_kernel(const float* __restrict__ A, AT* __restrict__ Aa, long long n,
                                     long long lo_off = 0) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    st_from_f32(Aa + i, A[i]);
    if (lo_off != 0) st_from_f32(Aa + lo_off + i, bf16_residual(A[i]));
  }
}

// ------------------------------------------------------ SIMT attention --

// Causal grouped-query attention inside one cell, fp32 arithmetic.
// qkv [L][rows][(Hq+2Hkv)*hd] (q and k already rotated), out [L][rows][Hq*hd].
// Block: 64 queries of one head of one layer; 4 threads per query, each
// owning hd/4 dimensions; keys processed in tiles of 64 with an online
// softmax.  Grid (ceil(rows/64), Hq, layers).
template <typename T, int HD>
__device__ __forceinline__ void attn_simt_kernel_block(const uint3 bid, const T* qkv, T* out,
                                                        int rows, int Hq, int Hkv, float scale,
                                                        int g_first) {
  constexpr int DPT = HD / 4;  // dims per thread
  extern __shared__ float kv[];  // K tile [64][HD], V tile [64][HD]
  float* Ks = kv;
  float* Vs = kv + 64 * HD;
  const int l = g_first + bid.z, h = bid.y, kvh = (h * Hkv) / Hq;
  const int qi = bid.x * 64 + (threadIdx.x >> 2), part = threadIdx.x & 3;
  const int ncols = (Hq + 2 * Hkv) * HD;
  const T* base = qkv + (long long)l * rows * ncols;
  float q[DPT], o[DPT];
  const bool qvalid = qi < rows;
#pragma unroll
  for (int e = 0; e < DPT; ++e) {
    q[e] = qvalid ? ld_as_f32(base + (long long)qi * ncols + h * HD + part * DPT + e) * scale : 0.f;
    o[e] = 0.f;
  }
  float m = -INFINITY, lsum = 0.f;
  const int q_last = min(bid.x * 64 + 63, rows - 1);
  for (int k0 = 0; k0 <= q_last; k0 += 64) {
    __syncthreads();
    for (int t = threadIdx.x; t < 64 * HD; t += blockDim.x) {
      const int kr = k0 + t / HD, c = t % HD;
      float kvv = 0.f, vvv = 0.f;
      if (kr < rows) {
        kvv = ld_as_f32(base + (long long)kr * ncols + (Hq + kvh) * HD + c);
        vvv = ld_as_f32(base + (long long)kr * ncols + (Hq + Hkv + kvh) * HD + c);
      }
      Ks[t] = kvv;
      Vs[t] = vvv;
    }
    __syncthreads();
    float s[64];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < DPT; ++e) a += q[e] * Ks[j * HD + part * DPT + e];
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      a += __shfl_xor_sync(0xffffffffu, a, 2);
      const bool ok = (k0 + j) <= qi && (k0 + j) < rows;
      s[j] = ok ? a : -INFINITY;
      tmax = fmaxf(tmax, s[j]);
    }
    const float mnew = fmaxf(m, tmax);
    if (mnew == -INFINITY) continue;  // nothing visible yet (padding query rows)
    const float corr = expf(m - mnew);
    lsum *= corr;
#pragma unroll
    for (int e = 0; e < DPT; ++e) o[e] *= corr;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const float p = expf(s[j] - mnew);
      lsum += p;
#pragma unroll
      for (int e = 0; e < DPT; ++e) o[e] += p * Vs[j * HD + part * DPT + e];
    }
    m = mnew;
  }
  if (qvalid) {
    T* orow = out + ((long long)l * rows + qi) * (Hq * HD) + h * HD + part * DPT;
    const float inv = 1.0f / lsum;
#pragma unroll
    for (int e = 0; e < DPT; ++e) st_from_f32(orow + e, o[e] * inv);
  }
}

template <typename T, int HD>
__global__ void __launch_bounds__(256) attn_simt_kernel(const T* __restrict__ qkv, T* __restrict__ out,
                                                        int rows, int Hq, int Hkv, float scale,
                                                        int g_first) {
  attn_simt_kernel_block<T, HD>(blockIdx, qkv, out, rows, Hq, Hkv, scale, g_first);
}

// --------------------------------------------------- fp32 SIMT GEMM ----

// C[l] = A[l] * B[l / b_div]^T, fp32, for l = g_first + blockIdx.z.  A
// [rows][K] (row stride lda) starting at row a_row0(l) of slot l + a_slot_off,
// B [N][K], C [rows][N] (row stride ldc).  64 x 64 tiles, 16-wide K steps,
// 4 x 4 outputs per thread, fixed K order.
struct SimtAMap {
  int row0, a_slot_off, b_div, alt_lo, alt_hi, alt_row0;
};
__device__ __forceinline__ void gemm_simt_f32_kernel_block(const uint3 bid, const float* A, long long a_gs,
                                                            int lda, const float* B,
                                                            long long b_gs, float* C,
                                                            long long c_gs, int ldc, int rows, int N,
                                                            int K, int g_first, SimtAMap am) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int l = g_first + bid.z;
  const int r0 = (l >= am.alt_lo && l < am.alt_hi) ? am.alt_row0 : am.row0;
  const float* Al = A + (l + am.a_slot_off) * a_gs + (long long)r0 * lda;
  const float* Bl = B + (l / am.b_div) * b_gs;
  float* Cl = C + l * c_gs;
  const int m0 = bid.y * 64, n0 = bid.x * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int t = threadIdx.x; t < 64 * 16; t += 256) {
      const int r = t / 16, c = t % 16;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + c;
      As[c][r] = (gm < rows && gk < K) ? Al[(long long)gm * lda + gk] : 0.f;
      Bs[c][r] = (gn < N && gk < K) ? Bl[(long long)gn * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += a[i] * b[j];
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + ty * 4 + i, gn = n0 + tx * 4 + j;
      if (gm < rows && gn < N) Cl[(long long)gm * ldc + gn] = acc[i][j];
    }
}

__global__ void __launch_bounds__(256) gemm_simt_f32_kernel(const float* __restrict__ A, long long a_gs,
                                                            int lda, const float* __restrict__ B,
                                                            long long b_gs, float* __restrict__ C,
                                                            long long c_gs, int ldc, int rows, int N,
                                                            int K, int g_first, SimtAMap am) {
  gemm_simt_f32_kernel_block(blockIdx, A, a_gs, lda, B, b_gs, C, c_gs, ldc, rows, N, K, g_first, am);
}

// Applies an epilogue functor to raw fp32 GEMM output rows (the fp32 path's
// counterpart of the tensor-core epilogue warps).  Grid (rows, layers).
template <class Epi>
__device__ __forceinline__ void epi_rows_kernel_block(const uint3 bid, const float* C, long long c_gs, int ldc, int N,
                                int g_first, Epi epi) {
  const int l = g_first + bid.y, row = bid.x;
  const float* cr = C + l * c_gs + (long long)row * ldc;
  // N must be a multiple of Epi::GROUP (checked when the model is created)
  for (int grp = threadIdx.x; grp < N / Epi::GROUP; grp += blockDim.x) {
    PtrSrc src{cr + grp * Epi::GROUP};
    epi(l, row, true, grp * Epi::GROUP, Epi::GROUP, src);
  }
}

template <class Epi>
__global__ void epi_rows_kernel(const float* __restrict__ C, long long c_gs, int ldc, int N,
                                int g_first, Epi epi) {
  epi_rows_kernel_block<Epi>(blockIdx, C, c_gs, ldc, N, g_first, epi);
}

}  // namespace armt
