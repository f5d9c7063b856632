// GEMM epilogues of the grouped layer.
//
// Each functor turns accumulator values of one output row segment into the
// next activation, so the projections of a cell write what the following
// step consumes with no extra pass over HBM:
//   EpiStore     C = acc (fp32)                        plain grouped GEMM
//   EpiAssocRead x' = x + acc / den[row]               associative read + residual
//                (+ gain-weighted row and partial sums for RMSNorm 1)
//   EpiQkvRope   q|k|v = acc / rms with rotate-half RoPE on q and k
//   EpiResidual  out = res + acc (fp32), optional act-dtype copy
//                (+ gain-weighted row and partial sums for RMSNorm 2)
//   EpiSwiGLU    u = silu(gate / rms) * (up / rms), gate/up interleaved in blocks of 128
// A functor is called once per (row, group of GROUP columns) with a source
// that yields accumulator columns `c .. c+n-1` relative to the group start.
// `valid` is false for padding rows past the end of the cell; the functor
// must still read its source (TMEM loads are warp-collective) but stores
// nothing.
#pragma once

#include "common.cuh"

namespace armt {

constexpr int GU_BLK = 128;  // gate/up interleave block (rows of W_gate then W_up)

// ---------------------------------------------------------------- stores --

__device__ __forceinline__ void store_row(float* dst, const float* v, int n) {
  if (n == 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
  } else {
    for (int i = 0; i < n; ++i) dst[i] = v[i];
  }
}

__device__ __forceinline__ void store_row(bf16* dst, const float* v, int n) {
  if (n == 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 p;
      p.x = pack_bf16x2(v[i], v[i + 1]);
      p.y = pack_bf16x2(v[i + 2], v[i + 3]);
      p.z = pack_bf16x2(v[i + 4], v[i + 5]);
      p.w = pack_bf16x2(v[i + 6], v[i + 7]);
      *reinterpret_cast<uint4*>(dst + i) = p;
    }
  } else {
    for (int i = 0; i < n; ++i) dst[i] = f2bf(v[i]);
  }
}

__device__ __forceinline__ void store_row(f16* dst, const float* v, int n) {
  if (n == 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 p;
      p.x = pack_f16x2(v[i], v[i + 1]);
      p.y = pack_f16x2(v[i + 2], v[i + 3]);
      p.z = pack_f16x2(v[i + 4], v[i + 5]);
      p.w = pack_f16x2(v[i + 6], v[i + 7]);
      *reinterpret_cast<uint4*>(dst + i) = p;
    }
  } else {
    for (int i = 0; i < n; ++i) dst[i] = __float2half_rn(v[i]);
  }
}

__device__ __forceinline__ void load_row(const float* src, float* v, int n) {
  if (n == 32 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float4 t = *reinterpret_cast<const float4*>(src + i);
      v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
    }
  } else {
    for (int i = 0; i < n; ++i) v[i] = src[i];
  }
}

// RMSNorm folded across two GEMMs: the producing epilogue writes the
// gain-weighted row (x * gain, activation dtype) and one partial sum of x^2
// per (row, column tile); the consuming GEMM scales its accumulator row by
// 1 / sqrt(sum / d + eps) -- the norm is linear in that factor, so
//   RMSNorm(x) W^T = (x * gain) W^T / rms(x).
// Partials are summed in a fixed order (deterministic).
struct RowNormIn {
  const float* ssq;  // [L][rows][npart] partial sums of squares, or nullptr
  int npart;
  float inv_d, eps;
  __device__ __forceinline__ float scale(int l, int rows, int row) const {
    if (ssq == nullptr) return 1.f;
    const float* p = ssq + ((long long)l * rows + row) * npart;
    float s = 0.f;
    if ((npart & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
      for (int i = 0; i < npart; i += 4) {  // fixed order: ((p0 + p1) + p2) + p3 ...
        const float4 q = *reinterpret_cast<const float4*>(p + i);
        s += q.x;
        s += q.y;
        s += q.z;
        s += q.w;
      }
    } else {
      for (int i = 0; i < npart; ++i) s += p[i];
    }
    return 1.0f / sqrtf(s * inv_d + eps);
  }
};

template <typename AT>
struct RowNormOut {
  const float* gain;  // [L][d] stacked gains, or nullptr (no norm output)
  AT* out;            // [groups][rows][d] gain-weighted row
  float* ssq;         // [groups][rows][npart]
  int gdiv = 1;       // group g uses the gains of layer g / gdiv
  long long lo_off = 0;  // split precision: bf16 low part at out + lo_off (staged path only)
  // v: 32 fp32 values of row `row` at columns col..col+31 (col0 = start of
  // this call's columns; the call's partial index is col0 / ncols).
  __device__ __forceinline__ void put(int l, int rows, int d, int row, int col, const float* v,
                                      float& acc) const {
    float w[32];
    const float* g = gain + (long long)(l / gdiv) * d + col;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      w[i] = v[i] * g[i];
      acc += v[i] * v[i];
    }
    store_row(out + ((long long)l * rows + row) * d + col, w, 32);
  }
  __device__ __forceinline__ void finish(int l, int rows, int row, int col0, int ncols, int d,
                                         float acc) const {
    ssq[((long long)l * rows + row) * (d / ncols) + col0 / ncols] = acc;
  }
};

// ------------------------------------------------------------- functors --

struct EpiStore {
  static constexpr int GROUP = 16;  // narrow outputs (e.g. a 16-wide key projection) too
  float* C;
  long long ld;        // row stride (elements)
  long long g_stride;  // stride between layers/groups (elements)
  template <class Src>
  __device__ __forceinline__ void operator()(int g, int row, bool valid, int col0, int ncols,
                                             Src& src) const {
    float* dst = C + g * g_stride + (long long)row * ld + col0;
    int c = 0;
    for (; c + 32 <= ncols; c += 32) {
      float v[32];
      src.template load<32>(c, v);
      if (valid) store_row(dst + c, v, 32);
    }
    for (; c < ncols; c += 16) {
      float v[16];
      src.template load<16>(c, v);
      if (valid)
        for (int i = 0; i < 16; ++i) dst[c + i] = v[i];
    }
  }
};

// x' = x + acc / den[row]: the associative read (numerator from the grouped
// GEMM of phi rows with the state) added to the residual stream; also the
// first half of RMSNorm 1 (gain-weighted row + partial sums of squares).
template <typename AT>
struct EpiAssocRead {
  static constexpr int GROUP = 32;
  const float* x;      // [slots][rows][d] layer input (slot = layer)
  const float* den;    // [L][rows]  z^T phi + eps
  float* out;          // [L][rows][d]
  int rows, d;
  RowNormOut<AT> norm;
  template <class Src>
  __device__ __forceinline__ void operator()(int l, int row, bool valid, int col0, int ncols,
                                             Src& src) const {
    const long long off = ((long long)l * rows + row) * d + col0;
    const float dn = valid ? den[(long long)l * rows + row] : 1.f;
    float ss = 0.f;
    for (int c = 0; c < ncols; c += 32) {
      float a[32], xv[32];
      src.template load<32>(c, a);
      if (valid) {
        load_row(x + off + c, xv, 32);
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = xv[i] + a[i] / dn;
        store_row(out + off + c, a, 32);
        norm.put(l, rows, d, row, col0 + c, a, ss);
      }
    }
    if (valid) norm.finish(l, rows, row, col0, ncols, d, ss);
  }
};

// Fused Q|K|V projection output with rotate-half RoPE on the q and k heads.
// Accumulator columns [0, Hq*hd) are q, then Hkv*hd of k, then Hkv*hd of v.
// q and k go to `out` (row stride `ld`); v goes to `out` too when vt is null
// (fp32 path), else transposed into vt[l][g][c][t] (row stride t_pad) so the
// tensor-core attention reads it K-major.  cos/sin tables are [rows][hd/2]
// (the position of each row within its cell).  With nb sequences per layer
// the rows of a layer are nb cells of cell_rows rows; cell b of layer l
// keeps its values at vt[l * nb + b].
template <typename OutT>
struct EpiQkvRope {
  // 64-column groups: whole heads for hd <= 64; for hd = 128 a group holds
  // half a head, and the group holding the first half rotates both halves
  // (the pairs are (i, i + hd/2)) while the other one does nothing
  static constexpr int GROUP = 64;
  OutT* out;
  const float* cosT;
  const float* sinT;
  int rows, hd, n_rope_cols, ld;    // n_rope_cols = (Hq+Hkv)*hd
  OutT* vt;                         // nullptr: v stays in `out`
  int n_kv, t_pad;
  RowNormIn norm;                   // RMSNorm 1 row scale
  int cell_rows = 0, nb = 1;        // rows per cell, cells per layer (rows = nb * cell_rows)

  template <int CH, class Src>
  __device__ __forceinline__ void rope_chunk(int l, int row, bool valid, int hcol, int h0, int i0,
                                             long long rbase, float rs, Src& src) const {
    const int half = hd >> 1;
    float x1[CH], x2[CH];
    src.template load<CH>(h0 + i0, x1);
    src.template load<CH>(h0 + half + i0, x2);
    if (!valid) return;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      x1[i] *= rs;
      x2[i] *= rs;
    }
    const bool rope = hcol < n_rope_cols;
    if (rope) {
      const float* cr = cosT + (long long)row * half + i0;
      const float* sr = sinT + (long long)row * half + i0;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const float c = cr[i], s = sr[i];
        const float a = x1[i], b = x2[i];
        x1[i] = a * c - b * s;
        x2[i] = b * c + a * s;
      }
    } else if (vt != nullptr) {
      const int g = (hcol - n_rope_cols) / hd;
      const int b = nb > 1 ? row / cell_rows : 0;
      OutT* col0 = vt + ((long long)((l * nb + b) * n_kv + g) * hd) * t_pad + (row - b * cell_rows);
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        st_from_f32(col0 + (long long)(i0 + i) * t_pad, x1[i]);
        st_from_f32(col0 + (long long)(half + i0 + i) * t_pad, x2[i]);
      }
      return;
    }
    store_row(out + rbase + hcol + i0, x1, CH);
    store_row(out + rbase + hcol + half + i0, x2, CH);
  }

  template <class Src>
  __device__ __forceinline__ void operator()(int l, int row, bool valid, int col0, int ncols,
                                             Src& src) const {
    const long long rbase = ((long long)l * rows + row) * ld;
    const int half = hd >> 1;
    const float rs = valid ? norm.scale(l, rows, row) : 1.f;
    if (hd > ncols && col0 % hd != 0) return;  // second half of a head: its first half's group writes it
    for (int h0 = 0; h0 < ncols; h0 += hd) {
      const int hcol = col0 + h0;
      if (half >= 32) {
        for (int i0 = 0; i0 < half; i0 += 32)
          rope_chunk<32>(l, row, valid, hcol, h0, i0, rbase, rs, src);
      } else {
        rope_chunk<16>(l, row, valid, hcol, h0, 0, rbase, rs, src);
      }
    }
  }
};

// out = res + acc (fp32 residual stream), plus an optional copy in the
// activation dtype (the next layer's associative-query GEMM operand) and an
// optional first half of RMSNorm 2 (norm.gain != nullptr).
template <typename CopyT>
struct EpiResidual {
  static constexpr int GROUP = 32;
  const float* res;    // [L][rows][n]
  float* out;          // [slots][rows][n] at slot l + out_slot_offset
  CopyT* copy;         // same indexing as out, or nullptr
  int rows, n, out_slot_offset;
  RowNormOut<CopyT> norm;
  template <class Src>
  __device__ __forceinline__ void operator()(int l, int row, bool valid, int col0, int ncols,
                                             Src& src) const {
    const long long ri = ((long long)l * rows + row) * n + col0;
    const long long oi = ((long long)(l + out_slot_offset) * rows + row) * n + col0;
    float ss = 0.f;
    for (int c = 0; c < ncols; c += 32) {
      float a[32], r[32];
      src.template load<32>(c, a);
      if (valid) {
        load_row(res + ri + c, r, 32);
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] += r[i];
        store_row(out + oi + c, a, 32);
        if (copy != nullptr) store_row(copy + oi + c, a, 32);
        if (norm.gain != nullptr) norm.put(l, rows, n, row, col0 + c, a, ss);
      }
    }
    if (valid && norm.gain != nullptr) norm.finish(l, rows, row, col0, ncols, n, ss);
  }
};

// SwiGLU over interleaved gate/up columns: block b of 2*GU_BLK accumulator
// columns holds gate rows [b*GU_BLK, (b+1)*GU_BLK) then the same up rows.
template <typename OutT>
struct EpiSwiGLU {
  static constexpr int GROUP = 2 * GU_BLK;
  OutT* out;           // [L][rows][F]
  int rows, F;
  RowNormIn norm;      // RMSNorm 2 row scale
  template <class Src>
  __device__ __forceinline__ void operator()(int l, int row, bool valid, int col0, int ncols,
                                             Src& src) const {
    const float rs = valid ? norm.scale(l, rows, row) : 1.f;
    for (int b0 = 0; b0 < ncols; b0 += 2 * GU_BLK) {
      const int f0 = (col0 + b0) / 2;
      OutT* dst = out + ((long long)l * rows + row) * F + f0;
      for (int c = 0; c < GU_BLK; c += 32) {
        float g[32], u[32];
        src.template load<32>(b0 + c, g);
        src.template load<32>(b0 + GU_BLK + c, u);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i] * rs) * (u[i] * rs);
          store_row(dst + c, g, 32);
        }
      }
    }
  }
};

// Accumulator sources.
struct TmemSrc {
  uint32_t taddr;  // lane base of this warp | column of the tile start
  template <int N>
  __device__ __forceinline__ void load(int c, float* v) const;
};
template <>
__device__ __forceinline__ void TmemSrc::load<32>(int c, float* v) const {
  tmem_ld32(taddr + (uint32_t)c, v);
}
template <>
__device__ __forceinline__ void TmemSrc::load<16>(int c, float* v) const {
  tmem_ld16(taddr + (uint32_t)c, v);
}

struct PtrSrc {
  const float* p;  // row pointer at the group start
  template <int N>
  __device__ __forceinline__ void load(int c, float* v) const {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = p[c + i];
  }
};

}  // namespace armt
