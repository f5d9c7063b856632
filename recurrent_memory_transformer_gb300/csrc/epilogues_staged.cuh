// Staged GEMM epilogues for the tensor-core path.
//
// The accumulator tile lives in TMEM with one row per lane (tcgen05.ld gives
// a thread one row).  Reading and writing global memory that way makes every
// warp instruction touch 32 different rows.  Here each epilogue warp instead
// moves its 32 rows x 64 columns through a swizzled shared-memory stage and
// then walks the rows with the lanes across columns in 16-byte pieces, so a
// warp's global accesses are contiguous runs of whole rows.  Per-row scalars
// (a denominator, an RMSNorm scale) are loaded by the lane that owns the row
// and broadcast with shuffles; per-row sums are reduced over the lanes that
// share a row.
//
// A staged functor defines:
//   ROWSUM                 process() accumulates a per-row sum,
//   unit(u, a, b)          the two 32-column groups (tile offsets) of unit u;
//                          a tile of BN columns has BN/64 units,
//   row_ctx(l, row, ok)    per-row scalar, computed by the row's lane,
//   process(...)           the epilogue of one unit, reading the stage,
//   finish(l, row, col0, ncols, sum)  consumes the row sum of one tile,
//   direct_tile(col0)      true for tiles handled thread-per-row instead
//                          (direct(...) then gets a TMEM source).
// The arithmetic matches the thread-per-row functors in epilogues.cuh, which
// the fp32 path uses.
#pragma once

#include "common.cuh"
#include "epilogues.cuh"

namespace armt {

// Stage: this warp's 32 rows x 64 accumulator columns (columns 0..31 = the
// unit's group a, 32..63 = group b), fp32, 16-byte chunks swizzled by
// (row & 7) so that both the row-per-thread writes and the chunk-per-lane
// reads are free of bank conflicts.
__device__ __forceinline__ float4 stage_ld4(const float* stage, int row, int chunk) {
  return reinterpret_cast<const float4*>(stage)[row * 16 + (chunk ^ (row & 7))];
}
__device__ __forceinline__ void stage_st4(float* stage, int row, int chunk, float a, float b,
                                          float c, float d) {
  reinterpret_cast<float4*>(stage)[row * 16 + (chunk ^ (row & 7))] = make_float4(a, b, c, d);
}

__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(bf16* p, float4 v) {
  uint2 u;
  u.x = pack_bf16x2(v.x, v.y);
  u.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void st4(f16* p, float4 v) {
  uint2 u;
  u.x = pack_f16x2(v.x, v.y);
  u.y = pack_f16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
// bf16 rounding residuals of four values (the low part of a split operand)
__device__ __forceinline__ float4 residual4(float4 v) {
  return make_float4(bf16_residual(v.x), bf16_residual(v.y), bf16_residual(v.z), bf16_residual(v.w));
}

// Sum over the 16 lanes of each half-warp (lanes sharing a row).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Elementwise functors: lane -> (row 2*it + lane/16, 4 columns at 4*(lane%16)
// of the unit's 64), i.e. every half-warp touches one contiguous 256-byte
// run of a row.  Two callbacks per 4-column piece:
//   pre(row, col) -> float4   global input the piece needs (e.g. the residual),
//   op(row, col, v, pre, ctx) -> float   the work; returns its row-sum part.
// The inputs of all 16 rows a lane handles are loaded before any of their
// outputs are stored, so a warp keeps 16 loads in flight even though the
// compiler must assume inputs and outputs alias (the epilogue waits on
// these loads: more in flight hides more of their latency).  Shuffles run on
// all lanes; the work is predicated on the row being valid.
template <class Pre, class Op>
__device__ __forceinline__ void staged_rows_elementwise(const float* stage, int row0, int rows,
                                                        int colA, int colB, float ctx, Pre&& pre,
                                                        Op&& op, float* rowsum) {
  const int lane = threadIdx.x & 31;
  const int q = lane & 15, half = lane >> 4;
  const int col = (q < 8 ? colA + 4 * q : colB + 4 * (q - 8));
  constexpr int PREF = 8;  // rows whose inputs are in flight together
#pragma unroll 1
  for (int it0 = 0; it0 < 16; it0 += PREF) {
    float4 in[PREF];
#pragma unroll
    for (int k = 0; k < PREF; ++k) {
      const int row = row0 + 2 * (it0 + k) + half;
      in[k] = row < rows ? pre(row, col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < PREF; ++k) {
      const int r = 2 * (it0 + k) + half;
      const float4 v = stage_ld4(stage, r, q);
      const float c = __shfl_sync(0xffffffffu, ctx, r);
      const int row = row0 + r;
      float part = 0.f;
      if (row < rows) part = op(row, col, v, in[k], c);
      if (rowsum != nullptr) {
        part = half_warp_sum(part);
        if (q == 0) rowsum[r] += part;  // shared: one float per row of this warp
      }
    }
  }
}

// Paired functors: lane -> (row 4*it + lane/8, pairs 4*(lane%8)..+3), reading
// chunk q of group a and chunk q of group b.  `op(row, i, float4 a, float4 b, ctx)`.
template <class Op>
__device__ __forceinline__ void staged_rows_paired(const float* stage, int row0, int rows, float ctx,
                                                   Op&& op) {
  const int lane = threadIdx.x & 31;
  const int q = lane & 7, sub = lane >> 3;
#pragma unroll 4
  for (int it = 0; it < 8; ++it) {
    const int r = 4 * it + sub;
    const float4 a = stage_ld4(stage, r, q);
    const float4 b = stage_ld4(stage, r, q + 8);
    const float c = __shfl_sync(0xffffffffu, ctx, r);
    const int row = row0 + r;
    if (row < rows) op(row, 4 * q, a, b, c);
  }
}

struct SEpiStore {
  static constexpr bool ROWSUM = false;
  float* C;
  long long ld, g_stride;
  __device__ static void unit(int u, int& a, int& b) { a = 64 * u; b = 64 * u + 32; }
  __device__ bool direct_tile(int) const { return false; }
  template <class Src> __device__ void direct(int, int, bool, int, int, Src&) const {}
  __device__ float row_ctx(int, int, bool) const { return 0.f; }
  __device__ __forceinline__ void process(int l, int row0, int rows, int colA, int colB,
                                          const float* stage, float, float*) const {
    staged_rows_elementwise(stage, row0, rows, colA, colB, 0.f,
                            [&](int, int) { return make_float4(0.f, 0.f, 0.f, 0.f); },
                            [&](int row, int col, float4 v, float4, float) {
                              st4(C + l * g_stride + (long long)row * ld + col, v);
                              return 0.f;
                            },
                            nullptr);
  }
  __device__ void finish(int, int, int, int, float) const {}
};

// Gain-weighted row for RMSNorm (activation dtype) at 4 columns; g = the
// gains of those columns (the same for every row, loaded once per unit).
template <typename AT>
__device__ __forceinline__ float norm_put4(const RowNormOut<AT>& n, int l, int rows, int d, int row,
                                           int col, float4 v, float4 g) {
  const long long i = ((long long)l * rows + row) * d + col;
  const float4 w = make_float4(v.x * g.x, v.y * g.y, v.z * g.z, v.w * g.w);
  st4(n.out + i, w);
  if (n.lo_off != 0) st4(n.out + i + n.lo_off, residual4(w));
  return v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
}

// The gains of the 4 columns a lane handles in staged_rows_elementwise.
__device__ __forceinline__ float4 lane_gain4(const float* gain, int l, int d, int colA, int colB) {
  const int q = threadIdx.x & 15;
  const int col = (q < 8 ? colA + 4 * q : colB + 4 * (q - 8));
  return ld4(gain + (long long)l * d + col);
}

template <typename AT>
struct SEpiAssocRead {
  static constexpr bool ROWSUM = true;
  const float* x;
  const float* den;
  float* out;
  int rows, d;
  RowNormOut<AT> norm;
  __device__ static void unit(int u, int& a, int& b) { a = 64 * u; b = 64 * u + 32; }
  __device__ bool direct_tile(int) const { return false; }
  template <class Src> __device__ void direct(int, int, bool, int, int, Src&) const {}
  __device__ float row_ctx(int l, int row, bool ok) const {  // 1 / den, once per row
    return ok ? 1.0f / den[(long long)l * rows + row] : 1.f;
  }
  __device__ __forceinline__ void process(int l, int row0, int rows_, int colA, int colB,
                                          const float* stage, float ctx, float* rowsum) const {
    const float4 g = lane_gain4(norm.gain, l / norm.gdiv, d, colA, colB);
    staged_rows_elementwise(stage, row0, rows_, colA, colB, ctx,
                            [&](int row, int col) { return ld4(x + ((long long)l * rows + row) * d + col); },
                            [&](int row, int col, float4 v, float4 xv, float inv) {
                              const long long off = ((long long)l * rows + row) * d + col;
                              const float4 y = make_float4(xv.x + v.x * inv, xv.y + v.y * inv,
                                                           xv.z + v.z * inv, xv.w + v.w * inv);
                              st4(out + off, y);
                              return norm_put4(norm, l, rows, d, row, col, y, g);
                            },
                            rowsum);
  }
  __device__ void finish(int l, int row, int col0, int ncols, float s) const {
    norm.ssq[((long long)l * rows + row) * (d / ncols) + col0 / ncols] = s;
  }
};

template <typename CopyT>
struct SEpiResidual {
  static constexpr bool ROWSUM = true;
  const float* res;
  float* out;
  CopyT* copy;
  int rows, n, out_slot_offset;
  RowNormOut<CopyT> norm;
  long long copy_lo_off = 0;  // split precision: low part of the copy at copy + copy_lo_off
  __device__ static void unit(int u, int& a, int& b) { a = 64 * u; b = 64 * u + 32; }
  __device__ bool direct_tile(int) const { return false; }
  template <class Src> __device__ void direct(int, int, bool, int, int, Src&) const {}
  __device__ float row_ctx(int, int, bool) const { return 0.f; }
  __device__ __forceinline__ void process(int l, int row0, int rows_, int colA, int colB,
                                          const float* stage, float, float* rowsum) const {
    const float4 g = norm.gain != nullptr ? lane_gain4(norm.gain, l / norm.gdiv, n, colA, colB)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    staged_rows_elementwise(stage, row0, rows_, colA, colB, 0.f,
                            [&](int row, int col) { return ld4(res + ((long long)l * rows + row) * n + col); },
                            [&](int row, int col, float4 v, float4 r, float) {
                              const long long oi =
                                  ((long long)(l + out_slot_offset) * rows + row) * n + col;
                              const float4 y = make_float4(r.x + v.x, r.y + v.y, r.z + v.z, r.w + v.w);
                              st4(out + oi, y);
                              if (copy != nullptr) {
                                st4(copy + oi, y);
                                if (copy_lo_off != 0) st4(copy + oi + copy_lo_off, residual4(y));
                              }
                              if (norm.gain == nullptr) return 0.f;
                              return norm_put4(norm, l, rows, n, row, col, y, g);
                            },
                            norm.gain != nullptr ? rowsum : nullptr);
  }
  __device__ void finish(int l, int row, int col0, int ncols, float s) const {
    if (norm.gain != nullptr) norm.ssq[((long long)l * rows + row) * (n / ncols) + col0 / ncols] = s;
  }
};

// Q|K with RoPE; V tiles go thread-per-row to the transposed store of the
// row functor.
template <typename OutT>
struct SEpiQkvRope {
  static constexpr bool ROWSUM = false;
  OutT* out;
  const float* cosT;
  const float* sinT;
  int rows, hd, n_rope_cols, ld;
  OutT* vt;
  int n_kv, t_pad;
  RowNormIn norm;
  int cell_rows = 0, nb = 1;
  // unit u: 32 rotation pairs (i0 + i, i0 + i + hd/2) of one head
  __device__ void unit_hd(int u, int& a, int& b) const {
    const int half = hd >> 1, per_head = half / 32;
    const int h = u / per_head, i0 = (u - h * per_head) * 32;
    a = h * hd + i0;
    b = a + half;
  }
  __device__ static void unit(int, int&, int&) {}
  __device__ bool direct_tile(int col0) const { return col0 >= n_rope_cols; }
  template <class Src>
  __device__ void direct(int l, int row, bool valid, int col0, int ncols, Src& src) const {
    EpiQkvRope<OutT> e{out, cosT, sinT, rows, hd, n_rope_cols, ld, vt, n_kv, t_pad, norm,
                       cell_rows, nb};
    e(l, row, valid, col0, ncols, src);
  }
  __device__ float row_ctx(int l, int row, bool ok) const {
    return ok ? norm.scale(l, rows, row) : 1.f;
  }
  __device__ __forceinline__ void process(int l, int row0, int rows_, int colA, int colB,
                                          const float* stage, float ctx, float*) const {
    const int half = hd >> 1;
    const int i0 = colA % hd;
    staged_rows_paired(stage, row0, rows_, ctx, [&](int row, int i, float4 a, float4 b, float rs) {
      const float4 c = ld4(cosT + (long long)row * half + i0 + i);
      const float4 s = ld4(sinT + (long long)row * half + i0 + i);
      a = make_float4(a.x * rs, a.y * rs, a.z * rs, a.w * rs);
      b = make_float4(b.x * rs, b.y * rs, b.z * rs, b.w * rs);
      OutT* o = out + ((long long)l * rows + row) * ld;
      st4(o + colA + i, make_float4(a.x * c.x - b.x * s.x, a.y * c.y - b.y * s.y,
                                    a.z * c.z - b.z * s.z, a.w * c.w - b.w * s.w));
      st4(o + colB + i, make_float4(b.x * c.x + a.x * s.x, b.y * c.y + a.y * s.y,
                                    b.z * c.z + a.z * s.z, b.w * c.w + a.w * s.w));
    });
  }
  __device__ void finish(int, int, int, int, float) const {}
};

template <typename OutT>
struct SEpiSwiGLU {
  static constexpr bool ROWSUM = false;
  OutT* out;
  int rows, F;
  RowNormIn norm;
  long long lo_off = 0;  // split precision: low part at out + lo_off
  // unit u: gate columns 32u..32u+31 and their up columns 128 later
  __device__ static void unit(int u, int& a, int& b) { a = 32 * u; b = 32 * u + GU_BLK; }
  __device__ bool direct_tile(int) const { return false; }
  template <class Src> __device__ void direct(int, int, bool, int, int, Src&) const {}
  __device__ float row_ctx(int l, int row, bool ok) const {
    return ok ? norm.scale(l, rows, row) : 1.f;
  }
  __device__ __forceinline__ void process(int l, int row0, int rows_, int colA, int,
                                          const float* stage, float ctx, float*) const {
    const int f0 = (colA / (2 * GU_BLK)) * GU_BLK + (colA % (2 * GU_BLK));
    staged_rows_paired(stage, row0, rows_, ctx, [&](int row, int i, float4 g, float4 u, float rs) {
      const long long o = ((long long)l * rows + row) * F + f0 + i;
      const float4 y = make_float4(silu_f(g.x * rs) * (u.x * rs), silu_f(g.y * rs) * (u.y * rs),
                                   silu_f(g.z * rs) * (u.z * rs), silu_f(g.w * rs) * (u.w * rs));
      st4(out + o, y);
      if (lo_off != 0) st4(out + o + lo_off, residual4(y));
    });
  }
  __device__ void finish(int, int, int, int, float) const {}
};

// DPFP features and the read denominator straight from the associative
// query GEMM, whose 64-wide tile holds the whole query q = Wq_a x of a row
// (key_dim 64, nu 3, P = 384; the tensor-core path supports only that):
//   r = [relu(q), relu(-q)],  phi_{128 (j-1) + c} = r_c r_{(c-j) mod 128}, j = 1..3,
//   den = z^T phi + eps with z of the row's (layer, sequence) group,
// phi stored in the activation dtype, den in fp32 (from the unrounded phi).
// Per row, lane L holds q_{2L}, q_{2L+1} and computes the pairs p, p + 1 with
// p = 64 t + 2 L, t < 6 (c = 2 L + 64 (t mod 2), j = t / 2 + 1), storing each
// as one bf16 pair.  The rolled factors r_{c-j}, r_{c+1-j} are q values of
// lanes L-1 and L-2 (three shuffles per row); where c - j falls below the
// start of its half (L = 0, or L <= 1 for j = 3) it wraps into the other half
// of r, i.e. the sign of the relu flips.  z is reloaded only when the rows
// pass into another sequence's cell.
template <typename AT>
struct SEpiPhi {
  static_assert(sizeof(AT) == 2, "bf16 features");
  static constexpr bool ROWSUM = false;
  AT* phi;         // [groups][rows][384]
  float* den;      // [groups][rows]
  const float* z;  // [L * nb][384]
  int rows, cell_rows, nb;
  float eps;
  long long lo_off = 0;  // split precision: bf16 low part of phi at phi + lo_off
  __device__ static void unit(int u, int& a, int& b) { a = 64 * u; b = 64 * u + 32; }
  __device__ bool direct_tile(int) const { return false; }
  template <class Src> __device__ void direct(int, int, bool, int, int, Src&) const {}
  __device__ float row_ctx(int, int, bool) const { return 0.f; }
  // relu(x) in the first half of r, relu(-x) in the second
  __device__ __forceinline__ static float rv(float x, bool neg) { return neg ? fmaxf(-x, 0.f) : fmaxf(x, 0.f); }
  __device__ __forceinline__ void process(int l, int row0, int rows_, int, int, const float* stage,
                                          float, float*) const {
    const int lane = threadIdx.x & 31;
    const bool w1 = lane == 0, w3 = lane <= 1;  // the lanes whose rolled factors wrap
    int cell = -1, next_cell_row = 0;
    float2 zz[6];
#pragma unroll 1
    for (int r = 0; r < 32; ++r) {
      const int row = row0 + r;
      if (row >= rows_) break;  // warp-uniform
      if (row >= next_cell_row) {
        const int cb = row / cell_rows;
        next_cell_row = (cb + 1) * cell_rows;
        if (cb != cell) {
          cell = cb;
          const float* zr = z + ((long long)l * nb + cb) * 384 + 2 * lane;
#pragma unroll
          for (int t = 0; t < 6; ++t) zz[t] = *reinterpret_cast<const float2*>(zr + 64 * t);
        }
      }
      // q_{2L}, q_{2L+1} of stage row r (16-byte chunks swizzled by r & 7)
      const float2 q = *reinterpret_cast<const float2*>(stage + r * 64 + ((((2 * lane) >> 2) ^ (r & 7)) << 2) +
                                                        ((2 * lane) & 3));
      const float a0 = __shfl_sync(0xffffffffu, q.x, (lane - 1) & 31);  // q_{2L-2}
      const float a1 = __shfl_sync(0xffffffffu, q.y, (lane - 1) & 31);  // q_{2L-1}
      const float b1 = __shfl_sync(0xffffffffu, q.y, (lane - 2) & 31);  // q_{2L-3}
      uint32_t* out = reinterpret_cast<uint32_t*>(phi + ((long long)l * rows + row) * 384) + lane;
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < 6; ++t) {
        const int j = t / 2 + 1;
        const bool h = (t & 1) != 0;  // c in the second half of r
        const float rc0 = rv(q.x, h), rc1 = rv(q.y, h);
        float f0, f1;
        if (j == 1) {
          f0 = rc0 * rv(a1, h != w1);
          f1 = rc1 * rc0;
        } else if (j == 2) {
          f0 = rc0 * rv(a0, h != w1);
          f1 = rc1 * rv(a1, h != w1);
        } else {
          f0 = rc0 * rv(b1, h != w3);
          f1 = rc1 * rv(a0, h != w1);
        }
        out[32 * t] = pack_bf16x2(f0, f1);
        if (lo_off != 0) out[lo_off / 2 + 32 * t] = pack_bf16x2(bf16_residual(f0), bf16_residual(f1));
        acc = fmaf(zz[t].x, f0, acc);
        acc = fmaf(zz[t].y, f1, acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) den[(long long)l * rows + row] = acc + eps;
    }
  }
  __device__ void finish(int, int, int, int, float) const {}
};

// Unit enumeration: functors with a runtime layout (RoPE heads) provide
// unit_hd(); the rest a static unit().
template <class E>
__device__ __forceinline__ void epi_unit(const E& e, int u, int& a, int& b) {
  E::unit(u, a, b);
}
template <typename T>
__device__ __forceinline__ void epi_unit(const SEpiQkvRope<T>& e, int u, int& a, int& b) {
  e.unit_hd(u, a, b);
}

// One tile's epilogue for the 32 rows of this warp.  `stage` is this warp's
// private area: 32 x 64 fp32 (the stage) followed by 32 floats (row sums);
// tbase = TMEM address of the warp's lane quarter at the tile's first column.
// All 32 lanes call this.
constexpr int STAGED_FLOATS_PER_WARP = 32 * 64 + 32;

// With EPI_WG warpgroups, warp part p handles units [p*U/EPI_WG, (p+1)*U/EPI_WG)
// of the tile's U = BN/64 units, and its row sums cover BN/EPI_WG columns.
template <int BN, int EPI_WG, class Epi>
__device__ __forceinline__ void staged_epilogue(const Epi& epi, int l, int row0, int rows,
                                                int tile_col0, int part, uint32_t tbase,
                                                float* stage) {
  const int lane = threadIdx.x & 31;
  constexpr int U = BN / 64, UP = U / EPI_WG, NCOLS = BN / EPI_WG;
  if (epi.direct_tile(tile_col0)) {
    // thread-per-row tiles: the first warpgroup does the whole tile
    if (part == 0) {
      TmemSrc src{tbase};
      const int row = row0 + lane;
      epi.direct(l, row, row < rows, tile_col0, BN, src);
    }
    return;
  }
  const float ctx = epi.row_ctx(l, row0 + lane, row0 + lane < rows);
  float* rowsum = stage + 32 * 64;
  if (Epi::ROWSUM) rowsum[lane] = 0.f;
#pragma unroll 1
  for (int u = part * UP; u < (part + 1) * UP; ++u) {
    int ca, cb;
    epi_unit(epi, u, ca, cb);
    {
      float va[32];
      tmem_ld32(tbase + (uint32_t)ca, va);
#pragma unroll
      for (int c = 0; c < 8; ++c) stage_st4(stage, lane, c, va[4 * c], va[4 * c + 1], va[4 * c + 2], va[4 * c + 3]);
    }
    {
      float vb[32];
      tmem_ld32(tbase + (uint32_t)cb, vb);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        stage_st4(stage, lane, 8 + c, vb[4 * c], vb[4 * c + 1], vb[4 * c + 2], vb[4 * c + 3]);
    }
    __syncwarp();
    epi.process(l, row0, rows, tile_col0 + ca, tile_col0 + cb, stage, ctx, rowsum);
    __syncwarp();
  }
  if (Epi::ROWSUM) {
    const int row = row0 + lane;
    if (row < rows) epi.finish(l, row, tile_col0 + part * NCOLS, NCOLS, rowsum[lane]);
    __syncwarp();
  }
}

}  // namespace armt
