// Backward pass of the ARMT forward (fp32): the kernels.
//
// Method: summary page of "Diagonal Batching Unlocks Parallelism in Recurrent
// Memory Transformers for Long Contexts", section 四: diagonal batching is
// carried over to the backward pass, so that training and inference share
// one schedule.  The backward of the recurrence is the adjoint of the
// forward cell by cell: cell (l, s) hands the adjoint of its input rows to
// cell (l-1, s) and the adjoint of the state it started from to cell
// (l, s-1), so the reverse anti-diagonals i = L + n - 2 .. 0 are again sets
// of independent cells, one per layer, and every launch below runs all cells
// of one diagonal side by side (group z of a launch is cell (l0 + z, s0 - z)).
//
// The forward keeps each cell's input rows and the state it started from; a
// cell's intermediates are recomputed from those (one cell of activations
// per layer is live at a time).  All arithmetic is fp32; every reduction runs
// in a fixed order, so results are bitwise reproducible.
//
// The per-op adjoints follow the forward definitions term by term:
//   RMSNorm  y = x s g,  s = (mean x^2 + eps)^-1/2:
//            x_bar = s t - s^3 (t . x) x / d,  t = y_bar g;   g_bar = sum_rows y_bar x s
//   RoPE     a rotation per (i, i + hd/2) pair: its transpose
//   softmax attention (per head, causal): with P = softmax(q k^T / sqrt(hd)),
//            v_bar = P^T o_bar,  S_bar = P (o_bar v^T - rowsum(o_bar . o)),
//            q_bar = S_bar k / sqrt(hd),  k_bar = S_bar^T q / sqrt(hd)
//   SwiGLU   u = silu(a) b:  a_bar = u_bar b sig(a) (1 + a (1 - sig(a))),  b_bar = u_bar silu(a)
//   DPFP     phi_{(j-1) 2k + c} = r_c r_{(c - j) mod 2k},  r = [relu(x), relu(-x)]:
//            each product sends phi_bar times the other factor to both factors
//   read     y = x + A phi / D,  D = z^T phi + eps  (section 二's associative read)
//   write    the delta rule over the memory rows in order (section 二), below.
#pragma once

#include "common.cuh"
#include "epilogues.cuh"

namespace armt {

// Where a cell's tensor lives: p + l * sl + s * ss + off, and the cell of
// layer alt_l (the last segment's, when it is short) adds alt_add.
struct CellPtr {
  float* p = nullptr;
  long long sl = 0, ss = 0;
  int alt_l = -1;
  long long alt_add = 0;
  long long off = 0;  // added last (e.g. -1 slot: layer l's output goes to slot l - 1)
  __host__ __device__ __forceinline__ float* at(int l, long long s) const {
    return p + ((long long)l * sl + s * ss + (l == alt_l ? alt_add : 0) + off);
  }
};

// ------------------------------------------------------------- GEMM --

// Operand element (r, c) at m.at(l, s)[trans ? c * ld + r : r * ld + c].
struct BwMat {
  CellPtr m;
  long long ld = 0;
  int trans = 0;
};

// C = E + alpha * rs[r] * sum_k A(r, k) B(k, c) for every cell of a
// diagonal; E may be C itself (accumulate) or absent (E.m.p == nullptr);
// rs absent: 1; rs_div: the row factor divides instead.  ksplit > 1: the K
// range is cut into ksplit chunks of kchunk (a multiple of 16); each chunk's
// raw product goes to part[(kz * groups + cell)][M][N] and bw_gemm_reduce
// sums the chunks in order and applies the epilogue (deterministic).
struct BwGemm {
  BwMat A, B, C, E;
  CellPtr rs;
  int rs_div = 0;
  float alpha = 1.f;
  int M = 0, N = 0, K = 0;
  int l0 = 0;
  long long s0 = 0;
  int groups = 1, ksplit = 1, kchunk = 0;
  float* part = nullptr;
};

// One thread's share of a BM x 16 A tile and a 16 x BN B tile: element q of
// the thread is e = tid + 256 q, laid out along the operand's contiguous
// dimension.
template <int BM, int BN>
__device__ __forceinline__ void bw_tile_index(int e, int trans_a, int trans_b, int& ia, int& ka, int& jb, int& kb) {
  if (trans_a) {
    ia = e % BM;
    ka = e / BM;
  } else {
    ka = e & 15;
    ia = e >> 4;
  }
  if (trans_b) {
    kb = e & 15;
    jb = e >> 4;
  } else {
    jb = e % BN;
    kb = e / BN;
  }
}

// A BM x BN output tile per 256-thread block (16 x 16 threads), TM x TN per
// thread (BM = 16 TM, BN = 16 TN), K in steps of 16 through two shared-memory
// buffers: the next step's operands are loaded into registers while the
// current step computes.  Every output element is summed over K in order by
// one thread (the same order for every tile shape).  64 x 64 tiles for small
// products, 128 x 128 (8 x 8 per thread, operands read as float4) where there
// are enough tiles: four shared-memory loads per 64 FMAs instead of eight per
// 16.  With TN = 8 a thread's columns are tx*4 .. +3 and 64 + tx*4 .. +3, so
// the eight float4 reads of a quarter-warp fall in distinct banks.
template <int BM, int BN>
__global__ void __launch_bounds__(256) bw_gemm_kernel(const BwGemm g) {
  constexpr int TM = BM / 16, TN = BN / 16, QA = BM / 16, QB = BN / 16;
  __shared__ __align__(16) float As[2][16][BM + 4];
  __shared__ __align__(16) float Bs[2][16][BN + 4];
  const int cell = blockIdx.z % g.groups, kz = blockIdx.z / g.groups;
  const int l = g.l0 + cell;
  const long long s = g.s0 - cell;
  const float* A = g.A.m.at(l, s);
  const float* B = g.B.m.at(l, s);
  const int i0 = blockIdx.y * BM, j0 = blockIdx.x * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int kbeg = g.ksplit > 1 ? kz * g.kchunk : 0;
  const int kend = g.ksplit > 1 ? min(g.K, kbeg + g.kchunk) : g.K;
  float acc[TM][TN];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
  float ra[QA], rb[QB];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < QA; ++q) {
      int ia, ka, jb, kb;
      bw_tile_index<BM, BN>(threadIdx.x + 256 * q, g.A.trans, g.B.trans, ia, ka, jb, kb);
      const int r = i0 + ia, c = k0 + ka;
      ra[q] = (r < g.M && c < kend) ? (g.A.trans ? A[(long long)c * g.A.ld + r] : A[(long long)r * g.A.ld + c]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      int ia, ka, jb, kb;
      bw_tile_index<BM, BN>(threadIdx.x + 256 * q, g.A.trans, g.B.trans, ia, ka, jb, kb);
      const int cb = j0 + jb, rk = k0 + kb;
      rb[q] = (cb < g.N && rk < kend) ? (g.B.trans ? B[(long long)cb * g.B.ld + rk] : B[(long long)rk * g.B.ld + cb])
                                      : 0.f;
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int q = 0; q < QA; ++q) {
      int ia, ka, jb, kb;
      bw_tile_index<BM, BN>(threadIdx.x + 256 * q, g.A.trans, g.B.trans, ia, ka, jb, kb);
      As[buf][ka][ia] = ra[q];
    }
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      int ia, ka, jb, kb;
      bw_tile_index<BM, BN>(threadIdx.x + 256 * q, g.A.trans, g.B.trans, ia, ka, jb, kb);
      Bs[buf][kb][jb] = rb[q];
    }
  };
  // column of this thread's v-th output
  auto col_of = [&](int v) { return TN == 8 ? (v < 4 ? tx * 4 + v : 64 + tx * 4 + v - 4) : tx * TN + v; };
  int buf = 0;
  if (kbeg < kend) {
    load(kbeg);
    stash(0);
  }
  __syncthreads();
  for (int k0 = kbeg; k0 < kend; k0 += 16) {
    const bool more = k0 + 16 < kend;
    if (more) load(k0 + 16);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int u = 0; u < TM; u += 4) {
        const float4 t = *reinterpret_cast<const float4*>(&As[buf][kk][ty * TM + u]);
        a[u] = t.x;
        a[u + 1] = t.y;
        a[u + 2] = t.z;
        a[u + 3] = t.w;
      }
#pragma unroll
      for (int v = 0; v < TN; v += 4) {
        const float4 t = *reinterpret_cast<const float4*>(&Bs[buf][kk][col_of(v)]);
        b[v] = t.x;
        b[v + 1] = t.y;
        b[v + 2] = t.z;
        b[v + 3] = t.w;
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) acc[u][v] += a[u] * b[v];
    }
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
  if (g.ksplit > 1) {
    float* pt = g.part + ((long long)kz * g.groups + cell) * g.M * g.N;
#pragma unroll
    for (int u = 0; u < TM; ++u) {
      const int r = i0 + ty * TM + u;
      if (r >= g.M) continue;
#pragma unroll
      for (int v = 0; v < TN; ++v) {
        const int c = j0 + col_of(v);
        if (c < g.N) pt[(long long)r * g.N + c] = acc[u][v];
      }
    }
    return;
  }
  float* C = g.C.m.at(l, s);
  const float* E = g.E.m.p != nullptr ? g.E.m.at(l, s) : nullptr;
  const float* rs = g.rs.p != nullptr ? g.rs.at(l, s) : nullptr;
#pragma unroll
  for (int u = 0; u < TM; ++u) {
    const int r = i0 + ty * TM + u;
    if (r >= g.M) continue;
    float f = g.alpha;
    if (rs != nullptr) f = g.rs_div ? f / rs[r] : f * rs[r];
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      const int c = j0 + col_of(v);
      if (c >= g.N) continue;
      float val = f * acc[u][v];
      if (E != nullptr) val += E[(long long)r * g.E.ld + c];
      C[(long long)r * g.C.ld + c] = val;
    }
  }
}

// The split-K epilogue: C = E + alpha rs[r] sum_kz part[kz], chunks in order.
__global__ void bw_gemm_reduce_kernel(const BwGemm g) {
  const int cell = blockIdx.y, l = g.l0 + cell;
  const long long s = g.s0 - cell;
  const long long mn = (long long)g.M * g.N;
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= mn) return;
  const int r = (int)(idx / g.N), c = (int)(idx - (long long)r * g.N);
  float acc = 0.f;
  for (int kz = 0; kz < g.ksplit; ++kz) acc += g.part[((long long)kz * g.groups + cell) * mn + idx];
  float f = g.alpha;
  if (g.rs.p != nullptr) {
    const float rv = g.rs.at(l, s)[r];
    f = g.rs_div ? f / rv : f * rv;
  }
  float val = f * acc;
  if (g.E.m.p != nullptr) val += g.E.m.at(l, s)[(long long)r * g.E.ld + c];
  g.C.m.at(l, s)[(long long)r * g.C.ld + c] = val;
}

// ------------------------------------------------------ row kernels --
// One block per (row, cell): blockIdx.x = row, blockIdx.y = cell.

// Z = X + Y over rows of width n.
__global__ void bw_add_rows_kernel(CellPtr X, CellPtr Y, CellPtr Z, int n, int l0, long long s0) {
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, r = blockIdx.x;
  const float* x = X.at(l, s) + r * n;
  const float* y = Y.at(l, s) + r * n;
  float* o = Z.at(l, s) + r * n;
  for (int c = threadIdx.x; c < n; c += blockDim.x) o[c] = x[c] + y[c];
}

// phi = DPFP_nu(q) for q rows of width k (row stride ldq), and
// D = z^T phi + eps.  phi rows of width P = 2 k nu.
__global__ void bw_dpfp_rows_kernel(CellPtr Q, long long ldq, CellPtr Z, CellPtr Phi, CellPtr Den, int k, int nu,
                                    float eps, int l0, long long s0) {
  extern __shared__ float r[];  // 2k
  __shared__ float red[32];
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const int k2 = 2 * k, P = k2 * nu;
  const float* q = Q.at(l, s) + row * ldq;
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    const float v = q[c];
    r[c] = v > 0.f ? v : 0.f;
    r[c + k] = v < 0.f ? -v : 0.f;
  }
  __syncthreads();
  const float* z = Z.at(l, s);
  float* ph = Phi.at(l, s) + row * P;
  float acc = 0.f;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int j = p / k2 + 1, c = p - (j - 1) * k2;
    const int src = c - j < 0 ? c - j + k2 : c - j;
    const float f = r[c] * r[src];
    ph[p] = f;
    acc += z[p] * f;
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0 && Den.p != nullptr) Den.at(l, s)[row] = acc + eps;
}

// Adjoint of DPFP for one row: phi_bar_eff = PhiBar + c1[row] v1 + c2[row] v2
// (either term absent when its pointer is null), then
//   r_bar_c     += phi_bar_{(j-1) 2k + c} r_{(c-j) mod 2k}
//   r_bar_{c-j} += phi_bar_{(j-1) 2k + c} r_c
//   q_bar = r_bar[:k] [q > 0] - r_bar[k:] [q < 0].
// c1/c2 are read at c1.at(l,s)[row * cstride + coff].
struct DpfpTerms {
  CellPtr c1, v1, c2, v2;
  int cstride = 1, c1off = 0, c2off = 0;
};

__global__ void bw_dpfp_bwd_rows_kernel(CellPtr Q, long long ldq, CellPtr PhiBar, DpfpTerms t, CellPtr QBar,
                                        long long ldqb, int k, int nu, int l0, long long s0) {
  extern __shared__ float sm[];  // r: 2k, pb: P, rb: 2k
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const int k2 = 2 * k, P = k2 * nu;
  float* r = sm;
  float* pb = sm + k2;
  float* rb = pb + P;
  const float* q = Q.at(l, s) + row * ldq;
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    const float v = q[c];
    r[c] = v > 0.f ? v : 0.f;
    r[c + k] = v < 0.f ? -v : 0.f;
  }
  const float* phb = PhiBar.at(l, s) + row * P;
  const float c1 = t.c1.p != nullptr ? t.c1.at(l, s)[row * t.cstride + t.c1off] : 0.f;
  const float c2 = t.c2.p != nullptr ? t.c2.at(l, s)[row * t.cstride + t.c2off] : 0.f;
  const float* v1 = t.v1.p != nullptr ? t.v1.at(l, s) : nullptr;
  const float* v2 = t.v2.p != nullptr ? t.v2.at(l, s) : nullptr;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    float v = phb[p];
    if (v1 != nullptr) v += c1 * v1[p];
    if (v2 != nullptr) v += c2 * v2[p];
    pb[p] = v;
  }
  __syncthreads();
  // r_bar_c collects, over j, phi_bar at (j, c) times r_{c-j} and phi_bar at
  // (j, c+j) times r_{c+j}: a fixed summation order per element
  for (int c = threadIdx.x; c < k2; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 1; j <= nu; ++j) {
      const int cm = c - j < 0 ? c - j + k2 : c - j;
      const int cp = c + j >= k2 ? c + j - k2 : c + j;
      acc += pb[(j - 1) * k2 + c] * r[cm];
      acc += pb[(j - 1) * k2 + cp] * r[cp];
    }
    rb[c] = acc;
  }
  __syncthreads();
  float* qb = QBar.at(l, s) + row * ldqb;
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    const float v = q[c];
    qb[c] = v > 0.f ? rb[c] : (v < 0.f ? -rb[c + k] : 0.f);
  }
}

// y = x s g with s = (mean x^2 + eps)^-1/2, rows of width d; also stores s.
__global__ void bw_rmsnorm_rows_kernel(CellPtr X, CellPtr G, CellPtr Y, CellPtr Srow, int d, float eps, int l0,
                                       long long s0) {
  __shared__ float red[32];
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const float* x = X.at(l, s) + row * d;
  const float* g = G.at(l, s);
  float acc = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) acc += x[c] * x[c];
  acc = block_sum(acc, red);
  const float sc = 1.0f / sqrtf(acc / (float)d + eps);
  float* y = Y.at(l, s) + row * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) y[c] = x[c] * sc * g[c];
  if (threadIdx.x == 0 && Srow.p != nullptr) Srow.at(l, s)[row] = sc;
}

// Adjoint of the RMSNorm above: X_bar = E + s t - s^3 (t . x) x / d with
// t = Y_bar g (E absent: 0).  Rows >= valid (alt_valid for layer alt_l) get
// X_bar = E (or 0) and do not read Y_bar.  Stores s per row (for the gain).
__global__ void bw_rmsnorm_bwd_rows_kernel(CellPtr X, CellPtr G, CellPtr Ybar, long long ldy, CellPtr E,
                                           CellPtr Xbar, CellPtr Srow, int d, float eps, int valid, int alt_l,
                                           int alt_valid, int l0, long long s0) {
  __shared__ float red[32];
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const bool ok = row < (l == alt_l ? alt_valid : valid);
  const float* x = X.at(l, s) + row * d;
  const float* g = G.at(l, s);
  const float* yb = ok ? Ybar.at(l, s) + row * ldy : nullptr;
  const float* e = E.p != nullptr ? E.at(l, s) + row * d : nullptr;
  float* xb = Xbar.at(l, s) + row * d;
  float ss = 0.f, tx = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    ss += x[c] * x[c];
    if (ok) tx += yb[c] * g[c] * x[c];
  }
  ss = block_sum(ss, red);
  tx = block_sum(tx, red);
  const float sc = 1.0f / sqrtf(ss / (float)d + eps);
  const float k3 = sc * sc * sc * tx / (float)d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float v = ok ? sc * yb[c] * g[c] - k3 * x[c] : 0.f;
    if (e != nullptr) v += e[c];
    xb[c] = v;
  }
  if (threadIdx.x == 0) Srow.at(l, s)[row] = sc;
}

// dg[c] += sum_{r < valid} Ybar[r][c] X[r][c] s[r]: the gain's gradient.  A
// block takes 32 columns (one per lane); warp w sums rows w, w + 8, ... and
// the 8 partial sums are added in warp order (deterministic).  256 threads.
__global__ void __launch_bounds__(256) bw_gain_grad_kernel(CellPtr X, CellPtr Ybar, long long ldy, CellPtr Srow,
                                                           CellPtr dG, int d, int valid, int alt_l, int alt_valid,
                                                           int l0, long long s0) {
  __shared__ float part[8][32];
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  const int v = l == alt_l ? alt_valid : valid;
  const float* x = X.at(l, s);
  const float* yb = Ybar.at(l, s);
  const float* sr = Srow.at(l, s);
  float acc = 0.f;
  if (c < d)
    for (int r = warp; r < v; r += 8) acc += yb[(long long)r * ldy + c] * x[(long long)r * d + c] * sr[r];
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && c < d) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w][lane];
    dG.at(l, s)[c] += t;
  }
}

// RoPE (rotate-half, positions 0 .. T-1 of the cell) on the first n_rope
// columns of rows of width ld, per head of hd columns; dir = +1 the
// rotation, -1 its transpose (the adjoint).
__global__ void bw_rope_rows_kernel(CellPtr QKV, int ld, int n_rope, int hd, const float* cosT, const float* sinT,
                                    int dir, int l0, long long s0) {
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const int half = hd / 2;
  float* x = QKV.at(l, s) + row * ld;
  const float* cr = cosT + row * half;
  const float* sr = sinT + row * half;
  for (int e = threadIdx.x; e < n_rope / 2; e += blockDim.x) {
    const int h = e / half, i = e - h * half;
    float* p = x + h * hd + i;
    const float a = p[0], b = p[half], c = cr[i], sn = sr[i] * (float)dir;
    p[0] = a * c - b * sn;
    p[half] = b * c + a * sn;
  }
}

__device__ __forceinline__ float bw_sigmoid(float a) { return 1.0f / (1.0f + expf(-a)); }

// u_f = silu(a_f) b_f from the fused gate-up rows (blocks of GU_BLK gate
// columns followed by the same up columns), rows of F outputs.
__global__ void bw_swiglu_rows_kernel(CellPtr GU, CellPtr U, int F, int l0, long long s0) {
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const float* gu = GU.at(l, s) + row * 2 * F;
  float* u = U.at(l, s) + row * F;
  for (int f = threadIdx.x; f < F; f += blockDim.x) {
    const int b = f / GU_BLK, i = f - b * GU_BLK;
    const float a = gu[2 * b * GU_BLK + i], bb = gu[2 * b * GU_BLK + GU_BLK + i];
    u[f] = a * bw_sigmoid(a) * bb;
  }
}

// Adjoint of the SwiGLU above, into the fused column order.
__global__ void bw_swiglu_bwd_rows_kernel(CellPtr GU, CellPtr Ubar, CellPtr GUbar, int F, int l0, long long s0) {
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const float* gu = GU.at(l, s) + row * 2 * F;
  const float* ub = Ubar.at(l, s) + row * F;
  float* o = GUbar.at(l, s) + row * 2 * F;
  for (int f = threadIdx.x; f < F; f += blockDim.x) {
    const int b = f / GU_BLK, i = f - b * GU_BLK;
    const int ca = 2 * b * GU_BLK + i, cb = ca + GU_BLK;
    const float a = gu[ca], bb = gu[cb], sa = bw_sigmoid(a);
    o[ca] = ub[f] * bb * sa * (1.0f + a * (1.0f - sa));
    o[cb] = ub[f] * a * sa;
  }
}

// ---------------------------------------------------------- attention --
// Causal GQA attention over the T rows of a cell, fp32: QKV rows hold q
// heads (Hq * hd), then k heads and v heads (Hkv * hd each); query head h
// reads kv head h * Hkv / Hq.  Blocks of 8 warps take 32 rows (4 per warp)
// against 32-row tiles in shared memory; lane j scores key j of the tile,
// lanes own output columns lane + 32 t.

struct BwAttn {
  CellPtr QKV, O, LSE, dO, Dsum, dQKV;
  int T, Hq, Hkv, ld, ldo;
  float scale;
  int l0;
  long long s0;
};

// Forward with the log-sum-exp of every (row, head) kept.
template <int HD>
__global__ void __launch_bounds__(256) bw_attn_fwd_kernel(const BwAttn a) {
  constexpr int NC = HD / 32;
  extern __shared__ float sm[];
  float(*Ks)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm);
  float(*Qs)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm + 32 * (HD + 1));
  float(*Vs)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm + 64 * (HD + 1));
  const int z = blockIdx.z, l = a.l0 + z, h = blockIdx.y;
  const long long s = a.s0 - z;
  const int g = (h * a.Hkv) / a.Hq;
  const float* qkv = a.QKV.at(l, s);
  const int q0 = blockIdx.x * 32, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < 32 * HD; e += 256) {
    const int r = e / HD, c = e - r * HD;
    Qs[r][c] = q0 + r < a.T ? qkv[(long long)(q0 + r) * a.ld + h * HD + c] : 0.f;
  }
  float m[4], lsum[4], o[4][NC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    m[rr] = -INFINITY;
    lsum[rr] = 0.f;
#pragma unroll
    for (int t = 0; t < NC; ++t) o[rr][t] = 0.f;
  }
  const int kend = min(a.T, q0 + 32);
  for (int k0 = 0; k0 < kend; k0 += 32) {
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * HD; e += 256) {
      const int r = e / HD, c = e - r * HD;
      const bool ok = k0 + r < a.T;
      Ks[r][c] = ok ? qkv[(long long)(k0 + r) * a.ld + (a.Hq + g) * HD + c] : 0.f;
      Vs[r][c] = ok ? qkv[(long long)(k0 + r) * a.ld + (a.Hq + a.Hkv + g) * HD + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int qr = warp * 4 + rr, qi = q0 + qr, kj = k0 + lane;
      float sc = 0.f;
      for (int c = 0; c < HD; ++c) sc += Qs[qr][c] * Ks[lane][c];
      sc = (kj <= qi && kj < a.T) ? sc * a.scale : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[rr], mx);
      if (mn == -INFINITY) continue;  // no visible key yet (rows past T)
      const float p = sc == -INFINITY ? 0.f : expf(sc - mn);
      const float corr = m[rr] == -INFINITY ? 0.f : expf(m[rr] - mn);
      const float ps = warp_sum(p);
      lsum[rr] = lsum[rr] * corr + ps;
#pragma unroll
      for (int t = 0; t < NC; ++t) o[rr][t] *= corr;
      for (int j = 0; j < 32; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int t = 0; t < NC; ++t) o[rr][t] += pj * Vs[j][lane + 32 * t];
      }
      m[rr] = mn;
    }
  }
  float* out = a.O.at(l, s);
  float* lse = a.LSE.at(l, s);
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int qi = q0 + warp * 4 + rr;
    if (qi >= a.T) continue;
    const float inv = 1.0f / lsum[rr];
#pragma unroll
    for (int t = 0; t < NC; ++t) out[(long long)qi * a.ldo + h * HD + lane + 32 * t] = o[rr][t] * inv;
    if (lane == 0) lse[(long long)qi * a.Hq + h] = m[rr] + logf(lsum[rr]);
  }
}

// Dsum[r][h] = dO[r, h] . O[r, h] (the softmax adjoint's row term).
template <int HD>
__global__ void bw_attn_dsum_kernel(const BwAttn a) {
  const int z = blockIdx.y, l = a.l0 + z;
  const long long s = a.s0 - z, row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* o = a.O.at(l, s) + row * a.ldo;
  const float* d = a.dO.at(l, s) + row * a.ldo;
  for (int h = warp; h < a.Hq; h += blockDim.x >> 5) {
    float acc = 0.f;
    for (int c = lane; c < HD; c += 32) acc += o[h * HD + c] * d[h * HD + c];
    acc = warp_sum(acc);
    if (lane == 0) a.Dsum.at(l, s)[row * a.Hq + h] = acc;
  }
}

// q_bar rows: for query i, sum over keys j <= i of S_bar_ij k_j / sqrt(hd).
template <int HD>
__global__ void __launch_bounds__(256) bw_attn_dq_kernel(const BwAttn a) {
  constexpr int NC = HD / 32;
  extern __shared__ float sm[];
  float(*Ks)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm);
  float(*Vs)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm + 32 * (HD + 1));
  float(*Qs)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm + 64 * (HD + 1));
  float(*Ds)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm + 96 * (HD + 1));
  const int z = blockIdx.z, l = a.l0 + z, h = blockIdx.y;
  const long long s = a.s0 - z;
  const int g = (h * a.Hkv) / a.Hq;
  const float* qkv = a.QKV.at(l, s);
  const float* dO = a.dO.at(l, s);
  const int q0 = blockIdx.x * 32, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < 32 * HD; e += 256) {
    const int r = e / HD, c = e - r * HD;
    const bool ok = q0 + r < a.T;
    Qs[r][c] = ok ? qkv[(long long)(q0 + r) * a.ld + h * HD + c] : 0.f;
    Ds[r][c] = ok ? dO[(long long)(q0 + r) * a.ldo + h * HD + c] : 0.f;
  }
  float lse[4], dsum[4], dq[4][NC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int qi = q0 + warp * 4 + rr;
    lse[rr] = qi < a.T ? a.LSE.at(l, s)[(long long)qi * a.Hq + h] : 0.f;
    dsum[rr] = qi < a.T ? a.Dsum.at(l, s)[(long long)qi * a.Hq + h] : 0.f;
#pragma unroll
    for (int t = 0; t < NC; ++t) dq[rr][t] = 0.f;
  }
  const int kend = min(a.T, q0 + 32);
  for (int k0 = 0; k0 < kend; k0 += 32) {
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * HD; e += 256) {
      const int r = e / HD, c = e - r * HD;
      const bool ok = k0 + r < a.T;
      Ks[r][c] = ok ? qkv[(long long)(k0 + r) * a.ld + (a.Hq + g) * HD + c] : 0.f;
      Vs[r][c] = ok ? qkv[(long long)(k0 + r) * a.ld + (a.Hq + a.Hkv + g) * HD + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int qr = warp * 4 + rr, qi = q0 + qr, kj = k0 + lane;
      float sc = 0.f, dp = 0.f;
      for (int c = 0; c < HD; ++c) {
        sc += Qs[qr][c] * Ks[lane][c];
        dp += Ds[qr][c] * Vs[lane][c];
      }
      const bool vis = kj <= qi && kj < a.T && qi < a.T;
      const float p = vis ? expf(sc * a.scale - lse[rr]) : 0.f;
      const float ds = p * (dp - dsum[rr]);
      for (int j = 0; j < 32; ++j) {
        const float dj = __shfl_sync(0xffffffffu, ds, j);
#pragma unroll
        for (int t = 0; t < NC; ++t) dq[rr][t] += dj * Ks[j][lane + 32 * t];
      }
    }
  }
  float* out = a.dQKV.at(l, s);
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int qi = q0 + warp * 4 + rr;
    if (qi >= a.T) continue;
#pragma unroll
    for (int t = 0; t < NC; ++t) out[(long long)qi * a.ld + h * HD + lane + 32 * t] = dq[rr][t] * a.scale;
  }
}

// k_bar and v_bar rows of kv head g: for key j, over the query heads of the
// group and queries i >= j: v_bar_j += P_ij dO_i, k_bar_j += S_bar_ij q_i / sqrt(hd).
template <int HD>
__global__ void __launch_bounds__(256) bw_attn_dkv_kernel(const BwAttn a) {
  constexpr int NC = HD / 32;
  extern __shared__ float sm[];
  float(*Qs)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm);
  float(*Ds)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm + 32 * (HD + 1));
  float(*Ks)[HD] = reinterpret_cast<float(*)[HD]>(sm + 64 * (HD + 1));
  float(*Vs)[HD] = reinterpret_cast<float(*)[HD]>(sm + 64 * (HD + 1) + 32 * HD);
  float* ls = sm + 64 * (HD + 1) + 64 * HD;  // lse of the query tile
  float* dss = ls + 32;                       // Dsum of the query tile
  const int z = blockIdx.z, l = a.l0 + z, g = blockIdx.y;
  const long long s = a.s0 - z;
  const float* qkv = a.QKV.at(l, s);
  const float* dO = a.dO.at(l, s);
  const int k0 = blockIdx.x * 32, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < 32 * HD; e += 256) {
    const int r = e / HD, c = e - r * HD;
    const bool ok = k0 + r < a.T;
    Ks[r][c] = ok ? qkv[(long long)(k0 + r) * a.ld + (a.Hq + g) * HD + c] : 0.f;
    Vs[r][c] = ok ? qkv[(long long)(k0 + r) * a.ld + (a.Hq + a.Hkv + g) * HD + c] : 0.f;
  }
  float dk[4][NC], dv[4][NC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr)
#pragma unroll
    for (int t = 0; t < NC; ++t) {
      dk[rr][t] = 0.f;
      dv[rr][t] = 0.f;
    }
  const int per = a.Hq / a.Hkv;
  for (int hh = 0; hh < per; ++hh) {
    const int h = g * per + hh;
    for (int q0 = k0; q0 < a.T; q0 += 32) {
      __syncthreads();
      for (int e = threadIdx.x; e < 32 * HD; e += 256) {
        const int r = e / HD, c = e - r * HD;
        const bool ok = q0 + r < a.T;
        Qs[r][c] = ok ? qkv[(long long)(q0 + r) * a.ld + h * HD + c] : 0.f;
        Ds[r][c] = ok ? dO[(long long)(q0 + r) * a.ldo + h * HD + c] : 0.f;
      }
      if (threadIdx.x < 32) {
        const int qi = q0 + threadIdx.x;
        ls[threadIdx.x] = qi < a.T ? a.LSE.at(l, s)[(long long)qi * a.Hq + h] : 0.f;
        dss[threadIdx.x] = qi < a.T ? a.Dsum.at(l, s)[(long long)qi * a.Hq + h] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int kr = warp * 4 + rr, kj = k0 + kr, qi = q0 + lane;
        float sc = 0.f, dp = 0.f;
        for (int c = 0; c < HD; ++c) {
          sc += Qs[lane][c] * Ks[kr][c];
          dp += Ds[lane][c] * Vs[kr][c];
        }
        const bool vis = kj <= qi && qi < a.T && kj < a.T;
        const float p = vis ? expf(sc * a.scale - ls[lane]) : 0.f;
        const float ds = p * (dp - dss[lane]);
        for (int i = 0; i < 32; ++i) {
          const float pi = __shfl_sync(0xffffffffu, p, i);
          const float di = __shfl_sync(0xffffffffu, ds, i);
#pragma unroll
          for (int t = 0; t < NC; ++t) {
            dv[rr][t] += pi * Ds[i][lane + 32 * t];
            dk[rr][t] += di * Qs[i][lane + 32 * t];
          }
        }
      }
    }
  }
  float* out = a.dQKV.at(l, s);
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int kj = k0 + warp * 4 + rr;
    if (kj >= a.T) continue;
#pragma unroll
    for (int t = 0; t < NC; ++t) {
      out[(long long)kj * a.ld + (a.Hq + g) * HD + lane + 32 * t] = dk[rr][t] * a.scale;
      out[(long long)kj * a.ld + (a.Hq + a.Hkv + g) * HD + lane + 32 * t] = dv[rr][t];
    }
  }
}

// dynamic shared memory of the three kernels
inline size_t bw_attn_fwd_smem(int hd) { return (size_t)96 * (hd + 1) * sizeof(float); }
inline size_t bw_attn_dq_smem(int hd) { return (size_t)128 * (hd + 1) * sizeof(float); }
inline size_t bw_attn_dkv_smem(int hd) { return (size_t)(64 * (hd + 1) + 64 * hd + 64) * sizeof(float); }

// ------------------------------------------------------ memory write --
//
// The M memory rows write in order (section 二): with phi_i = DPFP(k_i),
//   D_i = z_i^T phi_i + eps,  vbar_i = A_i phi_i / D_i,
//   Q_i = phi_i^T phi_i + eps, gu_i = 1 - z_i^T phi_i / Q_i, gamma_i = clip(gu_i, 0, 1),
//   c_i = beta_i (v_i - vbar_i),  A_{i+1} = A_i + c_i phi_i^T,  z_{i+1} = z_i + gamma_i phi_i.
// Every update is rank one, so with G = Phi Phi^T every product of a state
// with a feature unrolls into the entry state plus earlier (or later) rank-one
// terms.  Walking the writes backwards from the adjoints (A_bar, z_bar) of
// the final state, with w_i = -beta_i c_bar_i / D_i (the adjoint of A_i phi_i):
//   c_bar_i  = A_bar phi_i + sum_{j>i} w_j G_ji                 (per row of A)
//   A_bar_in = A_bar + sum_i w_i phi_i^T
//   zeta_i   = -(w_i . vbar_i) - gu_bar_i / Q_i                 (adjoint of z_i^T phi_i)
//   gu_bar_i = [0 <= gu_i <= 1] (z_bar^T phi_i + sum_{j>i} zeta_j G_ji)
//   z_bar_in = z_bar + sum_i zeta_i phi_i
//   phi_bar_i = A_bar^T c_i + A_in^T w_i + gamma_i z_bar + zeta_i z_in
//             + sum_{j>i} (w_j . c_i + gamma_i zeta_j) phi_j
//             + sum_{j<i} (c_j . w_i + zeta_i gamma_j) phi_j + 2 gu_bar_i z_i^T phi_i / Q_i^2 phi_i
//   b_bar_i = c_bar_i . (v_i - vbar_i),  v_bar_i = beta_i c_bar_i,  k_bar_i = DPFP^T(phi_bar_i),
// with A_bar, z_bar those of the final state and A_in, z_in the entry state.
// Rows of the state are independent given the scalars, as in the forward.

// Per-write scalars, row i of a [M][8] block.
enum { WS_BETA = 0, WS_D, WS_Q, WS_GU, WS_GAMMA, WS_ZPHI, WS_ZETA, WS_NSC = 8 };

// One block per cell: phi_i, the Gram matrix and the normaliser recurrence
// (z is not touched: the entry state comes from zin).  vkb rows [v | k |
// beta logit | pad] of stride nw.  M <= 32.
__global__ void __launch_bounds__(256) bw_write_feat_kernel(CellPtr VKB, CellPtr Zin, CellPtr PhiM, CellPtr Sc,
                                                            CellPtr Gm, int M, int k, int nu, float eps, int d,
                                                            int nw, int l0, long long s0) {
  extern __shared__ float sm[];  // r: M * 2k, phi: M * (P + 1)
  __shared__ float G[32][33];
  __shared__ float z0phi[32], logit[32];
  const int l = l0 + blockIdx.x;
  const long long s = s0 - blockIdx.x;
  const int k2 = 2 * k, P = k2 * nu, Pp = P + 1;
  float* r = sm;
  float* ph = sm + M * k2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const float* vkb = VKB.at(l, s);
  const float* zin = Zin.at(l, s);
  for (int i = warp; i < M; i += nwarp) {
    const float* src = vkb + (long long)i * nw + d;
    for (int c = lane; c < k; c += 32) {
      const float v = src[c];
      r[i * k2 + c] = v > 0.f ? v : 0.f;
      r[i * k2 + c + k] = v < 0.f ? -v : 0.f;
    }
    if (lane == 0) logit[i] = src[k];
  }
  __syncthreads();
  float* phiM = PhiM.at(l, s);
  for (int i = warp; i < M; i += nwarp)
    for (int p = lane; p < P; p += 32) {
      const int j = p / k2 + 1, c = p - (j - 1) * k2;
      const int src = c - j < 0 ? c - j + k2 : c - j;
      const float f = r[i * k2 + c] * r[i * k2 + src];
      ph[i * Pp + p] = f;
      phiM[(long long)i * P + p] = f;
    }
  __syncthreads();
  for (int t = warp; t < M * M + M; t += nwarp) {
    float acc = 0.f;
    if (t < M * M) {
      const int i = t / M, j = t - i * M;
      for (int p = lane; p < P; p += 32) acc += ph[i * Pp + p] * ph[j * Pp + p];
      acc = warp_sum(acc);
      if (lane == 0) G[i][j] = acc;
    } else {
      const int i = t - M * M;
      for (int p = lane; p < P; p += 32) acc += zin[p] * ph[i * Pp + p];
      acc = warp_sum(acc);
      if (lane == 0) z0phi[i] = acc;
    }
  }
  __syncthreads();
  float* sc = Sc.at(l, s);
  if (threadIdx.x == 0) {
    float gam[32];
    for (int i = 0; i < M; ++i) {
      float zp = z0phi[i];
      for (int j = 0; j < i; ++j) zp += gam[j] * G[j][i];
      const float Q = G[i][i] + eps;
      const float gu = 1.0f - zp / Q;
      gam[i] = fminf(fmaxf(gu, 0.0f), 1.0f);
      float* o = sc + i * WS_NSC;
      o[WS_BETA] = bw_sigmoid(logit[i]);
      o[WS_D] = zp + eps;
      o[WS_Q] = Q;
      o[WS_GU] = gu;
      o[WS_GAMMA] = gam[i];
      o[WS_ZPHI] = zp;
      o[WS_ZETA] = 0.f;
    }
  }
  float* gm = Gm.at(l, s);
  for (int t = threadIdx.x; t < M * M; t += blockDim.x) gm[t] = G[t / M][t % M];
}

// Per row j of the state (lanes over the P features; each warp runs RW rows
// side by side, independent chains): forward over the writes from A_in[j]
// (c_i[j], vbar_i[j]), then backward from A_bar[j] (c_bar_i[j], w_i[j]), and
// A_bar_in[j] = A_bar[j] + sum_i w_i[j] phi_i.  Stores C, Vb, CB, W as [M][d].
template <int NT>
__global__ void __launch_bounds__(128) bw_write_rows_kernel(CellPtr Ain, CellPtr Abar, CellPtr AbarIn, CellPtr PhiM,
                                                            CellPtr Sc, CellPtr VKB, CellPtr Cw, CellPtr Vb,
                                                            CellPtr CB, CellPtr Wv, int M, int d, int nw,
                                                            int rows_per_block, int l0, long long s0) {
  constexpr int P = 32 * NT, RW = 4;
  extern __shared__ float sm[];
  float* ps = sm;           // [M][P]
  float* cs = ps + M * P;   // [M][WS_NSC]
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y;
  const float* phiM = PhiM.at(l, s);
  const float* sc = Sc.at(l, s);
  for (int t = threadIdx.x; t < M * P; t += blockDim.x) ps[t] = phiM[t];
  for (int t = threadIdx.x; t < M * WS_NSC; t += blockDim.x) cs[t] = sc[t];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const float* ain = Ain.at(l, s);
  const float* abar = Abar.at(l, s);
  float* abin = AbarIn.at(l, s);
  const float* vkb = VKB.at(l, s);
  float *cw = Cw.at(l, s), *vb = Vb.at(l, s), *cb = CB.at(l, s), *wv = Wv.at(l, s);
  const int j_end = min(d, (int)(blockIdx.x + 1) * rows_per_block);
  for (int jb = blockIdx.x * rows_per_block + warp * RW; jb < j_end; jb += nwarps * RW) {
    float a[RW][NT], vj[RW], my_c[RW], my_vb[RW], my_cb[RW], my_w[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int j = jb + r;
      const bool ok = j < j_end;
#pragma unroll
      for (int t = 0; t < NT; ++t) a[r][t] = ok ? ain[(long long)j * P + lane + 32 * t] : 0.f;
      vj[r] = (ok && lane < M) ? vkb[(long long)lane * nw + j] : 0.f;  // lane i holds v_i[j]
      my_c[r] = my_vb[r] = my_cb[r] = my_w[r] = 0.f;
    }
    for (int i = 0; i < M; ++i) {
      const float* pi = ps + i * P + lane;
      float ph[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) ph[t] = pi[32 * t];
      float dot[RW];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        dot[r] = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) dot[r] += a[r][t] * ph[t];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < RW; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
      const float beta = cs[i * WS_NSC + WS_BETA], D = cs[i * WS_NSC + WS_D];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const float vbar = dot[r] / D;
        const float c = beta * (__shfl_sync(0xffffffffu, vj[r], i) - vbar);
#pragma unroll
        for (int t = 0; t < NT; ++t) a[r][t] += c * ph[t];
        if (lane == i) {
          my_c[r] = c;
          my_vb[r] = vbar;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int j = jb + r;
      const bool ok = j < j_end;
#pragma unroll
      for (int t = 0; t < NT; ++t) a[r][t] = ok ? abar[(long long)j * P + lane + 32 * t] : 0.f;
    }
    for (int i = M - 1; i >= 0; --i) {
      const float* pi = ps + i * P + lane;
      float ph[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) ph[t] = pi[32 * t];
      float dot[RW];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        dot[r] = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) dot[r] += a[r][t] * ph[t];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < RW; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
      const float beta = cs[i * WS_NSC + WS_BETA], D = cs[i * WS_NSC + WS_D];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const float w = -beta * dot[r] / D;
#pragma unroll
        for (int t = 0; t < NT; ++t) a[r][t] += w * ph[t];
        if (lane == i) {
          my_cb[r] = dot[r];
          my_w[r] = w;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int j = jb + r;
      if (j >= j_end) continue;
#pragma unroll
      for (int t = 0; t < NT; ++t) abin[(long long)j * P + lane + 32 * t] = a[r][t];
      if (lane < M) {
        cw[(long long)lane * d + j] = my_c[r];
        vb[(long long)lane * d + j] = my_vb[r];
        cb[(long long)lane * d + j] = my_cb[r];
        wv[(long long)lane * d + j] = my_w[r];
      }
    }
  }
}

// One block per cell: the reductions over the rows of the state and the
// scalar recurrence of zeta (above), then
//   Coef[i][j] (the phi_j coefficients of phi_bar_i),
//   VKBbar row i = [beta_i c_bar_i | (k part: later) | b_bar_i beta_i (1 - beta_i) | 0],
//   z_bar_in = z_bar + sum_i zeta_i phi_i,  Sc[i][WS_ZETA] = zeta_i.
__global__ void __launch_bounds__(256) bw_write_scalars_kernel(CellPtr Cw, CellPtr Vb, CellPtr CB, CellPtr Wv,
                                                               CellPtr VKB, CellPtr PhiM, CellPtr Gm, CellPtr Sc,
                                                               CellPtr Zbar, CellPtr ZbarIn, CellPtr Coef,
                                                               CellPtr VKBbar, int M, int P, int d, int k, int nw,
                                                               int l0, long long s0) {
  __shared__ float X[32][33];   // X[j][i] = w_j . c_i
  __shared__ float G[32][33];
  __shared__ float bbar[32], e[32], zfp[32], zeta[32], dg[32];
  const int l = l0 + blockIdx.x;
  const long long s = s0 - blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const float *cw = Cw.at(l, s), *vb = Vb.at(l, s), *cb = CB.at(l, s), *wv = Wv.at(l, s);
  const float* vkb = VKB.at(l, s);
  const float* phiM = PhiM.at(l, s);
  const float* zbar = Zbar.at(l, s);
  float* sc = Sc.at(l, s);
  const float* gm = Gm.at(l, s);
  for (int t = threadIdx.x; t < M * M; t += blockDim.x) G[t / M][t % M] = gm[t];
  // the dot products over the d rows of the state, 32 rows at a time through
  // shared memory: thread t owns pairs (j, i) = t, t + 256, ... of X and, for
  // t < M, b_bar_t and e_t; every sum runs in row order
  {
    __shared__ float sW[32][33], sC[32][33], sB[32][33], sE[32][33], sV[32][33];
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, ab = 0.f, ae = 0.f;
    for (int r0 = 0; r0 < d; r0 += 32) {
      __syncthreads();
      for (int e2 = threadIdx.x; e2 < M * 32; e2 += blockDim.x) {
        const int i = e2 >> 5, c = e2 & 31, r = r0 + c;
        const bool ok = r < d;
        const long long o = (long long)i * d + r;
        sW[i][c] = ok ? wv[o] : 0.f;
        sC[i][c] = ok ? cw[o] : 0.f;
        sB[i][c] = ok ? cb[o] : 0.f;
        sV[i][c] = ok ? vb[o] : 0.f;
        sE[i][c] = ok ? vkb[(long long)i * nw + r] - vb[o] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int t = threadIdx.x + 256 * q;
        if (t < M * M) {
          const int j = t / M, i = t - j * M;
          float a = acc[q];
          for (int c = 0; c < 32; ++c) a += sW[j][c] * sC[i][c];
          acc[q] = a;
        }
      }
      if (threadIdx.x < M) {
        const int i = threadIdx.x;
        for (int c = 0; c < 32; ++c) {
          ab += sB[i][c] * sE[i][c];
          ae += sW[i][c] * sV[i][c];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = threadIdx.x + 256 * q;
      if (t < M * M) X[t / M][t % M] = acc[q];
    }
    if (threadIdx.x < M) {
      bbar[threadIdx.x] = ab;
      e[threadIdx.x] = ae;
    }
  }
  for (int i = warp; i < M; i += nwarp) {
    float acc = 0.f;
    for (int p = lane; p < P; p += 32) acc += zbar[p] * phiM[(long long)i * P + p];
    acc = warp_sum(acc);
    if (lane == 0) zfp[i] = acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = M - 1; i >= 0; --i) {
      const float* o = sc + i * WS_NSC;
      float gb = zfp[i];
      for (int j = i + 1; j < M; ++j) gb += zeta[j] * G[j][i];
      const float gu = o[WS_GU], Q = o[WS_Q];
      const float gub = (gu >= 0.f && gu <= 1.f) ? gb : 0.f;
      zeta[i] = -e[i] - gub / Q;
      dg[i] = 2.0f * gub * o[WS_ZPHI] / (Q * Q);
    }
  }
  __syncthreads();
  float* coef = Coef.at(l, s);
  for (int t = threadIdx.x; t < M * M; t += blockDim.x) {
    const int i = t / M, j = t - i * M;
    const float gi = sc[i * WS_NSC + WS_GAMMA], gj = sc[j * WS_NSC + WS_GAMMA];
    float v;
    if (j > i)
      v = X[j][i] + gi * zeta[j];
    else if (j < i)
      v = X[i][j] + zeta[i] * gj;
    else
      v = dg[i];
    coef[t] = v;
  }
  if (threadIdx.x < M) sc[threadIdx.x * WS_NSC + WS_ZETA] = zeta[threadIdx.x];
  float* vbar_out = VKBbar.at(l, s);
  for (int i = warp; i < M; i += nwarp) {
    const float beta = sc[i * WS_NSC + WS_BETA];
    float* row = vbar_out + (long long)i * nw;
    for (int r = lane; r < d; r += 32) row[r] = beta * cb[(long long)i * d + r];
    for (int c = d + k + lane; c < nw; c += 32) row[c] = c == d + k ? bbar[i] * beta * (1.0f - beta) : 0.f;
  }
  float* zout = ZbarIn.at(l, s);
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    float acc = zbar[p];
    for (int i = 0; i < M; ++i) acc += zeta[i] * phiM[(long long)i * P + p];
    zout[p] = acc;
  }
}

// ------------------------------------------- read backward, embedding --

// Per row of the read y = x + r, r = A phi / D: XS = y_bar / D and the
// denominator's adjoint D_bar = -(y_bar . r) / D.  Then A_bar += XS^T Phi,
// z_bar += D_bar^T Phi and phi_bar = XS A + D_bar z.
__global__ void bw_read_rows_kernel(CellPtr X1bar, CellPtr Rr, CellPtr Den, CellPtr XS, CellPtr Dbar, int d,
                                    int l0, long long s0) {
  __shared__ float red[32];
  const int l = l0 + blockIdx.y;
  const long long s = s0 - blockIdx.y, row = blockIdx.x;
  const float* xb = X1bar.at(l, s) + row * d;
  const float* r = Rr.at(l, s) + row * d;
  float* xs = XS.at(l, s) + row * d;
  const float D = Den.at(l, s)[row];
  float acc = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    acc += xb[c] * r[c];
    xs[c] = xb[c] / D;
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) Dbar.at(l, s)[row] = -acc / D;
}

// Embedding and memory-token gradients from the layer-0 input adjoints
// XB0[s] (T rows per segment): dE[tok] += row, dMem[i] += row n_rows + i, in
// segment and row order (one thread per column; ids clamped like the
// forward's gather).
__global__ void bw_embed_grad_kernel(const float* XB0, const int32_t* tokens, long long n_tok, int S, int T,
                                     int M, int d, int vocab, long long n_seg, float* dE, float* dMem) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  for (long long s = 0; s < n_seg; ++s) {
    const long long t0 = s * S;
    const int n_rows = (int)min((long long)S, n_tok - t0);
    const float* xb = XB0 + s * T * (long long)d;
    // eight rows' loads in flight; the adds stay in row order
    for (int t = 0; t < n_rows; t += 8) {
      int id[8];
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool ok = t + u < n_rows;
        const int v = ok ? tokens[t0 + t + u] : 0;
        id[u] = v < 0 ? 0 : (v >= vocab ? vocab - 1 : v);
        x[u] = ok ? xb[(long long)(t + u) * d + c] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (t + u < n_rows) dE[(long long)id[u] * d + c] += x[u];
    }
    for (int i = 0; i < M; ++i) dMem[(long long)i * d + c] += xb[(long long)(n_rows + i) * d + c];
  }
}

}  // namespace armt
