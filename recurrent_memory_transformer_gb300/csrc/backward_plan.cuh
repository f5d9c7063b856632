// Backward pass of the ARMT forward (fp32): the host side.  One call of
// BwRun::diagonal runs every cell of reverse anti-diagonal i (section 四 of the
// summary page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
// Transformers for Long Contexts": the backward pass keeps the diagonal
// schedule) in the order recompute -> write adjoint -> block adjoint -> read
// adjoint, each step one launch over all cells of the diagonal.
#pragma once

#include <algorithm>

#include "backward.cuh"
#include "bw_plan.h"

namespace armt {

// Everything the backward reads and writes (fp32, device).  Per-layer
// workspace slots hold one cell per layer; saved tensors hold one cell per
// (layer, segment).
struct BwView {
  // sizes
  int L, d, k, nu, P, Hq, Hkv, hd, F, Nq, nw, T, S, M, vocab;
  float norm_eps, assoc_eps;
  long long n_seg, n_tok;
  int last_len;
  // weights (library layout: Wqkv fused [q; k; v], Wgu gate/up interleaved,
  // Ww [Wv_a; Wk_a; wbeta_a; 0] per layer)
  float *aWq, *Wqkv, *Wo, *Wgu, *Wd, *Ww, *g1, *g2, *gf;
  const float *cosT, *sinT;
  // saved by the forward: cell inputs and entry states
  float *Xs, *As, *zs;
  // cotangents (nullptr: zero)
  const float *cot_h;
  // recomputed forward, per-layer slots
  float *Qa, *Phi, *Den, *Rr, *X1, *N1, *QKV, *LSE, *Att, *Y, *N2, *GU, *U, *H;
  // write side, per-layer slots
  float *VKB, *PhiM, *Sc, *Gm, *Cw, *Vb, *CB, *Wv, *Coef, *VKBbar, *PhiBarM;
  // adjoints, per-layer slots
  float *Srow, *dAtt, *Dsum, *dQKV, *N2bar, *Ybar, *Ubar, *GUbar, *N1bar, *X1bar, *XS, *Dbar, *PhiBar, *QaBar;
  // adjoints handed between diagonals (ping-pong by parity), layer-0 input adjoints
  float *Hbar[2], *SA[2], *Sz[2], *XB0;
  // gradient accumulators (fused layouts as the weights)
  float *dWqkv, *dWo, *dWgu, *dWd, *daWq, *dWw, *dg1, *dg2, *dgf;
  // split-K partial products
  float* Part;
  long long part_cap;
  int num_sms;
};

struct BwRun {
  const BwView& v;
  cudaStream_t st;
  long long launches = 0;
  double flops = 0;  // algorithmic FLOPs of the products and of attention
  // the current diagonal
  int l0 = 0, g = 0, alt_l = -1;
  long long s0 = 0;

  // per-layer slot of `size` floats, saved per (layer, segment), per-layer weight
  CellPtr slot(float* p, long long size) const { return CellPtr{p, size, 0}; }
  CellPtr saved(float* p, long long size) const { return CellPtr{p, v.n_seg * size, size}; }
  static BwMat rowm(CellPtr p, long long ld) { return BwMat{p, ld, 0}; }
  static BwMat colm(CellPtr p, long long ld) { return BwMat{p, ld, 1}; }

  armt_status check() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ARMT_ERR_CUDA, std::string("backward launch: ") + cudaGetErrorString(e));
    ++launches;
    return ARMT_OK;
  }

  // C = E + alpha rs (A B) over the cells [gl0, gl0 + gg) of the diagonal
  armt_status gemm(BwMat A, BwMat B, BwMat C, BwMat E, int M, int N, int K, float alpha = 1.f,
                   CellPtr rs = CellPtr(), int rs_div = 0, int gl0 = -1, int gg = -1) {
    BwGemm p;
    p.A = A;
    p.B = B;
    p.C = C;
    p.E = E;
    p.rs = rs;
    p.rs_div = rs_div;
    p.alpha = alpha;
    p.M = M;
    p.N = N;
    p.K = K;
    p.l0 = gl0 < 0 ? l0 : gl0;
    p.s0 = s0 - (p.l0 - l0);
    const int groups = gg < 0 ? g : gg;
    if (M == 0 || N == 0 || groups == 0) return ARMT_OK;
    flops += 2.0 * M * N * K * groups;
    p.groups = groups;
    // partial products of a split K go to scratch and are summed in order by a second kernel
    const BwGemmPlan plan = bw_gemm_plan(M, N, K, groups, v.num_sms, v.part_cap);
    const int bm = plan.bm;
    if (plan.ksplit > 1) {
      p.kchunk = plan.kchunk;
      p.ksplit = plan.ksplit;
      p.part = v.Part;
    }
    const dim3 grid((N + bm - 1) / bm, (M + bm - 1) / bm, groups * p.ksplit);
    if (bm == 128)
      bw_gemm_kernel<128, 128><<<grid, 256, 0, st>>>(p);
    else
      bw_gemm_kernel<64, 64><<<grid, 256, 0, st>>>(p);
    CKS(check());
    if (p.ksplit > 1) {
      const long long mn = (long long)M * N;
      bw_gemm_reduce_kernel<<<dim3((unsigned)((mn + 255) / 256), groups), 256, 0, st>>>(p);
      CKS(check());
    }
    return ARMT_OK;
  }
  dim3 rows_grid(int rows) const { return dim3((unsigned)rows, (unsigned)g); }

  template <int HD>
  armt_status attention(const BwAttn& a, bool forward) {
    const dim3 grid((v.T + 31) / 32, v.Hq, g);
    // causal products of T (T + 1) / 2 row pairs over hd: two in the forward
    // (q k, p v), three for q_bar (q k, o_bar v, s_bar k), four for k_bar and v_bar
    flops += (forward ? 2.0 : 7.0) * v.T * (v.T + 1.0) * v.hd * v.Hq * g;
    if (forward) {
      bw_attn_fwd_kernel<HD><<<grid, 256, bw_attn_fwd_smem(HD), st>>>(a);
      return check();
    }
    bw_attn_dsum_kernel<HD><<<dim3(v.T, g), 128, 0, st>>>(a);
    CKS(check());
    bw_attn_dq_kernel<HD><<<grid, 256, bw_attn_dq_smem(HD), st>>>(a);
    CKS(check());
    bw_attn_dkv_kernel<HD><<<dim3((v.T + 31) / 32, v.Hkv, g), 256, bw_attn_dkv_smem(HD), st>>>(a);
    return check();
  }
  armt_status attention_any(const BwAttn& a, bool forward) {
    if (v.hd == 32) return attention<32>(a, forward);
    if (v.hd == 64) return attention<64>(a, forward);
    return attention<128>(a, forward);
  }

  template <int NT>
  armt_status write_rows(CellPtr Ain, CellPtr Abar, CellPtr AbarIn) {
    const int rpb = 16;  // 4 warps x 4 rows
    const size_t smem = ((size_t)v.M * v.P + (size_t)v.M * WS_NSC) * sizeof(float);
    bw_write_rows_kernel<NT><<<dim3((v.d + rpb - 1) / rpb, g), 128, smem, st>>>(
        Ain, Abar, AbarIn, slot(v.PhiM, (long long)v.M * v.P), slot(v.Sc, (long long)v.M * WS_NSC),
        slot(v.VKB, (long long)v.M * v.nw), slot(v.Cw, (long long)v.M * v.d), slot(v.Vb, (long long)v.M * v.d),
        slot(v.CB, (long long)v.M * v.d), slot(v.Wv, (long long)v.M * v.d), v.M, v.d, v.nw, rpb, l0, s0);
    return check();
  }

  // Every cell of reverse anti-diagonal i.
  armt_status diagonal(long long i) {
    const int L = v.L, d = v.d, T = v.T, P = v.P, k = v.k, M = v.M, S = v.S, F = v.F, Nq = v.Nq;
    const long long n = v.n_seg;
    const int lo = (int)std::max<long long>(0, i - (n - 1)), hi = (int)std::min<long long>(L - 1, i);
    l0 = lo;
    g = hi - lo + 1;
    s0 = i - lo;
    const long long l_last = i - (n - 1);  // layer of the last segment's cell
    const bool short_last = v.last_len < S && l_last >= lo && l_last <= hi;
    alt_l = short_last ? (int)l_last : -1;
    const int cur = bw_in_buf(i), nxt = bw_out_buf(i);
    const long long Td = (long long)T * d;
    const CellPtr none;
    const BwMat no;
    // cell tensors
    const CellPtr XIN = saved(v.Xs, Td), AIN = saved(v.As, (long long)d * P), ZIN = saved(v.zs, P);
    const CellPtr Qa = slot(v.Qa, (long long)T * k), Phi = slot(v.Phi, (long long)T * P), Den = slot(v.Den, T);
    const CellPtr Rr = slot(v.Rr, Td), X1 = slot(v.X1, Td), N1 = slot(v.N1, Td), Y = slot(v.Y, Td),
                  N2 = slot(v.N2, Td), H = slot(v.H, Td);
    const CellPtr QKV = slot(v.QKV, (long long)T * Nq), LSE = slot(v.LSE, (long long)T * v.Hq),
                  Att = slot(v.Att, (long long)T * v.Hq * v.hd);
    const CellPtr GU = slot(v.GU, (long long)T * 2 * F), U = slot(v.U, (long long)T * F);
    // weights per layer
    const CellPtr aWq = slot(v.aWq, (long long)k * d), Wqkv = slot(v.Wqkv, (long long)Nq * d),
                  Wo = slot(v.Wo, (long long)d * v.Hq * v.hd), Wgu = slot(v.Wgu, (long long)2 * F * d),
                  Wd = slot(v.Wd, (long long)d * F), Ww = slot(v.Ww, (long long)v.nw * d);
    const CellPtr g1 = slot(v.g1, d), g2 = slot(v.g2, d);
    // the memory rows of a cell: rows S .. S + M - 1, or last_len .. after a short last segment
    auto mem_rows = [&](float* base) {
      CellPtr c = slot(base, Td);
      c.off = (long long)S * d;
      c.alt_l = alt_l;
      c.alt_add = (long long)(v.last_len - S) * d;
      return c;
    };

    // ---------------------------------------------- recompute the cells --
    CKS(gemm(rowm(XIN, d), colm(aWq, d), rowm(Qa, k), no, T, k, d));
    bw_dpfp_rows_kernel<<<rows_grid(T), 128, 2 * k * sizeof(float), st>>>(Qa, k, ZIN, Phi, Den, k, v.nu,
                                                                         v.assoc_eps, l0, s0);
    CKS(check());
    CKS(gemm(rowm(Phi, P), colm(AIN, P), rowm(Rr, d), no, T, d, P, 1.f, Den, 1));
    bw_add_rows_kernel<<<rows_grid(T), 128, 0, st>>>(XIN, Rr, X1, d, l0, s0);
    CKS(check());
    bw_rmsnorm_rows_kernel<<<rows_grid(T), 128, 0, st>>>(X1, g1, N1, none, d, v.norm_eps, l0, s0);
    CKS(check());
    CKS(gemm(rowm(N1, d), colm(Wqkv, d), rowm(QKV, Nq), no, T, Nq, d));
    bw_rope_rows_kernel<<<rows_grid(T), 128, 0, st>>>(QKV, Nq, (v.Hq + v.Hkv) * v.hd, v.hd, v.cosT, v.sinT, 1,
                                                      l0, s0);
    CKS(check());
    BwAttn at;
    at.QKV = QKV;
    at.O = Att;
    at.LSE = LSE;
    at.dO = slot(v.dAtt, (long long)T * v.Hq * v.hd);
    at.Dsum = slot(v.Dsum, (long long)T * v.Hq);
    at.dQKV = slot(v.dQKV, (long long)T * Nq);
    at.T = T;
    at.Hq = v.Hq;
    at.Hkv = v.Hkv;
    at.ld = Nq;
    at.ldo = v.Hq * v.hd;
    at.scale = 1.0f / sqrtf((float)v.hd);
    at.l0 = l0;
    at.s0 = s0;
    CKS(attention_any(at, true));
    CKS(gemm(rowm(Att, v.Hq * v.hd), colm(Wo, v.Hq * v.hd), rowm(Y, d), rowm(X1, d), T, d, v.Hq * v.hd));
    bw_rmsnorm_rows_kernel<<<rows_grid(T), 128, 0, st>>>(Y, g2, N2, none, d, v.norm_eps, l0, s0);
    CKS(check());
    CKS(gemm(rowm(N2, d), colm(Wgu, d), rowm(GU, 2 * F), no, T, 2 * F, d));
    bw_swiglu_rows_kernel<<<rows_grid(T), 128, 0, st>>>(GU, U, F, l0, s0);
    CKS(check());
    CKS(gemm(rowm(U, F), colm(Wd, F), rowm(H, d), rowm(Y, d), T, d, F));
    const CellPtr VKB = slot(v.VKB, (long long)M * v.nw);
    CKS(gemm(rowm(mem_rows(v.H), d), colm(Ww, d), rowm(VKB, v.nw), no, M, v.nw, d));

    // ---------------------------- adjoint of the output rows (h_bar) --
    const CellPtr HB = slot(v.Hbar[cur], Td);
    if (hi == L - 1) {
      // the last layer's cell: the final RMSNorm of its segment rows
      const int ll = L - 1;
      const long long sl = i - ll;
      if (v.cot_h != nullptr) {
        CellPtr cot{const_cast<float*>(v.cot_h), 0, (long long)S * d};
        const CellPtr gf{v.gf, 0, 0}, dgf{v.dgf, 0, 0};
        const CellPtr Srow = slot(v.Srow, T);
        bw_rmsnorm_bwd_rows_kernel<<<dim3(T, 1), 128, 0, st>>>(H, gf, cot, d, none, HB, Srow, d, v.norm_eps, S,
                                                               alt_l, v.last_len, ll, sl);
        CKS(check());
        bw_gain_grad_kernel<<<dim3((d + 31) / 32, 1), 256, 0, st>>>(H, cot, d, Srow, dgf, d, S, alt_l,
                                                                      v.last_len, ll, sl);
        CKS(check());
      } else {
        CK(cudaMemsetAsync(HB.at(ll, sl), 0, Td * sizeof(float), st));
      }
    }

    // ------------------------------------------- adjoint of the writes --
    {
      const CellPtr PhiM = slot(v.PhiM, (long long)M * P), Sc = slot(v.Sc, (long long)M * WS_NSC),
                    Gm = slot(v.Gm, (long long)M * M), Cw = slot(v.Cw, (long long)M * d),
                    Vb = slot(v.Vb, (long long)M * d), CB = slot(v.CB, (long long)M * d),
                    Wv = slot(v.Wv, (long long)M * d), Coef = slot(v.Coef, (long long)M * M),
                    VKBbar = slot(v.VKBbar, (long long)M * v.nw), PhiBarM = slot(v.PhiBarM, (long long)M * P);
      const CellPtr SAc = slot(v.SA[cur], (long long)d * P), SAn = slot(v.SA[nxt], (long long)d * P);
      const CellPtr Szc = slot(v.Sz[cur], P), Szn = slot(v.Sz[nxt], P);
      const size_t feat_smem = ((size_t)M * 2 * k + (size_t)M * (P + 1)) * sizeof(float);
      bw_write_feat_kernel<<<g, 256, feat_smem, st>>>(VKB, ZIN, PhiM, Sc, Gm, M, k, v.nu, v.assoc_eps, d, v.nw,
                                                      l0, s0);
      CKS(check());
      if (P == 96)
        CKS(write_rows<3>(AIN, SAc, SAn));
      else if (P == 192)
        CKS(write_rows<6>(AIN, SAc, SAn));
      else
        CKS(write_rows<12>(AIN, SAc, SAn));
      bw_write_scalars_kernel<<<g, 256, 0, st>>>(Cw, Vb, CB, Wv, VKB, PhiM, Gm, Sc, Szc, Szn, Coef, VKBbar, M, P,
                                                 d, k, v.nw, l0, s0);
      CKS(check());
      // phi_bar_i = A_bar^T c_i + A_in^T w_i + sum_j Coef_ij phi_j (+ the vector terms below)
      CKS(gemm(rowm(Cw, d), rowm(SAc, P), rowm(PhiBarM, P), no, M, P, d));
      CKS(gemm(rowm(Wv, d), rowm(AIN, P), rowm(PhiBarM, P), rowm(PhiBarM, P), M, P, d));
      CKS(gemm(rowm(Coef, M), rowm(PhiM, P), rowm(PhiBarM, P), rowm(PhiBarM, P), M, P, M));
      DpfpTerms tw;
      tw.c1 = Sc;
      tw.c1off = WS_GAMMA;
      tw.v1 = Szc;
      tw.c2 = Sc;
      tw.c2off = WS_ZETA;
      tw.v2 = ZIN;
      tw.cstride = WS_NSC;
      CellPtr kcols = VKB, kbar = VKBbar;
      kcols.off = d;
      kbar.off = d;
      bw_dpfp_bwd_rows_kernel<<<rows_grid(M), 128, (4 * k + P) * sizeof(float), st>>>(
          kcols, v.nw, PhiBarM, tw, kbar, v.nw, k, v.nu, l0, s0);
      CKS(check());
      // h_bar of the memory rows += VKB_bar Ww;  dWw += VKB_bar^T h_mem
      const CellPtr HBm = mem_rows(v.Hbar[cur]);
      CKS(gemm(rowm(VKBbar, v.nw), rowm(Ww, d), rowm(HBm, d), rowm(HBm, d), M, d, v.nw));
      const CellPtr dWw = slot(v.dWw, (long long)v.nw * d);
      CKS(gemm(colm(VKBbar, v.nw), rowm(mem_rows(v.H), d), rowm(dWw, d), rowm(dWw, d), v.nw, d, M));
    }

    // ------------------------------------------ adjoint of the block --
    const CellPtr Srow = slot(v.Srow, T);
    const CellPtr Ubar = slot(v.Ubar, (long long)T * F), GUbar = slot(v.GUbar, (long long)T * 2 * F);
    const CellPtr N2bar = slot(v.N2bar, Td), Ybar = slot(v.Ybar, Td), N1bar = slot(v.N1bar, Td),
                  X1bar = slot(v.X1bar, Td);
    // h = y + u Wd^T
    CKS(gemm(rowm(HB, d), rowm(Wd, F), rowm(Ubar, F), no, T, F, d));
    {
      const CellPtr dWd = slot(v.dWd, (long long)d * F);
      CKS(gemm(colm(HB, d), rowm(U, F), rowm(dWd, F), rowm(dWd, F), d, F, T));
    }
    bw_swiglu_bwd_rows_kernel<<<rows_grid(T), 128, 0, st>>>(GU, Ubar, GUbar, F, l0, s0);
    CKS(check());
    {
      const CellPtr dWgu = slot(v.dWgu, (long long)2 * F * d);
      CKS(gemm(colm(GUbar, 2 * F), rowm(N2, d), rowm(dWgu, d), rowm(dWgu, d), 2 * F, d, T));
    }
    CKS(gemm(rowm(GUbar, 2 * F), rowm(Wgu, d), rowm(N2bar, d), no, T, d, 2 * F));
    // n2 = RMSNorm(y): y_bar = h_bar + its adjoint
    bw_rmsnorm_bwd_rows_kernel<<<rows_grid(T), 128, 0, st>>>(Y, g2, N2bar, d, HB, Ybar, Srow, d, v.norm_eps, T,
                                                             -1, 0, l0, s0);
    CKS(check());
    bw_gain_grad_kernel<<<dim3((d + 31) / 32, g), 256, 0, st>>>(Y, N2bar, d, Srow, slot(v.dg2, d), d, T, -1, 0,
                                                                  l0, s0);
    CKS(check());
    // y = x1 + att Wo^T
    CKS(gemm(rowm(Ybar, d), rowm(Wo, v.Hq * v.hd), rowm(at.dO, v.Hq * v.hd), no, T, v.Hq * v.hd, d));
    {
      const CellPtr dWo = slot(v.dWo, (long long)d * v.Hq * v.hd);
      CKS(gemm(colm(Ybar, d), rowm(Att, v.Hq * v.hd), rowm(dWo, v.Hq * v.hd), rowm(dWo, v.Hq * v.hd), d,
               v.Hq * v.hd, T));
    }
    CKS(attention_any(at, false));
    bw_rope_rows_kernel<<<rows_grid(T), 128, 0, st>>>(at.dQKV, Nq, (v.Hq + v.Hkv) * v.hd, v.hd, v.cosT, v.sinT, -1,
                                                      l0, s0);
    CKS(check());
    {
      const CellPtr dWqkv = slot(v.dWqkv, (long long)Nq * d);
      CKS(gemm(colm(at.dQKV, Nq), rowm(N1, d), rowm(dWqkv, d), rowm(dWqkv, d), Nq, d, T));
    }
    CKS(gemm(rowm(at.dQKV, Nq), rowm(Wqkv, d), rowm(N1bar, d), no, T, d, Nq));
    bw_rmsnorm_bwd_rows_kernel<<<rows_grid(T), 128, 0, st>>>(X1, g1, N1bar, d, Ybar, X1bar, Srow, d, v.norm_eps, T,
                                                             -1, 0, l0, s0);
    CKS(check());
    bw_gain_grad_kernel<<<dim3((d + 31) / 32, g), 256, 0, st>>>(X1, N1bar, d, Srow, slot(v.dg1, d), d, T, -1, 0,
                                                                  l0, s0);
    CKS(check());

    // -------------------------------------------- adjoint of the read --
    {
      const CellPtr XS = slot(v.XS, Td), Dbar = slot(v.Dbar, T), PhiBar = slot(v.PhiBar, (long long)T * P),
                    QaBar = slot(v.QaBar, (long long)T * k);
      const CellPtr SAn = slot(v.SA[nxt], (long long)d * P), Szn = slot(v.Sz[nxt], P);
      bw_read_rows_kernel<<<rows_grid(T), 128, 0, st>>>(X1bar, Rr, Den, XS, Dbar, d, l0, s0);
      CKS(check());
      CKS(gemm(colm(XS, d), rowm(Phi, P), rowm(SAn, P), rowm(SAn, P), d, P, T));
      CKS(gemm(rowm(Dbar, T), rowm(Phi, P), rowm(Szn, P), rowm(Szn, P), 1, P, T));
      CKS(gemm(rowm(XS, d), rowm(AIN, P), rowm(PhiBar, P), no, T, P, d));
      DpfpTerms tr;  // phi_bar + D_bar z_in
      tr.c1 = Dbar;
      tr.v1 = ZIN;
      tr.cstride = 1;
      bw_dpfp_bwd_rows_kernel<<<rows_grid(T), 128, (4 * k + P) * sizeof(float), st>>>(
          Qa, k, PhiBar, tr, QaBar, k, k, v.nu, l0, s0);
      CKS(check());
      {
        const CellPtr daWq = slot(v.daWq, (long long)k * d);
        CKS(gemm(colm(QaBar, k), rowm(XIN, d), rowm(daWq, d), rowm(daWq, d), k, d, T));
      }
      // x_bar = x1_bar + q_bar Wq_a: to cell (l-1, s), or the layer-0 input adjoints
      if (hi >= 1) {
        const int a0 = std::max(lo, 1);
        CellPtr out = slot(v.Hbar[nxt], Td);
        out.off = -Td;
        CKS(gemm(rowm(QaBar, k), rowm(aWq, d), rowm(out, d), rowm(X1bar, d), T, d, k, 1.f, CellPtr(), 0, a0,
                 hi - a0 + 1));
      }
      if (lo == 0) {
        CellPtr out{v.XB0, 0, Td};
        CKS(gemm(rowm(QaBar, k), rowm(aWq, d), rowm(out, d), rowm(X1bar, d), T, d, k, 1.f, CellPtr(), 0, 0, 1));
      }
    }
    return ARMT_OK;
  }
};

}  // namespace armt
