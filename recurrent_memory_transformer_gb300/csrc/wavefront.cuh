// Persistent wavefront over the layer x segment grid (fp32 model).
//
// Summary page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
// Transformers for Long Contexts", section 二: cell (l, s) needs only cell
// (l-1, s) (its input rows) and cell (l, s-1) (layer l's memory state), so
// every cell with l + s = i can run in step i.  The diagonal schedule
// realises that with one grouped launch per kernel per step, which puts a
// grid-wide barrier between every two kernels of a step and between steps.
// Here one persistent, cooperative launch runs the whole forward instead, and
// the dependencies are tracked on the device:
//   * the work is cut into tasks -- one thread block's share of one stage of
//     one cell (the blocks the separate kernels would launch) -- listed in a
//     dependency order: step, then stage, then cell, then block;
//   * a block takes the next task from a global counter, waits (bounded)
//     until the completion counters of the (cell, stage) pairs the task reads
//     from reach their block counts, runs the block, and adds one to its own
//     (cell, stage) counter;
//   * a stage waits only for what it reads: the previous stage of its cell;
//     the first stage of a cell also for the cell one layer down (its input
//     rows) and the previous cell of its layer (the state); the down
//     projection, which overwrites layer l+1's input slot, also for the
//     previous segment's readers of that slot.
// No stage waits for the whole grid, so a cell can run ahead of the rest of
// its diagonal wherever the recurrence allows.  Tasks are taken in list
// order and every dependency points to an earlier task, so the oldest
// unfinished task can always run: no deadlock with all blocks co-resident
// (the cooperative launch guarantees that).  Every wait is bounded; a
// timeout records DEV_TIMEOUT_DEP and the remaining tasks give up at once.
// The blocks run the same device code (the *_block functions) on the same
// data as the separate kernels, so the result is bit-identical to the
// diagonal and sequential schedules.
#pragma once

#include <vector>

#include "common.cuh"
#include "epilogues.cuh"
#include "kernels.cuh"

namespace armt {

constexpr int DEV_TIMEOUT_DEP = 5;  // a wavefront task waited too long for a dependency

enum WfStage : int {
  WF_GATHER = 0, WF_QGEMM, WF_QEPI, WF_PHI, WF_RGEMM, WF_REPI, WF_QKVGEMM, WF_QKVEPI, WF_ATTN,
  WF_OGEMM, WF_OEPI, WF_GUGEMM, WF_GUEPI, WF_DGEMM, WF_DEPI, WF_WGEMM, WF_WEPI, WF_FEAT, WF_UPD,
  WF_FINAL, WF_NSTAGE
};

// One fp32 product C = A B^T of a stage (the gemm_simt_f32 block arguments
// of cell layer l, with g_first = l).
struct WfGemm {
  const float* A;
  long long a_gs;
  int lda;
  const float* B;
  long long b_gs;
  int N, K, rows, nbx;  // nbx: 64-wide column blocks
  SimtAMap am;
};

struct WfTask {
  int stage, l, s, block;
  int dep[3];   // counter indices (-1: none)
  int need[3];  // block counts those counters must reach
  int self;     // this task's counter
};

// Everything the stages read, for the fp32 model with one sequence.
struct WfArgs {
  // model
  const float *embed, *memtok, *gf;
  int T, S, M, d, k, nu, vocab, Hq, Hkv, hd, P, nw, nmax, L;
  float assoc_eps, norm_eps, attn_scale;
  int upd_rows;
  // workspace (batch 1)
  float *X, *Cscr, *Qa, *Phi, *Den, *QKV, *Att, *VKB, *PhiM, *Coef;
  // caller
  const int32_t* tokens;
  int64_t n_tok, n_seg;
  int last_len;
  float *hidden, *A, *z;
  // products, in stage order: query, read, qkv, o, gate-up, down, write
  WfGemm gq, gr, gqkv, go, ggu, gd, gw;
  // epilogues
  EpiStore eq;
  EpiAssocRead<float> er;
  EpiQkvRope<float> eqkv;
  EpiResidual<float> eo, ed;
  EpiSwiGLU<float> egu;
  EpiStore ew;
  // failure handling
  int* err;
  WaitPolicy wp;
};

// Products land in one scratch region of T rows per layer, the same for every
// product of that layer: cells of different layers run at the same time, so
// the region's stride must not depend on the product's row count.
__device__ __forceinline__ void wf_gemm_block(const WfGemm& g, const WfArgs& a, int l, int block,
                                              float* C) {
  const uint3 bid = make_uint3((unsigned)(block % g.nbx), (unsigned)(block / g.nbx), 0u);
  gemm_simt_f32_kernel_block(bid, g.A, g.a_gs, g.lda, g.B, g.b_gs, C, (long long)a.T * a.nmax, a.nmax,
                             g.rows, g.N, g.K, l, g.am);
}

template <class Epi>
__device__ __forceinline__ void wf_epi_block(const WfArgs& a, int l, int row, int N, const Epi& epi) {
  epi_rows_kernel_block<Epi>(make_uint3((unsigned)row, 0u, 0u), a.Cscr, (long long)a.T * a.nmax, a.nmax, N, l,
                             epi);
}

template <int HD>
__device__ __forceinline__ void wf_run(const WfTask& t, const WfArgs& a) {
  const int l = t.l, b = t.block;
  const int64_t s = t.s;
  const bool last = s == a.n_seg - 1;
  switch (t.stage) {
    case WF_GATHER:
      embed_gather_kernel_block<float>(make_uint3((unsigned)b, 0u, 0u), a.tokens + s * a.S, a.n_tok, a.embed,
                                       a.memtok, a.X, a.X, a.T, last ? a.last_len : a.S, a.M, a.d, a.vocab, 0);
      break;
    case WF_QGEMM: wf_gemm_block(a.gq, a, l, b, a.Cscr); break;
    case WF_QEPI: wf_epi_block(a, l, b, a.k, a.eq); break;
    case WF_PHI:
      assoc_phi_kernel_block<float>(make_uint3((unsigned)b, 0u, 0u), a.Qa, a.z, a.Phi, a.Den, a.T, a.k, a.nu,
                                    a.assoc_eps, l, a.T, 1);
      break;
    case WF_RGEMM: wf_gemm_block(a.gr, a, l, b, a.Cscr); break;
    case WF_REPI: wf_epi_block(a, l, b, a.d, a.er); break;
    case WF_QKVGEMM: wf_gemm_block(a.gqkv, a, l, b, a.Cscr); break;
    case WF_QKVEPI: wf_epi_block(a, l, b, a.gqkv.N, a.eqkv); break;
    case WF_ATTN: {
      const int nqt = (a.T + 63) / 64;
      attn_simt_kernel_block<float, HD>(make_uint3((unsigned)(b % nqt), (unsigned)(b / nqt), 0u), a.QKV, a.Att,
                                        a.T, a.Hq, a.Hkv, a.attn_scale, l);
      break;
    }
    case WF_OGEMM: wf_gemm_block(a.go, a, l, b, a.Cscr); break;
    case WF_OEPI: wf_epi_block(a, l, b, a.d, a.eo); break;
    case WF_GUGEMM: wf_gemm_block(a.ggu, a, l, b, a.Cscr); break;
    case WF_GUEPI: wf_epi_block(a, l, b, a.ggu.N, a.egu); break;
    case WF_DGEMM: wf_gemm_block(a.gd, a, l, b, a.Cscr); break;
    case WF_DEPI: wf_epi_block(a, l, b, a.d, a.ed); break;
    case WF_WGEMM: {
      WfGemm g = a.gw;  // the write reads the memory rows, after a short last segment from last_len
      if (last && a.last_len < a.S) g.am.row0 = a.last_len;
      wf_gemm_block(g, a, l, b, a.Cscr);
      break;
    }
    case WF_WEPI: wf_epi_block(a, l, b, a.nw, a.ew); break;
    case WF_FEAT:
      assoc_write_feat_kernel_block(make_uint3(0u, 0u, 0u), a.VKB, a.z, a.PhiM, a.Coef, a.M, a.k, a.nu,
                                    a.assoc_eps, a.d, a.nw, l);
      break;
    case WF_UPD: {
      const uint3 bid = make_uint3((unsigned)b, 0u, 0u);
      switch (a.P / 32) {
        case 3:
          assoc_write_update_kernel_block<float, 3>(bid, a.VKB, a.nw, a.PhiM, a.Coef, a.A, a.A, a.M, a.d, a.upd_rows,
                                                    l, 0);
          break;
        case 6:
          assoc_write_update_kernel_block<float, 6>(bid, a.VKB, a.nw, a.PhiM, a.Coef, a.A, a.A, a.M, a.d, a.upd_rows,
                                                    l, 0);
          break;
        default:
          assoc_write_update_kernel_block<float, 12>(bid, a.VKB, a.nw, a.PhiM, a.Coef, a.A, a.A, a.M, a.d,
                                                     a.upd_rows, l, 0);
      }
      break;
    }
    case WF_FINAL:
      rmsnorm_kernel_block<float>(make_uint3((unsigned)b, 0u, 0u), a.X + (long long)a.L * a.T * a.d,
                                  (long long)a.T * a.d, a.gf, 0, a.hidden + s * a.S * (long long)a.d,
                                  a.n_tok * (long long)a.d, a.d, a.norm_eps, 0);
      break;
  }
}

// The persistent kernel: 256 threads per block, the block size of every
// separate kernel whose result depends on it (the feature kernel's
// denominator sum); the others' results do not depend on the block size
// (per-group epilogues, per-row updates).
template <int HD>
__global__ void __launch_bounds__(256) wavefront_kernel(const WfTask* __restrict__ tasks, int n_tasks,
                                                        int* next, int* counters, const WfArgs a) {
  __shared__ int s_task, s_ok;
  for (;;) {
    if (threadIdx.x == 0) s_task = atomicAdd(next, 1);
    __syncthreads();
    const int ti = s_task;
    if (ti >= n_tasks) break;
    const WfTask t = tasks[ti];
    if (threadIdx.x == 0) {
      // bounded wait for the dependencies; give up at once after an error
      bool ok = *reinterpret_cast<volatile int*>(a.err) == 0;
      const uint64_t t0 = global_timer_ns();
      for (int q = 0; ok && q < 3; ++q) {
        if (t.dep[q] < 0) continue;
        const volatile int* c = counters + t.dep[q];
        for (uint32_t it = 0; *c < t.need[q]; ++it) {
          if ((it & 63u) == 63u) {
            if (*reinterpret_cast<volatile int*>(a.err) != 0) { ok = false; break; }
            if (global_timer_ns() - t0 > a.wp.limit_ns) {
              atomicCAS(a.err, 0, DEV_TIMEOUT_DEP);
              ok = false;
              break;
            }
          }
        }
      }
      s_ok = ok;
    }
    __syncthreads();
    __threadfence();  // acquire: the dependencies' writes are visible to every thread below
    if (s_ok) {
      wf_run<HD>(t, a);
      __threadfence();  // release: this block's writes before its count
      __syncthreads();
      // test hook: from task stall_after on, completions are not counted, so
      // the tasks depending on them wait until their limit runs out
      if (threadIdx.x == 0 && (a.wp.stall_after < 0 || ti < a.wp.stall_after)) atomicAdd(counters + t.self, 1);
    }
    __syncthreads();  // s_task / s_ok are rewritten next
  }
}

// Blocks per cell of each stage (0: the stage does not apply to this layer).
struct WfShape {
  int blocks[WF_NSTAGE];
};

inline WfShape wf_shape(const WfArgs& a, int l, int n_rows_final) {
  WfShape s{};
  auto gb = [](const WfGemm& g) { return g.nbx * ((g.rows + 63) / 64); };
  s.blocks[WF_GATHER] = l == 0 ? a.T : 0;
  s.blocks[WF_QGEMM] = gb(a.gq);
  s.blocks[WF_QEPI] = a.T;
  s.blocks[WF_PHI] = a.T;
  s.blocks[WF_RGEMM] = gb(a.gr);
  s.blocks[WF_REPI] = a.T;
  s.blocks[WF_QKVGEMM] = gb(a.gqkv);
  s.blocks[WF_QKVEPI] = a.T;
  s.blocks[WF_ATTN] = ((a.T + 63) / 64) * a.Hq;
  s.blocks[WF_OGEMM] = gb(a.go);
  s.blocks[WF_OEPI] = a.T;
  s.blocks[WF_GUGEMM] = gb(a.ggu);
  s.blocks[WF_GUEPI] = a.T;
  s.blocks[WF_DGEMM] = gb(a.gd);
  s.blocks[WF_DEPI] = a.T;
  s.blocks[WF_WGEMM] = gb(a.gw);
  s.blocks[WF_WEPI] = a.M;
  s.blocks[WF_FEAT] = 1;
  s.blocks[WF_UPD] = (a.d + a.upd_rows - 1) / a.upd_rows;
  s.blocks[WF_FINAL] = l == a.L - 1 ? n_rows_final : 0;
  return s;
}

// The task list of a forward over n_seg segments: step-major, then stage,
// then cell, then block -- a topological order of the dependencies below.
inline std::vector<WfTask> wf_tasks(const WfArgs& a, int64_t n_seg) {
  const int L = a.L;
  auto ctr = [&](int l, int64_t s, int st) { return (int)(((int64_t)l * n_seg + s) * WF_NSTAGE + st); };
  auto shape = [&](int l, int64_t s) { return wf_shape(a, l, s == n_seg - 1 ? a.last_len : a.S); };
  std::vector<WfTask> out;
  for (int64_t i = 0; i < L + n_seg - 1; ++i) {
    const int lo = (int)std::max<int64_t>(0, i - n_seg + 1), hi = (int)std::min<int64_t>(L - 1, i);
    for (int st = 0; st < WF_NSTAGE; ++st) {
      for (int l = lo; l <= hi; ++l) {
        const int64_t s = i - l;
        const WfShape sh = shape(l, s);
        if (sh.blocks[st] == 0) continue;
        WfTask t;
        t.stage = st;
        t.l = l;
        t.s = (int)s;
        t.self = ctr(l, s, st);
        for (int q = 0; q < 3; ++q) {
          t.dep[q] = -1;
          t.need[q] = 0;
        }
        int nd = 0;
        auto add = [&](int dl, int64_t ds, int dst) {
          t.dep[nd] = ctr(dl, ds, dst);
          t.need[nd] = shape(dl, ds).blocks[dst];
          ++nd;
        };
        // the previous stage of this cell that runs (stages that do not apply
        // to this layer are skipped)
        int prev = st - 1;
        while (prev >= 0 && sh.blocks[prev] == 0) --prev;
        const bool first = prev < 0;
        if (st == WF_FINAL) {
          add(l, s, WF_DEPI);  // the final norm reads the last layer's output rows
        } else if (!first) {
          add(l, s, prev);
        }
        if (first) {
          if (s > 0) add(l, s - 1, WF_UPD);  // layer l's state (and its workspace) is free
          if (l > 0) add(l - 1, s, WF_DEPI);  // this cell's input rows
        }
        if (st == WF_DEPI) {
          // the down projection overwrites layer l+1's input slot: the
          // previous segment's readers of it must be done
          if (l + 1 < L && s > 0) add(l + 1, s - 1, WF_REPI);
          if (l + 1 == L && s > 0) add(l, s - 1, WF_FINAL);
        }
        for (int b = 0; b < sh.blocks[st]; ++b) {
          t.block = b;
          out.push_back(t);
        }
      }
    }
  }
  return out;
}

}  // namespace armt
