// C ABI, model state and the two cell schedules of the ARMT forward pass.
//
// Summary page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
// Transformers for Long Contexts":
//   section 二  cell (l, s) depends on (l-1, s) and (l, s-1) only, so every
//             cell with l + s = i runs in grouped step i (n_layers +
//             n_segments - 1 steps in all);
//   section 三  all layers become one grouped layer: stacked weights,
//             grouped matrix products with one preallocated output tensor
//             addressed per group, stacked norm gains, the rest batched.
// The cells of step i are the contiguous layer range
//   [max(0, i - n + 1), min(L - 1, i)],
// so every kernel of a step takes (first layer, layer count) and indexes all
// per-layer tensors -- weights, activations, memory -- by layer.  Buffers are
// per layer: layer l's input slot X[l] is written by cell (l-1, s+1) in the
// same step in which cell (l, s) reads it, but every read of X[l] in a step
// (associative query and read) is enqueued before the down projection that
// overwrites it, so one slot per layer suffices.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <type_traits>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/armt.h"
#include "common.cuh"
#include "epilogues.cuh"
#include "attn_tc.cuh"
#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "kernels.cuh"
#include "schedule.h"
#include "wavefront.cuh"

using namespace armt;

// ----------------------------------------------------------- errors --

static thread_local std::string g_last_error;

static armt_status fail(armt_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

namespace armt {
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace armt

#define CK(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) {                                                              \
      return fail(e_ == cudaErrorMemoryAllocation ? ARMT_ERR_OOM : ARMT_ERR_CUDA,         \
                  std::string(#call) + ": " + cudaGetErrorString(e_));                    \
    }                                                                                     \
  } while (0)

#define CKS(expr)                   \
  do {                              \
    armt_status s_ = (expr);        \
    if (s_ != ARMT_OK) return s_;   \
  } while (0)

// the backward's host plan reports through fail / CK / CKS
#include "backward_plan.cuh"

// --------------------------------------------------------- TMA maps --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

namespace armt {
bool encode_tmap_bf16_3d(CUtensorMap* map, const void* base, int K, int rows, int layers,
                         int box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (K * 2) % 16 != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)layers};
  cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace armt

// ------------------------------------------------------- allocation --

static long long alloc_cap_bytes() {
  const char* s = getenv("ARMT_ALLOC_CAP_BYTES");  // test hook: simulated device memory limit
  return s ? atoll(s) : -1;
}

struct DevAllocs {
  std::vector<void*> ptrs;
  long long total = 0;
  armt_status alloc(void** p, size_t bytes) {
    const long long cap = alloc_cap_bytes();
    if (cap >= 0 && total + (long long)bytes > cap)
      return fail(ARMT_ERR_OOM, "allocation cap exceeded (" + std::to_string(total + bytes) +
                                    " > " + std::to_string(cap) + " bytes)");
    cudaError_t e = cudaMalloc(p, bytes < 256 ? 256 : bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(ARMT_ERR_OOM, std::string("cudaMalloc: ") + cudaGetErrorString(e));
    }
    ptrs.push_back(*p);
    total += (long long)bytes;
    return ARMT_OK;
  }
  template <typename T>
  armt_status alloc_n(T** p, size_t n) {
    return alloc(reinterpret_cast<void**>(p), n * sizeof(T));
  }
  void free_all() {
    for (void* p : ptrs) cudaFree(p);
    ptrs.clear();
    total = 0;
  }
};

template <typename T>
__global__ void to_f32_kernel(const T* __restrict__ src, float* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = ld_as_f32(src + i);
}

// ------------------------------------------------------------ model --

struct ModelBase {
  armt_config cfg{};
  int device = 0, num_sms = 148;
  DevAllocs mem;
  long long weight_bytes = 0;  // part of mem.total holding the weights
  int* d_err = nullptr;
  WaitPolicy wp;  // refreshed from the environment at every public call
  // profiling: launches of the classes in prof_mask get an event pair
  bool profiling = false;
  uint32_t prof_mask = 0;
  // tracing: NVTX ranges around every step (armt_set_tracing)
  bool tracing = false;
  void trace_push(const char* what, long long i, int lo, int hi) const {
    if (!tracing) return;
    char name[96];
    std::snprintf(name, sizeof(name), "armt %s %lld (layers %d-%d)", what, i, lo, hi);
    nvtxRangePushA(name);
  }
  void trace_pop() const {
    if (tracing) nvtxRangePop();
  }
  bool prof_open = false;
  std::vector<cudaEvent_t> ev_start, ev_stop;
  std::vector<int> ev_class;
  size_t ev_used = 0;
  // host-buffer staging (armt_forward_host)
  int32_t* st_tokens = nullptr;
  float *st_hidden = nullptr, *st_A = nullptr, *st_z = nullptr;
  size_t st_tokens_n = 0, st_hidden_n = 0;
  // Results leave for the host while the forward still runs: once the
  // last-layer cell of a segment is done its hidden rows are final, and once
  // layer l has run its last cell its state is final.  forward() reports that
  // progress after every step; sink_progress() then queues the device-to-host
  // copies of what became final on a second stream (copy_stream), ordered
  // after the step by one event.  Set only inside armt_forward_host.
  struct HostSink {
    float *h_hidden, *h_A, *h_z;              // host destinations
    const float *d_hidden, *d_A, *d_z;        // device sources (the staging buffers)
    int64_t rows_done, rows_total;            // hidden rows queued / to queue
    int layers_done;                          // layers whose state is queued
    int64_t chunk_rows;                       // queue hidden rows in chunks of at least this
  };
  HostSink* sink = nullptr;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t copy_event = nullptr;

  virtual ~ModelBase() {
    for (cudaEvent_t e : ev_start) cudaEventDestroy(e);
    for (cudaEvent_t e : ev_stop) cudaEventDestroy(e);
    if (copy_stream) cudaStreamDestroy(copy_stream);
    if (copy_event) cudaEventDestroy(copy_event);
    if (st_tokens) cudaFree(st_tokens);
    if (st_hidden) cudaFree(st_hidden);
    if (st_A) cudaFree(st_A);
    if (st_z) cudaFree(st_z);
    mem.free_all();
  }
  virtual armt_status create(const armt_weights* w, cudaStream_t st) = 0;
  // n_tok tokens per sequence, nb sequences ([nb][n_tok] tokens, [nb][n_tok][d]
  // hidden states, state [L][nb][d][P] and [L][nb][P]).
  virtual armt_status forward(const int32_t* tokens, int64_t n_tok, int nb, float* hidden, float* A,
                              float* z, int mem_in_valid, int schedule, cudaStream_t st) = 0;
  virtual long long batch_workspace_bytes() const = 0;
  virtual armt_status forward_full(const int32_t* tokens, int64_t T, float* hidden,
                                   cudaStream_t st) = 0;
  virtual long long full_workspace_bytes() const = 0;
  virtual armt_status lm_head(const float* hidden, int64_t n_rows, const void* w_head, float* logits,
                              cudaStream_t st) = 0;
  // Gradients of <hidden, cot_h> + <A, cot_A> + <z, cot_z> for one sequence
  // of n_tok tokens (armt_backward).
  virtual armt_status backward(const int32_t* tokens, int64_t n_tok, const float* A0, const float* z0,
                               const float* cot_h, const float* cot_A, const float* cot_z, float* hidden,
                               float* A, float* z, const armt_grads& g, cudaStream_t st) = 0;
  virtual long long backward_workspace_bytes() const = 0;
  long long bw_launches = 0;  // kernel launches of the last backward
  double bw_flops = 0;        // and its algorithmic FLOPs (products and attention)

  int rows() const { return cfg.seg_len + cfg.n_mem; }

  // Queues the copies of everything that is final after a step: hidden rows
  // [rows_done, rows_final) and the states of layers [layers_done,
  // layers_final) (single sequence: the state is [L][d][P], [L][P]).
  armt_status sink_progress(int64_t rows_final, int layers_final, cudaStream_t st) {
    HostSink& k = *sink;
    const bool last = rows_final >= k.rows_total && layers_final >= cfg.n_layers;
    const bool rows_due = rows_final - k.rows_done >= k.chunk_rows || (last && rows_final > k.rows_done);
    const bool layers_due = layers_final > k.layers_done;
    if (!rows_due && !layers_due) return ARMT_OK;
    CK(cudaEventRecord(copy_event, st));
    CK(cudaStreamWaitEvent(copy_stream, copy_event, 0));
    const size_t d = cfg.d_model, P = phi_dim();
    if (rows_due) {
      CK(cudaMemcpyAsync(k.h_hidden + k.rows_done * d, k.d_hidden + k.rows_done * d,
                         (size_t)(rows_final - k.rows_done) * d * sizeof(float), cudaMemcpyDeviceToHost,
                         copy_stream));
      k.rows_done = rows_final;
    }
    if (layers_due) {
      const size_t l0 = (size_t)k.layers_done, nl = (size_t)(layers_final - k.layers_done);
      CK(cudaMemcpyAsync(k.h_A + l0 * d * P, k.d_A + l0 * d * P, nl * d * P * sizeof(float),
                         cudaMemcpyDeviceToHost, copy_stream));
      CK(cudaMemcpyAsync(k.h_z + l0 * P, k.d_z + l0 * P, nl * P * sizeof(float),
                         cudaMemcpyDeviceToHost, copy_stream));
      k.layers_done = layers_final;
    }
    return ARMT_OK;
  }
  int phi_dim() const { return 2 * cfg.key_dim * cfg.dpfp_nu; }
  int n_qkv() const { return (cfg.n_q_heads + 2 * cfg.n_kv_heads) * cfg.head_dim; }

  // Kernel launches of one step covering layers [lo, hi].
  int64_t step_launches(int lo, int hi) const {
    const int per_gemm = cfg.dtype == ARMT_BF16 ? 1 : 2;
    int64_t n = 0;
    if (lo == 0) n += 1;                    // layer-0 input gather
    n += per_gemm + (per_gemm == 1 ? 0 : 1) + per_gemm;  // query GEMM (+ phi on the fp32 path), read GEMM
    n += per_gemm + 1 + per_gemm;           // QKV GEMM, attention, O GEMM (norms fused)
    n += per_gemm + per_gemm;               // gate-up GEMM, down GEMM
    n += per_gemm + 2;                      // delta-rule write: projection GEMM, z, A rows
    if (hi == cfg.n_layers - 1) n += 1;     // final norm
    return n;
  }
  int64_t launches(int64_t n_seg, int schedule, int mem_in_valid) const {
    const int L = cfg.n_layers;
    int64_t total = (mem_in_valid && cfg.dtype == ARMT_BF16) ? 1 : 0;  // state copy
    if (schedule == ARMT_SCHEDULE_WAVEFRONT) return total + 1;     // one persistent launch
    if (schedule == ARMT_SCHEDULE_DIAGONAL) {
      for (int64_t i = 0; i < diagonal_steps(L, n_seg); ++i) {
        const CellRange c = diagonal_step(i, L, n_seg);
        total += step_launches(c.lo, c.hi);
      }
    } else {
      for (int64_t s = 0; s < n_seg; ++s)
        for (int l = 0; l < L; ++l) total += step_launches(l, l);
    }
    return total;
  }

  // Event pair around one launch when profiling.
  armt_status prof_begin(int cls, cudaStream_t st) {
    prof_open = profiling && ((prof_mask >> cls) & 1u) != 0;
    if (!prof_open) return ARMT_OK;
    if (ev_used == ev_start.size()) {
      cudaEvent_t a, b;
      CK(cudaEventCreate(&a));
      CK(cudaEventCreate(&b));
      ev_start.push_back(a);
      ev_stop.push_back(b);
      ev_class.push_back(cls);
    }
    ev_class[ev_used] = cls;
    CK(cudaEventRecord(ev_start[ev_used], st));
    return ARMT_OK;
  }
  armt_status prof_end(cudaStream_t st) {
    if (!prof_open) return ARMT_OK;
    prof_open = false;
    CK(cudaEventRecord(ev_stop[ev_used], st));
    ++ev_used;
    return ARMT_OK;
  }
};

struct armt_model {
  ModelBase* impl;
};

template <typename WT>
struct Model : ModelBase {
  static constexpr bool kTC = sizeof(WT) == 2;  // bf16: tensor-core GEMMs
  typedef WT AT;                               // activation dtype of GEMM operands
  // attention operands (q, k, v): fp16 on the tensor-core path -- they are
  // activations, not weights, so they may take the 16-bit type with the
  // longer mantissa at the same tensor-core rate; fp32 on the fp32 path
  typedef std::conditional_t<kTC, f16, float> QT;
  // epilogue functors: staged (lanes across columns) on the tensor-core
  // path, thread-per-row on the fp32 path
  using FStore = std::conditional_t<kTC, SEpiStore, EpiStore>;
  using FRead = std::conditional_t<kTC, SEpiAssocRead<AT>, EpiAssocRead<AT>>;
  using FQkv = std::conditional_t<kTC, SEpiQkvRope<QT>, EpiQkvRope<QT>>;
  using FRes = std::conditional_t<kTC, SEpiResidual<AT>, EpiResidual<AT>>;
  using FSwi = std::conditional_t<kTC, SEpiSwiGLU<AT>, EpiSwiGLU<AT>>;

  // weights (library layout)
  WT *embed = nullptr, *memtok = nullptr, *Wqkv = nullptr, *Wo = nullptr, *Wgu = nullptr,
     *Wd = nullptr, *aWq = nullptr, *Ww = nullptr;  // Ww: per layer [Wv_a; Wk_a; wbeta_a; 0]
  float *g1 = nullptr, *g2 = nullptr, *gf = nullptr;
  int npart = 0;  // partial sums of squares per row (one per epilogue column tile)
  int nw = 0;  // rows of Ww per layer (d + k + 1 rounded up to the tile width)
  int qkv_ld = 0, t_pad = 0;  // row stride of QKV; padded row count of Vt
  // split precision (ARMT_PRECISION_BF16X2): Nrm, Att, U and Xa hold a bf16
  // low part behind the high one (twice the slots), and the weight GEMMs read
  // both (GemmGroupMap::a_lo_slot)
  bool split = false;
  int nmax = 0;  // widest GEMM output (fp32 scratch row stride)
  // weight tensor maps (bf16 path); the *2 maps have 128-row boxes for CTA-pair tiles
  CUtensorMap tmAWq, tmWqkv, tmWo, tmWgu, tmWd, tmWw, tmWqkv2, tmWo2, tmWgu2, tmWd2;
  // The cell engine's activations for nb sequences run side by side (a
  // batch of requests).  With T = S + M rows per cell and R = nb * T rows per
  // layer, the per-layer tensors are [layer or slot][R][width]: cell b of a
  // layer owns rows [b T, (b + 1) T), so the weight GEMMs see one R-row
  // matrix per layer, while the per-(layer, sequence) tensors -- memory state,
  // attention, write projections -- are addressed as groups l * nb + b of T
  // rows (the same memory, a finer view).
  struct Work {
    int nb = 0;
    float *X = nullptr, *Res = nullptr, *Qa = nullptr, *Den = nullptr, *VKB = nullptr,
          *PhiM = nullptr, *Coef = nullptr, *Cscr = nullptr, *Ssq = nullptr, *cosT = nullptr,
          *sinT = nullptr;
    AT *Xa = nullptr, *Nrm = nullptr, *Att = nullptr, *U = nullptr, *Phi = nullptr, *Aa = nullptr;
    QT *QKV = nullptr, *Vt = nullptr;
    // row views {width, R, layers}; group views {width, T, layers * nb}
    CUtensorMap tmXa, tmNrm, tmAtt, tmU, tmXaW, tmPhi, tmAa, tmQK, tmVt;
  };
  Work w1;             // one sequence: allocated by armt_create
  Work wb;             // armt_forward_batch with nb > 1, sized on first use
  DevAllocs wb_mem;
  size_t upd_smem = 0, feat_smem = 0, attn_smem = 0;
  // full-causal-attention LLaMA over a whole sequence (baseline): one
  // activation slot, grown on demand
  DevAllocs full_mem;
  int64_t full_T = 0;
  // LM head: bf16 copy of a chunk of hidden rows (tensor-core path)
  DevAllocs lm_mem;
  AT* lm_rows = nullptr;
  static constexpr int64_t kLmChunk = 8192;
  float *Xf = nullptr, *Resf = nullptr, *Ssqf = nullptr, *cosF = nullptr, *sinF = nullptr;
  AT *Nrmf = nullptr, *Attf = nullptr, *Uf = nullptr;
  QT *QKVf = nullptr, *Vtf = nullptr;
  CUtensorMap tmNrmf, tmQKf, tmVtf, tmAttf, tmUf;
  // backward (fp32 models): saved cell inputs and entry states, workspace
  struct BwSave {
    float *Xs, *As, *zs;
    int64_t n;
  };
  const BwSave* bw_save = nullptr;  // set while the backward's forward runs
  DevAllocs bw_mem;
  BwView bwv{};
  int64_t bw_n_cap = 0, bw_tok_cap = 0;
  float *bw_hidden = nullptr, *bw_A = nullptr, *bw_z = nullptr;  // forward results nobody asked for
  // bf16 models: fp32 copies of the weight products' weights (the backward's
  // arithmetic is fp32), made on the first backward
  DevAllocs bw_w32_mem;
  float *aWq32 = nullptr, *Wqkv32 = nullptr, *Wo32 = nullptr, *Wgu32 = nullptr, *Wd32 = nullptr,
        *Ww32 = nullptr;
  ~Model() override {
    bw_w32_mem.free_all();
    bw_mem.free_all();
    wf_mem.free_all();
    full_mem.free_all();
    lm_mem.free_all();
    wb_mem.free_all();
  }
  long long full_workspace_bytes() const override { return full_mem.total; }
  long long backward_workspace_bytes() const override { return bw_mem.total + bw_w32_mem.total; }
  long long batch_workspace_bytes() const override { return wb_mem.total; }
  int upd_rows_per_block = 32;
  // persistent wavefront (fp32 models): task list and (cell, stage) counters
  DevAllocs wf_mem;
  WfTask* wf_tasks_d = nullptr;
  int* wf_ctr = nullptr;
  size_t wf_tasks_cap = 0, wf_ctr_cap = 0;
  std::vector<WfTask> wf_tasks_h;  // kept until the next call (the upload reads it)

  armt_status copy_in(void* dst, const void* src, size_t bytes, cudaStream_t st) {
    CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, st));
    return ARMT_OK;
  }

  armt_status gain_to_f32(float** dst, const void* src, size_t n, cudaStream_t st) {
    CKS(mem.alloc_n(dst, n));
    WT* tmp = nullptr;
    CK(cudaMalloc(&tmp, n * sizeof(WT)));
    cudaError_t e = cudaMemcpyAsync(tmp, src, n * sizeof(WT), cudaMemcpyDefault, st);
    if (e == cudaSuccess) {
      to_f32_kernel<WT><<<64, 256, 0, st>>>(tmp, *dst, (long long)n);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(tmp);
    if (e != cudaSuccess) return fail(ARMT_ERR_CUDA, std::string("gain copy: ") + cudaGetErrorString(e));
    return ARMT_OK;
  }

  armt_status create(const armt_weights* w, cudaStream_t st) override {
    const armt_config& c = cfg;
    const size_t L = c.n_layers, d = c.d_model, hd = c.head_dim, F = c.ffn_dim, T = rows();
    const size_t Hq = c.n_q_heads, Hkv = c.n_kv_heads, k = c.key_dim, P = phi_dim();
    const size_t Nq = n_qkv(), es = sizeof(WT);
    // weights
    CKS(mem.alloc_n(&embed, (size_t)c.vocab * d));
    CKS(copy_in(embed, w->embed, (size_t)c.vocab * d * es, st));
    CKS(mem.alloc_n(&memtok, (size_t)c.n_mem * d));
    CKS(copy_in(memtok, w->mem, (size_t)c.n_mem * d * es, st));
    CKS(mem.alloc_n(&Wqkv, L * Nq * d));
    // fused rows: per layer [wq; wk; wv]
    CK(cudaMemcpy2DAsync(Wqkv, Nq * d * es, w->wq, Hq * hd * d * es, Hq * hd * d * es, L,
                         cudaMemcpyDefault, st));
    CK(cudaMemcpy2DAsync(Wqkv + Hq * hd * d, Nq * d * es, w->wk, Hkv * hd * d * es,
                         Hkv * hd * d * es, L, cudaMemcpyDefault, st));
    CK(cudaMemcpy2DAsync(Wqkv + (Hq + Hkv) * hd * d, Nq * d * es, w->wv, Hkv * hd * d * es,
                         Hkv * hd * d * es, L, cudaMemcpyDefault, st));
    CKS(mem.alloc_n(&Wo, L * d * Hq * hd));
    CKS(copy_in(Wo, w->wo, L * d * Hq * hd * es, st));
    // gate/up interleaved in blocks of GU_BLK rows
    CKS(mem.alloc_n(&Wgu, L * 2 * F * d));
    const size_t blk = (size_t)GU_BLK * d * es, nblk = L * F / GU_BLK;
    CK(cudaMemcpy2DAsync(Wgu, 2 * blk, w->w_gate, blk, blk, nblk, cudaMemcpyDefault, st));
    CK(cudaMemcpy2DAsync(reinterpret_cast<char*>(Wgu) + blk, 2 * blk, w->w_up, blk, blk, nblk,
                         cudaMemcpyDefault, st));
    CKS(mem.alloc_n(&Wd, L * d * F));
    CKS(copy_in(Wd, w->w_down, L * d * F * es, st));
    CKS(mem.alloc_n(&aWq, L * k * d));
    CKS(copy_in(aWq, w->a_wq, L * k * d * es, st));
    // write projections stacked per layer: rows [0,d) Wv_a, [d,d+k) Wk_a, d+k wbeta_a
    nw = (int)((d + k + 1 + (kTC ? 255 : 15)) / (kTC ? 256 : 16) * (kTC ? 256 : 16));
    CKS(mem.alloc_n(&Ww, L * (size_t)nw * d));
    CK(cudaMemsetAsync(Ww, 0, L * (size_t)nw * d * es, st));
    CK(cudaMemcpy2DAsync(Ww, (size_t)nw * d * es, w->a_wv, d * d * es, d * d * es, L,
                         cudaMemcpyDefault, st));
    CK(cudaMemcpy2DAsync(Ww + d * d, (size_t)nw * d * es, w->a_wk, k * d * es, k * d * es, L,
                         cudaMemcpyDefault, st));
    CK(cudaMemcpy2DAsync(Ww + (d + k) * d, (size_t)nw * d * es, w->a_wbeta, d * es, d * es, L,
                         cudaMemcpyDefault, st));
    CKS(gain_to_f32(&g1, w->norm1, L * d, st));
    CKS(gain_to_f32(&g2, w->norm2, L * d, st));
    CKS(gain_to_f32(&gf, w->norm_f, d, st));
    weight_bytes = mem.total;
    qkv_ld = kTC ? (int)((Hq + Hkv) * hd) : (int)Nq;
    t_pad = (int)((T + 7) / 8 * 8);
    npart = (int)(kTC ? d / 128 : d / 32);  // one partial per 128 columns (two epilogue halves)
    nmax = (int)std::max(std::max(Nq, d), std::max(2 * F, std::max(k, (size_t)nw)));
    if (kTC && ((Hq + Hkv) * hd) % 256 != 0)
      return fail(ARMT_ERR_UNSUPPORTED, "(Hq + Hkv) * head_dim must be a multiple of 256");
    if (kTC) {
      bool ok = true;
      ok &= encode_tmap_bf16_3d(&tmAWq, aWq, (int)d, (int)k, (int)L, 64);
      ok &= encode_tmap_bf16_3d(&tmWqkv, Wqkv, (int)d, (int)Nq, (int)L, 256);
      ok &= encode_tmap_bf16_3d(&tmWo, Wo, (int)(Hq * hd), (int)d, (int)L, 256);
      ok &= encode_tmap_bf16_3d(&tmWgu, Wgu, (int)d, (int)(2 * F), (int)L, 256);
      ok &= encode_tmap_bf16_3d(&tmWd, Wd, (int)F, (int)d, (int)L, 256);
      // CTA-pair tiles: each CTA loads 128 of a tile's 256 B rows
      ok &= encode_tmap_bf16_3d(&tmWqkv2, Wqkv, (int)d, (int)Nq, (int)L, 128);
      ok &= encode_tmap_bf16_3d(&tmWo2, Wo, (int)(Hq * hd), (int)d, (int)L, 128);
      ok &= encode_tmap_bf16_3d(&tmWgu2, Wgu, (int)d, (int)(2 * F), (int)L, 128);
      ok &= encode_tmap_bf16_3d(&tmWd2, Wd, (int)F, (int)d, (int)L, 128);
      ok &= encode_tmap_bf16_3d(&tmWw, Ww, (int)d, nw, (int)L, 256);
      if (!ok) return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    }
    split = kTC && c.precision == ARMT_PRECISION_BF16X2;
    CKS(alloc_work(w1, 1, mem, st));
    CKS(mem.alloc_n(&d_err, 1));
    CK(cudaMemsetAsync(d_err, 0, sizeof(int), st));
    // kernel configuration
    upd_smem = ((size_t)c.n_mem * P + 2 * c.n_mem) * sizeof(float);
    feat_smem = ((size_t)c.n_mem * 2 * k + (size_t)c.n_mem * (P + 1) + P) * sizeof(float);
    attn_smem = 2 * 64 * hd * sizeof(float);
    CK(cudaFuncSetAttribute(assoc_write_feat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            (int)feat_smem));
    switch (P / 32) {
      case 3: CK(cudaFuncSetAttribute(assoc_write_update_kernel<AT, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)upd_smem)); break;
      case 6: CK(cudaFuncSetAttribute(assoc_write_update_kernel<AT, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)upd_smem)); break;
      case 12: CK(cudaFuncSetAttribute(assoc_write_update_kernel<AT, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)upd_smem)); break;
      default: return fail(ARMT_ERR_UNSUPPORTED, "2 * key_dim * dpfp_nu must be 96, 192 or 384");
    }
    if (hd == 64)
      CK(cudaFuncSetAttribute(attn_simt_kernel<AT, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem));
    else if (hd == 128)
      CK(cudaFuncSetAttribute(attn_simt_kernel<AT, 128>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem));
    CK(cudaStreamSynchronize(st));
    return ARMT_OK;
  }

  // Activations for nb sequences per cell, from `pool`.
  armt_status alloc_work(Work& w, int nb, DevAllocs& pool, cudaStream_t st) {
    const armt_config& c = cfg;
    const size_t L = c.n_layers, d = c.d_model, hd = c.head_dim, F = c.ffn_dim, T = rows();
    const size_t Hq = c.n_q_heads, Hkv = c.n_kv_heads, k = c.key_dim, P = phi_dim();
    const size_t R = (size_t)nb * T, M = c.n_mem;
    w = Work();
    // RoPE tables over the R rows of a layer: row r sits at position r % T
    // (double precision on the host, stored fp32)
    {
      std::vector<float> hc(R * (hd / 2)), hs(R * (hd / 2));
      for (size_t t = 0; t < T; ++t)
        for (size_t i = 0; i < hd / 2; ++i) {
          const double ang = (double)t * std::pow(c.rope_base, -2.0 * (double)i / (double)hd);
          hc[t * (hd / 2) + i] = (float)std::cos(ang);
          hs[t * (hd / 2) + i] = (float)std::sin(ang);
        }
      for (size_t b = 1; b < (size_t)nb; ++b) {
        std::copy(hc.begin(), hc.begin() + T * (hd / 2), hc.begin() + b * T * (hd / 2));
        std::copy(hs.begin(), hs.begin() + T * (hd / 2), hs.begin() + b * T * (hd / 2));
      }
      CKS(pool.alloc_n(&w.cosT, hc.size()));
      CKS(pool.alloc_n(&w.sinT, hs.size()));
      CK(cudaMemcpy(w.cosT, hc.data(), hc.size() * 4, cudaMemcpyHostToDevice));
      CK(cudaMemcpy(w.sinT, hs.data(), hs.size() * 4, cudaMemcpyHostToDevice));
    }
    const size_t halves = split ? 2 : 1;  // split precision: high and low parts
    CKS(pool.alloc_n(&w.X, (L + 1) * R * d));
    if (kTC) {
      CKS(pool.alloc_n(&w.Xa, halves * (L + 1) * R * d));
    } else {
      w.Xa = reinterpret_cast<AT*>(w.X);
    }
    CKS(pool.alloc_n(&w.Res, L * R * d));
    CKS(pool.alloc_n(&w.Nrm, halves * L * R * d));
    // bf16: q|k rows in QKV, v transposed into Vt; fp32: q|k|v rows in QKV
    CKS(pool.alloc_n(&w.QKV, L * R * (size_t)qkv_ld));
    if (kTC) CKS(pool.alloc_n(&w.Vt, L * nb * Hkv * hd * (size_t)t_pad));
    CKS(pool.alloc_n(&w.Att, halves * L * R * Hq * hd));
    CKS(pool.alloc_n(&w.U, halves * L * R * F));
    CKS(pool.alloc_n(&w.Qa, L * R * k));
    CKS(pool.alloc_n(&w.Phi, halves * L * R * P));
    CKS(pool.alloc_n(&w.Den, L * R));
    CKS(pool.alloc_n(&w.Ssq, L * R * (size_t)npart));
    CKS(pool.alloc_n(&w.VKB, L * nb * M * (size_t)nw));
    CKS(pool.alloc_n(&w.PhiM, L * nb * M * P));
    CKS(pool.alloc_n(&w.Coef, L * nb * M * 2));
    if (kTC) CKS(pool.alloc_n(&w.Aa, halves * L * nb * d * P));
    if (!kTC) CKS(pool.alloc_n(&w.Cscr, L * R * (size_t)nmax));
    if (kTC) {
      const int iR = (int)R, iT = (int)T, iL = (int)L, G = (int)L * nb, h = (int)halves;
      bool ok = true;
      ok &= encode_tmap_bf16_3d(&w.tmXa, w.Xa, (int)d, iR, h * (iL + 1), TC_BM);
      ok &= encode_tmap_bf16_3d(&w.tmNrm, w.Nrm, (int)d, iR, h * iL, TC_BM);
      ok &= encode_tmap_bf16_3d(&w.tmAtt, w.Att, (int)(Hq * hd), iR, h * iL, TC_BM);
      ok &= encode_tmap_bf16_3d(&w.tmU, w.U, (int)F, iR, h * iL, TC_BM);
      ok &= encode_tmap_bf16_3d(&w.tmXaW, w.Xa, (int)d, iT, h * (iL + 1) * nb, TC_BM);
      ok &= encode_tmap_bf16_3d(&w.tmPhi, w.Phi, (int)P, iT, h * G, TC_BM);
      ok &= encode_tmap_bf16_3d(&w.tmAa, w.Aa, (int)P, (int)d, h * G, 256);
      ok &= encode_tmap_bf16_3d(&w.tmQK, w.QKV, qkv_ld, iT, G, 128);
      ok &= encode_tmap_bf16_3d(&w.tmVt, w.Vt, t_pad, (int)hd, G * (int)Hkv, (int)hd);
      if (!ok) return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    }
    (void)st;
    w.nb = nb;
    return ARMT_OK;
  }

  // The batched workspace for exactly nb sequences (re-sized when nb changes).
  armt_status ensure_batch(int nb, cudaStream_t st) {
    if (wb.nb == nb) return ARMT_OK;
    CK(cudaStreamSynchronize(st));
    wb_mem.free_all();
    wb = Work();
    armt_status s = alloc_work(wb, nb, wb_mem, st);
    if (s != ARMT_OK) {
      wb_mem.free_all();
      wb = Work();
    }
    return s;
  }

  // One grouped GEMM over groups [lo, lo+g): tensor cores for bf16, SIMT +
  // row epilogue for fp32.  `rows` output rows per group; `map` places each
  // group's A rows and B slot (GemmGroupMap).  The fp32 path stages raw
  // products in w.Cscr.
  // tb2 != nullptr: a 128-row-box map of the same B, so that the product
  // may run as 256 x 256 tiles on CTA pairs (gemm_tc2.cuh) -- chosen when
  // `rows` pads to 256-row tiles almost as tightly as to 128-row ones
  // (pair_tiles_pay_off); otherwise 128 x BN tiles on single CTAs.
  template <int BN, class Epi, int EPI_WG = 1>
  armt_status gemm(int cls, Work& w, const CUtensorMap& ta, const CUtensorMap& tb, const AT* a,
                   long long a_gs, const WT* b, int N, int K, const Epi& epi, int lo, int g,
                   cudaStream_t st, int rows, const GemmGroupMap& map = GemmGroupMap(),
                   const CUtensorMap* tb2 = nullptr) {
    CKS(prof_begin(cls, st));
    if constexpr (kTC) {
      bool done = false;
      if constexpr (BN == 256) {
        if (tb2 != nullptr && pair_tiles_pay_off(rows)) {
          CK((launch_gemm_tc2<Epi, EPI_WG>(ta, *tb2, rows, N, K, lo, g, d_err, epi, num_sms, st, map, wp)));
          done = true;
        }
      }
      if (!done)
        CK((launch_gemm_tc<Epi, BN, EPI_WG>(ta, tb, rows, N, K, lo, g, d_err, epi, num_sms, st, map, wp)));
    } else {
      const SimtAMap am{map.row0, map.a_slot_off, map.b_div, map.alt_lo, map.alt_hi, map.alt_row0};
      const float* b0 = reinterpret_cast<const float*>(b) + (long long)map.b_slot_off * N * K;
      dim3 grid((N + 63) / 64, (rows + 63) / 64, g);
      gemm_simt_f32_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(a), a_gs, K, b0,
                                                 (long long)N * K, w.Cscr, (long long)rows * nmax,
                                                 nmax, rows, N, K, lo, am);
      CK(cudaGetLastError());
      epi_rows_kernel<Epi><<<dim3(rows, g), 128, 0, st>>>(w.Cscr, (long long)rows * nmax, nmax, N,
                                                          lo, epi);
      CK(cudaGetLastError());
    }
    CKS(prof_end(st));
    return ARMT_OK;
  }

  // All kernels of one grouped step: the cells (l, s_lo - (l - lo)) for l in
  // [lo, hi], each for the w.nb sequences of the batch.  The sequences hold
  // n_tok tokens each (n_seg segments; the last one may be short).
  armt_status step(Work& w, int lo, int hi, int64_t s_lo, const int32_t* tokens, int64_t n_tok,
                   int64_t n_seg, float* hidden, float* A, float* z, cudaStream_t st) {
    const armt_config& c = cfg;
    const int L = c.n_layers, d = c.d_model, hd = c.head_dim, F = c.ffn_dim, T = rows();
    const int Hq = c.n_q_heads, Hkv = c.n_kv_heads, k = c.key_dim, P = phi_dim(), M = c.n_mem;
    const int S = c.seg_len, Nq = n_qkv();
    const int g = hi - lo + 1, nb = w.nb, R = nb * T;
    const long long Rd = (long long)R * d;
    // the last segment holds last_len <= S tokens; its memory rows follow them
    const int last_len = last_segment_len(n_tok, S);
    // split precision: where the low parts live (elements, and A slots of the
    // GEMM operand maps); all zero when the model is not split
    const long long xa_lo = split ? (long long)(L + 1) * Rd : 0, nrm_lo = split ? (long long)L * Rd : 0;
    const long long att_lo = split ? (long long)L * R * Hq * hd : 0, u_lo = split ? (long long)L * R * F : 0;
    GemmGroupMap layer_lo;  // A slot l + L holds the low part of slot l
    layer_lo.a_lo_slot = split ? L : 0;
    GemmGroupMap xa_map;    // Xa slots: L + 1 of them
    xa_map.a_lo_slot = split ? L + 1 : 0;
    GemmGroupMap read_map;  // features x state copy, both split: L * nb groups each
    read_map.a_lo_slot = split ? L * nb : 0;
    read_map.b_lo_slot = split ? L * nb : 0;
    const long long phi_lo = split ? (long long)L * R * P : 0;
    const long long aa_lo = split ? (long long)L * nb * d * P : 0;
    const int64_t l_last = last_segment_layer(lo, s_lo, n_seg);  // layer of the last segment's cell
    const bool short_here = last_len < S && l_last >= lo && l_last <= hi;
    if (lo == 0) {
      const int n_rows = s_lo == n_seg - 1 ? last_len : S;
      CKS(prof_begin(ARMT_KC_OTHER, st));
      embed_gather_kernel<WT><<<dim3(T, nb), 256, 0, st>>>(tokens + s_lo * S, n_tok, embed, memtok,
                                                           w.X, w.Xa, T, n_rows, M, d, c.vocab, xa_lo);
      CK(cudaGetLastError());
      CKS(prof_end(st));
    }
    // associative read: q = Wq_a x, phi, den, then x' = x + A phi / den.  On the
    // tensor-core path phi and den come out of the query GEMM's epilogue.
    if constexpr (kTC) {
      SEpiPhi<AT> ph{w.Phi, w.Den, z, R, T, nb, c.assoc_eps};
      ph.lo_off = phi_lo;
      CKS((gemm<64, SEpiPhi<AT>>(ARMT_KC_ASSOC_READ, w, w.tmXa, tmAWq, w.Xa, Rd, aWq, k, d, ph, lo, g, st, R,
                                 xa_map)));
    } else {
      CKS((gemm<64>(ARMT_KC_ASSOC_READ, w, w.tmXa, tmAWq, w.Xa, Rd, aWq, k, d,
                    FStore{w.Qa, (long long)k, (long long)R * k}, lo, g, st, R)));
      CKS(prof_begin(ARMT_KC_ASSOC_READ, st));
      // 256 threads, as in the persistent wavefront: the denominator's
      // reduction order depends on the block size
      assoc_phi_kernel<AT><<<dim3(R, g), 256, 2 * k * sizeof(float), st>>>(
          w.Qa, z, w.Phi, w.Den, R, k, c.dpfp_nu, c.assoc_eps, lo, T, nb);
      CK(cudaGetLastError());
      CKS(prof_end(st));
    }
    // the read GEMM runs per (layer, sequence): groups lo*nb .. (hi+1)*nb - 1
    // of T rows, each with its own state
    const AT* Asrc = kTC ? w.Aa : reinterpret_cast<const AT*>(A);
    const RowNormIn norm_in{w.Ssq, npart, 1.0f / (float)d, c.norm_eps};
    {
      RowNormOut<AT> n1{g1, w.Nrm, w.Ssq};
      n1.gdiv = nb;
      n1.lo_off = nrm_lo;
      CKS((gemm<256, FRead, 2>(ARMT_KC_ASSOC_READ, w, w.tmPhi, w.tmAa, w.Phi, (long long)T * P,
                               reinterpret_cast<const WT*>(Asrc), d, P,
                               FRead{w.X, w.Den, w.Res, T, d, n1}, lo * nb, g * nb, st, T, read_map)));
    }
    // attention sub-layer (RMSNorm 1 completes in the QKV epilogue)
    CKS((gemm<256, FQkv, 1>(ARMT_KC_GEMM_QKV, w, w.tmNrm, tmWqkv, w.Nrm, Rd, Wqkv, Nq, d,
                            FQkv{w.QKV, w.cosT, w.sinT, R, hd, (Hq + Hkv) * hd, qkv_ld, w.Vt, Hkv,
                                 t_pad, norm_in, T, nb},
                            lo, g, st, R, layer_lo, &tmWqkv2)));
    CKS(prof_begin(ARMT_KC_ATTENTION, st));
    if constexpr (kTC) {
      AttnArgs aa;
      aa.out = w.Att;
      aa.T = T;
      aa.Hq = Hq;
      aa.Hkv = Hkv;
      aa.g_first = lo * nb;
      aa.n_qtiles = (T + 127) / 128;
      aa.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
      aa.err = d_err;
      aa.wp = wp;
      aa.out_lo_off = att_lo;
      if (hd == 64)
        CK((launch_attn_tc<64, QT>(w.tmQK, w.tmVt, aa, g * nb, num_sms, st)));
      else
        CK((launch_attn_tc<128, QT>(w.tmQK, w.tmVt, aa, g * nb, num_sms, st)));
    } else {
      dim3 grid((T + 63) / 64, Hq, g * nb);
      const float scale = 1.0f / sqrtf((float)hd);
      if (hd == 64)
        attn_simt_kernel<AT, 64><<<grid, 256, attn_smem, st>>>(w.QKV, w.Att, T, Hq, Hkv, scale, lo * nb);
      else if (hd == 128)
        attn_simt_kernel<AT, 128><<<grid, 256, attn_smem, st>>>(w.QKV, w.Att, T, Hq, Hkv, scale, lo * nb);
      else
        attn_simt_kernel<AT, 32><<<grid, 256, attn_smem, st>>>(w.QKV, w.Att, T, Hq, Hkv, scale, lo * nb);
      CK(cudaGetLastError());
    }
    CKS(prof_end(st));
    {
      RowNormOut<AT> n2{g2, w.Nrm, w.Ssq};
      n2.lo_off = nrm_lo;
      CKS((gemm<256, FRes, 2>(ARMT_KC_GEMM_O, w, w.tmAtt, tmWo, w.Att, (long long)R * Hq * hd, Wo, d,
                              Hq * hd, FRes{w.Res, w.Res, nullptr, R, d, 0, n2}, lo, g, st, R, layer_lo,
                              &tmWo2)));
    }
    // MLP sub-layer (RMSNorm 2 completes in the gate-up epilogue)
    {
      FSwi swi{w.U, R, F, norm_in};
      FRes down{w.Res, w.X, kTC ? w.Xa : nullptr, R, d, 1, RowNormOut<AT>{nullptr, nullptr, nullptr}};
      if constexpr (kTC) {
        swi.lo_off = u_lo;
        down.copy_lo_off = xa_lo;
      }
      CKS((gemm<256, FSwi, 1>(ARMT_KC_GEMM_GATEUP, w, w.tmNrm, tmWgu, w.Nrm, Rd, Wgu, 2 * F, d, swi, lo, g, st,
                              R, layer_lo, &tmWgu2)));
      CKS((gemm<256, FRes, 1>(ARMT_KC_GEMM_DOWN, w, w.tmU, tmWd, w.U, (long long)R * F, Wd, d, F, down, lo,
                              g, st, R, layer_lo, &tmWd2)));
    }
    // delta-rule write from the memory-token rows of this layer's output:
    // [v | k | beta] = h_mem [Wv_a; Wk_a; wbeta_a]^T on the tensor cores, per
    // (layer, sequence) group: A = the M memory rows of the cell in layer
    // slot l + 1 (rows S..S+M-1, or last_len.. after a short last segment),
    // B = layer l's projections.  Then the normaliser recurrence and the
    // row-wise update of A.
    {
      GemmGroupMap wm;
      wm.row0 = S;
      wm.a_slot_off = nb;
      wm.b_div = nb;
      wm.a_lo_slot = split ? (L + 1) * nb : 0;
      if (short_here) {
        wm.alt_lo = (int)l_last * nb;
        wm.alt_hi = (int)(l_last + 1) * nb;
        wm.alt_row0 = last_len;
      }
      CKS((gemm<256>(ARMT_KC_ASSOC_WRITE, w, w.tmXaW, tmWw, w.Xa, (long long)T * d, Ww, nw, d,
                     FStore{w.VKB, (long long)nw, (long long)M * nw}, lo * nb, g * nb, st, M, wm)));
    }
    CKS(prof_begin(ARMT_KC_ASSOC_WRITE, st));
    assoc_write_feat_kernel<<<g * nb, 256, feat_smem, st>>>(w.VKB, z, w.PhiM, w.Coef, M, k, c.dpfp_nu,
                                                            c.assoc_eps, d, nw, lo * nb);
    CK(cudaGetLastError());
    CKS(prof_end(st));
    CKS(prof_begin(ARMT_KC_ASSOC_WRITE, st));
    {
      dim3 grid((d + upd_rows_per_block - 1) / upd_rows_per_block, g * nb);
      AT* Adst = kTC ? w.Aa : reinterpret_cast<AT*>(A);
      const int gf0 = lo * nb;
      if (P == 96)
        assoc_write_update_kernel<AT, 3><<<grid, 128, upd_smem, st>>>(w.VKB, nw, w.PhiM, w.Coef, A, Adst,
                                                                      M, d, upd_rows_per_block, gf0, aa_lo);
      else if (P == 192)
        assoc_write_update_kernel<AT, 6><<<grid, 128, upd_smem, st>>>(w.VKB, nw, w.PhiM, w.Coef, A, Adst,
                                                                      M, d, upd_rows_per_block, gf0, aa_lo);
      else
        assoc_write_update_kernel<AT, 12><<<grid, 128, upd_smem, st>>>(w.VKB, nw, w.PhiM, w.Coef, A, Adst,
                                                                       M, d, upd_rows_per_block, gf0, aa_lo);
      CK(cudaGetLastError());
    }
    CKS(prof_end(st));
    if (hi == L - 1) {
      const int64_t segL = s_lo - (hi - lo);
      const int n_rows = segL == n_seg - 1 ? last_len : S;
      CKS(prof_begin(ARMT_KC_NORM, st));
      rmsnorm_kernel<float><<<dim3(n_rows, nb), 256, 0, st>>>(
          w.X + (long long)L * Rd, (long long)T * d, gf, 0, hidden + segL * S * (long long)d,
          n_tok * (long long)d, d, c.norm_eps, 0);
      CK(cudaGetLastError());
      CKS(prof_end(st));
    }
    return ARMT_OK;
  }

  // Workspace of the full-attention baseline for T tokens.
  armt_status ensure_full(int64_t T, cudaStream_t st) {
    if (T <= full_T) return ARMT_OK;
    CK(cudaStreamSynchronize(st));
    full_mem.free_all();
    full_T = 0;
    const armt_config& c = cfg;
    const size_t d = c.d_model, hd = c.head_dim, F = c.ffn_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
    const size_t tp = (size_t)((T + 7) / 8 * 8);
    CKS(full_mem.alloc_n(&Xf, T * d));
    CKS(full_mem.alloc_n(&Resf, T * d));
    CKS(full_mem.alloc_n(&Ssqf, T * (size_t)npart));
    CKS(full_mem.alloc_n(&Nrmf, T * d));
    CKS(full_mem.alloc_n(&QKVf, T * (Hq + Hkv) * hd));
    CKS(full_mem.alloc_n(&Vtf, Hkv * hd * tp));
    CKS(full_mem.alloc_n(&Attf, T * Hq * hd));
    CKS(full_mem.alloc_n(&Uf, T * F));
    {
      std::vector<float> hc((size_t)T * (hd / 2)), hs((size_t)T * (hd / 2));
      for (int64_t t = 0; t < T; ++t)
        for (size_t i = 0; i < hd / 2; ++i) {
          const double ang = (double)t * std::pow(c.rope_base, -2.0 * (double)i / (double)hd);
          hc[t * (hd / 2) + i] = (float)std::cos(ang);
          hs[t * (hd / 2) + i] = (float)std::sin(ang);
        }
      CKS(full_mem.alloc_n(&cosF, hc.size()));
      CKS(full_mem.alloc_n(&sinF, hs.size()));
      CK(cudaMemcpy(cosF, hc.data(), hc.size() * 4, cudaMemcpyHostToDevice));
      CK(cudaMemcpy(sinF, hs.data(), hs.size() * 4, cudaMemcpyHostToDevice));
    }
    bool ok = true;
    ok &= encode_tmap_bf16_3d(&tmNrmf, Nrmf, (int)d, (int)T, 1, TC_BM);
    ok &= encode_tmap_bf16_3d(&tmQKf, QKVf, (int)((Hq + Hkv) * hd), (int)T, 1, 128);
    ok &= encode_tmap_bf16_3d(&tmVtf, Vtf, (int)tp, (int)hd, (int)Hkv, (int)hd);
    ok &= encode_tmap_bf16_3d(&tmAttf, Attf, (int)(Hq * hd), (int)T, 1, TC_BM);
    ok &= encode_tmap_bf16_3d(&tmUf, Uf, (int)F, (int)T, 1, TC_BM);
    if (!ok) return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    full_T = T;
    return ARMT_OK;
  }

  // Plain causal LLaMA over T tokens with the same weights: no memory tokens,
  // no associative memory, one attention over the whole sequence.  Layers run
  // one after another; each launch reads activation slot 0 and weight slot l.
  // logits[r][v] = hidden[r] . head[v], head = w_head or the token embedding
  // (tied); rows in chunks of kLmChunk.  Tensor cores for bf16 models: the
  // fp32 hidden rows are rounded to bf16 first (the head's operand type).
  armt_status lm_head(const float* hidden, int64_t n_rows, const void* w_head, float* logits,
                      cudaStream_t st) override {
    const armt_config& c = cfg;
    const int d = c.d_model, V = c.vocab;
    const WT* head = w_head != nullptr ? reinterpret_cast<const WT*>(w_head) : embed;
    if (kTC && V % 256 != 0) return fail(ARMT_ERR_UNSUPPORTED, "bf16 LM head needs vocab % 256 == 0");
    if (kTC && lm_rows == nullptr) CKS(lm_mem.alloc_n(&lm_rows, (size_t)kLmChunk * d));
    CKS(prof_begin(ARMT_KC_OTHER, st));
    if constexpr (kTC) {
      CUtensorMap tb;
      CUtensorMap tb1;
      if (!encode_tmap_bf16_3d(&tb, head, d, V, 1, 128) || !encode_tmap_bf16_3d(&tb1, head, d, V, 1, 256))
        return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
      for (int64_t r0 = 0; r0 < n_rows; r0 += kLmChunk) {
        const int rows_c = (int)std::min<int64_t>(kLmChunk, n_rows - r0);
        convert_state_kernel<AT><<<num_sms * 4, 256, 0, st>>>(hidden + r0 * d, lm_rows, (long long)rows_c * d);
        CK(cudaGetLastError());
        CUtensorMap ta;
        if (!encode_tmap_bf16_3d(&ta, lm_rows, d, rows_c, 1, TC_BM))
          return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        SEpiStore epi{logits + r0 * V, (long long)V, 0};
        if (pair_tiles_pay_off(rows_c))
          CK((launch_gemm_tc2<SEpiStore, 1>(ta, tb, rows_c, V, d, 0, 1, d_err, epi, num_sms, st,
                                            GemmGroupMap(), wp)));
        else
          CK((launch_gemm_tc<SEpiStore, 256>(ta, tb1, rows_c, V, d, 0, 1, d_err, epi, num_sms, st,
                                             GemmGroupMap(), wp)));
      }
    } else {
      for (int64_t r0 = 0; r0 < n_rows; r0 += kLmChunk) {
        const int rows_c = (int)std::min<int64_t>(kLmChunk, n_rows - r0);
        dim3 grid((V + 63) / 64, (rows_c + 63) / 64, 1);
        gemm_simt_f32_kernel<<<grid, 256, 0, st>>>(hidden + r0 * d, 0, d,
                                                   reinterpret_cast<const float*>(head), 0,
                                                   logits + r0 * V, 0, V, rows_c, V, d, 0,
                                                   SimtAMap{0, 0, 1, 0, 0, 0});
        CK(cudaGetLastError());
      }
    }
    CKS(prof_end(st));
    return ARMT_OK;
  }

  template <class Epi, int EPI_WG>
  cudaError_t launch_weight_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2,
                                 int rows, int N, int K, int g_first, int g_count, int* err,
                                 const Epi& epi, int nsm, cudaStream_t st, const GemmGroupMap& map) {
    if (pair_tiles_pay_off(rows))
      return launch_gemm_tc2<Epi, EPI_WG>(ta, tb2, rows, N, K, g_first, g_count, err, epi, nsm, st, map, wp);
    return launch_gemm_tc<Epi, 256, EPI_WG>(ta, tb, rows, N, K, g_first, g_count, err, epi, nsm, st, map, wp);
  }

  static GemmGroupMap layer_map(int l) {
    GemmGroupMap m;
    m.b_slot_off = l;
    return m;
  }

  armt_status forward_full(const int32_t* tokens, int64_t T64, float* hidden,
                           cudaStream_t st) override {
    if constexpr (!kTC) {
      return fail(ARMT_ERR_UNSUPPORTED, "the full-attention baseline needs a bf16 model");
    } else {
      if (T64 > (1 << 20)) return fail(ARMT_ERR_SHAPE, "n_tokens > 1048576");
      CKS(ensure_full(T64, st));
      const armt_config& c = cfg;
      const int T = (int)T64, L = c.n_layers, d = c.d_model, hd = c.head_dim, F = c.ffn_dim;
      const int Hq = c.n_q_heads, Hkv = c.n_kv_heads, Nq = n_qkv();
      const int tp = (T + 7) / 8 * 8;
      const long long Td = (long long)T * d;
      CKS(prof_begin(ARMT_KC_OTHER, st));
      embed_gather_kernel<WT><<<dim3(T, 1), 256, 0, st>>>(tokens, 0, embed, memtok, Xf, (WT*)nullptr, T, T, 0,
                                                         d, c.vocab);
      CK(cudaGetLastError());
      CKS(prof_end(st));
      const RowNormIn no_scale{nullptr, 0, 0.f, 0.f};
      const RowNormIn norm_in{Ssqf, npart, 1.0f / (float)d, c.norm_eps};
      for (int l = 0; l < L; ++l) {
        CKS(prof_begin(ARMT_KC_NORM, st));
        rmsnorm_kernel<AT><<<dim3(T, 1), 256, 0, st>>>(Xf, 0, g1 + (long long)l * d, 0, Nrmf, 0, d,
                                                      c.norm_eps, 0);
        CK(cudaGetLastError());
        CKS(prof_end(st));
        CKS(prof_begin(ARMT_KC_GEMM_QKV, st));
        CK((launch_weight_gemm<FQkv, 1>(tmNrmf, tmWqkv, tmWqkv2, T, Nq, d, 0, 1, d_err,
                                      FQkv{QKVf, cosF, sinF, T, hd, (Hq + Hkv) * hd, (Hq + Hkv) * hd,
                                           Vtf, Hkv, tp, no_scale, T, 1},
                                      num_sms, st, layer_map(l))));
        CKS(prof_end(st));
        CKS(prof_begin(ARMT_KC_ATTENTION, st));
        {
          AttnArgs aa;
          aa.out = Attf;
          aa.T = T;
          aa.Hq = Hq;
          aa.Hkv = Hkv;
          aa.g_first = 0;
          aa.n_qtiles = (T + 127) / 128;
          aa.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
          aa.err = d_err;
          aa.wp = wp;
          if (hd == 64)
            CK((launch_attn_tc<64, QT>(tmQKf, tmVtf, aa, 1, num_sms, st)));
          else
            CK((launch_attn_tc<128, QT>(tmQKf, tmVtf, aa, 1, num_sms, st)));
        }
        CKS(prof_end(st));
        CKS(prof_begin(ARMT_KC_GEMM_O, st));
        CK((launch_weight_gemm<FRes, 2>(tmAttf, tmWo, tmWo2, T, d, Hq * hd, 0, 1, d_err,
                                      FRes{Xf, Resf, nullptr, T, d, 0,
                                           RowNormOut<AT>{g2 + (long long)l * d, Nrmf, Ssqf}},
                                      num_sms, st, layer_map(l))));
        CKS(prof_end(st));
        CKS(prof_begin(ARMT_KC_GEMM_GATEUP, st));
        CK((launch_weight_gemm<FSwi, 1>(tmNrmf, tmWgu, tmWgu2, T, 2 * F, d, 0, 1, d_err, FSwi{Uf, T, F, norm_in},
                                      num_sms, st, layer_map(l))));
        CKS(prof_end(st));
        CKS(prof_begin(ARMT_KC_GEMM_DOWN, st));
        CK((launch_weight_gemm<FRes, 1>(tmUf, tmWd, tmWd2, T, d, F, 0, 1, d_err,
                                      FRes{Resf, Xf, nullptr, T, d, 0,
                                           RowNormOut<AT>{nullptr, nullptr, nullptr}},
                                      num_sms, st, layer_map(l))));
        CKS(prof_end(st));
      }
      CKS(prof_begin(ARMT_KC_NORM, st));
      rmsnorm_kernel<float><<<dim3(T, 1), 256, 0, st>>>(Xf, 0, gf, 0, hidden, 0, d, c.norm_eps, 0);
      CK(cudaGetLastError());
      CKS(prof_end(st));
      (void)Td;
      return ARMT_OK;
    }
  }

  // The whole forward of one sequence as one persistent launch (fp32 models;
  // wavefront.cuh): the same block code and data as step(), with device-side
  // (cell, stage) counters in place of the launch boundaries.
  armt_status forward_wavefront(const int32_t* tokens, int64_t n_tok, int64_t n, float* hidden, float* A,
                                float* z, int mem_in_valid, cudaStream_t st) {
    if constexpr (kTC) {
      return fail(ARMT_ERR_UNSUPPORTED, "the wavefront schedule runs fp32 models");
    } else {
      const armt_config& c = cfg;
      const int L = c.n_layers, d = c.d_model, hd = c.head_dim, F = c.ffn_dim, T = rows();
      const int Hq = c.n_q_heads, Hkv = c.n_kv_heads, k = c.key_dim, P = phi_dim(), M = c.n_mem;
      const int S = c.seg_len, Nq = n_qkv();
      Work& w = w1;
      const long long Rd = (long long)T * d;
      if (!mem_in_valid) {
        CK(cudaMemsetAsync(A, 0, (size_t)L * d * P * sizeof(float), st));
        CK(cudaMemsetAsync(z, 0, (size_t)L * P * sizeof(float), st));
      }
      WfArgs a{};
      a.embed = embed;
      a.memtok = memtok;
      a.gf = gf;
      a.T = T; a.S = S; a.M = M; a.d = d; a.k = k; a.nu = c.dpfp_nu; a.vocab = c.vocab;
      a.Hq = Hq; a.Hkv = Hkv; a.hd = hd; a.P = P; a.nw = nw; a.nmax = nmax; a.L = L;
      a.assoc_eps = c.assoc_eps; a.norm_eps = c.norm_eps; a.attn_scale = 1.0f / sqrtf((float)hd);
      a.upd_rows = upd_rows_per_block;
      a.X = w.X; a.Cscr = w.Cscr; a.Qa = w.Qa; a.Phi = w.Phi; a.Den = w.Den; a.QKV = w.QKV;
      a.Att = w.Att; a.VKB = w.VKB; a.PhiM = w.PhiM; a.Coef = w.Coef;
      a.tokens = tokens; a.n_tok = n_tok; a.n_seg = n; a.last_len = last_segment_len(n_tok, S);
      a.hidden = hidden; a.A = A; a.z = z;
      auto g = [&](const float* Aop, long long a_gs, int K, const float* B, int N, int rows_, SimtAMap am) {
        WfGemm r;
        r.A = Aop; r.a_gs = a_gs; r.lda = K; r.B = B; r.b_gs = (long long)N * K;
        r.N = N; r.K = K; r.rows = rows_; r.nbx = (N + 63) / 64; r.am = am;
        return r;
      };
      const SimtAMap plain{0, 0, 1, 0, 0, 0};
      a.gq = g(w.X, Rd, d, reinterpret_cast<const float*>(aWq), k, T, plain);
      a.gr = g(w.Phi, (long long)T * P, P, A, d, T, plain);
      a.gqkv = g(w.Nrm, Rd, d, reinterpret_cast<const float*>(Wqkv), Nq, T, plain);
      a.go = g(w.Att, (long long)T * Hq * hd, Hq * hd, reinterpret_cast<const float*>(Wo), d, T, plain);
      a.ggu = g(w.Nrm, Rd, d, reinterpret_cast<const float*>(Wgu), 2 * F, T, plain);
      a.gd = g(w.U, (long long)T * F, F, reinterpret_cast<const float*>(Wd), d, T, plain);
      a.gw = g(w.X, Rd, d, reinterpret_cast<const float*>(Ww), nw, M, SimtAMap{S, 1, 1, 0, 0, 0});
      const RowNormIn norm_in{w.Ssq, npart, 1.0f / (float)d, c.norm_eps};
      a.eq = EpiStore{w.Qa, (long long)k, (long long)T * k};
      {
        RowNormOut<float> n1{g1, w.Nrm, w.Ssq};
        a.er = EpiAssocRead<float>{w.X, w.Den, w.Res, T, d, n1};
      }
      a.eqkv = EpiQkvRope<float>{w.QKV, w.cosT, w.sinT, T, hd, (Hq + Hkv) * hd, qkv_ld, nullptr, Hkv, t_pad,
                                 norm_in, T, 1};
      a.eo = EpiResidual<float>{w.Res, w.Res, nullptr, T, d, 0, RowNormOut<float>{g2, w.Nrm, w.Ssq}};
      a.egu = EpiSwiGLU<float>{w.U, T, F, norm_in};
      a.ed = EpiResidual<float>{w.Res, w.X, nullptr, T, d, 1, RowNormOut<float>{nullptr, nullptr, nullptr}};
      a.ew = EpiStore{w.VKB, (long long)nw, (long long)M * nw};
      a.err = d_err;
      a.wp = wp;
      wf_tasks_h = wf_tasks(a, n);
      const size_t nt = wf_tasks_h.size(), nc = (size_t)L * n * WF_NSTAGE + 1;
      if (nt > (size_t)INT32_MAX || nc > (size_t)INT32_MAX) return fail(ARMT_ERR_SHAPE, "too many wavefront tasks");
      if (nt > wf_tasks_cap || nc > wf_ctr_cap) {
        CK(cudaStreamSynchronize(st));
        wf_mem.free_all();
        wf_tasks_d = nullptr;
        wf_ctr = nullptr;
        wf_tasks_cap = wf_ctr_cap = 0;
        CKS(wf_mem.alloc_n(&wf_tasks_d, nt));
        CKS(wf_mem.alloc_n(&wf_ctr, nc));
        wf_tasks_cap = nt;
        wf_ctr_cap = nc;
      }
      CK(cudaMemcpyAsync(wf_tasks_d, wf_tasks_h.data(), nt * sizeof(WfTask), cudaMemcpyHostToDevice, st));
      CK(cudaMemsetAsync(wf_ctr, 0, nc * sizeof(int), st));
      int* next = wf_ctr + (nc - 1);  // the task counter
      const size_t smem = std::max(std::max(attn_smem, feat_smem), std::max(upd_smem, (size_t)2 * k * sizeof(float)));
      CKS(prof_begin(ARMT_KC_OTHER, st));
      armt_status r = ARMT_OK;
      if (hd == 32) r = launch_wavefront<32>(nt, next, smem, a, st);
      else if (hd == 64) r = launch_wavefront<64>(nt, next, smem, a, st);
      else r = launch_wavefront<128>(nt, next, smem, a, st);
      CKS(r);
      CKS(prof_end(st));
      return ARMT_OK;
    }
  }

  template <int HD>
  armt_status launch_wavefront(size_t nt, int* next, size_t smem, const WfArgs& a, cudaStream_t st) {
    auto kern = wavefront_kernel<HD>;
    CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    int per_sm = 0;
    CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem));
    if (per_sm <= 0) return fail(ARMT_ERR_UNSUPPORTED, "the wavefront kernel does not fit an SM");
    // every block resident at once (cooperative launch), none idle beyond the task count
    const long long grid = std::min<long long>((long long)per_sm * num_sms, (long long)nt);
    const WfTask* tasks = wf_tasks_d;
    int n_tasks = (int)nt;
    int* ctr = wf_ctr;
    void* args[] = {(void*)&tasks, (void*)&n_tasks, (void*)&next, (void*)&ctr, (void*)&a};
    CK(cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(256), args, smem, st));
    return ARMT_OK;
  }

  // The backward's forward keeps, for every cell, its input rows and the
  // state it starts from: before a step, the input slots l >= 1 (written by
  // the cell below in the previous step) and the states; after it, layer 0's
  // gathered input.  Batch 1.
  armt_status save_cells(Work& w, const CellRange& c, const float* A, const float* z, bool before,
                         cudaStream_t st) {
    const int d = cfg.d_model, P = phi_dim(), T = rows();
    const int64_t n = bw_save->n;
    const size_t Td = (size_t)T * d;
    for (int l = c.lo; l <= c.hi; ++l) {
      const int64_t s = c.s_lo - (l - c.lo);
      const size_t cell = (size_t)l * n + s;
      if (before) {
        CK(cudaMemcpyAsync(bw_save->As + cell * d * P, A + (size_t)l * d * P, (size_t)d * P * sizeof(float),
                           cudaMemcpyDeviceToDevice, st));
        CK(cudaMemcpyAsync(bw_save->zs + cell * P, z + (size_t)l * P, (size_t)P * sizeof(float),
                           cudaMemcpyDeviceToDevice, st));
      }
      if ((l >= 1) == before)
        CK(cudaMemcpyAsync(bw_save->Xs + cell * Td, w.X + (size_t)l * Td, Td * sizeof(float),
                           cudaMemcpyDeviceToDevice, st));
    }
    return ARMT_OK;
  }

  // Backward workspace for n segments of n_tok tokens (grown on demand).
  armt_status bw_alloc(int64_t n, int64_t n_tok, cudaStream_t st) {
    if (n <= bw_n_cap && n_tok <= bw_tok_cap) return ARMT_OK;
    CK(cudaStreamSynchronize(st));
    bw_mem.free_all();
    bw_n_cap = bw_tok_cap = 0;
    const armt_config& c = cfg;
    const size_t L = c.n_layers, d = c.d_model, k = c.key_dim, P = phi_dim(), T = rows(), M = c.n_mem;
    const size_t F = c.ffn_dim, Nq = n_qkv(), HA = (size_t)c.n_q_heads * c.head_dim, Td = T * d;
    BwView& v = bwv;
    v = BwView{};
    auto A = [&](float** p, size_t nel) { return bw_mem.alloc_n(p, nel); };
    CKS(A(&v.Xs, L * n * Td));
    CKS(A(&v.As, L * n * d * P));
    CKS(A(&v.zs, L * n * P));
    CKS(A(&v.Qa, L * T * k));
    CKS(A(&v.Phi, L * T * P));
    CKS(A(&v.Den, L * T));
    float** td_bufs[] = {&v.Rr, &v.X1, &v.N1, &v.Y, &v.N2, &v.H, &v.N2bar, &v.Ybar, &v.N1bar, &v.X1bar, &v.XS};
    for (float** b : td_bufs) CKS(A(b, L * Td));
    CKS(A(&v.QKV, L * T * Nq));
    CKS(A(&v.dQKV, L * T * Nq));
    CKS(A(&v.LSE, L * T * c.n_q_heads));
    CKS(A(&v.Dsum, L * T * c.n_q_heads));
    CKS(A(&v.Att, L * T * HA));
    CKS(A(&v.dAtt, L * T * HA));
    CKS(A(&v.GU, L * T * 2 * F));
    CKS(A(&v.GUbar, L * T * 2 * F));
    CKS(A(&v.U, L * T * F));
    CKS(A(&v.Ubar, L * T * F));
    CKS(A(&v.VKB, L * M * nw));
    CKS(A(&v.VKBbar, L * M * nw));
    CKS(A(&v.PhiM, L * M * P));
    CKS(A(&v.PhiBarM, L * M * P));
    CKS(A(&v.Sc, L * M * WS_NSC));
    CKS(A(&v.Gm, L * M * M));
    CKS(A(&v.Coef, L * M * M));
    float** md_bufs[] = {&v.Cw, &v.Vb, &v.CB, &v.Wv};
    for (float** b : md_bufs) CKS(A(b, L * M * d));
    CKS(A(&v.Srow, L * T));
    CKS(A(&v.Dbar, L * T));
    CKS(A(&v.PhiBar, L * T * P));
    CKS(A(&v.QaBar, L * T * k));
    for (int q = 0; q < 2; ++q) {
      CKS(A(&v.Hbar[q], L * Td));
      CKS(A(&v.SA[q], L * d * P));
      CKS(A(&v.Sz[q], L * P));
    }
    CKS(A(&v.XB0, n * Td));
    v.part_cap = (long long)1 << 22;  // 16 MB of split-K partial products
    CKS(A(&v.Part, (size_t)v.part_cap));
    CKS(A(&v.dWqkv, L * Nq * d));
    CKS(A(&v.dWgu, L * 2 * F * d));
    CKS(A(&v.dWw, L * nw * d));
    CKS(A(&bw_hidden, (size_t)n_tok * d));
    CKS(A(&bw_A, L * d * P));
    CKS(A(&bw_z, L * P));
    // kernels with more than 48 KB of dynamic shared memory
    const int hd = c.head_dim;
    const int fwd_smem = (int)bw_attn_fwd_smem(hd), dq_smem = (int)bw_attn_dq_smem(hd),
              dkv_smem = (int)bw_attn_dkv_smem(hd);
    if (hd == 32) {
      CK(cudaFuncSetAttribute(bw_attn_fwd_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_smem));
      CK(cudaFuncSetAttribute(bw_attn_dq_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_smem));
      CK(cudaFuncSetAttribute(bw_attn_dkv_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv_smem));
    } else if (hd == 64) {
      CK(cudaFuncSetAttribute(bw_attn_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_smem));
      CK(cudaFuncSetAttribute(bw_attn_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_smem));
      CK(cudaFuncSetAttribute(bw_attn_dkv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv_smem));
    } else {
      CK(cudaFuncSetAttribute(bw_attn_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_smem));
      CK(cudaFuncSetAttribute(bw_attn_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_smem));
      CK(cudaFuncSetAttribute(bw_attn_dkv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv_smem));
    }
    const int rows_smem = (int)((M * P + M * WS_NSC) * sizeof(float));
    if (P == 96)
      CK(cudaFuncSetAttribute(bw_write_rows_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, rows_smem));
    else if (P == 192)
      CK(cudaFuncSetAttribute(bw_write_rows_kernel<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, rows_smem));
    else
      CK(cudaFuncSetAttribute(bw_write_rows_kernel<12>, cudaFuncAttributeMaxDynamicSharedMemorySize, rows_smem));
    CK(cudaFuncSetAttribute(bw_write_feat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            (int)((M * 2 * k + M * (P + 1)) * sizeof(float))));
    bw_n_cap = n;
    bw_tok_cap = n_tok;
    return ARMT_OK;
  }

  // fp32 copies of the bf16 weights the backward multiplies with (once)
  armt_status bw_weights_f32(cudaStream_t st) {
    if (aWq32 != nullptr) return ARMT_OK;
    const armt_config& c = cfg;
    const size_t L = c.n_layers, d = c.d_model, k = c.key_dim, F = c.ffn_dim, Nq = n_qkv();
    const size_t HA = (size_t)c.n_q_heads * c.head_dim;
    struct Item {
      float** dst;
      const WT* src;
      size_t n;
    } items[] = {{&aWq32, aWq, L * k * d}, {&Wqkv32, Wqkv, L * Nq * d}, {&Wo32, Wo, L * d * HA},
                 {&Wgu32, Wgu, L * 2 * F * d}, {&Wd32, Wd, L * d * F}, {&Ww32, Ww, L * (size_t)nw * d}};
    for (const Item& it : items) {
      armt_status s = bw_w32_mem.alloc_n(it.dst, it.n);
      if (s != ARMT_OK) {
        bw_w32_mem.free_all();
        aWq32 = nullptr;
        return s;
      }
      to_f32_kernel<WT><<<4 * num_sms, 256, 0, st>>>(it.src, *it.dst, (long long)it.n);
      CK(cudaGetLastError());
    }
    return ARMT_OK;
  }

  armt_status backward(const int32_t* tokens, int64_t n_tok, const float* A0, const float* z0,
                       const float* cot_h, const float* cot_A, const float* cot_z, float* hidden, float* A,
                       float* z, const armt_grads& gr, cudaStream_t st) override {
    {
      if constexpr (kTC) CKS(bw_weights_f32(st));
      const armt_config& c = cfg;
      const int L = c.n_layers, d = c.d_model, P = phi_dim(), S = c.seg_len, M = c.n_mem, k = c.key_dim;
      const int F = c.ffn_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, hd = c.head_dim;
      const int64_t n = n_segments_for(n_tok, S);
      CKS(bw_alloc(n, n_tok, st));
      BwView& v = bwv;
      if (hidden == nullptr) hidden = bw_hidden;
      if (A == nullptr) A = bw_A;
      if (z == nullptr) z = bw_z;
      const size_t a_n = (size_t)L * d * P, z_n = (size_t)L * P;
      // the forward, keeping every cell's input rows and entry state
      const bool resume = A0 != nullptr;
      if (resume) {
        CK(cudaMemcpyAsync(A, A0, a_n * sizeof(float), cudaMemcpyDeviceToDevice, st));
        CK(cudaMemcpyAsync(z, z0, z_n * sizeof(float), cudaMemcpyDeviceToDevice, st));
      }
      const BwSave sv{v.Xs, v.As, v.zs, n};
      bw_save = &sv;
      const armt_status fs = forward(tokens, n_tok, 1, hidden, A, z, resume ? 1 : 0, ARMT_SCHEDULE_DIAGONAL, st);
      bw_save = nullptr;
      CKS(fs);
      // sizes and weights
      v.L = L;
      v.d = d;
      v.k = k;
      v.nu = c.dpfp_nu;
      v.P = P;
      v.Hq = Hq;
      v.Hkv = Hkv;
      v.hd = hd;
      v.F = F;
      v.Nq = (int)n_qkv();
      v.nw = nw;
      v.T = rows();
      v.S = S;
      v.M = M;
      v.vocab = c.vocab;
      v.norm_eps = c.norm_eps;
      v.assoc_eps = c.assoc_eps;
      v.n_seg = n;
      v.n_tok = n_tok;
      v.last_len = last_segment_len(n_tok, S);
      if constexpr (kTC) {
        v.aWq = aWq32;
        v.Wqkv = Wqkv32;
        v.Wo = Wo32;
        v.Wgu = Wgu32;
        v.Wd = Wd32;
        v.Ww = Ww32;
      } else {
        v.aWq = aWq;
        v.Wqkv = Wqkv;
        v.Wo = Wo;
        v.Wgu = Wgu;
        v.Wd = Wd;
        v.Ww = Ww;
      }
      v.g1 = g1;
      v.g2 = g2;
      v.gf = gf;
      v.cosT = w1.cosT;
      v.sinT = w1.sinT;
      v.cot_h = cot_h;
      v.num_sms = num_sms;
      // gradients accumulate from zero: the unfused ones in the caller's buffers
      v.dWo = gr.wo;
      v.dWd = gr.w_down;
      v.daWq = gr.a_wq;
      v.dg1 = gr.norm1;
      v.dg2 = gr.norm2;
      v.dgf = gr.norm_f;
      const size_t HA = (size_t)Hq * hd;
      CK(cudaMemsetAsync(gr.wo, 0, (size_t)L * d * HA * 4, st));
      CK(cudaMemsetAsync(gr.w_down, 0, (size_t)L * d * F * 4, st));
      CK(cudaMemsetAsync(gr.a_wq, 0, (size_t)L * k * d * 4, st));
      CK(cudaMemsetAsync(gr.norm1, 0, (size_t)L * d * 4, st));
      CK(cudaMemsetAsync(gr.norm2, 0, (size_t)L * d * 4, st));
      CK(cudaMemsetAsync(gr.norm_f, 0, (size_t)d * 4, st));
      CK(cudaMemsetAsync(gr.embed, 0, (size_t)c.vocab * d * 4, st));
      CK(cudaMemsetAsync(gr.mem, 0, (size_t)M * d * 4, st));
      CK(cudaMemsetAsync(v.dWqkv, 0, (size_t)L * v.Nq * d * 4, st));
      CK(cudaMemsetAsync(v.dWgu, 0, (size_t)L * 2 * F * d * 4, st));
      CK(cudaMemsetAsync(v.dWw, 0, (size_t)L * nw * d * 4, st));
      // the final state's adjoints enter layer l's first cell in reverse order,
      // (l, n - 1) on diagonal l + n - 1, which reads buffer (l + n - 1) & 1
      for (int l = 0; l < L; ++l) {
        const int q = bw_state_seed_buf(l, n);
        float* sa = v.SA[q] + (size_t)l * d * P;
        float* sz = v.Sz[q] + (size_t)l * P;
        if (cot_A != nullptr)
          CK(cudaMemcpyAsync(sa, cot_A + (size_t)l * d * P, (size_t)d * P * 4, cudaMemcpyDeviceToDevice, st));
        else
          CK(cudaMemsetAsync(sa, 0, (size_t)d * P * 4, st));
        if (cot_z != nullptr)
          CK(cudaMemcpyAsync(sz, cot_z + (size_t)l * P, (size_t)P * 4, cudaMemcpyDeviceToDevice, st));
        else
          CK(cudaMemsetAsync(sz, 0, (size_t)P * 4, st));
      }
      BwRun run{v, st};
      for (int64_t i = diagonal_steps(L, n) - 1; i >= 0; --i) {
        const CellRange cr = diagonal_step(i, L, n);
        trace_push("backward diagonal", i, cr.lo, cr.hi);
        const armt_status ds = run.diagonal(i);
        trace_pop();
        CKS(ds);
      }
      bw_embed_grad_kernel<<<(d + 127) / 128, 128, 0, st>>>(v.XB0, tokens, n_tok, S, rows(), M, d, c.vocab, n,
                                                            gr.embed, gr.mem);
      CKS(run.check());
      // the initial state's adjoints: layer l's cell (l, 0) ran on diagonal l
      for (int l = 0; l < L; ++l) {
        const int q = bw_state_result_buf(l);
        if (gr.mem_A != nullptr)
          CK(cudaMemcpyAsync(gr.mem_A + (size_t)l * d * P, v.SA[q] + (size_t)l * d * P, (size_t)d * P * 4,
                             cudaMemcpyDeviceToDevice, st));
        if (gr.mem_z != nullptr)
          CK(cudaMemcpyAsync(gr.mem_z + (size_t)l * P, v.Sz[q] + (size_t)l * P, (size_t)P * 4,
                             cudaMemcpyDeviceToDevice, st));
      }
      // fused accumulators to the caller's layout (the reverse of create()'s copies)
      const size_t Nq = v.Nq, es = sizeof(float);
      CK(cudaMemcpy2DAsync(gr.wq, HA * d * es, v.dWqkv, Nq * d * es, HA * d * es, L, cudaMemcpyDeviceToDevice, st));
      CK(cudaMemcpy2DAsync(gr.wk, (size_t)Hkv * hd * d * es, v.dWqkv + HA * d, Nq * d * es, (size_t)Hkv * hd * d * es,
                           L, cudaMemcpyDeviceToDevice, st));
      CK(cudaMemcpy2DAsync(gr.wv, (size_t)Hkv * hd * d * es, v.dWqkv + (HA + (size_t)Hkv * hd) * d, Nq * d * es,
                           (size_t)Hkv * hd * d * es, L, cudaMemcpyDeviceToDevice, st));
      const size_t blk = (size_t)GU_BLK * d * es, nblk = (size_t)L * F / GU_BLK;
      CK(cudaMemcpy2DAsync(gr.w_gate, blk, v.dWgu, 2 * blk, blk, nblk, cudaMemcpyDeviceToDevice, st));
      CK(cudaMemcpy2DAsync(gr.w_up, blk, reinterpret_cast<char*>(v.dWgu) + blk, 2 * blk, blk, nblk,
                           cudaMemcpyDeviceToDevice, st));
      CK(cudaMemcpy2DAsync(gr.a_wv, (size_t)d * d * es, v.dWw, (size_t)nw * d * es, (size_t)d * d * es, L,
                           cudaMemcpyDeviceToDevice, st));
      CK(cudaMemcpy2DAsync(gr.a_wk, (size_t)k * d * es, v.dWw + (size_t)d * d, (size_t)nw * d * es,
                           (size_t)k * d * es, L, cudaMemcpyDeviceToDevice, st));
      CK(cudaMemcpy2DAsync(gr.a_wbeta, (size_t)d * es, v.dWw + (size_t)(d + k) * d, (size_t)nw * d * es,
                           (size_t)d * es, L, cudaMemcpyDeviceToDevice, st));
      bw_launches = run.launches;
      bw_flops = run.flops;
      return ARMT_OK;
    }
  }

  armt_status forward(const int32_t* tokens, int64_t n_tok, int nb, float* hidden, float* A,
                      float* z, int mem_in_valid, int schedule, cudaStream_t st) override {
    const int L = cfg.n_layers, d = cfg.d_model, P = phi_dim(), S = cfg.seg_len;
    const int64_t n = n_segments_for(n_tok, S);
    if (schedule == ARMT_SCHEDULE_WAVEFRONT) {
      if constexpr (kTC) {
        return fail(ARMT_ERR_UNSUPPORTED, "the wavefront schedule runs fp32 models");
      } else {
        if (nb != 1) return fail(ARMT_ERR_UNSUPPORTED, "the wavefront schedule runs one sequence");
        trace_push("wavefront", n, 0, L - 1);
        const armt_status ws = forward_wavefront(tokens, n_tok, n, hidden, A, z, mem_in_valid, st);
        trace_pop();
        return ws;
      }
    }
    if (nb > 1) CKS(ensure_batch(nb, st));
    Work& w = nb == 1 ? w1 : wb;
    const size_t a_n = (size_t)L * nb * d * P, z_n = (size_t)L * nb * P;
    if (!mem_in_valid) {
      CK(cudaMemsetAsync(A, 0, a_n * sizeof(float), st));
      CK(cudaMemsetAsync(z, 0, z_n * sizeof(float), st));
      if (kTC) CK(cudaMemsetAsync(w.Aa, 0, (split ? 2 : 1) * a_n * sizeof(AT), st));
    } else if (kTC) {
      CKS(prof_begin(ARMT_KC_OTHER, st));
      convert_state_kernel<AT><<<4 * num_sms, 256, 0, st>>>(A, w.Aa, (long long)a_n, split ? (long long)a_n : 0);
      CK(cudaGetLastError());
      CKS(prof_end(st));
    }
    const bool report = sink != nullptr && nb == 1;
    if (schedule == ARMT_SCHEDULE_DIAGONAL) {
      for (int64_t i = 0; i < diagonal_steps(L, n); ++i) {
        const CellRange c = diagonal_step(i, L, n);
        if (bw_save != nullptr) CKS(save_cells(w, c, A, z, true, st));
        trace_push("diagonal", i, c.lo, c.hi);
        const armt_status ss = step(w, c.lo, c.hi, c.s_lo, tokens, n_tok, n, hidden, A, z, st);
        trace_pop();
        CKS(ss);
        if (bw_save != nullptr) CKS(save_cells(w, c, A, z, false, st));
        if (report)
          CKS(sink_progress(diagonal_rows_final(i, L, S, n_tok), diagonal_layers_final(i, n), st));
      }
    } else {
      for (int64_t s = 0; s < n; ++s) {
        for (int l = 0; l < L; ++l) {
          trace_push("segment", s, l, l);
          const armt_status ss = step(w, l, l, s, tokens, n_tok, n, hidden, A, z, st);
          trace_pop();
          CKS(ss);
        }
        if (report) CKS(sink_progress(sequential_rows_final(s, S, n_tok), sequential_layers_final(s, n, L), st));
      }
    }
    return ARMT_OK;
  }
};

// --------------------------------------------------------- checking --

static armt_status validate(const armt_config* c) {
  if (c->n_layers <= 0 || c->d_model <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 ||
      c->head_dim <= 0 || c->ffn_dim <= 0 || c->vocab <= 0 || c->seg_len <= 0 || c->n_mem <= 0 ||
      c->key_dim <= 0 || c->dpfp_nu <= 0)
    return fail(ARMT_ERR_ARG, "config sizes must be positive");
  if (!(c->norm_eps > 0.f) || !(c->assoc_eps > 0.f) || !(c->rope_base > 1.0))
    return fail(ARMT_ERR_ARG, "norm_eps, assoc_eps must be > 0 and rope_base > 1");
  if (c->dtype != ARMT_F32 && c->dtype != ARMT_BF16) return fail(ARMT_ERR_ARG, "unknown dtype");
  if (c->precision != ARMT_PRECISION_BF16 && c->precision != ARMT_PRECISION_BF16X2)
    return fail(ARMT_ERR_ARG, "unknown precision");
  if (c->precision == ARMT_PRECISION_BF16X2 && c->dtype != ARMT_BF16)
    return fail(ARMT_ERR_UNSUPPORTED, "split precision needs a bf16 model");
  if (c->n_q_heads % c->n_kv_heads != 0)
    return fail(ARMT_ERR_SHAPE, "n_q_heads must be a multiple of n_kv_heads");
  if (c->n_mem > 32) return fail(ARMT_ERR_UNSUPPORTED, "n_mem > 32");
  if (c->dpfp_nu >= 2 * c->key_dim) return fail(ARMT_ERR_SHAPE, "dpfp_nu must be < 2 * key_dim");
  {
    const int Pf = 2 * c->key_dim * c->dpfp_nu;
    if (Pf != 96 && Pf != 192 && Pf != 384)
      return fail(ARMT_ERR_UNSUPPORTED, "2 * key_dim * dpfp_nu must be 96, 192 or 384");
  }
  const int hd = c->head_dim, d = c->d_model, F = c->ffn_dim;
  const int Nq = (c->n_q_heads + 2 * c->n_kv_heads) * hd;
  const int P = 2 * c->key_dim * c->dpfp_nu;
  const int T = c->seg_len + c->n_mem;
  if (hd != 32 && hd != 64 && hd != 128) return fail(ARMT_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 128");
  if (F % GU_BLK != 0) return fail(ARMT_ERR_SHAPE, "ffn_dim must be a multiple of 128");
  if (d % 32 != 0 || Nq % 64 != 0) return fail(ARMT_ERR_SHAPE, "d_model % 32, qkv width % 64");
  if (c->key_dim % 16 != 0) return fail(ARMT_ERR_SHAPE, "key_dim must be a multiple of 16");
  if (c->dtype == ARMT_BF16) {
    if (hd == 32) return fail(ARMT_ERR_UNSUPPORTED, "bf16 models need head_dim 64 or 128");
    if (d % 256 != 0 || Nq % 256 != 0)
      return fail(ARMT_ERR_SHAPE, "bf16: d_model and (Hq+2Hkv)*head_dim must be multiples of 256");
    if (c->key_dim != 64 || c->dpfp_nu != 3)
      return fail(ARMT_ERR_UNSUPPORTED, "bf16: key_dim must be 64 and dpfp_nu 3");
    if (P % 64 != 0 || (c->n_q_heads * hd) % 64 != 0 || F % 64 != 0)
      return fail(ARMT_ERR_SHAPE, "bf16: P, Hq*head_dim, ffn_dim must be multiples of 64");
  }
  if (T > 65535) return fail(ARMT_ERR_SHAPE, "seg_len + n_mem too large");
  return ARMT_OK;
}

static armt_status sm_count(int dev, int* n) {
  *n = 0;
  CK(cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev));
  if (*n <= 0) return fail(ARMT_ERR_CUDA, "multiprocessor count query returned " + std::to_string(*n));
  return ARMT_OK;
}

// ------------------------------------------ building blocks' error word --
//
// armt_grouped_gemm_bf16 and armt_segment_attention_bf16 run without a model,
// so their bounded waits report into a device global: every device that
// loads the library has its own copy, and no call allocates for it.  Host
// code needs its device address, looked up once per device (with it current)
// and again if the device's context changed (e.g. after cudaDeviceReset).
static __device__ int g_block_err;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

namespace armt {
void* current_context() {
  static std::atomic<CtxGetCurrentFn> fn{nullptr};
  CtxGetCurrentFn f = fn.load();
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    f = reinterpret_cast<CtxGetCurrentFn>(p);
    fn.store(f);
  }
  CUcontext c = nullptr;
  return f(&c) == CUDA_SUCCESS ? static_cast<void*>(c) : nullptr;
}
}  // namespace armt

namespace {
constexpr int kMaxDevices = 64;
struct DeviceWord {
  std::atomic<void*> ctx{nullptr};
  std::atomic<int*> ptr{nullptr};
};
DeviceWord g_block_err_addr[kMaxDevices];
}  // namespace

static armt_status block_err_word(int dev, int** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(ARMT_ERR_NO_DEVICE, "device ordinal out of range");
  void* ctx = current_context();
  DeviceWord& w = g_block_err_addr[dev];
  int* p = w.ptr.load();
  if (p == nullptr || w.ctx.load() != ctx) {
    void* a = nullptr;
    CK(cudaGetSymbolAddress(&a, g_block_err));
    CK(cudaMemset(a, 0, sizeof(int)));
    w.ptr.store(static_cast<int*>(a));
    w.ctx.store(ctx);
    p = static_cast<int*>(a);
  }
  *out = p;
  return ARMT_OK;
}

// ------------------------------------------------------------- C ABI --

extern "C" {

const char* armt_status_string(armt_status s) {
  switch (s) {
    case ARMT_OK: return "ok";
    case ARMT_ERR_ARG: return "invalid argument";
    case ARMT_ERR_SHAPE: return "inconsistent shape";
    case ARMT_ERR_UNSUPPORTED: return "unsupported configuration";
    case ARMT_ERR_OOM: return "out of device memory";
    case ARMT_ERR_CUDA: return "CUDA error";
    case ARMT_ERR_TIMEOUT: return "device-side wait timed out";
    case ARMT_ERR_NO_DEVICE: return "no compute capability 10.3 device";
  }
  return "unknown status";
}

const char* armt_last_error(void) { return g_last_error.c_str(); }

static armt_status check_device(int* dev) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    cudaGetLastError();
    return fail(ARMT_ERR_NO_DEVICE, "no CUDA device");
  }
  CK(cudaGetDevice(dev));
  int major = 0, minor = 0;
  CK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev));
  CK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev));
  if (major != 10 || minor != 3)
    return fail(ARMT_ERR_NO_DEVICE, "device is sm_" + std::to_string(major * 10 + minor) +
                                        ", this library is built for sm_103a");
  return ARMT_OK;
}

armt_status armt_create(const armt_config* cfg, const armt_weights* w, void* stream,
                        armt_model** out) {
  if (cfg == nullptr || w == nullptr || out == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  *out = nullptr;
  const void* ptrs[] = {w->embed, w->mem, w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up,
                        w->w_down, w->a_wq, w->a_wk, w->a_wv, w->a_wbeta, w->norm1, w->norm2,
                        w->norm_f};
  for (const void* p : ptrs)
    if (p == nullptr) return fail(ARMT_ERR_ARG, "NULL weight pointer");
  CKS(validate(cfg));
  int dev = 0;
  CKS(check_device(&dev));
  ModelBase* m = cfg->dtype == ARMT_BF16 ? static_cast<ModelBase*>(new Model<bf16>())
                                         : static_cast<ModelBase*>(new Model<float>());
  m->cfg = *cfg;
  m->device = dev;
  m->wp = wait_policy_from_env();
  armt_status s = sm_count(dev, &m->num_sms);
  if (s == ARMT_OK) s = m->create(w, reinterpret_cast<cudaStream_t>(stream));
  if (s != ARMT_OK) {
    cudaDeviceSynchronize();
    delete m;
    return s;
  }
  *out = new armt_model{m};
  return ARMT_OK;
}

armt_status armt_destroy(armt_model* m) {
  if (m == nullptr) return ARMT_OK;
  cudaDeviceSynchronize();
  delete m->impl;
  delete m;
  return ARMT_OK;
}

static armt_status forward_common(armt_model* m, const int32_t* tokens, int64_t n, float* hidden,
                                  float* A, float* z, int32_t mem_in_valid, int schedule,
                                  void* stream) {
  if (m == nullptr || tokens == nullptr || hidden == nullptr || A == nullptr || z == nullptr)
    return fail(ARMT_ERR_ARG, "NULL argument");
  if (n <= 0) return fail(ARMT_ERR_ARG, "n_segments must be positive");
  if (mem_in_valid != 0 && mem_in_valid != 1) return fail(ARMT_ERR_ARG, "mem_in_valid must be 0 or 1");
  if (n > ((int64_t)1 << 24)) return fail(ARMT_ERR_SHAPE, "n_segments too large");
  m->impl->wp = wait_policy_from_env();
  return m->impl->forward(tokens, n * m->impl->cfg.seg_len, 1, hidden, A, z, mem_in_valid, schedule,
                          reinterpret_cast<cudaStream_t>(stream));
}

armt_status armt_forward_batch(armt_model* m, const int32_t* tokens, int32_t batch, int64_t n_tokens,
                               float* hidden_out, float* mem_A, float* mem_z, int32_t mem_in_valid,
                               int32_t schedule, void* stream) {
  if (m == nullptr || tokens == nullptr || hidden_out == nullptr || mem_A == nullptr || mem_z == nullptr)
    return fail(ARMT_ERR_ARG, "NULL argument");
  if (batch <= 0 || n_tokens <= 0) return fail(ARMT_ERR_ARG, "batch and n_tokens must be positive");
  if (mem_in_valid != 0 && mem_in_valid != 1) return fail(ARMT_ERR_ARG, "mem_in_valid must be 0 or 1");
  if (schedule != ARMT_SCHEDULE_DIAGONAL && schedule != ARMT_SCHEDULE_SEQUENTIAL &&
      schedule != ARMT_SCHEDULE_WAVEFRONT)
    return fail(ARMT_ERR_ARG, "unknown schedule");
  const armt_config& c = m->impl->cfg;
  if (n_tokens > ((int64_t)1 << 24) * c.seg_len) return fail(ARMT_ERR_SHAPE, "n_tokens too large");
  if (batch > ARMT_MAX_BATCH || (int64_t)batch * c.n_layers > 65535)
    return fail(ARMT_ERR_SHAPE, "batch > ARMT_MAX_BATCH or batch * n_layers > 65535");
  m->impl->wp = wait_policy_from_env();
  return m->impl->forward(tokens, n_tokens, batch, hidden_out, mem_A, mem_z, mem_in_valid, schedule,
                          reinterpret_cast<cudaStream_t>(stream));
}

armt_status armt_forward(armt_model* m, const int32_t* tokens, int64_t n_segments, float* hidden_out,
                         float* mem_A, float* mem_z, int32_t mem_in_valid, void* stream) {
  return forward_common(m, tokens, n_segments, hidden_out, mem_A, mem_z, mem_in_valid,
                        ARMT_SCHEDULE_DIAGONAL, stream);
}

armt_status armt_forward_sequential(armt_model* m, const int32_t* tokens, int64_t n_segments,
                                    float* hidden_out, float* mem_A, float* mem_z,
                                    int32_t mem_in_valid, void* stream) {
  return forward_common(m, tokens, n_segments, hidden_out, mem_A, mem_z, mem_in_valid,
                        ARMT_SCHEDULE_SEQUENTIAL, stream);
}

armt_status armt_backward(armt_model* m, const int32_t* tokens, int64_t n_tokens, const float* mem_A0,
                          const float* mem_z0, const float* cot_hidden, const float* cot_A, const float* cot_z,
                          float* hidden_out, float* mem_A_out, float* mem_z_out, const armt_grads* grads,
                          void* stream) {
  if (m == nullptr || tokens == nullptr || grads == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  const float* gp[] = {grads->embed, grads->mem, grads->wq, grads->wk, grads->wv, grads->wo, grads->w_gate,
                       grads->w_up, grads->w_down, grads->a_wq, grads->a_wk, grads->a_wv, grads->a_wbeta,
                       grads->norm1, grads->norm2, grads->norm_f};
  for (const float* p : gp)
    if (p == nullptr) return fail(ARMT_ERR_ARG, "NULL gradient pointer");
  if ((mem_A0 == nullptr) != (mem_z0 == nullptr))
    return fail(ARMT_ERR_ARG, "mem_A0 and mem_z0 must both be given or both be NULL");
  if (n_tokens <= 0) return fail(ARMT_ERR_ARG, "n_tokens must be positive");
  const armt_config& c = m->impl->cfg;
  if (n_tokens > ((int64_t)1 << 24) * c.seg_len) return fail(ARMT_ERR_SHAPE, "n_tokens too large");
  m->impl->wp = wait_policy_from_env();
  return m->impl->backward(tokens, n_tokens, mem_A0, mem_z0, cot_hidden, cot_A, cot_z, hidden_out, mem_A_out,
                           mem_z_out, *grads, reinterpret_cast<cudaStream_t>(stream));
}

armt_status armt_backward_stats(const armt_model* m, int64_t* launches, int64_t* workspace_bytes, double* flops) {
  if (m == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (launches != nullptr) *launches = m->impl->bw_launches;
  if (workspace_bytes != nullptr) *workspace_bytes = m->impl->backward_workspace_bytes();
  if (flops != nullptr) *flops = m->impl->bw_flops;
  return ARMT_OK;
}

static bool is_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

armt_status armt_forward_host(armt_model* m, const int32_t* h_tokens, int64_t n, float* h_hidden,
                              float* h_A, float* h_z, int32_t mem_in_valid, int32_t schedule,
                              void* stream) {
  if (m == nullptr || h_tokens == nullptr || h_hidden == nullptr || h_A == nullptr || h_z == nullptr)
    return fail(ARMT_ERR_ARG, "NULL argument");
  if (n <= 0) return fail(ARMT_ERR_ARG, "n_segments must be positive");
  if (schedule != ARMT_SCHEDULE_DIAGONAL && schedule != ARMT_SCHEDULE_SEQUENTIAL &&
      schedule != ARMT_SCHEDULE_WAVEFRONT)
    return fail(ARMT_ERR_ARG, "unknown schedule");
  ModelBase* b = m->impl;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const armt_config& c = b->cfg;
  const size_t ntok = (size_t)n * c.seg_len, nh = ntok * c.d_model;
  const size_t na = (size_t)c.n_layers * c.d_model * b->phi_dim(), nz = (size_t)c.n_layers * b->phi_dim();
  if (b->st_tokens_n < ntok) {
    if (b->st_tokens) cudaFree(b->st_tokens);
    b->st_tokens = nullptr;
    b->st_tokens_n = 0;
    CK(cudaMalloc(&b->st_tokens, ntok * sizeof(int32_t)));
    b->st_tokens_n = ntok;
  }
  if (b->st_hidden_n < nh) {
    if (b->st_hidden) cudaFree(b->st_hidden);
    b->st_hidden = nullptr;
    b->st_hidden_n = 0;
    CK(cudaMalloc(&b->st_hidden, nh * sizeof(float)));
    b->st_hidden_n = nh;
  }
  if (b->st_A == nullptr) {
    CK(cudaMalloc(&b->st_A, na * sizeof(float)));
    CK(cudaMalloc(&b->st_z, nz * sizeof(float)));
  }
  CK(cudaMemcpyAsync(b->st_tokens, h_tokens, ntok * sizeof(int32_t), cudaMemcpyHostToDevice, st));
  if (mem_in_valid) {
    CK(cudaMemcpyAsync(b->st_A, h_A, na * sizeof(float), cudaMemcpyHostToDevice, st));
    CK(cudaMemcpyAsync(b->st_z, h_z, nz * sizeof(float), cudaMemcpyHostToDevice, st));
  }
  if (b->copy_stream == nullptr) {
    CK(cudaStreamCreateWithFlags(&b->copy_stream, cudaStreamNonBlocking));
    CK(cudaEventCreateWithFlags(&b->copy_event, cudaEventDisableTiming));
  }
  // Pinned destinations: results stream back to the host while later
  // diagonals still run.  Pageable ones: a copy into pageable memory returns
  // only when it has finished, which would stall the launches, so they are
  // copied once the forward is done.
  const bool pinned = is_pinned(h_hidden) && is_pinned(h_A) && is_pinned(h_z);
  ModelBase::HostSink sink{h_hidden, h_A, h_z, b->st_hidden, b->st_A, b->st_z, 0, (int64_t)ntok, 0,
                           (int64_t)8 * c.seg_len};
  b->sink = pinned ? &sink : nullptr;
  const armt_status fs = forward_common(m, b->st_tokens, n, b->st_hidden, b->st_A, b->st_z,
                                        mem_in_valid, schedule, stream);
  b->sink = nullptr;
  if (fs == ARMT_OK && !pinned) {
    CK(cudaEventRecord(b->copy_event, st));
    CK(cudaStreamWaitEvent(b->copy_stream, b->copy_event, 0));
    CK(cudaMemcpyAsync(h_hidden, b->st_hidden, nh * sizeof(float), cudaMemcpyDeviceToHost, b->copy_stream));
    CK(cudaMemcpyAsync(h_A, b->st_A, na * sizeof(float), cudaMemcpyDeviceToHost, b->copy_stream));
    CK(cudaMemcpyAsync(h_z, b->st_z, nz * sizeof(float), cudaMemcpyDeviceToHost, b->copy_stream));
    sink.rows_done = (int64_t)ntok;
    sink.layers_done = c.n_layers;
  }
  // drain the copy stream whatever happened, so no copy outlives the call
  const cudaError_t e1 = cudaStreamSynchronize(b->copy_stream);
  CKS(fs);
  if (e1 != cudaSuccess) return fail(ARMT_ERR_CUDA, std::string("copy stream: ") + cudaGetErrorString(e1));
  CK(cudaStreamSynchronize(st));
  if (sink.rows_done != (int64_t)ntok || sink.layers_done != c.n_layers)
    return fail(ARMT_ERR_CUDA, "internal: results not fully copied");
  return ARMT_OK;
}

armt_status armt_forward_full_attention(armt_model* m, const int32_t* tokens, int64_t n_tokens,
                                       float* hidden_out, void* stream) {
  if (m == nullptr || tokens == nullptr || hidden_out == nullptr)
    return fail(ARMT_ERR_ARG, "NULL argument");
  if (n_tokens <= 0) return fail(ARMT_ERR_ARG, "n_tokens must be positive");
  m->impl->wp = wait_policy_from_env();
  return m->impl->forward_full(tokens, n_tokens, hidden_out, reinterpret_cast<cudaStream_t>(stream));
}

armt_status armt_lm_head(armt_model* m, const float* hidden, int64_t n_rows, const void* w_head,
                         float* logits, void* stream) {
  if (m == nullptr || hidden == nullptr || logits == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (n_rows <= 0) return fail(ARMT_ERR_ARG, "n_rows must be positive");
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(logits) |
       reinterpret_cast<uintptr_t>(w_head)) & 15)
    return fail(ARMT_ERR_ARG, "pointers must be 16-byte aligned");
  m->impl->wp = wait_policy_from_env();
  return m->impl->lm_head(hidden, n_rows, w_head, logits, reinterpret_cast<cudaStream_t>(stream));
}

armt_status armt_grouped_gemm_bf16(const void* A, const void* B, float* C, int32_t G, int32_t M,
                                   int32_t N, int32_t K, void* stream) {
  if (A == nullptr || B == nullptr || C == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (G <= 0 || M <= 0 || N <= 0 || K <= 0) return fail(ARMT_ERR_ARG, "sizes must be positive");
  if (K % TC_BK != 0 || N % 256 != 0) return fail(ARMT_ERR_SHAPE, "need K % 64 == 0 and N % 256 == 0");
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 15)
    return fail(ARMT_ERR_ARG, "pointers must be 16-byte aligned");
  if ((long long)M > (1ll << 30) || (long long)G * N > (1ll << 30))
    return fail(ARMT_ERR_SHAPE, "sizes too large");
  int dev = 0, nsm = 0;
  int* err = nullptr;
  CKS(check_device(&dev));
  CKS(sm_count(dev, &nsm));
  CKS(block_err_word(dev, &err));
  CUtensorMap ta, tb;
  const bool pairs = pair_tiles_pay_off(M);
  if (!encode_tmap_bf16_3d(&ta, A, K, M, G, TC_BM) || !encode_tmap_bf16_3d(&tb, B, K, N, G, pairs ? 128 : 256))
    return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  SEpiStore epi{C, (long long)N, (long long)M * N};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const WaitPolicy wp = wait_policy_from_env();
  if (pairs)
    CK((launch_gemm_tc2<SEpiStore, 1>(ta, tb, M, N, K, 0, G, err, epi, nsm, st, GemmGroupMap(), wp)));
  else
    CK((launch_gemm_tc<SEpiStore, 256>(ta, tb, M, N, K, 0, G, err, epi, nsm, st, GemmGroupMap(), wp)));
  return ARMT_OK;
}

armt_status armt_segment_attention_bf16(const void* qk, const void* vt, void* out, int32_t G,
                                        int32_t T, int32_t Hq, int32_t Hkv, int32_t hd,
                                        void* stream) {
  if (qk == nullptr || vt == nullptr || out == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (G <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0) return fail(ARMT_ERR_ARG, "sizes must be positive");
  if (Hq % Hkv != 0) return fail(ARMT_ERR_SHAPE, "Hq must be a multiple of Hkv");
  if (hd != 64 && hd != 128) return fail(ARMT_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (T % 8 != 0) return fail(ARMT_ERR_SHAPE, "T must be a multiple of 8");
  if ((reinterpret_cast<uintptr_t>(qk) | reinterpret_cast<uintptr_t>(vt) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(ARMT_ERR_ARG, "pointers must be 16-byte aligned");
  int dev = 0, nsm = 0;
  int* err = nullptr;
  CKS(check_device(&dev));
  CKS(sm_count(dev, &nsm));
  CKS(block_err_word(dev, &err));
  CUtensorMap tq, tv;
  if (!encode_tmap_bf16_3d(&tq, qk, (Hq + Hkv) * hd, T, G, 128) ||
      !encode_tmap_bf16_3d(&tv, vt, T, hd, G * Hkv, hd))
    return fail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  AttnArgs aa;
  aa.out = reinterpret_cast<bf16*>(out);
  aa.T = T;
  aa.Hq = Hq;
  aa.Hkv = Hkv;
  aa.g_first = 0;
  aa.n_qtiles = (T + 127) / 128;
  aa.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  aa.err = err;
  aa.wp = wait_policy_from_env();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hd == 64)
    CK(launch_attn_tc<64>(tq, tv, aa, G, nsm, st));
  else
    CK(launch_attn_tc<128>(tq, tv, aa, G, nsm, st));
  return ARMT_OK;
}

armt_status armt_block_sync_status(void* stream) {
  int dev = 0;
  int* err = nullptr;
  CKS(check_device(&dev));
  CKS(block_err_word(dev, &err));
  CK(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int h = 0;
  CK(cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost));
  if (h != 0) {
    CK(cudaMemset(err, 0, sizeof(int)));
    return fail(ARMT_ERR_TIMEOUT, "device wait timed out (code " + std::to_string(h) + ")");
  }
  return ARMT_OK;
}

armt_status armt_state_sizes(const armt_model* m, int64_t* a_elems, int64_t* z_elems) {
  if (m == nullptr || a_elems == nullptr || z_elems == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  const armt_config& c = m->impl->cfg;
  *a_elems = (int64_t)c.n_layers * c.d_model * m->impl->phi_dim();
  *z_elems = (int64_t)c.n_layers * m->impl->phi_dim();
  return ARMT_OK;
}

armt_status armt_memory_bytes(const armt_model* m, int64_t* weights, int64_t* workspace,
                              int64_t* full_workspace) {
  if (m == nullptr) return fail(ARMT_ERR_ARG, "NULL model");
  const ModelBase& b = *m->impl;
  if (weights) *weights = b.weight_bytes;
  if (workspace) *workspace = b.mem.total - b.weight_bytes + b.batch_workspace_bytes();
  if (full_workspace) *full_workspace = b.full_workspace_bytes();
  return ARMT_OK;
}

armt_status armt_launch_count(const armt_model* m, int64_t n, int32_t schedule, int64_t* launches) {
  if (m == nullptr || launches == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (n <= 0) return fail(ARMT_ERR_ARG, "n_segments must be positive");
  if (schedule != ARMT_SCHEDULE_DIAGONAL && schedule != ARMT_SCHEDULE_SEQUENTIAL &&
      schedule != ARMT_SCHEDULE_WAVEFRONT)
    return fail(ARMT_ERR_ARG, "unknown schedule");
  *launches = m->impl->launches(n, schedule, 0);
  return ARMT_OK;
}

armt_status armt_set_tracing(armt_model* m, int32_t enable) {
  if (m == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  m->impl->tracing = enable != 0;
  return ARMT_OK;
}

armt_status armt_set_profiling(armt_model* m, int32_t enable) {
  return armt_set_profiling_mask(m, enable != 0 ? (1u << ARMT_KC_COUNT) - 1u : 0u);
}

armt_status armt_set_profiling_mask(armt_model* m, uint32_t class_mask) {
  if (m == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (class_mask >> ARMT_KC_COUNT) return fail(ARMT_ERR_ARG, "class_mask has bits past ARMT_KC_COUNT");
  m->impl->prof_mask = class_mask;
  m->impl->profiling = class_mask != 0;
  m->impl->ev_used = 0;
  return ARMT_OK;
}

armt_status armt_kernel_times(armt_model* m, int64_t* launches, double* ms, int32_t n_classes) {
  if (m == nullptr || launches == nullptr || ms == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  if (n_classes <= 0 || n_classes > ARMT_KC_COUNT) return fail(ARMT_ERR_ARG, "bad n_classes");
  ModelBase* b = m->impl;
  for (int i = 0; i < n_classes; ++i) {
    launches[i] = 0;
    ms[i] = 0.0;
  }
  for (size_t i = 0; i < b->ev_used; ++i) {
    CK(cudaEventSynchronize(b->ev_stop[i]));
    float t = 0.f;
    CK(cudaEventElapsedTime(&t, b->ev_start[i], b->ev_stop[i]));
    const int c = b->ev_class[i];
    if (c < n_classes) {
      launches[c] += 1;
      ms[c] += t;
    }
  }
  b->ev_used = 0;
  return ARMT_OK;
}

armt_status armt_sync_status(armt_model* m, void* stream) {
  if (m == nullptr) return fail(ARMT_ERR_ARG, "NULL argument");
  CK(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int h = 0;
  CK(cudaMemcpy(&h, m->impl->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (h != 0) {
    CK(cudaMemset(m->impl->d_err, 0, sizeof(int)));
    return fail(ARMT_ERR_TIMEOUT, "device wait timed out (code " + std::to_string(h) + ")");
  }
  return ARMT_OK;
}

}  // extern "C"
