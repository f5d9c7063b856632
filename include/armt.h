/*
 * armt.h -- C ABI of the diagonal-batched ARMT forward pass (GB300, sm_103a).
 *
 * Source of the method: the summary page of "Diagonal Batching Unlocks
 * Parallelism in Recurrent Memory Transformers for Long Contexts" (Sivtsov,
 * Rodkin, Kuzmin, Kuratov, Oseledets; arXiv:2506.05229).
 *   - Section 二: in a parallel recurrent memory transformer (PRMT) such as
 *     ARMT every layer l owns an associative memory A_l, updated from that
 *     layer's output on the previous segment, so cell (layer l, segment s)
 *     depends only on (l-1, s) and (l, s-1); all cells with l + s = i can run
 *     together in iteration i ("one diagonal").
 *   - Section 三: all layers become one grouped layer -- stacked weights,
 *     grouped matrix multiplication with the outputs preallocated as one
 *     tensor and viewed per group, stacked norm gains, everything else run
 *     as a larger batch (attention batched over the layers of a diagonal).
 *   - Sections 一 and 五: the reordering keeps the exact recurrence.
 * The associative read/write equations are not printed on the page; the
 * reading implemented here is the delta rule with DPFP features:
 *   read  (every row x of a cell, before the attention sub-layer):
 *         x <- x + A_l phi(Wq_a x) / (z_l^T phi(Wq_a x) + assoc_eps)
 *   write (memory-token rows h_i of the cell's output, i = 0..M-1 in order,
 *         each against the state the previous write left -- a delta rule):
 *         k = Wk_a h_i, v = Wv_a h_i, beta = sigmoid(wbeta_a^T h_i), p = phi(k),
 *         vbar = A_l p / (z_l^T p + assoc_eps),
 *         gamma = clip(1 - z_l^T p / (p^T p + assoc_eps), 0, 1),
 *         A_l <- A_l + beta (v - vbar) p^T,  z_l <- z_l + gamma p
 *   phi = DPFP of order nu: r = [relu(k), relu(-k)], blocks r * roll(r, j),
 *         j = 1..nu, roll(r, j)_i = r_{(i-j) mod 2k};  P = 2 * key_dim * nu.
 * Each cell runs a LLaMA decoder layer (RMSNorm, rotate-half RoPE at cell
 * positions 0..S+M-1, causal grouped-query attention, SwiGLU, no biases) on
 * its S segment rows followed by the M memory-token rows.
 *
 * Conventions for every entry point
 *   - Sizes are element counts.  Matrices are row-major; a linear map is
 *     stored (out, in) like torch.nn.Linear.weight.
 *   - Device pointers must come from the current CUDA device; `stream` is a
 *     cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *     asynchronously on `stream`; nothing synchronises the host unless the
 *     entry point says so.
 *   - Errors are returned as armt_status and never abort the process.
 *     Argument and shape checks happen before any work is enqueued; on an
 *     argument error nothing is written.  A device-side bounded wait that
 *     gives up records ARMT_ERR_TIMEOUT, reported by armt_sync_status() (or
 *     armt_block_sync_status / armt_noalloc_sync_status for the building
 *     blocks); the kernel then lets the copies and tensor-core operations it
 *     already issued finish, frees its tensor memory and returns.
 *   - Environment (read at every call; for tests of the failure paths):
 *     ARMT_ALLOC_CAP_BYTES  cap on the bytes a model allocates (ARMT_ERR_OOM
 *                           beyond it);
 *     ARMT_WAIT_LIMIT_MS    limit of every bounded device-side wait
 *                           (default 2000 ms);
 *     ARMT_TEST_STALL_AFTER the tensor-core kernels' copy producers stop
 *                           after that many stage loads, as a stuck producer
 *                           would, so that the waits run out; the wavefront
 *                           schedule stops counting completed tasks from
 *                           that task index on (unset: off).
 *   - Not thread-safe per model: one host thread at a time per armt_model,
 *     and calls on one model must not overlap on the device (they share the
 *     model's activation workspace).  Different models are independent.
 */
#ifndef ARMT_H
#define ARMT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ARMT_API __attribute__((visibility("default")))
#else
#define ARMT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum armt_status {
  ARMT_OK = 0,
  ARMT_ERR_ARG = 1,          /* NULL pointer, non-positive count, bad enum value */
  ARMT_ERR_SHAPE = 2,        /* sizes inconsistent with the config or the kernels' tiling */
  ARMT_ERR_UNSUPPORTED = 3,  /* a config the kernels do not cover (e.g. head_dim 96) */
  ARMT_ERR_OOM = 4,          /* device allocation failed or exceeded the allocation cap */
  ARMT_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  ARMT_ERR_TIMEOUT = 6,      /* a bounded device-side wait gave up (kernel returned early) */
  ARMT_ERR_NO_DEVICE = 7     /* no CUDA device, or not a compute capability 10.3 device */
} armt_status;

typedef enum armt_dtype {
  ARMT_F32 = 0,   /* weights fp32, all matrix products in fp32 on CUDA cores */
  ARMT_BF16 = 1   /* weights bf16, matrix products on tcgen05 tensor cores, fp32 accumulation */
} armt_dtype;

/* Operand precision of the bf16 model's weight products (ignored by
 * ARMT_F32 models).  The weights are bf16 either way.
 *   ARMT_PRECISION_BF16    activations rounded to bf16 before every weight
 *                          product (fastest);
 *   ARMT_PRECISION_BF16X2  split operands: each activation operand of a
 *                          weight product is carried as a bf16 high part plus
 *                          a bf16 low part (its rounding residual), so the
 *                          tensor cores see it with about 16 significant
 *                          bits; the weight products run their K loop twice
 *                          (about twice the tensor-core time).  The
 *                          associative read splits both of its operands (the
 *                          features and the state copy: four K passes).  The
 *                          model holds a low copy of every split tensor.
 * In both, the attention's own operands (q, k, v, probabilities) are fp16,
 * and accumulation, the residual stream, norms, softmax statistics and the
 * memory state are fp32.  The full-attention baseline and the LM head use
 * plain bf16 operands. */
typedef enum armt_precision {
  ARMT_PRECISION_BF16 = 0,
  ARMT_PRECISION_BF16X2 = 1
} armt_precision;

typedef enum armt_schedule {
  ARMT_SCHEDULE_DIAGONAL = 0,   /* one grouped launch per anti-diagonal l + s = i */
  ARMT_SCHEDULE_SEQUENTIAL = 1, /* segment by segment, layer by layer, one cell per launch */
  ARMT_SCHEDULE_WAVEFRONT = 2   /* one persistent launch for the whole forward: each stage of
                                   each cell starts as soon as the stages it reads from are done,
                                   tracked by device-side (layer, segment, stage) counters;
                                   ARMT_F32 models, one sequence (armt_forward_batch with batch 1,
                                   armt_forward_host); ARMT_ERR_UNSUPPORTED otherwise */
} armt_schedule;

/* Model shape.  LLaMA decoder layer + per-layer associative memory. */
typedef struct armt_config {
  int32_t n_layers;    /* L */
  int32_t d_model;     /* d */
  int32_t n_q_heads;   /* Hq */
  int32_t n_kv_heads;  /* Hkv, divides Hq */
  int32_t head_dim;    /* hd (even; 64 or 128 for ARMT_BF16) */
  int32_t ffn_dim;     /* F, SwiGLU hidden size */
  int32_t vocab;       /* V, rows of the token embedding */
  int32_t seg_len;     /* S, segment tokens per cell */
  int32_t n_mem;       /* M, memory tokens appended after the segment rows */
  int32_t key_dim;     /* k, associative key dim */
  int32_t dpfp_nu;     /* nu, DPFP order; P = 2 * k * nu */
  float norm_eps;      /* RMSNorm epsilon */
  float assoc_eps;     /* epsilon in the associative denominators */
  double rope_base;    /* RoPE base (theta) */
  int32_t dtype;       /* armt_dtype */
  int32_t precision;   /* armt_precision (ARMT_BF16 models) */
} armt_config;

/* Weights, stacked over layers (section 三: one grouped layer holds every
 * layer's parameters).  Element type: float for ARMT_F32, bf16 (raw 16-bit
 * patterns) for ARMT_BF16.  Either all host pointers (on_device = 0) or all
 * device pointers (on_device = 1).  armt_create copies them into its own
 * layout; the caller may free them once armt_create returns. */
typedef struct armt_weights {
  const void* embed;    /* [V, d] token embedding */
  const void* mem;      /* [M, d] memory-token embeddings (same for every segment) */
  const void* wq;       /* [L, Hq*hd, d] */
  const void* wk;       /* [L, Hkv*hd, d] */
  const void* wv;       /* [L, Hkv*hd, d] */
  const void* wo;       /* [L, d, Hq*hd] */
  const void* w_gate;   /* [L, F, d] */
  const void* w_up;     /* [L, F, d] */
  const void* w_down;   /* [L, d, F] */
  const void* a_wq;     /* [L, k, d] associative query projection */
  const void* a_wk;     /* [L, k, d] associative key projection */
  const void* a_wv;     /* [L, d, d] associative value projection */
  const void* a_wbeta;  /* [L, d]    write-strength projection (sigmoid) */
  const void* norm1;    /* [L, d] RMSNorm gain before attention */
  const void* norm2;    /* [L, d] RMSNorm gain before the MLP */
  const void* norm_f;   /* [d]    final RMSNorm gain */
  int32_t on_device;    /* 1: device pointers, 0: host pointers */
} armt_weights;

typedef struct armt_model armt_model;  /* opaque */

/* Builds a model on the current device: validates `cfg` (uniform layers are
 * implied by the stacked layout; unsupported shapes -> ARMT_ERR_UNSUPPORTED),
 * copies the weights into the library's stacked device layout (fused Q|K|V
 * rows, gate/up rows interleaved in blocks of 128, TMA descriptors per
 * projection) and allocates the activation workspace for every layer.  The
 * copies are enqueued on `stream` and finished before return (synchronous).
 * On success *out owns all of it until armt_destroy. */
ARMT_API armt_status armt_create(const armt_config* cfg, const armt_weights* w, void* stream,
                        armt_model** out);

/* Releases everything armt_create allocated (synchronises the device first).
 * NULL is accepted. */
ARMT_API armt_status armt_destroy(armt_model* m);

/* ARMT forward over n_segments * S tokens with the diagonal schedule
 * (section 二): for i = 0 .. L + n_segments - 2 one grouped step runs every
 * cell (l, s = i - l) with 0 <= s < n_segments, each with layer l's weights
 * and layer l's memory.
 *   tokens      device int32 [n_segments * S], each in [0, V) (out-of-range
 *               ids are clamped to V-1 on the device; they are not checked)
 *   hidden_out  device fp32 [n_segments * S, d]: last layer's segment rows
 *               after the final RMSNorm (memory-token rows are not returned)
 *   mem_A       device fp32 [L, d, P], mem_z device fp32 [L, P]: the memory
 *               state, updated in place.  mem_in_valid = 0: the state starts
 *               at zero (the buffers are overwritten); 1: the buffers hold
 *               the state to resume from (e.g. a previous call's result).
 * Caller owns all buffers; they must not alias each other.  Results are
 * bit-identical to armt_forward_sequential on the same inputs. */
ARMT_API armt_status armt_forward(armt_model* m, const int32_t* tokens, int64_t n_segments,
                         float* hidden_out, float* mem_A, float* mem_z, int32_t mem_in_valid,
                         void* stream);

/* Same arguments and results; cells run one per step, segment by segment and
 * layer by layer (the schedule the diagonal one reorders), through the same
 * kernels.  For checking and as the speed-up denominator.  The third
 * schedule, ARMT_SCHEDULE_WAVEFRONT, is reached through armt_forward_batch
 * (batch 1) and armt_forward_host; all three give bit-identical results. */
ARMT_API armt_status armt_forward_sequential(armt_model* m, const int32_t* tokens, int64_t n_segments,
                                    float* hidden_out, float* mem_A, float* mem_z,
                                    int32_t mem_in_valid, void* stream);

/* Largest batch armt_forward_batch accepts (also batch * n_layers <= 65535). */
#define ARMT_MAX_BATCH 1024

/* Batched forward over `batch` independent sequences of n_tokens tokens each,
 * with the diagonal or the sequential schedule.  Every cell (l, s) runs the
 * batch's sequences side by side: the weight GEMMs of a layer see the
 * batch * (S + M) rows of its cells as one matrix, while attention and the
 * memory read / write run per (layer, sequence) with that sequence's own
 * state.  With the sequential schedule this is the micro-batching the
 * summary page compares diagonal batching with (section 三: per-segment
 * time of diagonal batching vs micro-batching); with the diagonal schedule
 * the two kinds of batching combine.
 * A short last segment is allowed: n_tokens need not be a multiple of S.
 * The last segment then holds the remaining S' = n_tokens - (n - 1) S
 * tokens (n = ceil(n_tokens / S)) followed as usual by the M memory tokens,
 * at positions 0 .. S' + M - 1; the page does not discuss partial segments,
 * this is the plain reading (the segment is just shorter).
 *   tokens      device int32 [batch][n_tokens] (ids clamped to [0, V))
 *   hidden_out  device fp32 [batch][n_tokens][d]
 *   mem_A       device fp32 [L][batch][d][P] (layer-major: the state of
 *               layer l, sequence b is at (l * batch + b) * d * P)
 *   mem_z       device fp32 [L][batch][P]
 *   mem_in_valid, schedule: as for armt_forward / armt_forward_sequential.
 * batch == 1 uses the workspace built by armt_create; batch > 1 uses a second
 * workspace of about batch times that size, allocated on the first call with
 * that batch size and re-allocated when the batch size changes (the
 * re-allocation synchronises `stream`; ARMT_ERR_OOM if it does not fit).
 * Per sequence the results are bit-identical to a batch-1 call with the same
 * tokens and state, and the diagonal and sequential schedules agree bitwise.
 * batch <= ARMT_MAX_BATCH and batch * L <= 65535 (ARMT_ERR_SHAPE). */
ARMT_API armt_status armt_forward_batch(armt_model* m, const int32_t* tokens, int32_t batch,
                                        int64_t n_tokens, float* hidden_out, float* mem_A,
                                        float* mem_z, int32_t mem_in_valid, int32_t schedule,
                                        void* stream);

/* End-to-end variant with HOST buffers (pinned or pageable): copies tokens
 * (and the state when mem_in_valid) to the device, runs `schedule`, copies
 * hidden states and state back, and synchronises `stream` before returning.
 * Device staging buffers are owned by the model and grow on demand.  When
 * h_hidden_out, h_mem_A and h_mem_z are all pinned (cudaHostAlloc /
 * cudaHostRegister) the results leave while the forward still runs: on a
 * second, library-owned stream, hidden rows in chunks of 8 segments as soon
 * as their segments have left the last layer, and each layer's state once
 * that layer has run its last segment.  Pageable buffers are copied after
 * the forward.  Either way everything has arrived when the call returns. */
ARMT_API armt_status armt_forward_host(armt_model* m, const int32_t* h_tokens, int64_t n_segments,
                              float* h_hidden_out, float* h_mem_A, float* h_mem_z,
                              int32_t mem_in_valid, int32_t schedule, void* stream);

/* Full-causal-attention baseline on the same weights: the plain LLaMA stack
 * (RMSNorm, RoPE at positions 0..n_tokens-1, causal GQA attention over the
 * whole sequence, SwiGLU, final RMSNorm) without memory tokens and without
 * the associative memory -- the "standard" model the ARMT forward is compared
 * with (summary page, sections 一 and 五: diagonal-batched ARMT vs the full
 * LLaMA-1B at 131,072 tokens).
 *   tokens      device int32 [n_tokens] (ids clamped to [0, V))
 *   hidden_out  device fp32 [n_tokens, d]
 * bf16 models only (ARMT_ERR_UNSUPPORTED otherwise).  The model grows a
 * separate activation workspace for n_tokens on first use (synchronises
 * `stream` when it grows); n_tokens <= 2^20. */
ARMT_API armt_status armt_forward_full_attention(armt_model* m, const int32_t* tokens,
                                                 int64_t n_tokens, float* hidden_out, void* stream);

/* Grouped matrix multiplication, the building block of the grouped layer
 * (section 三: weights stacked per group, outputs preallocated as one tensor
 * and viewed per group):  C[g] = A[g] * B[g]^T for g = 0..G-1, with
 *   A device bf16 [G, M, K] row-major, B device bf16 [G, N, K] (out, in),
 *   C device fp32 [G, M, N].  fp32 accumulation on tcgen05 tensor cores.
 * Requires K % 64 == 0, N % 256 == 0, 16-byte aligned base pointers, any
 * M >= 1.  A fixed reduction order per element independent of G. */
ARMT_API armt_status armt_grouped_gemm_bf16(const void* A, const void* B, float* C, int32_t G, int32_t M,
                                   int32_t N, int32_t K, void* stream);

/* Segment-local causal grouped-query attention, batched over G cells
 * (section 三: attention is left as it is and batched over the cells of a
 * diagonal).  For g = 0..G-1, query head h = 0..Hq-1 reads kv head
 * h / (Hq/Hkv); row t attends to rows 0..t of the same cell:
 *   out[g][t][h*hd : (h+1)*hd] = softmax_u(q_t . k_u / sqrt(hd)) v_u
 *   qk  device bf16 [G][T][(Hq+Hkv)*hd]: q heads then k heads (already rotated)
 *   vt  device bf16 [G][Hkv][hd][T]: v transposed (token index innermost)
 *   out device bf16 [G][T][Hq*hd]
 * tcgen05 tensor cores, fp32 softmax and accumulation.  hd in {64, 128},
 * T % 8 == 0, 16-byte aligned pointers. */
ARMT_API armt_status armt_segment_attention_bf16(const void* qk, const void* vt, void* out, int32_t G,
                                                 int32_t T, int32_t Hq, int32_t Hkv, int32_t hd,
                                                 void* stream);

/* Status of the two building blocks above, which run without a model: waits
 * for `stream`, then reports ARMT_ERR_TIMEOUT if a bounded device-side wait
 * of either gave up on the current device since the last call, and clears it.
 * Their error word is a device global of the library (one per device, looked
 * up on the first call with the device current); it stays set until read,
 * and while it is set the blocks' waits give up early, so their outputs are
 * then undefined.  Allocates nothing. */
ARMT_API armt_status armt_block_sync_status(void* stream);

/* Fixed device scratch of armt_segment_attention_bf16_noalloc (bytes). */
#define ARMT_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* armt_segment_attention_bf16 for callers that cannot allocate device
 * memory -- for example a serving process whose device memory is owned by
 * its own arena or capped, or a latency-critical path that must not hit
 * cudaMalloc's implicit device-wide synchronisation.  The paper has no
 * counterpart to this entry point; it is a deployment convenience.
 *   qkv device bf16 [G][T][(Hq+2Hkv)*hd]: q heads, k heads (already
 *       rotated), then v heads -- the plain fused row layout
 *   out device bf16 [G][T][Hq*hd]; same result as armt_segment_attention_bf16.
 * It calls no cudaMalloc, cudaFree or allocating library routine.  Its
 * scratch (the transposed values, G * Hkv * hd * round_up(T, 8) * 2 bytes,
 * plus a 256-byte error word) lives in one file-scope device array of
 * ARMT_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits; larger problems are rejected with ARMT_ERR_SHAPE before
 * anything is enqueued.  The first call on a device (with that device
 * current, and again after its context changed, e.g. after cudaDeviceReset)
 * looks up the array's device address and clears the error word; make that
 * first call before any stream capture.  Every call on a device shares the
 * one array, which keeps the last call's contents, so calls that overlap on
 * the GPU (e.g. on two streams without ordering) race -- order them.  A
 * bounded device-side wait that gives up records a code in the error word;
 * it stays set, and later calls' waits give up early, until
 * armt_noalloc_sync_status reads and clears it.  hd in {64, 128}, any T >= 1,
 * 16-byte aligned pointers. */
ARMT_API armt_status armt_segment_attention_bf16_noalloc(const void* qkv, void* out, int32_t G,
                                                         int32_t T, int32_t Hq, int32_t Hkv,
                                                         int32_t hd, void* stream);

/* Waits for `stream`, then reports ARMT_ERR_TIMEOUT if the no-allocation
 * attention recorded a timeout on the current device since the last call,
 * and clears it.  Allocates nothing. */
ARMT_API armt_status armt_noalloc_sync_status(void* stream);

/* LM head over hidden states (the logits behind the error-accumulation
 * study of section 四 of the summary page: diagonal batching vs the
 * sequential recurrence):
 *   logits[r][v] = sum_c hidden[r][c] * head[v][c],  r < n_rows, v < vocab
 *   hidden  device fp32 [n_rows][d_model] (e.g. armt_forward's output)
 *   w_head  device [vocab][d_model] in the model's dtype, or NULL for the
 *           model's own token embedding (tied head)
 *   logits  device fp32 [n_rows][vocab], caller-owned
 * bf16 models: the hidden rows are rounded to bf16 and the product runs on
 * the tensor cores (fp32 accumulation, the grouped GEMM), 8192 rows per
 * launch; vocab % 256 == 0 (ARMT_ERR_UNSUPPORTED otherwise).  fp32 models:
 * fp32 SIMT product.  16-byte aligned pointers.  Asynchronous on `stream`;
 * the first call allocates a 8192 x d_model bf16 staging buffer owned by the
 * model. */
ARMT_API armt_status armt_lm_head(armt_model* m, const float* hidden, int64_t n_rows,
                                  const void* w_head, float* logits, void* stream);

/* Gradient buffers of armt_backward: device fp32, each in the layout of the
 * armt_weights field of the same name, overwritten (not accumulated).  All
 * required except mem_A / mem_z, the gradients with respect to the initial
 * memory state ([L, d, P] and [L, P]; NULL skips them). */
typedef struct armt_grads {
  float *embed, *mem, *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
  float *a_wq, *a_wk, *a_wv, *a_wbeta, *norm1, *norm2, *norm_f;
  float *mem_A, *mem_z;
} armt_grads;

/* Backward pass (training support; section 四 of the summary page: diagonal
 * batching carries over to the backward pass, so training and inference
 * share one schedule).  Runs the forward over n_tokens tokens of one
 * sequence with the diagonal schedule, keeping each cell's input rows and
 * the memory state it starts from, then the adjoint cell by cell over the
 * anti-diagonals in reverse order: every cell (l, s) of a reverse diagonal
 * recomputes its forward, then hands the adjoint of its input rows to cell
 * (l-1, s) and that of its entry state to cell (l, s-1), and adds its share
 * of layer l's weight gradients; the cells of one diagonal run side by side.
 * The gradient is that of the scalar
 *   loss = <hidden, cot_hidden> + <A_final, cot_A> + <z_final, cot_z>,
 * i.e. the vector-Jacobian product of the forward with those cotangents.
 *   tokens       device int32 [n_tokens] (ids clamped to [0, V) as in the
 *                forward; a short last segment is allowed)
 *   mem_A0/z0    device fp32 [L, d, P] / [L, P] initial state, or both NULL
 *                (zero state)
 *   cot_hidden   device fp32 [n_tokens, d], cot_A [L, d, P], cot_z [L, P];
 *                each may be NULL (zero)
 *   hidden_out, mem_A_out, mem_z_out: the forward's results (as from
 *                armt_forward_batch with batch 1), each may be NULL
 *   grads        see armt_grads
 * fp32 models: everything in fp32.  bf16 models: the forward runs as
 * armt_forward does (the model's precision mode, tensor cores) and keeps its
 * fp32 cell inputs and states; the adjoint runs in fp32 against fp32 copies
 * of the bf16 weights, made on the first call (kept by the model) -- the
 * gradients of the exact model at the bf16 forward's cell inputs.  Every
 * reduction runs in a fixed order: repeated calls give bitwise equal
 * gradients.  The first call (and one with more segments or tokens than
 * before) allocates the backward's workspace, which grows with the number
 * of segments (saved cell inputs and states); the allocation synchronises
 * `stream`; ARMT_ERR_OOM if it does not fit.  Asynchronous on `stream`
 * otherwise.  Buffers must not alias. */
ARMT_API armt_status armt_backward(armt_model* m, const int32_t* tokens, int64_t n_tokens,
                                   const float* mem_A0, const float* mem_z0, const float* cot_hidden,
                                   const float* cot_A, const float* cot_z, float* hidden_out,
                                   float* mem_A_out, float* mem_z_out, const armt_grads* grads,
                                   void* stream);

/* Of the last armt_backward (its forward not included): kernel launches and
 * the algorithmic FLOPs of its products and attention (recompute included:
 * 2 M N K per product, 2 T (T + 1) hd per head for the causal attention
 * recompute and 7 T (T + 1) hd for its adjoint); and the bytes of the
 * backward's workspace.  Any output pointer may be NULL. */
ARMT_API armt_status armt_backward_stats(const armt_model* m, int64_t* launches, int64_t* workspace_bytes,
                                         double* flops);

/* Sizes of the memory state buffers of one sequence (elements); a batch of
 * B sequences needs B times these. */
ARMT_API armt_status armt_state_sizes(const armt_model* m, int64_t* a_elems, int64_t* z_elems);

/* Device memory the library holds for this model, in bytes (its own
 * cudaMalloc calls; the caller's tokens, outputs and memory state are not
 * counted -- armt_state_sizes gives the state):
 *   weights         stacked per-layer weights, embeddings and norm gains
 *   workspace       the cell engine's activations and scratch, one slot per
 *                   layer: fixed at armt_create, independent of the number of
 *                   segments (the recurrence's constant-memory property,
 *                   section 一 of the summary page); plus, once
 *                   armt_forward_batch has run with batch > 1, the batched
 *                   workspace for the last batch size used
 *   full_workspace  the full-attention baseline's workspace, 0 until
 *                   armt_forward_full_attention has run; it grows with the
 *                   sequence length
 * Any pointer may be NULL to skip that figure.  ARMT_ERR_ARG if m is NULL. */
ARMT_API armt_status armt_memory_bytes(const armt_model* m, int64_t* weights, int64_t* workspace,
                                       int64_t* full_workspace);

/* Number of kernel launches one forward of n_segments makes with `schedule`. */
ARMT_API armt_status armt_launch_count(const armt_model* m, int64_t n_segments, int32_t schedule,
                              int64_t* launches);

/* Per-kernel timing with CUDA events recorded on the launch stream around
 * every launch of each kernel class (off by default; enable != 0 times all
 * classes).  armt_kernel_times
 * synchronises, then returns for class c (see armt_kernel_class) the number
 * of launches and total milliseconds since the last reset, and resets. */
typedef enum armt_kernel_class {
  ARMT_KC_GEMM_QKV = 0, ARMT_KC_GEMM_O = 1, ARMT_KC_GEMM_GATEUP = 2, ARMT_KC_GEMM_DOWN = 3,
  ARMT_KC_ATTENTION = 4, ARMT_KC_ASSOC_READ = 5, ARMT_KC_ASSOC_WRITE = 6, ARMT_KC_NORM = 7,
  ARMT_KC_OTHER = 8, ARMT_KC_COUNT = 9
} armt_kernel_class;
ARMT_API armt_status armt_set_profiling(armt_model* m, int32_t enable);
/* Same, for the classes whose bit (1 << armt_kernel_class) is set in
 * class_mask only (0 = off): the other launches get no events, so timing one
 * class disturbs the rest of the forward as little as possible.  Resets the
 * recorded times.  ARMT_ERR_ARG for bits at or past ARMT_KC_COUNT. */
ARMT_API armt_status armt_set_profiling_mask(armt_model* m, uint32_t class_mask);
ARMT_API armt_status armt_kernel_times(armt_model* m, int64_t* launches, double* ms, int32_t n_classes);

/* Tracing (off by default): with enable != 0 every step is wrapped in an
 * NVTX range -- "armt diagonal i (layers lo-hi)" for the diagonal schedule,
 * "armt segment s (layers l-l)" per cell of the sequential one, "armt
 * wavefront n (layers 0-L-1)" for a persistent launch, "armt backward
 * diagonal i (layers lo-hi)" for the reverse diagonals of armt_backward --
 * so that a profiler (nsys, ncu --nvtx) can attribute or select the kernels
 * of one step.  The ranges are host-side markers on the calling thread; with
 * no profiler attached they cost a function call each, with tracing off a
 * branch. */
ARMT_API armt_status armt_set_tracing(armt_model* m, int32_t enable);

/* Waits for `stream` and reports a device-side error recorded since the last
 * call (ARMT_ERR_TIMEOUT when a bounded wait gave up), then clears it. */
ARMT_API armt_status armt_sync_status(armt_model* m, void* stream);

/* Static description of a status code; never NULL. */
ARMT_API const char* armt_status_string(armt_status s);

/* Thread-local detail of the last error returned on this thread ("" if none). */
ARMT_API const char* armt_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ARMT_H */
