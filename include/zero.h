/*
 * zero.h — C ABI of the GB300 data-parallel optimizer-step library (libzero_gb300.so).
 *
 * What it computes: the per-step state update of DDP / ZeRO-1/2/3 / FSDP with the N
 * data-parallel ranks simulated as separate buffers on ONE GPU, plus the FSDP unit's
 * gather + linear. Sources (cited by page title and section):
 *   [Wiring]    "Behind the scenes of distributed training, and why your GPU wiring matters as
 *               much as your strategy" (automationscribe.com), Part 1: DDP, FSDP, "ZeRO: The
 *               Dial Between DDP and FSDP".
 *   [Interview] "DP、ZeRO-1/2/3、FSDP:每卡显存多少、通信多多少?" (charliedreemur.github.io,
 *               ml-interview / dp-zero-fsdp): concepts, Fig. 1, Fig. 2, key formulas, the
 *               7B / N = 8 worked table, and the follow-up on a hand-written FSDP linear.
 *   [Concepts]  "Data Parallel, ZeRO and FSDP" (k8ai.app): DDP steps, communication cost,
 *               the ZeRO / FSDP stage table, full sharding.
 *
 * Conventions (every call):
 *   - Returns zero_status: ZERO_OK (0) or a negative error. On error nothing is launched
 *     and zero_last_error() returns a thread-local message describing the cause.
 *   - Tensor arguments are raw DEVICE pointers owned by the caller (e.g. allocated by
 *     PyTorch); zero_fused_step_host alone takes page-locked host buffers. bf16 tensors
 *     are passed as zero_bf16 (raw IEEE bfloat16 bits). No call is given buffer lengths:
 *     each buffer must hold what the call's description states.
 *   - The step calls, fsdp_gather_rows and fsdp_transpose_cat accept any alignment:
 *     16-byte-aligned buffers take the vectorised path, others a scalar path with
 *     bit-identical results. The GEMM-based FSDP calls (fsdp_unit_forward and its static-
 *     scratch variant, fsdp_unit_backward, fsdp_mlp_forward), whose operands are TMA tensor
 *     maps, require 16-byte-aligned buffers and return ZERO_ERR_INVALID_ARG otherwise.
 *   - Arrays of per-rank pointers (grads[], masters[], w_shards[]) are HOST arrays of
 *     n_ranks device pointers; they are copied into the kernel's parameters, so the host
 *     array may be reused as soon as the call returns.
 *   - Every launch is asynchronous on the caller's stream (cudaStream_t; NULL = legacy
 *     default stream). Nothing on the step path allocates device memory.
 *   - Device-side checks (bounded waits in the pipelined kernels) never trap: they set a
 *     device error word that zero_device_status() reads.
 *   - Thread safety: calls may be made from several host threads; a plan is read-only
 *     after zero_plan() and may be shared.
 *
 * Arithmetic of the step (identical in every call that performs it; bit-exact with the
 * CPU oracle when buffers hold the same bytes):
 *   reduced gradient g = ((grad_0 + grad_1) + ... + grad_{N-1}) in fp32, rank order,
 *                        times f32(1/N) (the fp32 nearest 1/N);
 *   Adam (Kingma & Ba, bias-corrected, eps outside the root, decoupled weight decay),
 *   one IEEE fp32 operation per line, no fused multiply-add:
 *        m  = b1*m + (1-b1)*g;         v  = b2*v + (1-b2)*(g*g)
 *        mh = m / bc1;                 vh = v / bc2       bc_i = f32(1 - b_i^t), t >= 1
 *        den = sqrt(vh) + eps
 *        if (wd != 0) master = master - f32(lr*wd)*master
 *        master = master - lr*(mh/den)
 *   bf16 param = round-to-nearest-even(master).
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define ZERO_API __attribute__((visibility("default")))
#else
#define ZERO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* zero_stream_t; /* the same type as cudaStream_t */
typedef uint16_t zero_bf16;                /* raw bfloat16 bits */

typedef enum {
  ZERO_OK = 0,
  ZERO_ERR_INVALID_ARG = -1, /* a bad argument; nothing launched */
  ZERO_ERR_OOM = -2,         /* host allocation failed (plan object), or a plan's buffers do not fit
                                the device memory (zero_plan_check_memory) */
  ZERO_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed; message has the code */
  ZERO_ERR_UNSUPPORTED = -4, /* valid request this build / device cannot run */
  ZERO_ERR_DEVICE = -5       /* a kernel's device-side check fired (see zero_device_status) */
} zero_status;

/* Strategies ([Concepts] "ZeRO and FSDP" stage table; [Interview] Fig. 1). */
enum {
  ZERO_STAGE_DDP = 0, /* nothing sharded */
  ZERO_STAGE_1 = 1,   /* optimizer state sharded */
  ZERO_STAGE_2 = 2,   /* + gradients */
  ZERO_STAGE_3 = 3,   /* + parameters (ZeRO-3 / FSDP full shard) */
  ZERO_STAGE_MEGATRON = 4 /* Megatron distributed optimizer: bf16 params and fp32 gradients
                             kept in full, fp32 master / m / v sharded ([Interview] worked
                             table, Megatron row: 6P + 12P/N bytes) */
};

/* `rank` argument values besides 0..N-1 */
#define ZERO_RANK_VIEW (-1) /* one rank's view: per-rank pointers address S-element chunks */
#define ZERO_ALL_RANKS (-2) /* every rank's shard in one launch (full simulation) */
#define ZERO_MAX_RANKS 64

typedef struct zero_plan zero_plan_t; /* opaque; owned by the library until destroyed */

/* Layout and accounting of a plan. Element counts unless named *_bytes. */
typedef struct {
  uint64_t psi;          /* parameters */
  uint64_t psi_padded;   /* P = ceil(psi/N)*N; entries [psi, P) are padding (kept zero) */
  uint64_t shard_elems;  /* S = P/N; rank r owns flat [r*S, (r+1)*S) */
  uint64_t bucket_bytes; /* as passed to zero_plan */
  uint64_t bucket_elems; /* C = floor(bucket_bytes/(2N)) elements of every rank's shard */
  uint64_t n_buckets;    /* ceil(S/C); bucket k of rank r = flat [r*S+k*C, r*S+min((k+1)*C,S)) */
  int32_t n_ranks;
  int32_t stage;
  /* model-state bytes ONE rank keeps between steps for this stage ([Interview] "手算例子:
   * 7B、N = 8" / Fig. 1; [Concepts] stage table): DDP 16P; ZeRO-1 4P+12S; ZeRO-2 2P+14S;
   * ZeRO-3 16S; Megatron 6P+12S. Transient buffers (incoming gradient chunks, fp32 reduced
   * gradient) are not model state and are not counted. */
  uint64_t state_param_bytes, state_grad_bytes, state_master_bytes, state_m_bytes, state_v_bytes;
  uint64_t state_total_bytes;
  /* elements ONE rank moves per step per collective ([Interview] "每卡通信量"):
   * DDP and ZeRO-1/2: reduce-scatter P + all-gather P = 2P; ZeRO-3: + backward all-gather P = 3P */
  uint64_t comm_reduce_scatter, comm_all_gather_fwd, comm_all_gather_bwd, comm_total;
  /* elements one rank sends per step when each collective is a ring: (N-1)/N * comm_total
   * ([Concepts] "Communication cost": 2(N-1)/N * S bytes for an all-reduce) */
  uint64_t ring_sent_elems;
  /* algorithmic HBM bytes of one fused step over all P elements: P*(2N + 26) (read N bf16
   * grads, read+write fp32 master/m/v, write bf16 param); P*(4N + 26) for the Megatron
   * stage, whose gradients are fp32 */
  uint64_t fused_step_bytes;
} zero_layout;

/* Adam hyper-parameters (fp32). beta1, beta2 in [0, 1); eps > 0; lr, weight_decay >= 0. */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
} zero_adam;

/* ------------------------------------------------------------------------------------ */
/* plan: flat-buffer shard / bucket layout (host only; launches nothing)                  */
/* ------------------------------------------------------------------------------------ */

/* Build the layout for psi parameters over n_ranks (1..ZERO_MAX_RANKS) at `stage`, with
 * gradient buckets of bucket_bytes (bf16 bytes across all N rank segments; must be
 * >= 2*n_ranks). [Interview] "ZeRO-1 / 2 / 3": model states are cut by data-parallel rank
 * into N parts, each card keeps and updates only its 1/N; [Interview] follow-up "FSDP2 和
 * FSDP1": the flat parameter is flattened and concatenated before it is cut; [Concepts]
 * "Plain data parallel (DDP)": gradients are reduced in buckets. psi is padded to a
 * multiple of N. *out receives a new plan (free it with zero_plan_destroy). */
ZERO_API int zero_plan(uint64_t psi, int n_ranks, int stage, uint64_t bucket_bytes, zero_plan_t** out);

/* Copy the plan's layout and accounting into *out. */
ZERO_API int zero_plan_query(const zero_plan_t* plan, zero_layout* out);

/* Flat index range [*begin, *end) of bucket `bucket` in rank `rank`'s shard. */
ZERO_API int zero_bucket_range(const zero_plan_t* plan, int rank, uint64_t bucket, uint64_t* begin, uint64_t* end);

/* Free a plan (NULL is accepted). */
ZERO_API int zero_plan_destroy(zero_plan_t* plan);

/* Memory check before any buffer is allocated ([Wiring] "Fully Sharded Data Parallel
 * (FSDP)": Mistral-7B ran out of memory under DDP, where every GPU holds the whole model
 * state; the sharded stages exist so that it fits). *need_bytes receives the bytes of the
 * device buffers one step call addresses in rank mode `rank` (the pointer conventions
 * below), with G = 2 bytes per gradient element (4 for a ZERO_STAGE_MEGATRON plan):
 *   rank = r:              N * P * G (every rank's gradient buffer) + 12 S (master, m, v)
 *                          + 2 P (bf16 parameters; 2 S for ZeRO-3);
 *   ZERO_RANK_VIEW:        N * S * G + 12 S + 2 S;
 *   ZERO_ALL_RANKS:        N * P * G + 12 P + 2 P.
 * budget_bytes: the memory the caller can give the step; 0 = this device's free memory
 * (cudaMemGetInfo on the current device). *budget_out (nullable) receives the budget used.
 * Returns ZERO_OK when need <= budget, ZERO_ERR_OOM when it is not (the message states both
 * figures), ZERO_ERR_CUDA if the free memory cannot be read. Launches and allocates
 * nothing. */
ZERO_API int zero_plan_check_memory(const zero_plan_t* plan, int rank, uint64_t budget_bytes, uint64_t* need_bytes,
                                    uint64_t* budget_out);

/* ------------------------------------------------------------------------------------ */
/* the step                                                                              */
/* ------------------------------------------------------------------------------------ */
/* Pointer conventions by `rank` (S = shard_elems, P = psi_padded):
 *   rank = r in [0, N): grads[q] = rank q's full P-element bf16 gradient; the call reads
 *       elements [r*S, (r+1)*S) of each. g_shard / master / m / v address rank r's
 *       S-element shard. param_out: stages 0-2 = the full P-element bf16 parameter buffer,
 *       written at [r*S, (r+1)*S) (the all-gather's destination); stage 3 = rank r's own
 *       S-element bf16 shard.
 *   rank = ZERO_RANK_VIEW: grads[q] = the S-element chunk rank q contributes to this shard;
 *       every other buffer is S elements.
 *   rank = ZERO_ALL_RANKS: every rank's shard at once; grads[q] full P-element buffers and
 *       g / master / m / v / param_out all P-element flat buffers (rank r's shard at r*S).
 */

/* Reduce-scatter ([Wiring] "ZeRO: The Dial Between DDP and FSDP": sums everyone's gradients
 * but gives each GPU only its slice; [Interview] "reduce-scatter 与 all-gather"):
 * g_shard[i] = fp32 rank-order sum of the N bf16 contributions times f32(1/N). */
ZERO_API int zero_reduce_scatter(const zero_plan_t* plan, int rank, const zero_bf16* const grads[],
                        float* g_shard, zero_stream_t stream);

/* Adam on a shard's fp32 master/m/v with the fp32 reduced gradient g_shard (updated in
 * place). step counts from 1. param_out may be NULL (no bf16 cast); otherwise it receives
 * bf16(master) as described above. ([Interview] DDP item: bf16 param + bf16 grad + fp32
 * master, m, v = 16 bytes per parameter; [Wiring] Adam keeps momentum and variance.) */
ZERO_API int zero_adam_step(const zero_plan_t* plan, int rank, const float* g_shard, float* master, float* m,
                   float* v, zero_bf16* param_out, const zero_adam* hp, int64_t step,
                   zero_stream_t stream);

/* Reduce-scatter + Adam + bf16 cast / all-gather write in ONE pass over HBM: each byte of
 * gradient and state is read once and each result written once. Same arguments as the two
 * calls above without g_shard. Results are bit-identical to zero_reduce_scatter followed
 * by zero_adam_step. */
ZERO_API int zero_fused_step(const zero_plan_t* plan, int rank, const zero_bf16* const grads[], float* master,
                    float* m, float* v, zero_bf16* param_out, const zero_adam* hp, int64_t step,
                    zero_stream_t stream);

/* zero_fused_step with the gradients and the bf16 parameters in HOST memory: host_grads[q]
 * and host_param_out must be page-locked (cudaHostAlloc / cudaMallocHost /
 * cudaHostRegister) and mapped for the device; the kernel reads every rank's gradient
 * straight from host memory and writes the parameters straight back over the host link
 * (NVLink-C2C on Grace-Blackwell), so each byte crosses the link once and no device
 * staging buffer exists. master / m / v stay in device memory. Pointer conventions and
 * results as zero_fused_step; a buffer that is not page-locked host memory the device
 * can address is rejected with ZERO_ERR_INVALID_ARG (checked with
 * cudaPointerGetAttributes before anything is launched). */
ZERO_API int zero_fused_step_host(const zero_plan_t* plan, int rank, const zero_bf16* const host_grads[],
                                  float* master, float* m, float* v, zero_bf16* host_param_out, const zero_adam* hp,
                                  int64_t step, zero_stream_t stream);

/* zero_fused_step with fp32 gradient contributions: grads[q] are fp32 (Megatron
 * distributed optimizer, gradients accumulated and reduced in fp32 — [Interview] worked
 * table, Megatron row and note). Same pointer conventions and arithmetic (the widening of
 * the gradient is the identity); 4N + 26 bytes per parameter. Valid with any plan; the
 * ZERO_STAGE_MEGATRON plan accounts its memory. */
ZERO_API int zero_fused_step_fp32_grads(const zero_plan_t* plan, int rank, const float* const grads[], float* master,
                                        float* m, float* v, zero_bf16* param_out, const zero_adam* hp, int64_t step,
                                        zero_stream_t stream);

/* As zero_fused_step, restricted to buckets [bucket_begin, bucket_end) of the shard(s):
 * the unit DDP / ZeRO reduce as soon as backward has produced a bucket ([Concepts] "Plain
 * data parallel (DDP)"). Pointers follow the same convention (whole-shard / whole-buffer
 * bases); the call offsets them to the buckets. Calls on disjoint bucket ranges touch
 * disjoint memory, so a caller may issue them on different streams and let them overlap
 * (one launch's ramp-up runs during another's drain; the results are the same bits). */
ZERO_API int zero_fused_step_buckets(const zero_plan_t* plan, int rank, uint64_t bucket_begin, uint64_t bucket_end,
                            const zero_bf16* const grads[], float* master, float* m, float* v,
                            zero_bf16* param_out, const zero_adam* hp, int64_t step, zero_stream_t stream);

/* Parameter all-gather ([Interview] "reduce-scatter 与 all-gather"; ZeRO-1/2 after the
 * update): full_param[r*S + i] = bf16(masters[r][i]) for every rank r, masters[r] being
 * rank r's S-element fp32 master shard. full_param has P elements. */
ZERO_API int zero_allgather_params(const zero_plan_t* plan, const float* const masters[], zero_bf16* full_param,
                          zero_stream_t stream);

/* DDP all-reduce = reduce-scatter + all-gather ([Wiring] "ZeRO: The Dial Between DDP and
 * FSDP"; [Concepts] "Plain data parallel (DDP)" step 2): g_full[j] = fp32 rank-order sum
 * of grads[q][j] times f32(1/N) for all j < P. Each rank's reduce-scatter result lands at
 * its own offset r*S of g_full, so the all-gather is in place. */
ZERO_API int ddp_allreduce(const zero_plan_t* plan, const zero_bf16* const grads[], float* g_full,
                  zero_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* FSDP unit ([Interview] follow-up "手写 FSDP 的一层 linear"; Fig. 2)                     */
/* ------------------------------------------------------------------------------------ */

/* All-gather of dim-0 row shards: w_full[r*R/N + j][c] = w_shards[r][j][c] (bit copy).
 * w_shards[r]: row-major [rows_out/N, k_in] bf16; w_full: row-major [rows_out, k_in].
 * rows_out % n_ranks must be 0. */
ZERO_API int fsdp_gather_rows(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out, int64_t k_in,
                     zero_bf16* w_full, zero_stream_t stream);

/* Forward of an FSDP unit's linear on the local batch: Y = A * W^T with W [rows_out, k_in]
 * (the [out, in] layout of a linear layer) assembled from its N row shards, fp32
 * accumulation on the tensor cores. A: row-major [m_tokens, k_in] bf16. Y: row-major
 * [m_tokens, rows_out] fp32. Y_bf16 (nullable): bf16 copy of Y (round-to-nearest-even).
 * Y may be NULL when Y_bf16 is given (needs rows_out % 8 == 0): only the bf16 result is
 * written, with the same bits as the bf16 copy, and half the output bytes.
 * scratch_w (nullable): a [rows_out, k_in] bf16 buffer; if given, the shards are first
 * gathered into it (fsdp_gather_rows) and the GEMM reads the gathered W, which the caller
 * frees after use; if NULL the gather is fused into the GEMM's loads (each tile is loaded
 * straight from its shard), which needs (rows_out/n_ranks) % 128 == 0 (% 256 under
 * zero_set_gemm_kernel(1)).
 * Requires k_in % 8 == 0 (16-byte rows for the tensor-memory copies), and 16-byte-aligned
 * A, shards and scratch_w. Results are fp32 sums of exact bf16 products in an unspecified
 * order: within K * 2^-23 * sum|a*w| of the exact value. */
ZERO_API int fsdp_unit_forward(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out, int64_t k_in,
                      const zero_bf16* A, int64_t m_tokens, float* Y, zero_bf16* Y_bf16, zero_bf16* scratch_w,
                      zero_stream_t stream);

/* The backward's operand layout step, as a call of its own (fsdp_unit_backward uses it on
 * shapes its in-place GEMMs do not take): dst[c][q*rows + r] = srcs[q][r][c] for q <
 * n_srcs — the n_srcs row-major [rows, cols] bf16 sources transposed and concatenated into
 * one row-major [cols, n_srcs*rows] bf16 buffer (W^T from W's row shards is the backward
 * all-gather of [Interview] follow-up "手写 FSDP 的一层 linear", landing transposed; the
 * ranks' dY^T and X^T are the operands of the reduced dW). Any alignment; 16-byte-aligned
 * buffers with cols and n_srcs*rows multiples of 8 take 16-byte accesses. */
ZERO_API int fsdp_transpose_cat(int n_srcs, const zero_bf16* const srcs[], int64_t rows, int64_t cols, zero_bf16* dst,
                                zero_stream_t stream);

/* Bytes of device workspace fsdp_unit_backward needs. When R/N, k_in and m_tokens are
 * multiples of 64 and N <= 16, every operand is read where it lies (W from its row shards
 * for dX, dY and X for dW, as MN-major tensor-core operands): 0 bytes. Other shapes need
 * transposed copies W^T (2*R*K bytes), dY^T (2*R*N*M) and X^T (2*K*N*M), each rounded up
 * to 256 bytes. */
ZERO_API int fsdp_unit_backward_workspace(int n_ranks, int64_t rows_out, int64_t k_in, int64_t m_tokens,
                                          uint64_t* bytes);

/* Backward of the FSDP unit's linear for all N simulated ranks ([Interview] follow-up
 * "手写 FSDP 的一层 linear": all-gather W again, dX, full-shape dW, reduce-scatter of dW into
 * each rank's 1/N of the rows; [Concepts] "ZeRO and FSDP" full-shard steps 2-3).
 * w_shards[r]: row-major [rows_out/N, k_in] bf16 (rank r's rows of W [R, K]);
 * A[q]: rank q's local activations, row-major [m_tokens, k_in] bf16;
 * dY[q]: rank q's upstream gradient, row-major [m_tokens, rows_out] bf16;
 * dX[q]: out, row-major [m_tokens, k_in] fp32: dX_q = dY_q W;
 * dW: out, row-major [rows_out, k_in] fp32: dW = (1/N) sum_q dY_q^T X_q; rank r's
 *     reduce-scattered shard is rows [r*R/N, (r+1)*R/N).
 * workspace: device buffer of fsdp_unit_backward_workspace() bytes (caller-owned scratch);
 *     may be NULL when that size is 0.
 * Requires rows_out % N == 0 and k_in, rows_out, N*m_tokens multiples of 8; all buffers
 * 16-byte aligned. fp32 accumulation on the tensor cores in an unspecified order: each dX
 * entry is within (R+1) 2^-23 sum|dy w| and each dW entry within (N M + 1) 2^-23 (1/N)
 * sum|dy x| (+ half an ulp for the 1/N scale) of the exact value. */
ZERO_API int fsdp_unit_backward(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out, int64_t k_in,
                                const zero_bf16* const A[], const zero_bf16* const dY[], int64_t m_tokens,
                                float* const dX[], float* dW, void* workspace, uint64_t workspace_bytes,
                                zero_stream_t stream);

/* Forward of a full FSDP MLP unit (Mistral-style): H = silu(X W_gate^T) * (X W_up^T) and
 * Y = H W_down^T, each weight all-gathered from its N row shards ([Interview] Fig. 2 and
 * the follow-up on hiding FSDP communication; [Concepts] full sharding with prefetch).
 * gate_shards[r], up_shards[r]: row-major [d_ff/N, d_model] bf16; down_shards[r]:
 * row-major [d_model/N, d_ff] bf16; X: row-major [m_tokens, d_model] bf16.
 * H: out, row-major [m_tokens, d_ff] bf16 (silu(g) u computed in fp32 from the fp32
 * accumulators, one rounding to bf16); Y: out, row-major [m_tokens, d_model] fp32.
 * The gate and up projections run in one kernel sharing every X tile, with the SiLU-gate
 * product as its epilogue (needs d_ff/N % 128 == 0). W_down is gathered inside the loads
 * when d_model/N % 128 == 0 (% 256 under zero_set_gemm_kernel(1)) and scratch_down is
 * NULL; otherwise pass scratch_down
 * ([d_model, d_ff] bf16): its gather then runs on prefetch_stream (NULL = `stream`)
 * while the gate-up GEMM runs, and `stream` waits for it before the down projection.
 * d_model, d_ff multiples of 8; all buffers 16-byte aligned. */
ZERO_API int fsdp_mlp_forward(int n_ranks, const zero_bf16* const gate_shards[], const zero_bf16* const up_shards[],
                              const zero_bf16* const down_shards[], int64_t d_model, int64_t d_ff, const zero_bf16* X,
                              int64_t m_tokens, zero_bf16* H, float* Y, zero_bf16* scratch_down, zero_stream_t stream,
                              zero_stream_t prefetch_stream);

/* ------------------------------------------------------------------------------------ */
/* ZeRO-3 / FSDP training step over a stack of units ([Interview] Fig. 2 and the follow-up */
/* "FSDP 怎么把通信藏起来?"; [Concepts] "ZeRO and FSDP", full-shard steps 1-3)             */
/* ------------------------------------------------------------------------------------ */

/* One FSDP unit: a linear layer Y = X W^T whose weight W [rows_out, k_in] is held as N
 * dim-0 row shards, its ZeRO-3 state, and the activations of every simulated rank. With
 * M tokens per rank, rank q's rows of the [N*M, .] buffers are [q*M, (q+1)*M). */
typedef struct {
  int64_t rows_out, k_in;  /* W [rows_out, k_in]; rows_out % N == 0; unit i+1's k_in == unit i's rows_out */
  const zero_plan_t* plan; /* zero_plan(rows_out * k_in, N, ZERO_STAGE_3, any bucket): rank r's shard = rows
                              [r*R/N, (r+1)*R/N) of W, flat elements [r*S, (r+1)*S) */
  zero_bf16* w;            /* [rows_out, k_in] bf16, the N shards back to back; the step writes the new shards */
  float *master, *m, *v;   /* [rows_out * k_in] fp32 each, rank r's shard at r*S; updated in place */
  zero_bf16* x;            /* [N*M, k_in] bf16: the unit's input. Unit 0: the caller's batch (read); unit i > 0:
                              written by the forward (unit i-1's output) and kept for the backward */
  zero_bf16* dy;           /* [N*M, rows_out] bf16: the gradient of the unit's output. Last unit: the caller's
                              loss gradient (read); unit i < last: written by unit i+1's backward (its dX) */
  float* dw;               /* out, [rows_out, k_in] fp32: dW = (1/N) sum_q dY_q^T X_q; rank r's reduce-scattered
                              gradient = rows [r*R/N, (r+1)*R/N), which its Adam consumes. May be NULL (not
                              written) unless the optimizer runs as its own launch */
} fsdp_unit_state;

/* flags of fsdp_zero3_step */
#define FSDP_GATHER_MATERIALIZE 1 /* gather each unit's W into a workspace slot (the all-gather's receive
                                     buffer: sharded model + the unit in use) before its forward and again
                                     before its backward; without it both GEMMs read every tile straight
                                     from its shard */
#define FSDP_BACKWARD_PREFETCH 2  /* with FSDP_GATHER_MATERIALIZE: issue unit i-1's gather on prefetch_stream
                                     while unit i's backward runs on `stream`; without it, no effect */
#define FSDP_OVERLAP_OPTIMIZER 4  /* run unit i's Adam as its own launch on prefetch_stream once its dW is
                                     done, beside the following units' backward GEMMs on `stream` */
#define FSDP_SEPARATE_OPTIMIZER 8 /* run each Adam as its own launch (zero_adam_step) after the dW GEMM on
                                     `stream`. Without this flag or the one above, each rank's Adam is fused
                                     into the dW GEMM's epilogue: it updates the shard's fp32 state and writes
                                     its bf16 values from the fp32 result as it leaves the accumulator (the
                                     same operations, the same bits), and dW is written only if given */

/* Bytes of device workspace fsdp_zero3_step needs for these units, M tokens per rank and
 * flags: 0 without FSDP_GATHER_MATERIALIZE; with it, one slot (two with
 * FSDP_BACKWARD_PREFETCH) for the gathered W of the largest unit, 2*rows_out*k_in bytes
 * rounded up to 256. Only the units' sizes are read. */
ZERO_API int fsdp_zero3_step_workspace(int n_ranks, int n_units, const fsdp_unit_state* units, int64_t m_tokens,
                                       int flags, uint64_t* bytes);

/* One training step of a stack of n_units FSDP units under ZeRO-3, for all N simulated
 * ranks (M = m_tokens each), following a unit's life on a card ([Interview] Fig. 2):
 *   forward, unit 0 -> last: gather W_i (fused into the GEMM's loads, or into a workspace
 *     slot), X_{i+1} = bf16(X_i W_i^T) for every rank (the last unit's output goes to y_out;
 *     with y_out NULL that product is skipped), W_i freed;
 *   backward, last -> unit 0: gather W_i again (fused into the dX GEMM's loads, which read
 *     W_i's shards as an MN-major operand, or into the slot), dY_{i-1} = bf16(dY_i W_i)
 *     (unit 0: into dx_out, skipped when NULL), dW_i = (1/N) sum_q dY_{i,q}^T X_{i,q} (dY_i
 *     and X_i read in place as MN-major operands; the reduce of the reduce-scatter inside
 *     the fp32 tensor-core accumulation, rank r keeping its rows),
 *     then each rank's Adam on its shard (the operations of zero_adam_step, fused into the
 *     dW GEMM's epilogue by default) writing the new bf16 shards of W_i — after W_i's last
 *     use;
 *   with FSDP_GATHER_MATERIALIZE and FSDP_BACKWARD_PREFETCH, unit i-1's gather runs on
 *     prefetch_stream while unit i computes ([Interview] follow-up "FSDP 怎么把通信藏起来?":
 *     the all-gather on its own stream, the backward prefetching the next unit's);
 *   with FSDP_OVERLAP_OPTIMIZER, unit i's Adam runs on prefetch_stream after its dW, while
 *     the backward of the units below it runs on `stream`.
 * All work is ordered on `stream` by the time the call returns (prefetch_stream joins it).
 * Results do not depend on the flags (same bits). dX / dY products are fp32 sums of exact
 * bf16 products in an unspecified order (bounds as fsdp_unit_backward), rounded once to
 * bf16; Adam is bit-exact as zero_adam_step.
 * Requires 1 <= N <= 16, 1 <= n_units <= 64, N*M % 8 == 0; per unit rows_out a multiple of
 * N with rows_out / N and k_in multiples of 64 (the backward reads W's shards, dY and X in
 * place), and without FSDP_GATHER_MATERIALIZE the fused gather's shard rule ((rows_out /
 * N) % 128 == 0; 256 under zero_set_gemm_kernel(1)); 16-byte-aligned buffers; workspace of
 * fsdp_zero3_step_workspace() bytes (NULL when 0). prefetch_stream may be NULL (then
 * everything runs on `stream`). */
ZERO_API int fsdp_zero3_step(int n_ranks, int n_units, const fsdp_unit_state* units, int64_t m_tokens,
                             zero_bf16* y_out, zero_bf16* dx_out, const zero_adam* hp, int64_t step, int flags,
                             void* workspace, uint64_t workspace_bytes, zero_stream_t stream,
                             zero_stream_t prefetch_stream);

/* The ZeRO-3 state of one weight [rows, cols] of an FSDP unit. */
typedef struct {
  const zero_plan_t* plan; /* zero_plan(rows * cols, N, ZERO_STAGE_3, any bucket): rank r's shard = rows
                              [r*rows/N, (r+1)*rows/N), flat elements [r*S, (r+1)*S) */
  zero_bf16* w;            /* [rows, cols] bf16, the N row shards back to back; the step writes the new shards */
  float *master, *m, *v;   /* [rows * cols] fp32 each, rank r's shard at r*S; updated in place */
} fsdp_weight_state;

/* One Mistral-style FSDP MLP unit: H = silu(X W_gate^T) * (X W_up^T), Y = H W_down^T, for all
 * N simulated ranks (M tokens each; rank q's rows of every [N*M, .] buffer are [q*M, (q+1)*M)). */
typedef struct {
  int64_t d_model, d_ff;
  fsdp_weight_state gate, up; /* W_gate, W_up [d_ff, d_model] */
  fsdp_weight_state down;     /* W_down [d_model, d_ff] */
  zero_bf16* x;     /* [N*M, d_model]: the input. Unit 0: the caller's batch (read); unit i > 0: written by
                       the forward (unit i-1's output) */
  zero_bf16* gu;    /* out, [N*M, 2*d_ff]: G | U = X W_gate^T | X W_up^T, rounded from the fp32 accumulators
                       (the activations the backward reads) */
  zero_bf16* h;     /* out, [N*M, d_ff]: H, the down projection's input */
  zero_bf16* dy;    /* [N*M, d_model]: the gradient of the unit's output. Last unit: the caller's (read);
                       unit i < last: written by unit i+1's backward */
  zero_bf16* dh;    /* out, [N*M, d_ff]: dH = dY W_down */
  zero_bf16* dgu;   /* out, [N*M, 2*d_ff]: dG | dU, the SiLU-gate backward of dH */
  float* dw_gu;     /* out, [2*d_ff, d_model]: (1/N) sum_q [dG | dU]_q^T X_q = dW_gate (rows 0..d_ff-1)
                       stacked on dW_up (rows d_ff..): each rank's reduce-scattered rows feed its Adam.
                       May be NULL (not written) unless FSDP_SEPARATE_OPTIMIZER */
  float* dw_down;   /* out, [d_model, d_ff]: (1/N) sum_q dY_q^T H_q; NULL as dw_gu */
} fsdp_mlp_unit_state;

/* Bytes of device workspace fsdp_zero3_mlp_step needs: 0 for N <= 8, where every backward
 * GEMM reads its operands in place (the dX GEMM takes the 2N shards of W_gate and W_up as
 * its pieces); for N > 8 one slot for the gathered [W_gate; W_up] of the largest unit,
 * 4*d_ff*d_model bytes rounded up to 256. */
ZERO_API int fsdp_zero3_mlp_step_workspace(int n_ranks, int n_units, const fsdp_mlp_unit_state* units,
                                           int64_t m_tokens, uint64_t* bytes);

/* One ZeRO-3 training step of a stack of n_units FSDP MLP units for all N ranks, each unit
 * following its life on a card ([Interview] Fig. 2; "FSDP" item: gather before use, free
 * after, reduce-scatter the gradient):
 *   forward, unit 0 -> last: G | U and H = silu(G) * U in one tensor-core kernel (the gate
 *     and up shards gathered inside its loads), then X_{i+1} = bf16(H W_down^T) (the last
 *     unit's output to y_out; skipped when NULL);
 *   backward, last -> unit 0 (every GEMM operand read where it lies, K-major or MN-major):
 *     dH = bf16(dY W_down), W_down's shards gathered again inside the loads;
 *     dW_down = (1/N) sum_q dY_q^T H_q with each rank's Adam on its W_down shard in the GEMM's
 *     epilogue (or, with FSDP_SEPARATE_OPTIMIZER in flags, as its own launch); dG | dU by the
 *     SiLU-gate backward (s = 1/(1 + exp(-g)): dU = dH g s, dG = dH U s (1 + g (1 - s)), fp32
 *     from the saved bf16 G, U and dH, rounded to bf16); dY_{i-1} = bf16([dG | dU] [W_gate;
 *     W_up]) over the 2N shards of both (gathered into the workspace first when N > 8;
 *     unit 0: into dx_out, skipped when NULL); dW_gate | dW_up = (1/N) sum_q [dG | dU]_q^T X_q with each rank's Adam on its
 *     W_gate and W_up shards in the same way. Every weight's update follows its last read.
 * The reduce over ranks happens inside the fp32 accumulation of each dW GEMM; rank r's
 * reduce-scattered gradient is its rows. GEMM outputs are fp32 sums of exact bf16 products
 * in an unspecified order, rounded once to bf16 where the output is bf16; Adam is bit-exact as
 * zero_adam_step. All work is ordered on `stream`.
 * Requires 1 <= N <= 16, 1 <= n_units <= 64, N*M % 8 == 0, d_model and d_ff multiples of 64,
 * unit i+1's d_model equal to unit i's, (d_ff / N) % 128 == 0 and d_model / N tiling the fused
 * gather ((d_model / N) % 128 == 0; 256 under zero_set_gemm_kernel(1)); 16-byte-aligned
 * buffers; workspace of fsdp_zero3_mlp_step_workspace() bytes (NULL when 0). */
ZERO_API int fsdp_zero3_mlp_step(int n_ranks, int n_units, const fsdp_mlp_unit_state* units, int64_t m_tokens,
                                 zero_bf16* y_out, zero_bf16* dx_out, const zero_adam* hp, int64_t step, int flags,
                                 void* workspace, uint64_t workspace_bytes, zero_stream_t stream);

/* Allocation-free variant of fsdp_unit_forward, for callers that cannot allocate device
 * memory where they run the unit (e.g. a plug-in inside a framework that owns all device
 * memory through its own pool, or a latency-critical path that cannot take cudaMalloc's
 * device-wide synchronisation). The pages have no counterpart to this call.
 * Arguments as fsdp_unit_forward without scratch_w. When the shards tile the GEMM (the
 * fused gather of fsdp_unit_forward applies: n_ranks <= 16 and rows_out/n_ranks a multiple
 * of 128, of 256 under zero_set_gemm_kernel(1)), W is read straight from its shards and no
 * scratch is used. Otherwise W is gathered first into a 16 MiB array inside this library
 * (8,388,608 bf16 elements; rows_out * k_in above that returns ZERO_ERR_INVALID_ARG), then
 * the same GEMM runs. It allocates nothing. Every GPU that loads the library holds the
 * array until the process exits. Each call outside stream capture looks up the array's
 * address in the current device's current context; a call during capture reuses the
 * address found in that same context, so make the first call on a device (and the first
 * after a cudaDeviceReset) before any stream capture. All calls share the array and it
 * keeps the last call's W; calls that overlap on the GPU race on it. */
ZERO_API int fsdp_unit_forward_static_scratch(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out,
                                              int64_t k_in, const zero_bf16* A, int64_t m_tokens, float* Y,
                                              zero_bf16* Y_bf16, zero_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* status                                                                                */
/* ------------------------------------------------------------------------------------ */

/* Message for the last error on this host thread ("" if none). Valid until the next call
 * on this thread. */
ZERO_API const char* zero_last_error(void);

/* Synchronise `stream`, then read and clear the device error word that bounded waits set
 * (current device). Returns ZERO_OK, ZERO_ERR_DEVICE (message names the kernel and wait)
 * or ZERO_ERR_CUDA. */
ZERO_API int zero_device_status(zero_stream_t stream);

/* Check of the library's failure path, not part of the method: launches one thread that
 * waits on an mbarrier nothing arrives on, through the same bounded wait the pipelined
 * kernels use, with a limit of timeout_ms (1..2000). The wait runs out, records its code
 * (0x301) in the device error word and the kernel returns; the next zero_device_status()
 * reports ZERO_ERR_DEVICE and the context stays usable. Nothing traps or faults. */
ZERO_API int zero_selftest_bounded_wait(uint32_t timeout_ms, zero_stream_t stream);

/* Select the fused-step kernel: 0 = default (the register-streaming kernel), 1 = TMA
 * bulk-copy pipeline staging the N rank chunks in shared memory, 2 = register-streaming.
 * All give bit-identical results (misaligned buffers always take a scalar kernel). */
ZERO_API int zero_set_fused_kernel(int which);

/* Select the tensor-core GEMM kernel of the FSDP calls. 0 = default: the CTA-pair kernel
 * (tcgen05.mma.cta_group::2, a cluster of two CTAs on two SMs per 256-row tile) for every
 * GEMM, K-major or MN-major operands alike. 1 = the one-CTA kernel everywhere; 2 = the
 * CTA-pair kernel everywhere (the same as 0). All give bit-identical
 * results (each output sums the same products in the same order). The fused gather needs
 * rows_out / n_ranks to be a multiple of 128 on the pair kernel, of 256 on the one-CTA
 * kernel. Process-wide; affects calls made after it returns. */
ZERO_API int zero_set_gemm_kernel(int which);

/* Library version, e.g. 100 for 0.1.0. */
ZERO_API int zero_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_GB300_H */
