// Internal declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/zero.h"

struct zero_plan {
  zero_layout lay;
};

namespace zgb {

// Scalars of one Adam step, prepared once on the host (bias corrections, 1 - beta,
// lr * wd, 1 / N) and passed by value to every kernel that updates state.
struct AdamScalars {
  float lr, beta1, beta2, omb1, omb2, eps, bc1, bc2, lr_wd, inv_n;
  int wd_on;
};

// N device pointers carried in kernel parameter space.
template <typename T>
struct RankPtrs {
  const T* p[ZERO_MAX_RANKS];
};
using GradPtrs = RankPtrs<uint16_t>;   // bf16 gradients (raw bits)
using F32GradPtrs = RankPtrs<float>;   // fp32 gradients (Megatron distributed optimizer)
using MasterPtrs = RankPtrs<float>;

// The elements a launch covers: n_seg segments of seg_len elements; element e of segment
// s is at flat offset s * seg_stride + e of EVERY stream of the launch (the host offsets
// each stream's base pointer before the launch).
struct Domain {
  uint64_t n_seg, seg_len, seg_stride;
};

// ---- launchers (step_kernels.cu, fused_step.cu) ----
cudaError_t launch_reduce(const GradPtrs& gp, int n, float* out, const Domain& d, float inv_n, bool vec,
                          cudaStream_t st);
cudaError_t launch_adam(const float* g, float* master, float* m, float* v, uint16_t* param, const Domain& d,
                        const AdamScalars& sc, bool vec, cudaStream_t st);
// variant: 1 = TMA bulk pipeline, 2 = register streaming, 3 = scalar (unaligned inputs)
cudaError_t launch_fused(const GradPtrs& gp, int n, float* master, float* m, float* v, uint16_t* param,
                         const Domain& d, const AdamScalars& sc, int variant, cudaStream_t st);
// fused step with fp32 gradients: variant 2 = register streaming, 3 = scalar
cudaError_t launch_fused_f32g(const F32GradPtrs& gp, int n, float* master, float* m, float* v, uint16_t* param,
                              const Domain& d, const AdamScalars& sc, int variant, cudaStream_t st);
cudaError_t launch_allgather(const MasterPtrs& mp, int n, uint64_t shard, uint16_t* full, bool vec,
                             cudaStream_t st);
cudaError_t launch_gather_rows(const GradPtrs& shards, int n, uint64_t shard_elems, uint16_t* full, bool vec,
                               cudaStream_t st);
unsigned int step_kernels_read_clear_error();
unsigned int fused_step_read_clear_error();
cudaError_t launch_wait_selftest(unsigned long long timeout_ns, cudaStream_t st);
// dst[c][q * rows + r] = srcs[q][r][c] for q < n: the N row-major [rows, cols] bf16 sources
// transposed and concatenated into one row-major [cols, n * rows] buffer
cudaError_t launch_transpose_cat(const GradPtrs& srcs, int n, int64_t rows, int64_t cols, uint16_t* dst,
                                 cudaStream_t st);
// SiLU-gate backward of H = silu(G) * U: dG | dU [rows, 2 d_ff] bf16 from dH [rows, d_ff]
// and the saved G | U [rows, 2 d_ff], elementwise in fp32
cudaError_t launch_silu_gate_backward(const uint16_t* dh, const uint16_t* gu, uint16_t* dgu, int64_t rows, int64_t d_ff,
                                      cudaStream_t st);

// ---- FSDP GEMM (fsdp_gemm.cu) ----
// Adam fused into a weight-gradient GEMM's epilogue: output element (row, col) of the
// [rows, r] fp32 result is the reduced gradient of parameter (row - split*s) * r + col of
// weight set s = (row >= split), whose fp32 master / m / v are updated and whose bf16 value
// is written, in the same operation order as zero_adam_step (same bits). Two sets serve a
// result that stacks two weights (W_gate rows, then W_up rows).
struct AdamFuse {
  float* master[2];
  float* m[2];
  float* v[2];
  uint16_t* w[2];
  int64_t split;  // rows of set 0 (>= rows for one set)
  AdamScalars sc;
};
// Y[M, R] = alpha * A[M, K] * W^T with W given as n_ranks row shards of R/n_ranks rows
// each (n_ranks = 1 with the full W for the materialised path). Both operands K-major.
int launch_fsdp_gemm(int n_ranks, const uint16_t* const* w_shards, int64_t rows_out, int64_t k_in,
                     const uint16_t* A, int64_t m_tokens, float* Y, uint16_t* Y_bf16, float alpha, cudaStream_t st);
// Y_s[rows_per_shard, R] = alpha * A_s W^T for s < a_shards in ONE persistent launch
// (rows_per_shard % 128 == 0, a_shards <= 16, R % 4 == 0, 16-byte-aligned Y_s).
int launch_fsdp_gemm_row_split(int a_shards, const uint16_t* const* A, float* const* Y, int64_t rows_per_shard,
                               const uint16_t* W, int64_t rows_out, int64_t k_in, float alpha, cudaStream_t st);
// H[M, d_ff] (bf16) = silu(X W_gate^T) * (X W_up^T), gate and up given as n_ranks row
// shards each (d_ff / n_ranks rows, a multiple of 128, or n_ranks = 1 with full weights).
// GU (nullable, [M, 2 d_ff] bf16) also receives the two projections G | U, rounded from the
// same fp32 accumulators (the activations the backward needs).
int launch_fsdp_gate_up(int n_ranks, const uint16_t* const* gate_shards, const uint16_t* const* up_shards,
                        int64_t d_ff, int64_t d_model, const uint16_t* X, int64_t m_tokens, uint16_t* H,
                        cudaStream_t st, uint16_t* GU = nullptr);
// Backward GEMMs reading every operand where it lies: a tensor stored [K, M] (or [K, N])
// for a GEMM that contracts over K is read as MN-major tiles, so no transpose is ever laid
// out. Operands given as several pieces are split along K into whole 64-row K blocks (at
// most kGemmMaxPieces pieces per operand); the results are bit-identical to the K-major
// forms over transposed copies.
// dX_q[M, K] = dY_q W (fp32) for the dy_pieces row pieces of dY / dX (dy_pieces = 1: one
// rank), W read in place from its n_ranks row shards (R / n_ranks a multiple of 64).
constexpr int kGemmMaxPieces = 16;
int launch_fsdp_bwd_dx(int n_ranks, const uint16_t* const* dY, int64_t dy_pieces_rows, int dy_pieces,
                       const uint16_t* const* w_shards, int64_t rows_out, int64_t k_in, float* const* dX,
                       cudaStream_t st);
// Y[m, n_out] = alpha A W, A [m, K] K-major, W [K, n_out] given as w_pieces row pieces of
// w_piece_rows rows (K = w_pieces * w_piece_rows; n_out a multiple of 64): a unit's input
// gradient from its weight's row shards, or from [W_gate; W_up]'s 2N shards. fp32 Y and/or
// bf16 Y_bf16 (a bf16-only output needs n_out % 8 == 0).
int launch_fsdp_gemm_w_mn(int w_pieces, const uint16_t* const* W, int64_t w_piece_rows, int64_t n_out,
                          const uint16_t* A, int64_t m, float* Y, uint16_t* Y_bf16, float alpha, cudaStream_t st,
                          const char* who);
// dW[R, K] = alpha sum over the tokens of dY^T X, dY [T, R] and X [T, K] both read in place
// as MN-major operands given as `pieces` token pieces of piece_rows rows (each rank's
// tokens, or one piece for all T = pieces * piece_rows); the K loop runs over every token,
// so the sum over ranks (the reduce of the reduce-scatter) happens in the fp32 accumulator.
// R and K multiples of 64. With adam, each row's optimizer update runs in the epilogue.
int launch_fsdp_bwd_dw_in_place(int pieces, const uint16_t* const* dY, const uint16_t* const* X, int64_t piece_rows,
                                int64_t rows_out, int64_t k_in, float* dW, float alpha, cudaStream_t st,
                                const AdamFuse* adam, const char* who);
unsigned int fsdp_gemm_read_clear_error();
int set_gemm_kernel(int which);  // 0 = default (CTA-pair kernel), 1 = one-CTA kernel everywhere, 2 = CTA-pair kernel

// Runs a set-up step (a kernel attribute) once per device until it succeeds. Unlike
// std::call_once, a failed attempt (say, under an error left pending by an earlier launch)
// leaves the device's flag clear, so the next call tries again instead of launching with
// the attribute unset.
class OncePerDevice {
 public:
  template <class F>
  cudaError_t run(int dev, F&& setup) {
    std::atomic<bool>& flag = done_[dev & 63];
    if (flag.load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (flag.load(std::memory_order_relaxed)) return cudaSuccess;
    const cudaError_t e = setup();
    if (e == cudaSuccess) flag.store(true, std::memory_order_release);
    return e;
  }

 private:
  std::atomic<bool> done_[64] = {};
  std::mutex mu_;
};

// True when fsdp_unit_forward can read W straight from its n_ranks row shards (the fused
// gather, no scratch) under the current zero_set_gemm_kernel choice.
bool fsdp_fused_gather_ok(int n_ranks, int64_t rows_out);

// ---- errors (capi.cu) ----
int set_error(int code, const char* fmt, ...);
// Adam hyper-parameters and step validated as the step calls do (ZERO_ERR_INVALID_ARG)
int check_adam_args(const zero_adam* hp, int64_t step, const char* who);
// ... and turned into the scalars every Adam kernel takes (bias corrections of `step`)
int make_adam_scalars(const zero_adam* hp, int64_t step, const char* who, AdamScalars* sc);
int num_sms();

}  // namespace zgb
