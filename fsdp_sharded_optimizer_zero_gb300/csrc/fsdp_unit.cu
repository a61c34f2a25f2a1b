// FSDP unit backward ([Interview] follow-up "手写 FSDP 的一层 linear": all-gather W again,
// compute dX, compute the full-shape dW locally, reduce-scatter dW into each rank's 1/N of
// the rows; [Concepts] "ZeRO and FSDP": gather before backward, then reduce-scatter).
//
// With the N ranks on one GPU the step is, for every rank q with local batch X_q [M, K] and
// upstream gradient dY_q [M, R]:
//   dX_q = dY_q W                                  (W [R, K] gathered from its row shards)
//   dW   = (1/N) sum_q dY_q^T X_q                  (all ranks' contributions, reduced)
// and rank r's reduce-scatter result is rows [r R/N, (r+1) R/N) of dW, a contiguous block.
//
// Both products run on the tcgen05 GEMM (CTA-pair kernel). When R / N, K and M are
// multiples of 64 (and N <= 16) every operand is read where it lies, with no workspace:
//   dX_q = dY_q W   with dY_q a K-major A and W read from its row shards as an MN-major B
//                   (the backward all-gather fused into the loads, as in the forward: the
//                   shard is picked by K block). One launch over all ranks' row pieces when
//                   M % 128 == 0, else one per rank;
//   dW = (1/N) sum_q dY_q^T X_q   with dY_q and X_q both read as MN-major operands and the
//                   K loop over every rank's tokens in turn,
// so the sum over ranks happens inside the fp32 tensor-core accumulation, and the 1/N scale
// is applied in the epilogue. With the operand layouts compiled into the kernel, an
// MN-major operand costs the pair kernel 0-3 % on GB300 (Mistral W_up, 8 ranks x 2048
// tokens: dX 1.047 ms with W in place against 1.045 ms over a laid-out W^T, dW 1.016 ms
// with both operands in place), so laying out W^T, X^T or dY^T (44-49 us each) no longer
// pays. Other shapes take the transposed path: W^T [K, R], dY^T [R, N M] and X^T [K, N M]
// in the workspace, then K-major GEMMs. Every path gives the same bits.
#include <string.h>

#include <algorithm>

#include "internal.h"

using namespace zgb;

namespace {

uint64_t align256(uint64_t b) { return (b + 255) & ~uint64_t(255); }

struct BackwardWorkspace {
  uint64_t wt, dyt, xt, total;  // byte offsets of W^T, dY^T, X^T and the total size
  uint64_t min_total;           // the smallest workspace the call accepts
};

// The backward reads W, dY and X in place (MN-major GEMM operands) when every K piece is
// a whole number of 64-row K blocks (the W shards' R / N rows for dX, each rank's m_tokens
// rows for dW) and every MN-major operand's rows are whole 64-column chunks (k_in % 64 ==
// 0; R % 64 follows from R / N).
bool backward_in_place(int n, int64_t rows_out, int64_t k_in, int64_t m_tokens) {
  return n <= kGemmMaxPieces && (rows_out / n) % 64 == 0 && m_tokens % 64 == 0 && k_in % 64 == 0;
}

BackwardWorkspace backward_workspace(int n, int64_t rows_out, int64_t k_in, int64_t m_tokens) {
  BackwardWorkspace w{0, 0, 0, 0, 0};
  const uint64_t R = static_cast<uint64_t>(rows_out), K = static_cast<uint64_t>(k_in);
  const uint64_t NM = static_cast<uint64_t>(n) * static_cast<uint64_t>(m_tokens);
  if (backward_in_place(n, rows_out, k_in, m_tokens)) return w;  // no workspace
  w.wt = 0;
  w.dyt = align256(2 * R * K);
  w.xt = w.dyt + align256(2 * R * NM);
  w.total = w.min_total = w.xt + align256(2 * K * NM);
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int fsdp_transpose_cat(int n_srcs, const zero_bf16* const srcs[], int64_t rows, int64_t cols,
                                  zero_bf16* dst, zero_stream_t stream) {
  const char* who = "fsdp_transpose_cat";
  if (n_srcs < 1 || n_srcs > ZERO_MAX_RANKS)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_srcs %d outside 1..%d", who, n_srcs, ZERO_MAX_RANKS);
  if (rows < 1 || cols < 1) return set_error(ZERO_ERR_INVALID_ARG, "%s: rows and cols must be >= 1", who);
  if (!srcs || !dst) return set_error(ZERO_ERR_INVALID_ARG, "%s: NULL argument", who);
  GradPtrs sp;
  memset(&sp, 0, sizeof(sp));
  for (int q = 0; q < n_srcs; ++q) {
    if (!srcs[q]) return set_error(ZERO_ERR_INVALID_ARG, "%s: srcs[%d] is NULL", who, q);
    sp.p[q] = srcs[q];
  }
  cudaError_t e = launch_transpose_cat(sp, n_srcs, rows, cols, dst, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
  return ZERO_OK;
}

extern "C" int fsdp_unit_backward_workspace(int n_ranks, int64_t rows_out, int64_t k_in, int64_t m_tokens,
                                            uint64_t* bytes) {
  if (!bytes) return set_error(ZERO_ERR_INVALID_ARG, "fsdp_unit_backward_workspace: bytes is NULL");
  if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || rows_out < 1 || k_in < 1 || m_tokens < 1)
    return set_error(ZERO_ERR_INVALID_ARG, "fsdp_unit_backward_workspace: bad sizes");
  *bytes = backward_workspace(n_ranks, rows_out, k_in, m_tokens).total;
  return ZERO_OK;
}

extern "C" int fsdp_unit_backward(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out, int64_t k_in,
                                  const zero_bf16* const A[], const zero_bf16* const dY[], int64_t m_tokens,
                                  float* const dX[], float* dW, void* workspace, uint64_t workspace_bytes,
                                  zero_stream_t stream) {
  const char* who = "fsdp_unit_backward";
  if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_ranks %d outside 1..%d", who, n_ranks, ZERO_MAX_RANKS);
  if (rows_out < 1 || k_in < 1 || m_tokens < 1) return set_error(ZERO_ERR_INVALID_ARG, "%s: sizes must be >= 1", who);
  if (rows_out % n_ranks != 0)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: rows_out %lld is not a multiple of n_ranks %d", who,
                     (long long)rows_out, n_ranks);
  const int64_t nm = static_cast<int64_t>(n_ranks) * m_tokens;
  if (k_in % 8 || rows_out % 8 || nm % 8)
    return set_error(ZERO_ERR_INVALID_ARG,
                     "%s: k_in, rows_out and n_ranks * m_tokens must be multiples of 8 (16-byte GEMM rows)", who);
  if (!w_shards || !A || !dY || !dX || !dW) return set_error(ZERO_ERR_INVALID_ARG, "%s: NULL argument", who);
  const BackwardWorkspace ws = backward_workspace(n_ranks, rows_out, k_in, m_tokens);
  if (ws.min_total && (!workspace || workspace_bytes < ws.min_total))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: workspace of %llu bytes is below the %llu needed", who,
                     workspace ? (unsigned long long)workspace_bytes : 0ull, (unsigned long long)ws.min_total);
  if (!aligned16(dW) || (ws.min_total && !aligned16(workspace)))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: dW and workspace must be 16-byte aligned", who);
  GradPtrs wp, ap, dyp;
  memset(&wp, 0, sizeof(wp));
  memset(&ap, 0, sizeof(ap));
  memset(&dyp, 0, sizeof(dyp));
  for (int q = 0; q < n_ranks; ++q) {
    if (!w_shards[q] || !A[q] || !dY[q] || !dX[q])
      return set_error(ZERO_ERR_INVALID_ARG, "%s: a pointer of rank %d is NULL (missing rank)", who, q);
    if (!aligned16(w_shards[q]) || !aligned16(A[q]) || !aligned16(dY[q]) || !aligned16(dX[q]))
      return set_error(ZERO_ERR_INVALID_ARG, "%s: buffers of rank %d must be 16-byte aligned", who, q);
    wp.p[q] = w_shards[q];
    ap.p[q] = A[q];
    dyp.p[q] = dY[q];
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (backward_in_place(n_ranks, rows_out, k_in, m_tokens)) {
    const uint16_t* const* dy = reinterpret_cast<const uint16_t* const*>(dY);
    const uint16_t* const* wsh = reinterpret_cast<const uint16_t* const*>(w_shards);
    int rc;
    // dX_q = dY_q W with W read as its row shards: one launch over all ranks' rows when
    // each rank's M is a whole number of 128-row tiles, else one launch per rank
    if (m_tokens % 128 == 0) {
      if ((rc = launch_fsdp_bwd_dx(n_ranks, dy, m_tokens, n_ranks, wsh, rows_out, k_in, dX, st))) return rc;
    } else {
      for (int q = 0; q < n_ranks; ++q)
        if ((rc = launch_fsdp_bwd_dx(n_ranks, dy + q, m_tokens, 1, wsh, rows_out, k_in, dX + q, st))) return rc;
    }
    // dW = (1/N) sum_q dY_q^T X_q: both read in place, the K loop over every rank's tokens
    return launch_fsdp_bwd_dw_in_place(n_ranks, dy, reinterpret_cast<const uint16_t* const*>(A), m_tokens, rows_out,
                                       k_in, dW, 1.0f / static_cast<float>(n_ranks), st, nullptr, who);
  }
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint16_t* wt = reinterpret_cast<uint16_t*>(base + ws.wt);
  uint16_t* dyt = reinterpret_cast<uint16_t*>(base + ws.dyt);
  uint16_t* xt = reinterpret_cast<uint16_t*>(base + ws.xt);

  cudaError_t e = launch_transpose_cat(wp, n_ranks, rows_out / n_ranks, k_in, wt, st);
  if (e == cudaSuccess) e = launch_transpose_cat(dyp, n_ranks, m_tokens, rows_out, dyt, st);
  if (e == cudaSuccess) e = launch_transpose_cat(ap, n_ranks, m_tokens, k_in, xt, st);
  if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: transpose: %s", who, cudaGetErrorString(e));

  // dX_q [M, K] = dY_q [M, R] * (W^T [K, R])^T for every rank: one launch over all ranks'
  // rows when each rank's M is a whole number of 128-row tiles, else one launch per rank
  const uint16_t* wt1[1] = {wt};
  if (m_tokens % 128 == 0 && n_ranks <= 16) {
    int rc = launch_fsdp_gemm_row_split(n_ranks, reinterpret_cast<const uint16_t* const*>(dY), dX, m_tokens, wt,
                                        k_in, rows_out, 1.0f, st);
    if (rc) return rc;
  } else {
    for (int q = 0; q < n_ranks; ++q) {
      int rc = launch_fsdp_gemm(1, wt1, k_in, rows_out, dY[q], m_tokens, dX[q], nullptr, 1.0f, st);
      if (rc) return rc;
    }
  }
  // dW [R, K] = (1/N) dY^T [R, NM] * (X^T [K, NM])^T
  const uint16_t* xt1[1] = {xt};
  return launch_fsdp_gemm(1, xt1, k_in, nm, dyt, rows_out, dW, nullptr, 1.0f / static_cast<float>(n_ranks), st);
}

// ======================================================================================
// The full MLP unit forward of a Mistral-style block under FSDP:
//   H = silu(X W_gate^T) * (X W_up^T)      (one kernel: both projections share every X
//                                           tile; the SiLU-gate product is the epilogue)
//   Y = H W_down^T
// Each weight is all-gathered from its row shards inside the GEMM's loads. When W_down's
// shards do not tile the GEMM (or the caller prefers it), the caller passes scratch_down
// and the gather of W_down into it runs on prefetch_stream while the gate-up GEMM runs on
// `stream` — the overlap FSDP gets from issuing the next unit's all-gather on a separate
// stream ([Interview] follow-up "FSDP 怎么把通信藏起来?"; [Concepts] full sharding:
// prefetch the next layer's all-gather while the current layer computes).
// ======================================================================================

namespace {

// per-thread, per-device pair of events ordering the prefetch stream (no timing)
thread_local cudaEvent_t t_events[64][2] = {};

int prefetch_events(cudaEvent_t* ev) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64)
    return set_error(ZERO_ERR_CUDA, "fsdp_mlp_forward: cudaGetDevice failed");
  for (int i = 0; i < 2; ++i) {
    if (!t_events[dev][i]) {
      e = cudaEventCreateWithFlags(&t_events[dev][i], cudaEventDisableTiming);
      if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "fsdp_mlp_forward: cudaEventCreate: %s", cudaGetErrorString(e));
    }
    ev[i] = t_events[dev][i];
  }
  return ZERO_OK;
}

}  // namespace

extern "C" int fsdp_mlp_forward(int n_ranks, const zero_bf16* const gate_shards[], const zero_bf16* const up_shards[],
                                const zero_bf16* const down_shards[], int64_t d_model, int64_t d_ff,
                                const zero_bf16* X, int64_t m_tokens, zero_bf16* H, float* Y, zero_bf16* scratch_down,
                                zero_stream_t stream, zero_stream_t prefetch_stream) {
  const char* who = "fsdp_mlp_forward";
  if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_ranks %d outside 1..%d", who, n_ranks, ZERO_MAX_RANKS);
  if (d_model < 1 || d_ff < 1 || m_tokens < 1) return set_error(ZERO_ERR_INVALID_ARG, "%s: sizes must be >= 1", who);
  if (d_model % n_ranks || d_ff % n_ranks)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: d_model and d_ff must be multiples of n_ranks", who);
  if (d_model % 8 || d_ff % 8)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: d_model and d_ff must be multiples of 8 (16-byte rows)", who);
  if (!gate_shards || !up_shards || !down_shards || !X || !H || !Y)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: NULL argument", who);
  if (!aligned16(X) || !aligned16(H) || !aligned16(Y) || (scratch_down && !aligned16(scratch_down)))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: X, H, Y and scratch_down must be 16-byte aligned", who);
  GradPtrs dp;
  memset(&dp, 0, sizeof(dp));
  for (int q = 0; q < n_ranks; ++q) {
    if (!gate_shards[q] || !up_shards[q] || !down_shards[q])
      return set_error(ZERO_ERR_INVALID_ARG, "%s: a shard of rank %d is NULL (missing rank)", who, q);
    if (!aligned16(gate_shards[q]) || !aligned16(up_shards[q]) || !aligned16(down_shards[q]))
      return set_error(ZERO_ERR_INVALID_ARG, "%s: shards of rank %d must be 16-byte aligned", who, q);
    dp.p[q] = down_shards[q];
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t pf = prefetch_stream ? reinterpret_cast<cudaStream_t>(prefetch_stream) : st;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  if (scratch_down) {
    int rc = 0;
    if (pf != st) {
      if ((rc = prefetch_events(ev))) return rc;
      // the gather must see everything the caller queued on `stream` before this call
      cudaError_t e = cudaEventRecord(ev[0], st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(pf, ev[0], 0);
      if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
    }
    cudaError_t e = launch_gather_rows(dp, n_ranks, static_cast<uint64_t>(d_model / n_ranks) * d_ff, scratch_down,
                                       true, pf);
    if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: gather of W_down: %s", who, cudaGetErrorString(e));
    if (pf != st) {
      e = cudaEventRecord(ev[1], pf);
      if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
    }
  }
  int rc = launch_fsdp_gate_up(n_ranks, gate_shards, up_shards, d_ff, d_model, X, m_tokens, H, st);
  if (rc) return rc;
  if (scratch_down) {
    if (pf != st) {
      cudaError_t e = cudaStreamWaitEvent(st, ev[1], 0);
      if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
    }
    const uint16_t* w1[1] = {scratch_down};
    return launch_fsdp_gemm(1, w1, d_model, d_ff, H, m_tokens, Y, nullptr, 1.0f, st);
  }
  return launch_fsdp_gemm(n_ranks, down_shards, d_model, d_ff, H, m_tokens, Y, nullptr, 1.0f, st);
}
