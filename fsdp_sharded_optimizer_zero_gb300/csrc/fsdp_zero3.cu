// One ZeRO-3 / FSDP training step over a stack of FSDP units, for all N simulated ranks.
//
// A unit's life on a card ([Interview] Fig. 2; [Concepts] "ZeRO and FSDP", full-shard
// steps 1-3): only its 1/N row shard is kept between uses; the full W exists only while
// the unit computes (gathered before the forward, freed, gathered again before the
// backward); after the backward the weight gradient is reduce-scattered so each rank keeps
// the rows of its own shard, and each rank's Adam updates that shard alone.
//
// Here both gathers (before the forward and again before the backward) read the N shards
// where they lie: inside the GEMMs' operand loads (the default: no copy of W exists at
// all; the backward's dX GEMM reads the shards as an MN-major operand, picking the shard by
// K block), or, with FSDP_GATHER_MATERIALIZE, by a gather kernel into a workspace slot
// that plays the all-gather's receive buffer. The dW GEMM reads dY and X where they lie
// too (both MN-major), so the backward lays out no transpose. The reduce of the
// reduce-scatter happens inside the dW GEMM's fp32 accumulation (its K loop runs over
// every rank's tokens), so rank r's reduce-scattered gradient is simply rows
// [r R/N, (r+1) R/N) of dW, contiguous with its flat-parameter shard.
//
// Overlap ([Interview] follow-up "FSDP 怎么把通信藏起来?": the all-gather on its own CUDA
// stream, the backward prefetching the next unit's): with FSDP_GATHER_MATERIALIZE,
// FSDP_BACKWARD_PREFETCH and a prefetch stream, unit i-1's gather is issued on the
// prefetch stream once unit i's dX GEMM is enqueued, into the other of two slots; events
// order each slot's reuse and each unit's start. With the fused gather there is no copy to
// prefetch and the flag changes nothing. Forward prefetch stays off (the pages' default).
//
// Ordering inside a unit's backward: dX (reads W_i), then dW with each rank's Adam, which
// writes the new W_i shards. Unit i's W is not read again in this step (unit i-1's backward
// reads W_{i-1} and the dY that unit i produced from the old W_i), so the update can follow
// each unit. By default the update is fused into the dW GEMM's epilogue: rank r's
// reduce-scattered gradient is rows [r R/N, (r+1) R/N) of dW, the same flat elements as its
// shard, so the epilogue applies Adam to each fp32 result as it leaves the accumulator
// (the same operations as zero_adam_step, the same bits). dW then needs no HBM round trip
// (it is written only when the caller passes dw), and the update's state traffic runs
// beside the GEMM's tensor work instead of after it. FSDP_SEPARATE_OPTIMIZER keeps
// zero_adam_step as its own launch after the dW GEMM; FSDP_OVERLAP_OPTIMIZER puts that
// launch on the prefetch stream, beside the following units' GEMMs.
#include <string.h>

#include <algorithm>
#include <vector>

#include "internal.h"

using namespace zgb;

namespace {

const char* const kWho = "fsdp_zero3_step";

uint64_t align256(uint64_t b) { return (b + 255) & ~uint64_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct Zero3Workspace {
  int slots;           // gathered-W slots: 2 with a materialised gather and backward prefetch, 1
                       // with a materialised gather, 0 with the fused gather
  uint64_t w_off[2];   // the unit's gathered W [rows_out, k_in] bf16
  uint64_t total;
};

Zero3Workspace zero3_workspace(int n_units, const fsdp_unit_state* u, int flags) {
  Zero3Workspace w;
  memset(&w, 0, sizeof(w));
  if (!(flags & FSDP_GATHER_MATERIALIZE)) return w;
  uint64_t wmax = 0;
  for (int i = 0; i < n_units; ++i)
    wmax = std::max<uint64_t>(wmax, static_cast<uint64_t>(u[i].rows_out) * static_cast<uint64_t>(u[i].k_in));
  w.slots = (flags & FSDP_BACKWARD_PREFETCH) ? 2 : 1;
  for (int s = 0; s < w.slots; ++s) w.w_off[s] = static_cast<uint64_t>(s) * align256(2 * wmax);
  w.total = static_cast<uint64_t>(w.slots) * align256(2 * wmax);
  return w;
}

// per-thread, per-device events ordering the prefetch stream (no timing)
thread_local std::vector<cudaEvent_t> t_events[64];

int get_events(size_t count, cudaEvent_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return set_error(ZERO_ERR_CUDA, "%s: cudaGetDevice failed", kWho);
  std::vector<cudaEvent_t>& v = t_events[dev];
  while (v.size() < count) {
    cudaEvent_t ev = nullptr;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: cudaEventCreate: %s", kWho, cudaGetErrorString(e));
    v.push_back(ev);
  }
  *out = v.data();
  return ZERO_OK;
}

int check_units(int n, int n_units, const fsdp_unit_state* u, int64_t m, int flags, bool buffers) {
  if (n < 1 || n > kGemmMaxPieces)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_ranks %d outside 1..%d", kWho, n, kGemmMaxPieces);
  if (n_units < 1 || n_units > 64) return set_error(ZERO_ERR_INVALID_ARG, "%s: n_units %d outside 1..64", kWho, n_units);
  if (!u) return set_error(ZERO_ERR_INVALID_ARG, "%s: units is NULL", kWho);
  if (m < 1 || (static_cast<int64_t>(n) * m) % 8)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_ranks * m_tokens must be a positive multiple of 8", kWho);
  if (flags & ~(FSDP_GATHER_MATERIALIZE | FSDP_BACKWARD_PREFETCH | FSDP_OVERLAP_OPTIMIZER | FSDP_SEPARATE_OPTIMIZER))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: unknown flags 0x%x", kWho, flags);
  for (int i = 0; i < n_units; ++i) {
    const fsdp_unit_state& s = u[i];
    if (s.rows_out < 1 || s.k_in < 1 || s.rows_out > (1 << 30) || s.k_in > (1 << 30))
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: sizes outside 1..2^30", kWho, i);
    // the backward reads W's shards (dX) and dY [N M, rows_out], X [N M, k_in] (dW) in place
    // as MN-major operands: rows of whole 64-column chunks, shards of whole 64-row K blocks
    if (s.rows_out % n || s.k_in % 64 || (s.rows_out / n) % 64)
      return set_error(ZERO_ERR_INVALID_ARG,
                       "%s: unit %d: rows_out / n_ranks and k_in must each be a multiple of 64 (got %lld / %d, %lld)",
                       kWho, i, (long long)s.rows_out, n, (long long)s.k_in);
    if (!(flags & FSDP_GATHER_MATERIALIZE) && !fsdp_fused_gather_ok(n, s.rows_out))
      return set_error(ZERO_ERR_INVALID_ARG,
                       "%s: unit %d: shards of %lld rows do not tile the GEMM for the fused gather; pass "
                       "FSDP_GATHER_MATERIALIZE",
                       kWho, i, (long long)(s.rows_out / n));
    if (i + 1 < n_units && u[i + 1].k_in != s.rows_out)
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d's k_in %lld is not unit %d's rows_out %lld", kWho, i + 1,
                       (long long)u[i + 1].k_in, i, (long long)s.rows_out);
    if (!buffers) continue;
    if (!s.plan) return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: plan is NULL", kWho, i);
    zero_layout L;
    zero_plan_query(s.plan, &L);
    if (L.psi != static_cast<uint64_t>(s.rows_out) * static_cast<uint64_t>(s.k_in) || L.n_ranks != n ||
        L.stage != ZERO_STAGE_3)
      return set_error(ZERO_ERR_INVALID_ARG,
                       "%s: unit %d: the plan must be zero_plan(rows_out * k_in, n_ranks, ZERO_STAGE_3, ...)", kWho, i);
    // dw is read by a separate optimizer launch; with the fused update it is optional
    const bool need_dw = (flags & (FSDP_OVERLAP_OPTIMIZER | FSDP_SEPARATE_OPTIMIZER)) != 0;
    if (!s.w || !s.master || !s.m || !s.v || !s.x || !s.dy || (need_dw && !s.dw))
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: a buffer is NULL", kWho, i);
    if (!aligned16(s.w) || !aligned16(s.master) || !aligned16(s.m) || !aligned16(s.v) || !aligned16(s.x) ||
        !aligned16(s.dy) || !aligned16(s.dw))
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: buffers must be 16-byte aligned", kWho, i);
  }
  return ZERO_OK;
}

}  // namespace

extern "C" int fsdp_zero3_step_workspace(int n_ranks, int n_units, const fsdp_unit_state* units, int64_t m_tokens,
                                         int flags, uint64_t* bytes) {
  if (!bytes) return set_error(ZERO_ERR_INVALID_ARG, "fsdp_zero3_step_workspace: bytes is NULL");
  int rc = check_units(n_ranks, n_units, units, m_tokens, flags, false);
  if (rc) return rc;
  *bytes = zero3_workspace(n_units, units, flags).total;
  return ZERO_OK;
}

extern "C" int fsdp_zero3_step(int n_ranks, int n_units, const fsdp_unit_state* units, int64_t m_tokens,
                               zero_bf16* y_out, zero_bf16* dx_out, const zero_adam* hp, int64_t step, int flags,
                               void* workspace, uint64_t workspace_bytes, zero_stream_t stream,
                               zero_stream_t prefetch_stream) {
  const int n = n_ranks, L = n_units;
  int rc = check_units(n, L, units, m_tokens, flags, true);
  if (rc) return rc;
  if ((rc = check_adam_args(hp, step, kWho))) return rc;
  if ((y_out && !aligned16(y_out)) || (dx_out && !aligned16(dx_out)))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: y_out and dx_out must be 16-byte aligned", kWho);
  const Zero3Workspace ws = zero3_workspace(L, units, flags);
  if (ws.total && (!workspace || !aligned16(workspace) || workspace_bytes < ws.total))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: workspace of %llu bytes (16-byte aligned) is below the %llu needed",
                     kWho, workspace ? (unsigned long long)workspace_bytes : 0ull, (unsigned long long)ws.total);
  const bool materialize = (flags & FSDP_GATHER_MATERIALIZE) != 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t side = prefetch_stream ? reinterpret_cast<cudaStream_t>(prefetch_stream) : st;
  cudaStream_t pf = materialize && (flags & FSDP_BACKWARD_PREFETCH) ? side : st;
  const bool overlap = pf != st;
  const bool adam_side = (flags & FSDP_OVERLAP_OPTIMIZER) && side != st;
  const bool adam_separate = (flags & (FSDP_OVERLAP_OPTIMIZER | FSDP_SEPARATE_OPTIMIZER)) != 0;
  AdamScalars sc;
  if ((rc = make_adam_scalars(hp, step, kWho, &sc))) return rc;
  const int64_t nm = static_cast<int64_t>(n) * m_tokens;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  auto w_slot = [&](int i) { return reinterpret_cast<uint16_t*>(base + ws.w_off[i % std::max(ws.slots, 1)]); };
  // events: [0] forward done, [1 + i] unit i's gathered W ready, [1 + L + i] unit i's dX
  // GEMM done (its slot is free), [1 + 2L + i] unit i's dW GEMM done, [1 + 3L] the side
  // stream's last launch
  cudaEvent_t* ev = nullptr;
  if ((overlap || adam_side) && (rc = get_events(static_cast<size_t>(3 * L + 2), &ev))) return rc;
  const auto ev_ready = [&](int i) { return ev[1 + i]; };
  const auto ev_free = [&](int i) { return ev[1 + L + i]; };
  const auto ev_done = [&](int i) { return ev[1 + 2 * L + i]; };

  // the N row shards of unit i (rank r's rows at r R/N), or its gathered copy
  const uint16_t* shard_ptrs[kGemmMaxPieces];
  auto shards_of = [&](int i) {
    const fsdp_unit_state& s = units[i];
    const int64_t per = (s.rows_out / n) * s.k_in;
    for (int r = 0; r < n; ++r) shard_ptrs[r] = s.w + r * per;
    return static_cast<const uint16_t* const*>(shard_ptrs);
  };
  auto gather = [&](int i, cudaStream_t s) {
    return fsdp_gather_rows(n, shards_of(i), units[i].rows_out, units[i].k_in, w_slot(i),
                            reinterpret_cast<zero_stream_t>(s));
  };
  auto wait = [&](cudaStream_t s, cudaEvent_t e) {
    const cudaError_t err = cudaStreamWaitEvent(s, e, 0);
    return err == cudaSuccess ? ZERO_OK : set_error(ZERO_ERR_CUDA, "%s: %s", kWho, cudaGetErrorString(err));
  };
  auto record = [&](cudaEvent_t e, cudaStream_t s) {
    const cudaError_t err = cudaEventRecord(e, s);
    return err == cudaSuccess ? ZERO_OK : set_error(ZERO_ERR_CUDA, "%s: %s", kWho, cudaGetErrorString(err));
  };

  // ---- forward, unit 0 -> last: gather, X_{i+1} = bf16(X_i W_i^T), free ----
  for (int i = 0; i < L; ++i) {
    const fsdp_unit_state& s = units[i];
    zero_bf16* out = i + 1 < L ? units[i + 1].x : y_out;
    if (!out) continue;
    if (materialize) {
      if ((rc = gather(i, st))) return rc;
      const uint16_t* w1[1] = {w_slot(i)};
      rc = launch_fsdp_gemm(1, w1, s.rows_out, s.k_in, s.x, nm, nullptr, out, 1.0f, st);
    } else {
      rc = launch_fsdp_gemm(n, shards_of(i), s.rows_out, s.k_in, s.x, nm, nullptr, out, 1.0f, st);
    }
    if (rc) return rc;
  }

  // ---- backward, last -> unit 0 ----
  // with a materialised gather, unit i's W gathered again into its slot
  auto prepare = [&](int i, cudaStream_t s) {
    int r = ZERO_OK;
    if (overlap && i + ws.slots < L && (r = wait(s, ev_free(i + ws.slots)))) return r;  // slot reuse
    if ((r = gather(i, s))) return r;
    return overlap ? record(ev_ready(i), s) : ZERO_OK;
  };
  if (overlap) {
    // the prefetch stream starts once the forward (which writes every unit's input) is done
    if ((rc = record(ev[0], st)) || (rc = wait(pf, ev[0])) || (rc = prepare(L - 1, pf))) return rc;
  }
  for (int i = L - 1; i >= 0; --i) {
    const fsdp_unit_state& s = units[i];
    if (overlap) {
      if ((rc = wait(st, ev_ready(i)))) return rc;
    } else if (materialize && (rc = prepare(i, st))) {
      return rc;
    }
    // dY_{i-1} [N M, K] = bf16(dY_i [N M, R] * W_i [R, K]), W_i read as an MN-major operand
    // from its N row shards (or its gathered copy)
    zero_bf16* dx = i > 0 ? units[i - 1].dy : dx_out;
    const uint16_t* w1[1] = {materialize ? w_slot(i) : nullptr};
    const uint16_t* const* wp = materialize ? w1 : shards_of(i);
    const int w_pieces = materialize ? 1 : n;
    if (dx && (rc = launch_fsdp_gemm_w_mn(w_pieces, wp, s.rows_out / w_pieces, s.k_in, s.dy, nm, nullptr, dx, 1.0f,
                                          st, kWho)))
      return rc;
    if (overlap) {
      if ((rc = record(ev_free(i), st))) return rc;
      if (i > 0 && (rc = prepare(i - 1, pf))) return rc;  // overlaps this unit's dW GEMM and Adam
    }
    // dW = (1/N) dY_i^T X_i with dY_i and X_i read in place; by default with each rank's
    // Adam on its rows in the epilogue
    const float inv_n = 1.0f / static_cast<float>(n);
    const AdamFuse fuse = {{s.master, s.master}, {s.m, s.m}, {s.v, s.v}, {s.w, s.w}, s.rows_out, sc};
    const uint16_t* dy1[1] = {s.dy};
    const uint16_t* x1[1] = {s.x};
    if ((rc = launch_fsdp_bwd_dw_in_place(1, dy1, x1, nm, s.rows_out, s.k_in, s.dw, inv_n, st,
                                          adam_separate ? nullptr : &fuse, kWho)))
      return rc;
    if ((overlap || adam_side) && (rc = record(ev_done(i), st))) return rc;
    // with a separate optimizer: each rank's Adam on its shard (rows r R/N .. of dW), every
    // rank's shard in one launch, on `stream` or, overlapped, on the side stream
    if (!adam_separate) {
    } else if (adam_side) {
      if ((rc = wait(side, ev_done(i))) ||
          (rc = zero_adam_step(s.plan, ZERO_ALL_RANKS, s.dw, s.master, s.m, s.v, s.w, hp, step,
                               reinterpret_cast<zero_stream_t>(side))))
        return rc;
    } else if ((rc = zero_adam_step(s.plan, ZERO_ALL_RANKS, s.dw, s.master, s.m, s.v, s.w, hp, step, stream))) {
      return rc;
    }
  }
  // join: `stream` waits for the side stream's last launch (its last Adam; without Adam on
  // it, unit 0's gather, which `stream` has already awaited)
  if (overlap || adam_side) {
    if ((rc = record(ev[1 + 3 * L], side)) || (rc = wait(st, ev[1 + 3 * L]))) return rc;
  }
  return ZERO_OK;
}

// ======================================================================================
// The same step over Mistral-style MLP units (H = silu(X W_gate^T) * (X W_up^T), Y = H
// W_down^T), each of the three weights with its own ZeRO-3 state. Forward: the gate-up
// kernel (both projections in one N = 256 MMA stream, SiLU-gate epilogue) also saves G | U
// for the backward, then the down projection. Backward, per unit: dH from W_down's shards
// read in place, dW_down (dY and H read in place) with W_down's Adam; the SiLU-gate
// backward; dX over the concatenated K of both projections from the 2N shards of [W_gate;
// W_up] read in place, dW_gate | dW_up in one GEMM (dG | dU and X read in place) with
// their Adam. No transpose is laid out; only more than 8 ranks (2N pieces above the
// GEMM's 16) gather [W_gate; W_up] into the workspace first. Serial on one stream: on one
// GPU the side-stream forms of the linear step above measured slower.
// ======================================================================================

namespace {

const char* const kWhoMlp = "fsdp_zero3_mlp_step";

struct MlpWorkspace {
  uint64_t total;  // [W_gate; W_up] gathered [2 d_ff, d_model] bf16 when 2 n_ranks > 16, else 0
};

MlpWorkspace mlp_workspace(int n, int L, const fsdp_mlp_unit_state* u) {
  MlpWorkspace w{0};
  if (2 * n <= kGemmMaxPieces) return w;
  for (int i = 0; i < L; ++i)
    w.total = std::max<uint64_t>(w.total, align256(4ull * static_cast<uint64_t>(u[i].d_ff) *
                                                   static_cast<uint64_t>(u[i].d_model)));
  return w;
}

int check_weight(const fsdp_weight_state& w, int64_t rows, int64_t cols, int n, int i, const char* name) {
  if (!w.plan) return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: %s.plan is NULL", kWhoMlp, i, name);
  zero_layout L;
  zero_plan_query(w.plan, &L);
  if (L.psi != static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols) || L.n_ranks != n || L.stage != ZERO_STAGE_3)
    return set_error(ZERO_ERR_INVALID_ARG,
                     "%s: unit %d: %s.plan must be zero_plan(%lld * %lld, n_ranks, ZERO_STAGE_3, ...)", kWhoMlp, i,
                     name, (long long)rows, (long long)cols);
  if (!w.w || !w.master || !w.m || !w.v)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: a buffer of %s is NULL", kWhoMlp, i, name);
  if (!aligned16(w.w) || !aligned16(w.master) || !aligned16(w.m) || !aligned16(w.v))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: buffers of %s must be 16-byte aligned", kWhoMlp, i, name);
  return ZERO_OK;
}

int check_mlp_units(int n, int L, const fsdp_mlp_unit_state* u, int64_t m, bool buffers, bool need_dw = false) {
  if (n < 1 || n > kGemmMaxPieces)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_ranks %d outside 1..%d", kWhoMlp, n, kGemmMaxPieces);
  if (L < 1 || L > 64) return set_error(ZERO_ERR_INVALID_ARG, "%s: n_units %d outside 1..64", kWhoMlp, L);
  if (!u) return set_error(ZERO_ERR_INVALID_ARG, "%s: units is NULL", kWhoMlp);
  if (m < 1 || (static_cast<int64_t>(n) * m) % 8)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: n_ranks * m_tokens must be a positive multiple of 8", kWhoMlp);
  for (int i = 0; i < L; ++i) {
    const fsdp_mlp_unit_state& s = u[i];
    const int64_t d = s.d_model, f = s.d_ff;
    if (d < 64 || f < 64 || d > (1 << 28) || f > (1 << 28) || d % 64 || f % 64)
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: d_model and d_ff must be multiples of 64 (got %lld, %lld)",
                       kWhoMlp, i, (long long)d, (long long)f);
    if (f % n || (f / n) % 128)
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: d_ff / n_ranks must be a multiple of 128 (got %lld / %d)",
                       kWhoMlp, i, (long long)f, n);
    if (!fsdp_fused_gather_ok(n, d))
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: W_down's shards of %lld rows do not tile the fused gather",
                       kWhoMlp, i, (long long)(d % n ? -1 : d / n));
    if (i + 1 < L && u[i + 1].d_model != d)
      return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d's d_model %lld differs from unit %d's %lld", kWhoMlp, i + 1,
                       (long long)u[i + 1].d_model, i, (long long)d);
    if (!buffers) continue;
    int rc;
    if ((rc = check_weight(s.gate, f, d, n, i, "gate")) || (rc = check_weight(s.up, f, d, n, i, "up")) ||
        (rc = check_weight(s.down, d, f, n, i, "down")))
      return rc;
    const void* bufs[] = {s.x, s.gu, s.h, s.dy, s.dh, s.dgu, s.dw_gu, s.dw_down};
    for (int k = 0; k < 8; ++k) {
      const void* b = bufs[k];
      // dw_gu and dw_down (the last two) are optional when the optimizer is fused
      if (!b && (k < 6 || need_dw))
        return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: an activation or gradient buffer is NULL", kWhoMlp, i);
      if (!aligned16(b))
        return set_error(ZERO_ERR_INVALID_ARG, "%s: unit %d: activation and gradient buffers must be 16-byte aligned",
                         kWhoMlp, i);
    }
  }
  return ZERO_OK;
}

}  // namespace

extern "C" int fsdp_zero3_mlp_step_workspace(int n_ranks, int n_units, const fsdp_mlp_unit_state* units,
                                             int64_t m_tokens, uint64_t* bytes) {
  if (!bytes) return set_error(ZERO_ERR_INVALID_ARG, "fsdp_zero3_mlp_step_workspace: bytes is NULL");
  int rc = check_mlp_units(n_ranks, n_units, units, m_tokens, false);
  if (rc) return rc;
  *bytes = mlp_workspace(n_ranks, n_units, units).total;
  return ZERO_OK;
}

extern "C" int fsdp_zero3_mlp_step(int n_ranks, int n_units, const fsdp_mlp_unit_state* units, int64_t m_tokens,
                                   zero_bf16* y_out, zero_bf16* dx_out, const zero_adam* hp, int64_t step, int flags,
                                   void* workspace, uint64_t workspace_bytes, zero_stream_t stream) {
  const int n = n_ranks, L = n_units;
  if (flags & ~FSDP_SEPARATE_OPTIMIZER)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: unknown flags 0x%x", kWhoMlp, flags);
  const bool separate = (flags & FSDP_SEPARATE_OPTIMIZER) != 0;
  int rc = check_mlp_units(n, L, units, m_tokens, true, separate);
  if (rc) return rc;
  AdamScalars sc;
  if ((rc = make_adam_scalars(hp, step, kWhoMlp, &sc))) return rc;
  if ((y_out && !aligned16(y_out)) || (dx_out && !aligned16(dx_out)))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: y_out and dx_out must be 16-byte aligned", kWhoMlp);
  const MlpWorkspace ws = mlp_workspace(n, L, units);
  if (ws.total && (!workspace || !aligned16(workspace) || workspace_bytes < ws.total))
    return set_error(ZERO_ERR_INVALID_ARG, "%s: workspace of %llu bytes (16-byte aligned) is below the %llu needed",
                     kWhoMlp, workspace ? (unsigned long long)workspace_bytes : 0ull, (unsigned long long)ws.total);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t nm = static_cast<int64_t>(n) * m_tokens;
  uint16_t* wgu = static_cast<uint16_t*>(workspace);  // gathered [W_gate; W_up] (more than 8 ranks)
  const float inv_n = 1.0f / static_cast<float>(n);

  // the N row shards of a weight (rank r's rows at r rows/N), into ptrs[first .. first + N)
  auto shards = [&](const fsdp_weight_state& w, int64_t rows, int64_t cols, const uint16_t** ptrs, int first) {
    const int64_t per = (rows / n) * cols;
    for (int r = 0; r < n; ++r) ptrs[first + r] = w.w + r * per;
  };

  // ---- forward, unit 0 -> last ----
  for (int i = 0; i < L; ++i) {
    const fsdp_mlp_unit_state& s = units[i];
    const int64_t d = s.d_model, f = s.d_ff;
    const uint16_t *gsh[kGemmMaxPieces], *ush[kGemmMaxPieces], *dsh[kGemmMaxPieces];
    shards(s.gate, f, d, gsh, 0);
    shards(s.up, f, d, ush, 0);
    shards(s.down, d, f, dsh, 0);
    if ((rc = launch_fsdp_gate_up(n, gsh, ush, f, d, s.x, nm, s.h, st, s.gu))) return rc;
    zero_bf16* out = i + 1 < L ? units[i + 1].x : y_out;
    if (out && (rc = launch_fsdp_gemm(n, dsh, d, f, s.h, nm, nullptr, out, 1.0f, st))) return rc;
  }

  // ---- backward, last -> unit 0 ----
  for (int i = L - 1; i >= 0; --i) {
    const fsdp_mlp_unit_state& s = units[i];
    const int64_t d = s.d_model, f = s.d_ff;
    const uint16_t* wsh[2 * kGemmMaxPieces];
    // dH [nm, f] = bf16(dY [nm, d] * W_down [d, f]), W_down read from its row shards
    shards(s.down, d, f, wsh, 0);
    if ((rc = launch_fsdp_gemm_w_mn(n, wsh, d / n, f, s.dy, nm, nullptr, s.dh, 1.0f, st, kWhoMlp))) return rc;
    // dW_down [d, f] = (1/N) dY^T H with W_down's Adam fused into its epilogue (or as its
    // own launch)
    const AdamFuse fd = {{s.down.master, s.down.master}, {s.down.m, s.down.m}, {s.down.v, s.down.v},
                         {s.down.w, s.down.w}, d, sc};
    const uint16_t* dy1[1] = {s.dy};
    const uint16_t* h1[1] = {s.h};
    if ((rc = launch_fsdp_bwd_dw_in_place(1, dy1, h1, nm, d, f, s.dw_down, inv_n, st, separate ? nullptr : &fd,
                                          kWhoMlp)))
      return rc;
    if (separate && (rc = zero_adam_step(s.down.plan, ZERO_ALL_RANKS, s.dw_down, s.down.master, s.down.m, s.down.v,
                                         s.down.w, hp, step, stream)))
      return rc;
    // dG | dU from dH and the saved G | U
    cudaError_t e = launch_silu_gate_backward(s.dh, s.gu, s.dgu, nm, f, st);
    if (e != cudaSuccess)
      return set_error(ZERO_ERR_CUDA, "%s: SiLU-gate backward: %s", kWhoMlp, cudaGetErrorString(e));
    // dX [nm, d] = bf16([dG | dU] [nm, 2f] * [W_gate; W_up] [2f, d]): the sum of both
    // projections' input gradients over the concatenated K, [W_gate; W_up] read from the
    // 2N shards of both (or, past 8 ranks, from its gathered copy)
    zero_bf16* dx = i > 0 ? units[i - 1].dy : dx_out;
    if (dx) {
      shards(s.gate, f, d, wsh, 0);
      shards(s.up, f, d, wsh, n);
      int pieces = 2 * n;
      if (2 * n > kGemmMaxPieces) {
        if ((rc = fsdp_gather_rows(n, wsh, f, d, wgu, stream)) ||
            (rc = fsdp_gather_rows(n, wsh + n, f, d, wgu + f * d, stream)))
          return rc;
        wsh[0] = wgu;
        pieces = 1;
      }
      if ((rc = launch_fsdp_gemm_w_mn(pieces, wsh, 2 * f / pieces, d, s.dgu, nm, nullptr, dx, 1.0f, st, kWhoMlp)))
        return rc;
    }
    // dW_gate | dW_up [2f, d] = (1/N) [dG | dU]^T X with both weights' Adam fused into its
    // epilogue (rows < d_ff: W_gate)
    const AdamFuse fgu = {{s.gate.master, s.up.master}, {s.gate.m, s.up.m}, {s.gate.v, s.up.v}, {s.gate.w, s.up.w},
                          f, sc};
    const uint16_t* dgu1[1] = {s.dgu};
    const uint16_t* x1[1] = {s.x};
    if ((rc = launch_fsdp_bwd_dw_in_place(1, dgu1, x1, nm, 2 * f, d, s.dw_gu, inv_n, st, separate ? nullptr : &fgu,
                                          kWhoMlp)))
      return rc;
    if (separate &&
        ((rc = zero_adam_step(s.gate.plan, ZERO_ALL_RANKS, s.dw_gu, s.gate.master, s.gate.m, s.gate.v, s.gate.w, hp,
                              step, stream)) ||
         (rc = zero_adam_step(s.up.plan, ZERO_ALL_RANKS, s.dw_gu + f * d, s.up.master, s.up.m, s.up.v, s.up.w, hp,
                              step, stream))))
      return rc;
  }
  return ZERO_OK;
}
