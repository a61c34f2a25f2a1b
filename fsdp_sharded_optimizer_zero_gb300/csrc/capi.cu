// C ABI of the library: argument validation, the flat-buffer plan, pointer resolution for
// the three rank modes, and dispatch to the kernels. Nothing here allocates device memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <new>

#include "internal.h"

namespace zgb {

namespace {
thread_local char g_msg[512] = {0};
std::atomic<int> g_fused_variant{0};
std::atomic<int> g_sms[64];
}  // namespace

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

static void clear_error() { g_msg[0] = 0; }

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  int v = g_sms[dev & 63].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    g_sms[dev & 63].store(v, std::memory_order_relaxed);
  }
  return v;
}

}  // namespace zgb

using namespace zgb;

#define CHECK_ARG(cond, ...)                                         \
  do {                                                               \
    if (!(cond)) return set_error(ZERO_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define CUDA_LAUNCH(expr)                                                                                  \
  do {                                                                                                     \
    cudaError_t e_ = (expr);                                                                               \
    if (e_ != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s (%s)", #expr, cudaGetErrorName(e_),      \
                                            cudaGetErrorString(e_));                                       \
  } while (0)

static inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ======================================================================================
// plan
// ======================================================================================

extern "C" int zero_plan(uint64_t psi, int n_ranks, int stage, uint64_t bucket_bytes, zero_plan_t** out) {
  clear_error();
  CHECK_ARG(out != nullptr, "zero_plan: out is NULL");
  *out = nullptr;
  CHECK_ARG(psi >= 1, "zero_plan: psi must be >= 1");
  CHECK_ARG(psi <= (1ull << 50), "zero_plan: psi %llu too large", (unsigned long long)psi);
  CHECK_ARG(n_ranks >= 1 && n_ranks <= ZERO_MAX_RANKS, "zero_plan: n_ranks %d outside 1..%d", n_ranks,
            ZERO_MAX_RANKS);
  CHECK_ARG(stage >= ZERO_STAGE_DDP && stage <= ZERO_STAGE_MEGATRON, "zero_plan: stage %d outside 0..4", stage);
  CHECK_ARG(bucket_bytes >= 2ull * (uint64_t)n_ranks,
            "zero_plan: bucket_bytes %llu holds less than one bf16 element per rank (need >= %d)",
            (unsigned long long)bucket_bytes, 2 * n_ranks);

  const uint64_t n = static_cast<uint64_t>(n_ranks);
  zero_layout L;
  memset(&L, 0, sizeof(L));
  L.psi = psi;
  L.n_ranks = n_ranks;
  L.stage = stage;
  L.bucket_bytes = bucket_bytes;
  L.psi_padded = (psi + n - 1) / n * n;
  L.shard_elems = L.psi_padded / n;
  L.bucket_elems = bucket_bytes / (2 * n);
  L.n_buckets = (L.shard_elems + L.bucket_elems - 1) / L.bucket_elems;

  const uint64_t P = L.psi_padded, S = L.shard_elems;
  // bytes one rank keeps: bf16 param (2), bf16 grad (2), fp32 master/m/v (4 each)
  const bool megatron = stage == ZERO_STAGE_MEGATRON;
  L.state_param_bytes = 2 * (stage == ZERO_STAGE_3 ? S : P);
  // Megatron keeps the full gradient in fp32; ZeRO-2/3 keep a bf16 slice
  L.state_grad_bytes = megatron ? 4 * P : 2 * (stage == ZERO_STAGE_2 || stage == ZERO_STAGE_3 ? S : P);
  const uint64_t opt_elems = stage >= ZERO_STAGE_1 ? S : P;
  L.state_master_bytes = L.state_m_bytes = L.state_v_bytes = 4 * opt_elems;
  L.state_total_bytes =
      L.state_param_bytes + L.state_grad_bytes + L.state_master_bytes + L.state_m_bytes + L.state_v_bytes;
  // elements one rank moves per step: reduce-scatter P + all-gather P (+ backward all-gather P for ZeRO-3)
  L.comm_reduce_scatter = P;
  L.comm_all_gather_fwd = P;
  L.comm_all_gather_bwd = stage == ZERO_STAGE_3 ? P : 0;
  L.comm_total = L.comm_reduce_scatter + L.comm_all_gather_fwd + L.comm_all_gather_bwd;
  L.ring_sent_elems = (n - 1) * (L.comm_total / n);
  L.fused_step_bytes = P * ((megatron ? 4 : 2) * n + 26);

  zero_plan_t* p = new (std::nothrow) zero_plan_t;
  if (!p) return set_error(ZERO_ERR_OOM, "zero_plan: host allocation failed");
  p->lay = L;
  *out = p;
  return ZERO_OK;
}

extern "C" int zero_plan_query(const zero_plan_t* plan, zero_layout* out) {
  clear_error();
  CHECK_ARG(plan && out, "zero_plan_query: NULL argument");
  *out = plan->lay;
  return ZERO_OK;
}

extern "C" int zero_bucket_range(const zero_plan_t* plan, int rank, uint64_t bucket, uint64_t* begin,
                                 uint64_t* end) {
  clear_error();
  CHECK_ARG(plan && begin && end, "zero_bucket_range: NULL argument");
  const zero_layout& L = plan->lay;
  CHECK_ARG(rank >= 0 && rank < L.n_ranks, "zero_bucket_range: rank %d outside 0..%d", rank, L.n_ranks - 1);
  CHECK_ARG(bucket < L.n_buckets, "zero_bucket_range: bucket %llu >= n_buckets %llu", (unsigned long long)bucket,
            (unsigned long long)L.n_buckets);
  const uint64_t base = static_cast<uint64_t>(rank) * L.shard_elems;
  const uint64_t hi = (bucket + 1) * L.bucket_elems;
  *begin = base + bucket * L.bucket_elems;
  *end = base + (hi < L.shard_elems ? hi : L.shard_elems);
  return ZERO_OK;
}

extern "C" int zero_plan_destroy(zero_plan_t* plan) {
  clear_error();
  delete plan;
  return ZERO_OK;
}

extern "C" int zero_plan_check_memory(const zero_plan_t* plan, int rank, uint64_t budget_bytes, uint64_t* need_bytes,
                                      uint64_t* budget_out) {
  clear_error();
  const char* who = "zero_plan_check_memory";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  CHECK_ARG(rank == ZERO_RANK_VIEW || rank == ZERO_ALL_RANKS || (rank >= 0 && rank < L.n_ranks),
            "%s: rank %d is not 0..%d, ZERO_RANK_VIEW or ZERO_ALL_RANKS", who, rank, L.n_ranks - 1);
  const uint64_t P = L.psi_padded, S = L.shard_elems, n = static_cast<uint64_t>(L.n_ranks);
  // the buffers one step call addresses in this rank mode: n gradient buffers (bf16, fp32
  // for a Megatron plan), fp32 master / m / v, the bf16 parameter output
  const uint64_t grad_elems = rank == ZERO_RANK_VIEW ? S : P;
  const uint64_t state_elems = rank == ZERO_ALL_RANKS ? P : S;
  const uint64_t param_elems = rank == ZERO_RANK_VIEW ? S : (rank >= 0 && L.stage == ZERO_STAGE_3 ? S : P);
  const uint64_t gsz = L.stage == ZERO_STAGE_MEGATRON ? 4 : 2;
  const uint64_t need = n * grad_elems * gsz + 12 * state_elems + 2 * param_elems;
  if (need_bytes) *need_bytes = need;
  uint64_t budget = budget_bytes;
  if (budget == 0) {
    size_t free_b = 0, total_b = 0;
    CUDA_LAUNCH(cudaMemGetInfo(&free_b, &total_b));
    budget = static_cast<uint64_t>(free_b);
  }
  if (budget_out) *budget_out = budget;
  if (need > budget)
    return set_error(ZERO_ERR_OOM,
                     "%s: one step of this plan (psi %llu, N %d, stage %d, rank mode %d) addresses %llu bytes of "
                     "device buffers; %s is %llu bytes",
                     who, (unsigned long long)L.psi, L.n_ranks, L.stage, rank, (unsigned long long)need,
                     budget_bytes ? "the caller's budget" : "this device's free memory", (unsigned long long)budget);
  return ZERO_OK;
}

// ======================================================================================
// the step
// ======================================================================================

namespace {

// the element range of one call and where each stream's element 0 sits
struct Resolved {
  Domain d;
  uint64_t grad_off;   // into each grads[q]
  uint64_t state_off;  // into g / master / m / v
  uint64_t param_off;  // into param_out
};

int resolve(const zero_layout& L, int rank, uint64_t b0, uint64_t b1, const char* who, Resolved* r) {
  CHECK_ARG(rank == ZERO_RANK_VIEW || rank == ZERO_ALL_RANKS || (rank >= 0 && rank < L.n_ranks),
            "%s: rank %d is not 0..%d, ZERO_RANK_VIEW or ZERO_ALL_RANKS", who, rank, L.n_ranks - 1);
  CHECK_ARG(b0 < b1 && b1 <= L.n_buckets, "%s: bucket range [%llu, %llu) not inside [0, %llu)", who,
            (unsigned long long)b0, (unsigned long long)b1, (unsigned long long)L.n_buckets);
  const uint64_t S = L.shard_elems, C = L.bucket_elems;
  const uint64_t lo = b0 * C, hi = (b1 * C < S) ? b1 * C : S, len = hi - lo;
  if (rank >= 0) {
    const uint64_t rs = static_cast<uint64_t>(rank) * S;
    r->d = {1, len, 0};
    r->grad_off = rs + lo;
    r->state_off = lo;
    r->param_off = (L.stage == ZERO_STAGE_3 ? 0 : rs) + lo;
  } else if (rank == ZERO_RANK_VIEW) {
    r->d = {1, len, 0};
    r->grad_off = r->state_off = r->param_off = lo;
  } else {
    r->d = (lo == 0 && hi == S) ? Domain{1, L.psi_padded, 0} : Domain{static_cast<uint64_t>(L.n_ranks), len, S};
    r->grad_off = r->state_off = r->param_off = lo;
  }
  return ZERO_OK;
}

int make_scalars(const zero_adam* hp, int64_t step, int n, const char* who, AdamScalars* sc) {
  CHECK_ARG(hp != nullptr, "%s: hp is NULL", who);
  CHECK_ARG(step >= 1, "%s: step %lld must count from 1", who, (long long)step);
  CHECK_ARG(isfinite(hp->lr) && hp->lr >= 0.f, "%s: lr must be finite and >= 0", who);
  CHECK_ARG(hp->beta1 >= 0.f && hp->beta1 < 1.f, "%s: beta1 must be in [0, 1)", who);
  CHECK_ARG(hp->beta2 >= 0.f && hp->beta2 < 1.f, "%s: beta2 must be in [0, 1)", who);
  CHECK_ARG(isfinite(hp->eps) && hp->eps > 0.f, "%s: eps must be finite and > 0", who);
  CHECK_ARG(isfinite(hp->weight_decay) && hp->weight_decay >= 0.f, "%s: weight_decay must be finite and >= 0", who);
  sc->lr = hp->lr;
  sc->beta1 = hp->beta1;
  sc->beta2 = hp->beta2;
  sc->omb1 = 1.0f - hp->beta1;
  sc->omb2 = 1.0f - hp->beta2;
  sc->eps = hp->eps;
  // 1 - beta^t in binary64, rounded once to fp32
  sc->bc1 = static_cast<float>(1.0 - pow(static_cast<double>(hp->beta1), static_cast<double>(step)));
  sc->bc2 = static_cast<float>(1.0 - pow(static_cast<double>(hp->beta2), static_cast<double>(step)));
  const float lr = hp->lr, wd = hp->weight_decay;
  sc->lr_wd = lr * wd;
  sc->wd_on = wd != 0.f ? 1 : 0;
  sc->inv_n = 1.0f / static_cast<float>(n);
  return ZERO_OK;
}

}  // namespace

// hp and step checked as every Adam call checks them (nothing launched)
int zgb::check_adam_args(const zero_adam* hp, int64_t step, const char* who) {
  AdamScalars sc;
  return make_scalars(hp, step, 1, who, &sc);
}

int zgb::make_adam_scalars(const zero_adam* hp, int64_t step, const char* who, AdamScalars* sc) {
  return make_scalars(hp, step, 1, who, sc);
}

namespace {

int load_grads(const zero_bf16* const grads[], int n, uint64_t off, const char* who, GradPtrs* gp) {
  CHECK_ARG(grads != nullptr, "%s: grads array is NULL", who);
  memset(gp, 0, sizeof(*gp));
  for (int q = 0; q < n; ++q) {
    CHECK_ARG(grads[q] != nullptr, "%s: grads[%d] is NULL (missing rank)", who, q);
    gp->p[q] = grads[q] + off;
  }
  return ZERO_OK;
}

bool grads_aligned(const GradPtrs& gp, int n, uintptr_t a) {
  for (int q = 0; q < n; ++q)
    if (!aligned(gp.p[q], a)) return false;
  return true;
}

// vector paths need: grads 8 B (register) / 16 B (bulk) aligned, fp32 state 16 B, bf16
// param 8 B, and a segment stride that keeps every segment start aligned the same way
bool stride_ok(const Domain& d, uint64_t elems) { return d.n_seg == 1 || d.seg_stride % elems == 0; }

}  // namespace

extern "C" int zero_reduce_scatter(const zero_plan_t* plan, int rank, const zero_bf16* const grads[], float* g_shard,
                                   zero_stream_t stream) {
  clear_error();
  const char* who = "zero_reduce_scatter";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  Resolved r;
  int rc = resolve(L, rank, 0, L.n_buckets, who, &r);
  if (rc) return rc;
  CHECK_ARG(g_shard != nullptr, "%s: g_shard is NULL", who);
  GradPtrs gp;
  if ((rc = load_grads(grads, L.n_ranks, r.grad_off, who, &gp))) return rc;
  float* out = g_shard + r.state_off;
  const bool vec = grads_aligned(gp, L.n_ranks, 8) && aligned(out, 16) && stride_ok(r.d, 4);
  CUDA_LAUNCH(launch_reduce(gp, L.n_ranks, out, r.d, 1.0f / static_cast<float>(L.n_ranks), vec,
                            reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

extern "C" int zero_adam_step(const zero_plan_t* plan, int rank, const float* g_shard, float* master, float* m,
                              float* v, zero_bf16* param_out, const zero_adam* hp, int64_t step, zero_stream_t stream) {
  clear_error();
  const char* who = "zero_adam_step";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  Resolved r;
  int rc = resolve(L, rank, 0, L.n_buckets, who, &r);
  if (rc) return rc;
  CHECK_ARG(g_shard && master && m && v, "%s: g_shard / master / m / v must not be NULL", who);
  AdamScalars sc;
  if ((rc = make_scalars(hp, step, L.n_ranks, who, &sc))) return rc;
  const float* g = g_shard + r.state_off;
  float *w = master + r.state_off, *mm = m + r.state_off, *vv = v + r.state_off;
  uint16_t* p = param_out ? param_out + r.param_off : nullptr;
  const bool vec = aligned(g, 16) && aligned(w, 16) && aligned(mm, 16) && aligned(vv, 16) && (!p || aligned(p, 8)) &&
                   stride_ok(r.d, 4);
  CUDA_LAUNCH(launch_adam(g, w, mm, vv, p, r.d, sc, vec, reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

static int fused_impl(const zero_plan_t* plan, int rank, uint64_t b0, uint64_t b1, const zero_bf16* const grads[],
                      float* master, float* m, float* v, zero_bf16* param_out, const zero_adam* hp, int64_t step,
                      zero_stream_t stream, const char* who) {
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  Resolved r;
  int rc = resolve(L, rank, b0, b1, who, &r);
  if (rc) return rc;
  CHECK_ARG(master && m && v && param_out, "%s: master / m / v / param_out must not be NULL", who);
  AdamScalars sc;
  if ((rc = make_scalars(hp, step, L.n_ranks, who, &sc))) return rc;
  GradPtrs gp;
  if ((rc = load_grads(grads, L.n_ranks, r.grad_off, who, &gp))) return rc;
  float *w = master + r.state_off, *mm = m + r.state_off, *vv = v + r.state_off;
  uint16_t* p = param_out + r.param_off;
  const bool state16 = aligned(w, 16) && aligned(mm, 16) && aligned(vv, 16) && aligned(p, 8);
  const bool tma_ok = state16 && grads_aligned(gp, L.n_ranks, 16) && stride_ok(r.d, 8);
  const bool vec_ok = state16 && grads_aligned(gp, L.n_ranks, 8) && stride_ok(r.d, 4);
  // default (0) and 2: register streaming, at the copy roofline for every N on GB300;
  // 1: the TMA bulk pipeline (ablation). Misaligned buffers take the scalar kernel.
  const int want = g_fused_variant.load(std::memory_order_relaxed);
  int variant;
  if (want == 1)
    variant = tma_ok ? 1 : (vec_ok ? 2 : 3);
  else
    variant = vec_ok ? 2 : 3;
  CUDA_LAUNCH(launch_fused(gp, L.n_ranks, w, mm, vv, p, r.d, sc, variant, reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

extern "C" int zero_fused_step(const zero_plan_t* plan, int rank, const zero_bf16* const grads[], float* master,
                               float* m, float* v, zero_bf16* param_out, const zero_adam* hp, int64_t step,
                               zero_stream_t stream) {
  clear_error();
  if (!plan) return set_error(ZERO_ERR_INVALID_ARG, "zero_fused_step: plan is NULL");
  return fused_impl(plan, rank, 0, plan->lay.n_buckets, grads, master, m, v, param_out, hp, step, stream,
                    "zero_fused_step");
}

extern "C" int zero_fused_step_fp32_grads(const zero_plan_t* plan, int rank, const float* const grads[],
                                          float* master, float* m, float* v, zero_bf16* param_out,
                                          const zero_adam* hp, int64_t step, zero_stream_t stream) {
  clear_error();
  const char* who = "zero_fused_step_fp32_grads";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  Resolved r;
  int rc = resolve(L, rank, 0, L.n_buckets, who, &r);
  if (rc) return rc;
  CHECK_ARG(master && m && v && param_out, "%s: master / m / v / param_out must not be NULL", who);
  CHECK_ARG(grads != nullptr, "%s: grads array is NULL", who);
  AdamScalars sc;
  if ((rc = make_scalars(hp, step, L.n_ranks, who, &sc))) return rc;
  F32GradPtrs gp;
  memset(&gp, 0, sizeof(gp));
  bool grads16 = true;
  for (int q = 0; q < L.n_ranks; ++q) {
    CHECK_ARG(grads[q] != nullptr, "%s: grads[%d] is NULL (missing rank)", who, q);
    gp.p[q] = grads[q] + r.grad_off;
    grads16 = grads16 && aligned(gp.p[q], 16);
  }
  float *w = master + r.state_off, *mm = m + r.state_off, *vv = v + r.state_off;
  uint16_t* p = param_out + r.param_off;
  const bool vec = grads16 && aligned(w, 16) && aligned(mm, 16) && aligned(vv, 16) && aligned(p, 8) &&
                   stride_ok(r.d, 4);
  CUDA_LAUNCH(launch_fused_f32g(gp, L.n_ranks, w, mm, vv, p, r.d, sc, vec ? 2 : 3,
                                reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

// device address of a page-locked host buffer, or null (with the message set) when the
// buffer is not page-locked host memory the device can address
static const void* host_buffer_device_address(const void* p, const char* who, const char* what, int idx) {
  if (!p) {
    set_error(ZERO_ERR_INVALID_ARG, "%s: %s[%d] is NULL (missing rank)", who, what, idx);
    return nullptr;
  }
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error(ZERO_ERR_INVALID_ARG, "%s: %s[%d]: cudaPointerGetAttributes: %s", who, what, idx, cudaGetErrorString(e));
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) {
    set_error(ZERO_ERR_INVALID_ARG, "%s: %s[%d] is not page-locked host memory mapped for the device", who, what, idx);
    return nullptr;
  }
  return a.devicePointer;
}

extern "C" int zero_fused_step_host(const zero_plan_t* plan, int rank, const zero_bf16* const host_grads[],
                                    float* master, float* m, float* v, zero_bf16* host_param_out, const zero_adam* hp,
                                    int64_t step, zero_stream_t stream) {
  clear_error();
  const char* who = "zero_fused_step_host";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  CHECK_ARG(host_grads != nullptr, "%s: host_grads array is NULL", who);
  const zero_layout& L = plan->lay;
  const zero_bf16* dev_grads[ZERO_MAX_RANKS];
  for (int q = 0; q < L.n_ranks; ++q) {
    dev_grads[q] = static_cast<const zero_bf16*>(host_buffer_device_address(host_grads[q], who, "host_grads", q));
    if (!dev_grads[q]) return ZERO_ERR_INVALID_ARG;
  }
  zero_bf16* dev_param =
      static_cast<zero_bf16*>(const_cast<void*>(host_buffer_device_address(host_param_out, who, "host_param_out", 0)));
  if (!dev_param) return ZERO_ERR_INVALID_ARG;
  return fused_impl(plan, rank, 0, L.n_buckets, dev_grads, master, m, v, dev_param, hp, step, stream, who);
}

extern "C" int zero_fused_step_buckets(const zero_plan_t* plan, int rank, uint64_t bucket_begin, uint64_t bucket_end,
                                       const zero_bf16* const grads[], float* master, float* m, float* v,
                                       zero_bf16* param_out, const zero_adam* hp, int64_t step, zero_stream_t stream) {
  clear_error();
  return fused_impl(plan, rank, bucket_begin, bucket_end, grads, master, m, v, param_out, hp, step, stream,
                    "zero_fused_step_buckets");
}

extern "C" int zero_allgather_params(const zero_plan_t* plan, const float* const masters[], zero_bf16* full_param,
                                     zero_stream_t stream) {
  clear_error();
  const char* who = "zero_allgather_params";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  CHECK_ARG(masters != nullptr && full_param != nullptr, "%s: NULL argument", who);
  MasterPtrs mp;
  memset(&mp, 0, sizeof(mp));
  bool vec = L.shard_elems % 4 == 0 && aligned(full_param, 8);
  for (int q = 0; q < L.n_ranks; ++q) {
    CHECK_ARG(masters[q] != nullptr, "%s: masters[%d] is NULL (missing rank)", who, q);
    mp.p[q] = masters[q];
    vec = vec && aligned(masters[q], 16);
  }
  CUDA_LAUNCH(launch_allgather(mp, L.n_ranks, L.shard_elems, full_param, vec, reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

extern "C" int ddp_allreduce(const zero_plan_t* plan, const zero_bf16* const grads[], float* g_full,
                             zero_stream_t stream) {
  clear_error();
  const char* who = "ddp_allreduce";
  CHECK_ARG(plan != nullptr, "%s: plan is NULL", who);
  const zero_layout& L = plan->lay;
  CHECK_ARG(g_full != nullptr, "%s: g_full is NULL", who);
  GradPtrs gp;
  int rc = load_grads(grads, L.n_ranks, 0, who, &gp);
  if (rc) return rc;
  // every rank's reduce-scatter result written at its own offset r*S: the all-gather of
  // the fp32 shards is in place, so the whole padded buffer is one domain
  const Domain d{1, L.psi_padded, 0};
  const bool vec = grads_aligned(gp, L.n_ranks, 8) && aligned(g_full, 16);
  CUDA_LAUNCH(launch_reduce(gp, L.n_ranks, g_full, d, 1.0f / static_cast<float>(L.n_ranks), vec,
                            reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

// ======================================================================================
// FSDP unit
// ======================================================================================

extern "C" int fsdp_gather_rows(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out, int64_t k_in,
                                zero_bf16* w_full, zero_stream_t stream) {
  clear_error();
  const char* who = "fsdp_gather_rows";
  CHECK_ARG(n_ranks >= 1 && n_ranks <= ZERO_MAX_RANKS, "%s: n_ranks %d outside 1..%d", who, n_ranks, ZERO_MAX_RANKS);
  CHECK_ARG(rows_out >= 1 && k_in >= 1, "%s: rows_out and k_in must be >= 1", who);
  CHECK_ARG(rows_out % n_ranks == 0, "%s: rows_out %lld is not a multiple of n_ranks %d", who, (long long)rows_out,
            n_ranks);
  CHECK_ARG(w_shards != nullptr && w_full != nullptr, "%s: NULL argument", who);
  GradPtrs sp;
  int rc = load_grads(w_shards, n_ranks, 0, who, &sp);
  if (rc) return rc;
  const uint64_t shard_elems = static_cast<uint64_t>(rows_out / n_ranks) * static_cast<uint64_t>(k_in);
  const bool vec = shard_elems % 8 == 0 && grads_aligned(sp, n_ranks, 16) && aligned(w_full, 16);
  CUDA_LAUNCH(launch_gather_rows(sp, n_ranks, shard_elems, w_full, vec, reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

extern "C" int fsdp_unit_forward(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out, int64_t k_in,
                                 const zero_bf16* A, int64_t m_tokens, float* Y, zero_bf16* Y_bf16,
                                 zero_bf16* scratch_w, zero_stream_t stream) {
  clear_error();
  const char* who = "fsdp_unit_forward";
  CHECK_ARG(n_ranks >= 1 && n_ranks <= ZERO_MAX_RANKS, "%s: n_ranks %d outside 1..%d", who, n_ranks, ZERO_MAX_RANKS);
  CHECK_ARG(rows_out >= 1 && k_in >= 1 && m_tokens >= 1, "%s: sizes must be >= 1", who);
  CHECK_ARG(rows_out % n_ranks == 0, "%s: rows_out %lld is not a multiple of n_ranks %d", who, (long long)rows_out,
            n_ranks);
  CHECK_ARG(k_in % 8 == 0, "%s: k_in %lld must be a multiple of 8 (16-byte rows)", who, (long long)k_in);
  CHECK_ARG(A != nullptr && w_shards != nullptr, "%s: NULL argument", who);
  CHECK_ARG(Y != nullptr || Y_bf16 != nullptr, "%s: Y and Y_bf16 are both NULL", who);
  CHECK_ARG(Y != nullptr || rows_out % 8 == 0, "%s: a bf16-only output needs rows_out %% 8 == 0", who);
  CHECK_ARG(aligned(A, 16) && aligned(Y, 16) && (!Y_bf16 || aligned(Y_bf16, 16)) &&
                (!scratch_w || aligned(scratch_w, 16)),
            "%s: A, Y, Y_bf16 and scratch_w must be 16-byte aligned", who);
  for (int q = 0; q < n_ranks; ++q) {
    CHECK_ARG(w_shards[q] != nullptr, "%s: w_shards[%d] is NULL (missing rank)", who, q);
    CHECK_ARG(aligned(w_shards[q], 16), "%s: w_shards[%d] must be 16-byte aligned", who, q);
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (scratch_w) {
    int rc = fsdp_gather_rows(n_ranks, w_shards, rows_out, k_in, scratch_w, stream);
    if (rc) return rc;
    const uint16_t* w1[1] = {scratch_w};
    return launch_fsdp_gemm(1, w1, rows_out, k_in, A, m_tokens, Y, Y_bf16, 1.0f, st);
  }
  return launch_fsdp_gemm(n_ranks, w_shards, rows_out, k_in, A, m_tokens, Y, Y_bf16, 1.0f, st);
}

// ======================================================================================
// status
// ======================================================================================

extern "C" const char* zero_last_error(void) { return g_msg; }

extern "C" int zero_device_status(zero_stream_t stream) {
  clear_error();
  CUDA_LAUNCH(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  const unsigned int a = step_kernels_read_clear_error();
  const unsigned int f = fused_step_read_clear_error();
  const unsigned int b = fsdp_gemm_read_clear_error();
  if (a == 0xffffffffu || f == 0xffffffffu || b == 0xffffffffu)
    return set_error(ZERO_ERR_CUDA, "zero_device_status: cannot read the device error word");
  if (a || f || b)
    return set_error(ZERO_ERR_DEVICE,
                     "zero_device_status: a bounded wait gave up (step kernels code 0x%x, fused step code 0x%x, "
                     "FSDP GEMM code 0x%x; high byte = kernel, low byte = wait)",
                     a, f, b);
  return ZERO_OK;
}

extern "C" int zero_selftest_bounded_wait(uint32_t timeout_ms, zero_stream_t stream) {
  clear_error();
  CHECK_ARG(timeout_ms >= 1 && timeout_ms <= 2000, "zero_selftest_bounded_wait: timeout_ms %u outside 1..2000",
            timeout_ms);
  CUDA_LAUNCH(launch_wait_selftest(static_cast<unsigned long long>(timeout_ms) * 1000000ull,
                                   reinterpret_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

extern "C" int zero_set_fused_kernel(int which) {
  clear_error();
  CHECK_ARG(which >= 0 && which <= 2, "zero_set_fused_kernel: %d is not 0, 1 or 2", which);
  g_fused_variant.store(which, std::memory_order_relaxed);
  return ZERO_OK;
}

extern "C" int zero_set_gemm_kernel(int which) {
  clear_error();
  CHECK_ARG(which >= 0 && which <= 2, "zero_set_gemm_kernel: %d is not 0, 1 or 2", which);
  set_gemm_kernel(which);
  return ZERO_OK;
}

extern "C" int zero_version(void) { return 100; }
