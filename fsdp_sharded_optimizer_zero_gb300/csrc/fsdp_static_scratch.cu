// fsdp_unit_forward_static_scratch: the FSDP unit forward for callers that cannot allocate
// device memory. When W's shards do not tile the GEMM, the gathered weight goes into a
// fixed device array of this library instead of a buffer the caller allocates.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at the point where
// they run the unit — for example a plug-in hosted by a framework that owns all device
// memory through its own pool and forbids other allocations, or code on a latency-
// critical path where cudaMalloc's implicit device-wide synchronisation is not
// acceptable. They still pass the shards, A and Y (and Y_bf16); only the scratch is
// provided here.
//
// Limits and behaviour:
//   - When the shards tile the GEMM (fsdp_unit_forward's fused gather applies: at most 16
//     shards of a multiple of 128 rows, 256 under zero_set_gemm_kernel(1)), the GEMM reads
//     W straight from its shards: no scratch is used and no size limit applies.
//   - Otherwise W is gathered into the array, which holds kStaticScratchElems = 8,388,608
//     bf16 elements (16 MiB); larger weights (rows_out * k_in above that) are rejected with
//     ZERO_ERR_INVALID_ARG.
//   - The array is part of the library's device image: every GPU on which the library's
//     module is loaded holds those 16 MiB until the process exits.
//   - Host code cannot use the array's name as a device address. Each call made outside
//     stream capture looks the address up with cudaGetSymbolAddress (current device and
//     context), checks the result and caches it with the context it belongs to; a call
//     made during capture uses the cached address, and only if it was taken in the
//     current context (else ZERO_ERR_INVALID_ARG). So the first call on a device, and the
//     first after a cudaDeviceReset, must come before any stream capture.
//   - Every call shares the one array and leaves the last call's gathered W in it. The
//     gather rewrites every element the GEMM reads, so nothing needs clearing; but two
//     calls that overlap on the GPU (different streams, no ordering) race on the array.
//   - No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace zgb {
namespace {

constexpr uint64_t kStaticScratchElems = 8ull << 20;  // bf16 elements (16 MiB)

static __device__ __align__(256) uint16_t g_static_w[kStaticScratchElems];

struct ScratchEntry {
  CUcontext ctx;
  uint16_t* ptr;
};

std::mutex g_scratch_mu;
ScratchEntry g_scratch[64] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

const char* const kWho = "fsdp_unit_forward_static_scratch";

int current_context(CUcontext* ctx) {
  std::call_once(g_ctx_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  if (!g_ctx_current) return set_error(ZERO_ERR_CUDA, "%s: cuCtxGetCurrent unavailable", kWho);
  *ctx = nullptr;
  if (g_ctx_current(ctx) != CUDA_SUCCESS || *ctx == nullptr)
    return set_error(ZERO_ERR_CUDA, "%s: no current CUDA context", kWho);
  return ZERO_OK;
}

// The array's device address in the current device's current context.
int static_scratch(cudaStream_t st, uint16_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: cudaGetDevice: %s", kWho, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(ZERO_ERR_UNSUPPORTED, "%s: device %d", kWho, dev);
  // a call cudaStreamIsCapturing cannot answer is treated as captured: no look-up then
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    cs = cudaStreamCaptureStatusActive;
  }
  CUcontext ctx = nullptr;
  int rc = current_context(&ctx);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_w);
    if (e != cudaSuccess || p == nullptr)
      return set_error(ZERO_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", kWho, cudaGetErrorString(e));
    ent.ctx = ctx;
    ent.ptr = static_cast<uint16_t*>(p);
  } else if (ent.ptr == nullptr || ent.ctx != ctx) {
    return set_error(ZERO_ERR_INVALID_ARG,
                     "%s: called during stream capture before any call outside capture in this device's current "
                     "context; make one call first, outside capture",
                     kWho);
  }
  *out = ent.ptr;
  return ZERO_OK;
}

}  // namespace
}  // namespace zgb

using namespace zgb;

extern "C" int fsdp_unit_forward_static_scratch(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out,
                                                int64_t k_in, const zero_bf16* A, int64_t m_tokens, float* Y,
                                                zero_bf16* Y_bf16, zero_stream_t stream) {
  // shards that tile the GEMM need no gathered copy of W at all
  if (fsdp_fused_gather_ok(n_ranks, rows_out))
    return fsdp_unit_forward(n_ranks, w_shards, rows_out, k_in, A, m_tokens, Y, Y_bf16, nullptr, stream);
  if (rows_out < 1 || k_in < 1 ||
      static_cast<uint64_t>(rows_out) > kStaticScratchElems / static_cast<uint64_t>(k_in))
    return set_error(ZERO_ERR_INVALID_ARG,
                     "%s: rows_out * k_in = %lld x %lld exceeds the static scratch of %llu bf16 elements (16 MiB) "
                     "and the shards do not tile the GEMM",
                     kWho, (long long)rows_out, (long long)k_in, (unsigned long long)kStaticScratchElems);
  uint16_t* scratch = nullptr;
  int rc = static_scratch(reinterpret_cast<cudaStream_t>(stream), &scratch);
  if (rc) return rc;
  return fsdp_unit_forward(n_ranks, w_shards, rows_out, k_in, A, m_tokens, Y, Y_bf16, scratch, stream);
}
