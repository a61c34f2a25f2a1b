// fsdp_unit_forward_static_scratch: the FSDP unit forward with a materialised gather whose
// scratch (the gathered weight W) lives in a fixed device array of this library instead
// of a buffer the caller allocates.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at the point where
// they run the unit — for example a plug-in hosted by a framework that owns all device
// memory through its own pool and forbids other allocations, or code on a latency-
// critical path where cudaMalloc's implicit device-wide synchronisation is not
// acceptable. They still pass the shards, A and Y (and Y_bf16); only the scratch is
// provided here.
//
// Limits and behaviour:
//   - The array holds kStaticScratchElems = 8,388,608 bf16 elements (16 MiB); larger
//     weights (rows_out * k_in above that) are rejected with ZERO_ERR_INVALID_ARG.
//   - The array is part of the library's device image: every GPU on which the library's
//     module is loaded holds those 16 MiB until the process exits.
//   - Host code cannot use the array's name as a device address. The first call on each
//     device (that device current) looks the address up with cudaGetSymbolAddress, checks
//     the result and caches it; make that first call before any stream capture.
//   - Every call shares the one array and leaves the last call's gathered W in it. The
//     gather rewrites every element the GEMM reads, so nothing needs clearing; but two
//     calls that overlap on the GPU (different streams, no ordering) race on the array.
//   - No cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>

#include "internal.h"

namespace zgb {
namespace {

constexpr uint64_t kStaticScratchElems = 8ull << 20;  // bf16 elements (16 MiB)

static __device__ __align__(256) uint16_t g_static_w[kStaticScratchElems];

std::mutex g_scratch_mu;
uint16_t* g_scratch_ptr[64] = {nullptr};

int static_scratch(uint16_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "fsdp_unit_forward_static_scratch: cudaGetDevice: %s",
                                         cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(ZERO_ERR_UNSUPPORTED, "fsdp_unit_forward_static_scratch: device %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_w);
    if (e != cudaSuccess || p == nullptr)
      return set_error(ZERO_ERR_CUDA, "fsdp_unit_forward_static_scratch: cudaGetSymbolAddress: %s",
                       cudaGetErrorString(e));
    g_scratch_ptr[dev] = static_cast<uint16_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return ZERO_OK;
}

}  // namespace
}  // namespace zgb

using namespace zgb;

extern "C" int fsdp_unit_forward_static_scratch(int n_ranks, const zero_bf16* const w_shards[], int64_t rows_out,
                                                int64_t k_in, const zero_bf16* A, int64_t m_tokens, float* Y,
                                                zero_bf16* Y_bf16, zero_stream_t stream) {
  if (rows_out < 1 || k_in < 1 ||
      static_cast<uint64_t>(rows_out) > kStaticScratchElems / static_cast<uint64_t>(k_in))
    return set_error(ZERO_ERR_INVALID_ARG,
                     "fsdp_unit_forward_static_scratch: rows_out * k_in = %lld x %lld exceeds the static scratch of "
                     "%llu bf16 elements (16 MiB)",
                     (long long)rows_out, (long long)k_in, (unsigned long long)kStaticScratchElems);
  uint16_t* scratch = nullptr;
  int rc = static_scratch(&scratch);
  if (rc) return rc;
  return fsdp_unit_forward(n_ranks, w_shards, rows_out, k_in, A, m_tokens, Y, Y_bf16, scratch, stream);
}
