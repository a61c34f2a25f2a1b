// FSDP unit GEMM (tcgen05 / TMEM / TMA) — under construction.
#include "device_common.cuh"

namespace zgb {
ZGB_DECLARE_ERROR_WORD();

int launch_fsdp_gemm(int, const uint16_t* const*, int64_t, int64_t, const uint16_t*, int64_t, float*, uint16_t*,
                     cudaStream_t) {
  return set_error(ZERO_ERR_UNSUPPORTED, "fsdp_unit_forward: GEMM kernel not built yet");
}

unsigned int fsdp_gemm_read_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_zgb_dev_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v) cudaMemcpyToSymbol(g_zgb_dev_error, &zero, sizeof(zero));
  return v;
}
}  // namespace zgb
