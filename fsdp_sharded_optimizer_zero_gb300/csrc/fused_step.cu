// The fused optimizer step: reduce-scatter + Adam + bf16 cast / all-gather write in one
// pass over HBM, 2N + 26 bytes per parameter (4N + 26 with fp32 gradients): the
// register-streaming kernel (the default), the TMA bulk-copy pipeline and the scalar
// kernel for unaligned buffers. All three run the same per-element arithmetic
// (step_common.cuh, device_common.cuh) and give identical bits.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "step_common.cuh"

namespace zgb {

ZGB_DECLARE_ERROR_WORD();

namespace {

// device error codes of this file: (kernel id << 8) | wait id
constexpr unsigned int kErrTmaEmpty = (1u << 8) | 1u;  // producer waiting for a free stage
constexpr unsigned int kErrTmaFull = (1u << 8) | 2u;   // consumer waiting for a loaded stage
constexpr unsigned int kErrTmaDrain = (1u << 8) | 3u;  // producer draining copies after an abort

// ------------------------------------------------------------------------------------
// fused step, register-streaming variant: every thread loads its N gradient vectors and
// its state straight into registers (no shared memory)
// ------------------------------------------------------------------------------------
template <int NR, typename G>
__global__ void __launch_bounds__(kThreads) fused_vec_kernel(RankPtrs<G> gp, int n, float* __restrict__ master,
                                                             float* __restrict__ m, float* __restrict__ v,
                                                             uint16_t* __restrict__ param, Domain d,
                                                             AdamScalars sc) {
  const uint64_t ups = (d.seg_len + 3) / 4, total = ups * d.n_seg;
  const uint64_t stride = (uint64_t)gridDim.x * kThreads;
  for (uint64_t u = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u < total; u += stride) {
    const UnitPos p = unit_pos(d, ups, u);
    if (p.count == 4) {
      const float4 w = __ldcs(reinterpret_cast<const float4*>(master + p.base));
      const float4 mm = __ldcs(reinterpret_cast<const float4*>(m + p.base));
      const float4 vv = __ldcs(reinterpret_cast<const float4*>(v + p.base));
      float g[4];
      reduce4<NR, G>(gp, n, p.base, g);
      adam4_store(g, w, mm, vv, master, m, v, param, p.base, sc);
    } else {
      for (uint32_t k = 0; k < p.count; ++k) fused_elem(gp, n, master, m, v, param, p.base + k, sc);
    }
  }
}

// Blocks per SM of the register-streaming kernel's grid on long launches. With 40
// registers per thread six 256-thread blocks fit on an SM, but on GB300 four held the
// highest share of the copy bandwidth for N = 1, 2, 8, 12, 16, 32, 64 and both gradient
// types; one full wave (six per SM) or several waves of the full grid lost 2-8 %. For
// N = 3..7 (fewer bytes in flight per thread) the full grid held 0.5-2 % more (N = 4 showed
// no grid that won on every domain shape).
inline unsigned int fused_vec_blocks_per_sm(int n) { return n >= 3 && n <= 7 ? 16u : 4u; }

// scalar variant for buffers whose alignment rules out vector accesses
template <typename G>
__global__ void __launch_bounds__(kThreads) fused_scalar_kernel(RankPtrs<G> gp, int n, float* master, float* m,
                                                                float* v, uint16_t* param, Domain d,
                                                                AdamScalars sc) {
  const uint64_t total = d.seg_len * d.n_seg;
  for (uint64_t e = blockIdx.x * (uint64_t)kThreads + threadIdx.x; e < total; e += (uint64_t)gridDim.x * kThreads) {
    const uint64_t seg = d.n_seg > 1 ? e / d.seg_len : 0;
    const uint64_t j = seg * d.seg_stride + (e - seg * d.seg_len);
    fused_elem(gp, n, master, m, v, param, j, sc);
  }
}

// ------------------------------------------------------------------------------------
// fused step, TMA bulk-copy pipeline.
// One CTA per SM, persistent over tiles of `tile` elements. The last warp (one elected
// lane) is the producer: for each tile it issues N + 3 one-dimensional bulk copies (the N
// ranks' gradient chunks and the master / m / v slices) into a shared-memory stage and
// arms the stage's "full" mbarrier with the byte count. The other warps consume: they
// wait for the stage, reduce the N chunks in rank order, run Adam, store master / m / v /
// param to HBM with streaming stores, and release the stage through its "empty" mbarrier.
// A tile's ragged end (< 8 elements, below the 16-byte copy granule) is read directly
// from global memory by the consumers.
// Measured on GB300 (GPT-2-small list, N = 8): 16 consumer warps reach 97.5 % of the
// copy bandwidth (8 warps: 88 %, the IEEE divide / square-root chains need the extra
// warps); at large N the per-rank chunk of a tile shrinks (512 B at N = 64) and the
// pipeline falls far behind the register-streaming kernel, which is therefore the default.
// ------------------------------------------------------------------------------------
#ifndef ZGB_TMA_CONSUMER_WARPS
#define ZGB_TMA_CONSUMER_WARPS 16
#endif
#ifndef ZGB_TMA_CTAS_PER_SM
#define ZGB_TMA_CTAS_PER_SM 1
#endif
#ifndef ZGB_TMA_SMEM_BUDGET
#define ZGB_TMA_SMEM_BUDGET (200u * 1024u)
#endif
constexpr int kTmaConsumerWarps = ZGB_TMA_CONSUMER_WARPS;
constexpr int kTmaThreads = (kTmaConsumerWarps + 1) * 32;
constexpr int kTmaCtasPerSm = ZGB_TMA_CTAS_PER_SM;
constexpr int kTmaMaxStages = 8;
constexpr uint32_t kTmaSmemBudget = ZGB_TMA_SMEM_BUDGET;  // bytes of all stages of one CTA
constexpr uint32_t kTmaStageBudget = kTmaSmemBudget / 3 < 64u * 1024u ? kTmaSmemBudget / 3 : 64u * 1024u;

struct TileSpan {
  uint64_t base;  // flat index of the tile's first element
  uint32_t len;   // elements in the tile
};
__device__ __forceinline__ TileSpan tile_span(const Domain& d, uint64_t tiles_per_seg, uint32_t tile, uint64_t t) {
  uint64_t seg = 0, local = t;
  if (d.n_seg > 1) {
    seg = t / tiles_per_seg;
    local = t - seg * tiles_per_seg;
  }
  const uint64_t e0 = local * tile, rem = d.seg_len - e0;
  return {seg * d.seg_stride + e0, static_cast<uint32_t>(rem < tile ? rem : tile)};
}

__global__ void __launch_bounds__(kTmaThreads, kTmaCtasPerSm)
    fused_tma_kernel(GradPtrs gp, int n, float* __restrict__ master, float* __restrict__ m, float* __restrict__ v,
                     uint16_t* __restrict__ param, Domain d, AdamScalars sc, uint32_t tile, uint32_t stages) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kTmaMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kTmaMaxStages];
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;

  const uint32_t grad_bytes = tile * 2u;
  const uint32_t stage_bytes = static_cast<uint32_t>(n) * grad_bytes + 12u * tile;
  const uint64_t tps = (d.seg_len + tile - 1) / tile;
  const uint64_t n_tiles = tps * d.n_seg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kTmaConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kTmaConsumerWarps) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int64_t last_issue[kTmaMaxStages];
    for (uint32_t s = 0; s < kTmaMaxStages; ++s) last_issue[s] = -1;
    uint32_t it = 0;
    for (uint64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
      const uint32_t s = it % stages, ph = (it / stages) & 1u;
      const uint32_t fb = smem_u32(&full_bar[s]);
      if (it >= stages && !mbar_wait_bounded(smem_u32(&empty_bar[s]), ph ^ 1u, abort, &g_zgb_dev_error, kErrTmaEmpty))
        break;
      const TileSpan sp = tile_span(d, tps, tile, t);
      const uint32_t body = sp.len & ~7u;
      mbar_arrive_expect_tx(fb, body * (2u * static_cast<uint32_t>(n) + 12u));
      if (body) {
        const uint32_t sb = smem_u32(smem + static_cast<size_t>(s) * stage_bytes);
        for (int r = 0; r < n; ++r) bulk_g2s(sb + r * grad_bytes, gp.p[r] + sp.base, body * 2u, fb);
        const uint32_t fs = sb + n * grad_bytes;
        bulk_g2s(fs, master + sp.base, body * 4u, fb);
        bulk_g2s(fs + tile * 4u, m + sp.base, body * 4u, fb);
        bulk_g2s(fs + tile * 8u, v + sp.base, body * 4u, fb);
      }
      last_issue[s] = it;
    }
    if (*abort) {
      // no copy may still be writing this CTA's shared memory when it exits
      int never = 0;
      for (uint32_t s = 0; s < stages; ++s)
        if (last_issue[s] >= 0)
          mbar_wait_bounded(smem_u32(&full_bar[s]), static_cast<uint32_t>(last_issue[s] / stages) & 1u, &never,
                            &g_zgb_dev_error, kErrTmaDrain);
    }
    return;
  }

  // ---------------- consumers ----------------
  uint32_t it = 0;
  for (uint64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
    const uint32_t s = it % stages, ph = (it / stages) & 1u;
    if (!mbar_wait_bounded(smem_u32(&full_bar[s]), ph, abort, &g_zgb_dev_error, kErrTmaFull)) break;
    const TileSpan sp = tile_span(d, tps, tile, t);
    const uint32_t body = sp.len & ~7u;
    const uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes;
    const uint16_t* sg = reinterpret_cast<const uint16_t*>(st);
    const float* sw = reinterpret_cast<const float*>(st + n * grad_bytes);
    const float* sm = sw + tile;
    const float* sv = sm + tile;
    for (uint32_t e = threadIdx.x * 4u; e < sp.len; e += kTmaConsumerWarps * 32u * 4u) {
      const uint64_t j = sp.base + e;
      if (e < body) {
        float g[4];
        widen4(*reinterpret_cast<const uint2*>(sg + e), g);
        for (int r = 1; r < n; ++r) accum4(*reinterpret_cast<const uint2*>(sg + static_cast<size_t>(r) * tile + e), g);
        adam4_store(g, *reinterpret_cast<const float4*>(sw + e), *reinterpret_cast<const float4*>(sm + e),
                    *reinterpret_cast<const float4*>(sv + e), master, m, v, param, j, sc);
      } else {
        const uint32_t stop = min(e + 4u, sp.len);
        for (uint32_t k = e; k < stop; ++k) fused_elem(gp, n, master, m, v, param, sp.base + k, sc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
  }
}

}  // namespace

namespace {
struct TmaConfig {
  uint32_t tile, stages, smem;
};
TmaConfig tma_config(int n) {
  const uint32_t per_elem = 2u * static_cast<uint32_t>(n) + 12u;
  uint32_t tile = 4096;
  while (tile > 256 && per_elem * tile > kTmaStageBudget) tile /= 2;
  const uint32_t stage_bytes = per_elem * tile;
  uint32_t stages = std::min<uint32_t>(kTmaMaxStages, kTmaSmemBudget / stage_bytes);
  if (stages < 2) stages = 2;
  return {tile, stages, stages * stage_bytes};
}

OncePerDevice g_tma_attr_once;
}  // namespace

cudaError_t launch_fused(const GradPtrs& gp, int n, float* master, float* m, float* v, uint16_t* param,
                         const Domain& d, const AdamScalars& sc, int variant, cudaStream_t st) {
  const uint64_t total = d.seg_len * d.n_seg;
  if (total == 0) return cudaSuccess;
  if (variant == 1) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const cudaError_t attr_err = g_tma_attr_once.run(dev, [] {
      return cudaFuncSetAttribute(fused_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kTmaSmemBudget));
    });
    if (attr_err != cudaSuccess) return attr_err;
    const TmaConfig c = tma_config(n);
    const uint64_t tiles = (d.seg_len + c.tile - 1) / c.tile * d.n_seg;
    const unsigned int grid =
        static_cast<unsigned int>(std::max<uint64_t>(1, std::min<uint64_t>(tiles, num_sms() * kTmaCtasPerSm)));
    fused_tma_kernel<<<grid, kTmaThreads, c.smem, st>>>(gp, n, master, m, v, param, d, sc, c.tile, c.stages);
    return cudaGetLastError();
  }
  if (variant == 2) {
    const unsigned int grid = grid_streaming((d.seg_len + 3) / 4 * d.n_seg, fused_vec_blocks_per_sm(n));
    return dispatch_nr(n, [&](auto nr) {
      fused_vec_kernel<decltype(nr)::value, uint16_t><<<grid, kThreads, 0, st>>>(gp, n, master, m, v, param, d, sc);
      return cudaGetLastError();
    });
  }
  fused_scalar_kernel<uint16_t><<<grid_for(total), kThreads, 0, st>>>(gp, n, master, m, v, param, d, sc);
  return cudaGetLastError();
}

cudaError_t launch_fused_f32g(const F32GradPtrs& gp, int n, float* master, float* m, float* v, uint16_t* param,
                              const Domain& d, const AdamScalars& sc, int variant, cudaStream_t st) {
  const uint64_t total = d.seg_len * d.n_seg;
  if (total == 0) return cudaSuccess;
  if (variant == 2) {
    const unsigned int grid = grid_streaming((d.seg_len + 3) / 4 * d.n_seg, fused_vec_blocks_per_sm(n));
    return dispatch_nr(n, [&](auto nr) {
      fused_vec_kernel<decltype(nr)::value, float><<<grid, kThreads, 0, st>>>(gp, n, master, m, v, param, d, sc);
      return cudaGetLastError();
    });
  }
  fused_scalar_kernel<float><<<grid_for(total), kThreads, 0, st>>>(gp, n, master, m, v, param, d, sc);
  return cudaGetLastError();
}

unsigned int fused_step_read_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_zgb_dev_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v) cudaMemcpyToSymbol(g_zgb_dev_error, &zero, sizeof(zero));
  return v;
}

}  // namespace zgb
