// Memory-bound kernels of the optimizer step: reduce-scatter, Adam, the fused
// reduce-scatter + Adam + bf16 cast, the parameter all-gather and the FSDP row gather.
//
// All of them are elementwise over a Domain (see internal.h) and HBM-bandwidth bound:
// the fused step moves 2N + 26 bytes per parameter (N bf16 gradient reads, fp32 master /
// m / v read and written, one bf16 parameter write) and does ~N + 20 flops.
//
// Work unit: 4 consecutive elements per thread-iteration, so every global access of a
// warp is one contiguous run (bf16 grads: 8 B per lane; fp32 state: 16 B per lane) and
// every shared-memory read is bank-conflict free.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"

namespace zgb {

ZGB_DECLARE_ERROR_WORD();

namespace {

constexpr int kThreads = 256;

// device error codes of this file: (kernel id << 8) | wait id
constexpr unsigned int kErrTmaEmpty = (1u << 8) | 1u;  // producer waiting for a free stage
constexpr unsigned int kErrTmaFull = (1u << 8) | 2u;   // consumer waiting for a loaded stage
constexpr unsigned int kErrTmaDrain = (1u << 8) | 3u;  // producer draining copies after an abort
constexpr unsigned int kErrSelftest = (3u << 8) | 1u;  // the bounded-wait self-test

// ------------------------------------------------------------------------------------
// the reduced gradient: fp32 sum in rank order 0..N-1
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void widen4(uint2 u, float s[4]) {
  s[0] = bf16_lo(u.x);
  s[1] = bf16_hi(u.x);
  s[2] = bf16_lo(u.y);
  s[3] = bf16_hi(u.y);
}
__device__ __forceinline__ void accum4(uint2 u, float s[4]) {
  s[0] = __fadd_rn(s[0], bf16_lo(u.x));
  s[1] = __fadd_rn(s[1], bf16_hi(u.x));
  s[2] = __fadd_rn(s[2], bf16_lo(u.y));
  s[3] = __fadd_rn(s[3], bf16_hi(u.y));
}
// fp32 gradients: widening is the identity
__device__ __forceinline__ void widen4(float4 u, float s[4]) {
  s[0] = u.x;
  s[1] = u.y;
  s[2] = u.z;
  s[3] = u.w;
}
__device__ __forceinline__ void accum4(float4 u, float s[4]) {
  s[0] = __fadd_rn(s[0], u.x);
  s[1] = __fadd_rn(s[1], u.y);
  s[2] = __fadd_rn(s[2], u.z);
  s[3] = __fadd_rn(s[3], u.w);
}
// 4 consecutive gradient elements of one rank (8 B of bf16 or 16 B of fp32)
__device__ __forceinline__ uint2 load4(const uint16_t* p) { return __ldcs(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ float4 load4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float to_f32(uint16_t b) { return bf16_bits_to_f32(b); }
__device__ __forceinline__ float to_f32(float x) { return x; }

// NR > 0: rank count known at compile time, all N loads in flight at once.
// NR == 0: any N; loads issued in groups of 8 ranks, added strictly in rank order.
template <int NR, typename G>
__device__ __forceinline__ void reduce4(const RankPtrs<G>& gp, int n, uint64_t idx, float s[4]) {
  using V = decltype(load4(gp.p[0]));
  if constexpr (NR > 0) {
    V u[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) u[r] = load4(gp.p[r] + idx);
    widen4(u[0], s);
#pragma unroll
    for (int r = 1; r < NR; ++r) accum4(u[r], s);
  } else {
    for (int r0 = 0; r0 < n; r0 += 8) {
      const int cnt = min(8, n - r0);
      V u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < cnt) u[j] = load4(gp.p[r0 + j] + idx);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < cnt) {
          if (r0 + j == 0)
            widen4(u[0], s);
          else
            accum4(u[j], s);
        }
      }
    }
  }
}

template <typename G>
__device__ __forceinline__ float reduce1(const RankPtrs<G>& gp, int n, uint64_t j) {
  float s = to_f32(gp.p[0][j]);
  for (int r = 1; r < n; ++r) s = __fadd_rn(s, to_f32(gp.p[r][j]));
  return s;
}

template <typename G>
__device__ __forceinline__ void fused_elem(const RankPtrs<G>& gp, int n, float* master, float* m, float* v,
                                           uint16_t* param, uint64_t j, const AdamScalars& sc) {
  const float g = __fmul_rn(reduce1(gp, n, j), sc.inv_n);
  float w = master[j], mm = m[j], vv = v[j];
  adam_elem(g, w, mm, vv, sc);
  master[j] = w;
  m[j] = mm;
  v[j] = vv;
  param[j] = f32_to_bf16_bits(w);
}

__device__ __forceinline__ void adam4_store(float g[4], float4 w, float4 mm, float4 vv, float* master, float* m,
                                            float* v, uint16_t* param, uint64_t j, const AdamScalars& sc) {
  adam_elem(__fmul_rn(g[0], sc.inv_n), w.x, mm.x, vv.x, sc);
  adam_elem(__fmul_rn(g[1], sc.inv_n), w.y, mm.y, vv.y, sc);
  adam_elem(__fmul_rn(g[2], sc.inv_n), w.z, mm.z, vv.z, sc);
  adam_elem(__fmul_rn(g[3], sc.inv_n), w.w, mm.w, vv.w, sc);
  __stcs(reinterpret_cast<float4*>(master + j), w);
  __stcs(reinterpret_cast<float4*>(m + j), mm);
  __stcs(reinterpret_cast<float4*>(v + j), vv);
  __stcs(reinterpret_cast<uint2*>(param + j), make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w)));
}

// position of 4-element unit u of a domain: flat index of its first element and the
// number of valid elements (4, or fewer at a segment's ragged end)
struct UnitPos {
  uint64_t base;
  uint32_t count;
};
__device__ __forceinline__ UnitPos unit_pos(const Domain& d, uint64_t units_per_seg, uint64_t u) {
  uint64_t seg = 0, local = u;
  if (d.n_seg > 1) {
    seg = u / units_per_seg;
    local = u - seg * units_per_seg;
  }
  const uint64_t e0 = local * 4, rem = d.seg_len - e0;
  return {seg * d.seg_stride + e0, static_cast<uint32_t>(rem < 4 ? rem : 4)};
}

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
  for (uint64_t u = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u < total; u += (uint64_t)gridDim.x * kThreads) {
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

// ------------------------------------------------------------------------------------
// standalone reduce-scatter / all-reduce: out = (sum_r grads_r) * (1/N), fp32
// ------------------------------------------------------------------------------------
template <int NR>
__global__ void __launch_bounds__(kThreads) reduce_vec_kernel(GradPtrs gp, int n, float* __restrict__ out, Domain d,
                                                              float inv_n) {
  const uint64_t ups = (d.seg_len + 3) / 4, total = ups * d.n_seg;
  for (uint64_t u = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u < total; u += (uint64_t)gridDim.x * kThreads) {
    const UnitPos p = unit_pos(d, ups, u);
    if (p.count == 4) {
      float g[4];
      reduce4<NR, uint16_t>(gp, n, p.base, g);
      __stcs(reinterpret_cast<float4*>(out + p.base),
             make_float4(__fmul_rn(g[0], inv_n), __fmul_rn(g[1], inv_n), __fmul_rn(g[2], inv_n),
                         __fmul_rn(g[3], inv_n)));
    } else {
      for (uint32_t k = 0; k < p.count; ++k) out[p.base + k] = __fmul_rn(reduce1(gp, n, p.base + k), inv_n);
    }
  }
}

__global__ void __launch_bounds__(kThreads) reduce_scalar_kernel(GradPtrs gp, int n, float* out, Domain d,
                                                                 float inv_n) {
  const uint64_t total = d.seg_len * d.n_seg;
  for (uint64_t e = blockIdx.x * (uint64_t)kThreads + threadIdx.x; e < total; e += (uint64_t)gridDim.x * kThreads) {
    const uint64_t seg = d.n_seg > 1 ? e / d.seg_len : 0;
    const uint64_t j = seg * d.seg_stride + (e - seg * d.seg_len);
    out[j] = __fmul_rn(reduce1(gp, n, j), inv_n);
  }
}

// ------------------------------------------------------------------------------------
// standalone Adam on an fp32 reduced gradient (param may be null: no cast)
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void adam_one(const float* g, float* master, float* m, float* v, uint16_t* param,
                                         uint64_t j, const AdamScalars& sc) {
  float w = master[j], mm = m[j], vv = v[j];
  adam_elem(g[j], w, mm, vv, sc);
  master[j] = w;
  m[j] = mm;
  v[j] = vv;
  if (param) param[j] = f32_to_bf16_bits(w);
}

__global__ void __launch_bounds__(kThreads) adam_vec_kernel(const float* __restrict__ g, float* __restrict__ master,
                                                            float* __restrict__ m, float* __restrict__ v,
                                                            uint16_t* __restrict__ param, Domain d, AdamScalars sc) {
  const uint64_t ups = (d.seg_len + 3) / 4, total = ups * d.n_seg;
  for (uint64_t u = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u < total; u += (uint64_t)gridDim.x * kThreads) {
    const UnitPos p = unit_pos(d, ups, u);
    if (p.count == 4) {
      const float4 gg = __ldcs(reinterpret_cast<const float4*>(g + p.base));
      float4 w = __ldcs(reinterpret_cast<const float4*>(master + p.base));
      float4 mm = __ldcs(reinterpret_cast<const float4*>(m + p.base));
      float4 vv = __ldcs(reinterpret_cast<const float4*>(v + p.base));
      adam_elem(gg.x, w.x, mm.x, vv.x, sc);
      adam_elem(gg.y, w.y, mm.y, vv.y, sc);
      adam_elem(gg.z, w.z, mm.z, vv.z, sc);
      adam_elem(gg.w, w.w, mm.w, vv.w, sc);
      __stcs(reinterpret_cast<float4*>(master + p.base), w);
      __stcs(reinterpret_cast<float4*>(m + p.base), mm);
      __stcs(reinterpret_cast<float4*>(v + p.base), vv);
      if (param)
        __stcs(reinterpret_cast<uint2*>(param + p.base), make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w)));
    } else {
      for (uint32_t k = 0; k < p.count; ++k) adam_one(g, master, m, v, param, p.base + k, sc);
    }
  }
}

__global__ void __launch_bounds__(kThreads) adam_scalar_kernel(const float* g, float* master, float* m, float* v,
                                                               uint16_t* param, Domain d, AdamScalars sc) {
  const uint64_t total = d.seg_len * d.n_seg;
  for (uint64_t e = blockIdx.x * (uint64_t)kThreads + threadIdx.x; e < total; e += (uint64_t)gridDim.x * kThreads) {
    const uint64_t seg = d.n_seg > 1 ? e / d.seg_len : 0;
    adam_one(g, master, m, v, param, seg * d.seg_stride + (e - seg * d.seg_len), sc);
  }
}

// ------------------------------------------------------------------------------------
// parameter all-gather with the bf16 cast: full[r*S + i] = bf16(masters[r][i])
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) allgather_kernel(MasterPtrs mp, int n, uint64_t shard,
                                                             uint16_t* __restrict__ full, int vec) {
  if (vec) {  // shard % 4 == 0 and aligned: a 4-element unit never straddles two ranks
    const uint64_t upr = shard / 4, total = upr * static_cast<uint64_t>(n);
    for (uint64_t u = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u < total; u += (uint64_t)gridDim.x * kThreads) {
      const uint64_t r = u / upr, i = (u - r * upr) * 4;
      const float4 w = __ldcs(reinterpret_cast<const float4*>(mp.p[r] + i));
      __stcs(reinterpret_cast<uint2*>(full + r * shard + i), make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w)));
    }
  } else {
    const uint64_t total = shard * static_cast<uint64_t>(n);
    for (uint64_t j = blockIdx.x * (uint64_t)kThreads + threadIdx.x; j < total; j += (uint64_t)gridDim.x * kThreads) {
      const uint64_t r = j / shard;
      full[j] = f32_to_bf16_bits(mp.p[r][j - r * shard]);
    }
  }
}

// ------------------------------------------------------------------------------------
// FSDP row gather: shard r's rows land at rows [r*R/N, (r+1)*R/N) of W, i.e. at the
// contiguous element range [r*E, (r+1)*E) with E = (R/N) * K
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(GradPtrs shards, int n, uint64_t shard_elems,
                                                               uint16_t* __restrict__ full, int vec) {
  if (vec) {  // shard_elems % 8 == 0 and 16-byte aligned: 16-byte units
    const uint64_t upr = shard_elems / 8, total = upr * static_cast<uint64_t>(n);
    for (uint64_t u = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u < total; u += (uint64_t)gridDim.x * kThreads) {
      const uint64_t r = u / upr, i = (u - r * upr) * 8;
      __stcs(reinterpret_cast<uint4*>(full + r * shard_elems + i), __ldcs(reinterpret_cast<const uint4*>(shards.p[r] + i)));
    }
  } else {
    const uint64_t total = shard_elems * static_cast<uint64_t>(n);
    for (uint64_t j = blockIdx.x * (uint64_t)kThreads + threadIdx.x; j < total; j += (uint64_t)gridDim.x * kThreads) {
      const uint64_t r = j / shard_elems;
      full[j] = shards.p[r][j - r * shard_elems];
    }
  }
}

// ------------------------------------------------------------------------------------
// FSDP backward operand layout: dst[c][q * rows + r] = srcs[q][r][c], i.e. the N row-major
// [rows, cols] bf16 sources transposed and concatenated along the new column axis. It
// produces W^T from W's row shards (the backward all-gather of W) and the rank-concatenated
// dY^T and X^T whose product sums the ranks' weight gradients inside one GEMM. 64 x 64
// tiles through shared memory; 16-byte loads and stores when rows and columns allow.
// ------------------------------------------------------------------------------------
constexpr int kTT = 64;

__global__ void __launch_bounds__(256) transpose_cat_kernel(GradPtrs srcs, int64_t rows, int64_t cols,
                                                            int64_t total_rows, uint16_t* __restrict__ dst, int vec) {
  __shared__ uint16_t tile[kTT][kTT + 2];
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTT;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTT;
  const int t = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int v = t + i * 256, rr = v >> 3, cv = (v & 7) * 8;
    const int64_t gr = r0 + rr;
    if (gr >= total_rows) continue;
    const int64_t q = gr / rows, lr = gr - q * rows;
    const uint16_t* src = srcs.p[q] + lr * cols + c0 + cv;
    if (vec && c0 + cv + 8 <= cols) {
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(src));
      uint32_t* trow = reinterpret_cast<uint32_t*>(&tile[rr][cv]);
      trow[0] = u.x;
      trow[1] = u.y;
      trow[2] = u.z;
      trow[3] = u.w;
    } else {
      for (int j = 0; j < 8; ++j) tile[rr][cv + j] = (c0 + cv + j < cols) ? src[j] : uint16_t(0);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int v = t + i * 256, cc = v >> 3, rv = (v & 7) * 8;
    const int64_t dc = c0 + cc;
    if (dc >= cols) continue;
    uint16_t* out = dst + dc * total_rows + r0 + rv;
    if (vec && r0 + rv + 8 <= total_rows) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = static_cast<uint32_t>(tile[rv + 2 * j][cc]) | (static_cast<uint32_t>(tile[rv + 2 * j + 1][cc]) << 16);
      __stcs(reinterpret_cast<uint4*>(out), make_uint4(w[0], w[1], w[2], w[3]));
    } else {
      for (int j = 0; j < 8; ++j)
        if (r0 + rv + j < total_rows) out[j] = tile[rv + j][cc];
    }
  }
}

// One thread waits on an mbarrier that nothing arrives on, through the same bounded wait
// the pipelined kernels use; after timeout_ns it records kErrSelftest and returns.
__global__ void wait_selftest_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, &g_zgb_dev_error, kErrSelftest, timeout_ns);
}

unsigned int grid_for(uint64_t work_items) {
  const uint64_t want = (work_items + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(num_sms()) * 16u;
  return static_cast<unsigned int>(std::max<uint64_t>(1, std::min(want, cap)));
}

template <typename F>
cudaError_t dispatch_nr(int n, F&& f) {
  switch (n) {
    case 1: return f(std::integral_constant<int, 1>{});
    case 2: return f(std::integral_constant<int, 2>{});
    case 4: return f(std::integral_constant<int, 4>{});
    case 8: return f(std::integral_constant<int, 8>{});
    case 16: return f(std::integral_constant<int, 16>{});
    default: return f(std::integral_constant<int, 0>{});
  }
}

}  // namespace

cudaError_t launch_reduce(const GradPtrs& gp, int n, float* out, const Domain& d, float inv_n, bool vec,
                          cudaStream_t st) {
  const uint64_t total = d.seg_len * d.n_seg;
  if (total == 0) return cudaSuccess;
  if (!vec) {
    reduce_scalar_kernel<<<grid_for(total), kThreads, 0, st>>>(gp, n, out, d, inv_n);
    return cudaGetLastError();
  }
  const unsigned int grid = grid_for((d.seg_len + 3) / 4 * d.n_seg);
  return dispatch_nr(n, [&](auto nr) {
    reduce_vec_kernel<decltype(nr)::value><<<grid, kThreads, 0, st>>>(gp, n, out, d, inv_n);
    return cudaGetLastError();
  });
}

cudaError_t launch_adam(const float* g, float* master, float* m, float* v, uint16_t* param, const Domain& d,
                        const AdamScalars& sc, bool vec, cudaStream_t st) {
  const uint64_t total = d.seg_len * d.n_seg;
  if (total == 0) return cudaSuccess;
  if (vec)
    adam_vec_kernel<<<grid_for((d.seg_len + 3) / 4 * d.n_seg), kThreads, 0, st>>>(g, master, m, v, param, d, sc);
  else
    adam_scalar_kernel<<<grid_for(total), kThreads, 0, st>>>(g, master, m, v, param, d, sc);
  return cudaGetLastError();
}

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

std::once_flag g_tma_attr_once[64];
}  // namespace

cudaError_t launch_fused(const GradPtrs& gp, int n, float* master, float* m, float* v, uint16_t* param,
                         const Domain& d, const AdamScalars& sc, int variant, cudaStream_t st) {
  const uint64_t total = d.seg_len * d.n_seg;
  if (total == 0) return cudaSuccess;
  if (variant == 1) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(g_tma_attr_once[dev & 63], [&] {
      attr_err = cudaFuncSetAttribute(fused_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    const unsigned int grid = grid_for((d.seg_len + 3) / 4 * d.n_seg);
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
    const unsigned int grid = grid_for((d.seg_len + 3) / 4 * d.n_seg);
    return dispatch_nr(n, [&](auto nr) {
      fused_vec_kernel<decltype(nr)::value, float><<<grid, kThreads, 0, st>>>(gp, n, master, m, v, param, d, sc);
      return cudaGetLastError();
    });
  }
  fused_scalar_kernel<float><<<grid_for(total), kThreads, 0, st>>>(gp, n, master, m, v, param, d, sc);
  return cudaGetLastError();
}

cudaError_t launch_allgather(const MasterPtrs& mp, int n, uint64_t shard, uint16_t* full, bool vec,
                             cudaStream_t st) {
  const uint64_t total = shard * static_cast<uint64_t>(n);
  if (total == 0) return cudaSuccess;
  allgather_kernel<<<grid_for(vec ? total / 4 : total), kThreads, 0, st>>>(mp, n, shard, full, vec ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const GradPtrs& shards, int n, uint64_t shard_elems, uint16_t* full, bool vec,
                               cudaStream_t st) {
  const uint64_t total = shard_elems * static_cast<uint64_t>(n);
  if (total == 0) return cudaSuccess;
  gather_rows_kernel<<<grid_for(vec ? total / 8 : total), kThreads, 0, st>>>(shards, n, shard_elems, full,
                                                                             vec ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_transpose_cat(const GradPtrs& srcs, int n, int64_t rows, int64_t cols, uint16_t* dst,
                                 cudaStream_t st) {
  const int64_t total_rows = rows * n;
  if (total_rows == 0 || cols == 0) return cudaSuccess;
  bool vec = cols % 8 == 0 && total_rows % 8 == 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
  for (int q = 0; q < n; ++q) vec = vec && (reinterpret_cast<uintptr_t>(srcs.p[q]) & 15) == 0;
  const int64_t gy = (total_rows + kTT - 1) / kTT, gx = (cols + kTT - 1) / kTT;
  if (gy > 65535 || gx > 0x7fffffff) return cudaErrorInvalidConfiguration;
  transpose_cat_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0, st>>>(
      srcs, rows, cols, total_rows, dst, vec ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned long long timeout_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns);
  return cudaGetLastError();
}

unsigned int step_kernels_read_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_zgb_dev_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v) cudaMemcpyToSymbol(g_zgb_dev_error, &zero, sizeof(zero));
  return v;
}

}  // namespace zgb
