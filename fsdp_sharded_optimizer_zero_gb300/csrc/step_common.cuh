// Element-level helpers shared by the optimizer-step kernels (fused_step.cu,
// step_kernels.cu): the rank-order fp32 reduction of N gradient contributions (bf16 or
// fp32), the per-element fused update, 4-element vector units, and launch sizing.
#pragma once

#include <algorithm>
#include <type_traits>

#include "device_common.cuh"

namespace zgb {
namespace {

constexpr int kThreads = 256;

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

// grid of a grid-stride kernel: one thread per work item, at most blocks_per_sm blocks of
// kThreads threads per SM
inline unsigned int grid_for(uint64_t work_items, unsigned int blocks_per_sm = 16) {
  const uint64_t want = (work_items + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(num_sms()) * blocks_per_sm;
  return static_cast<unsigned int>(std::max<uint64_t>(1, std::min(want, cap)));
}

// Grid of a streaming kernel with a tuned, smaller number of blocks per SM for long
// launches. Measured on GB300 (fused step, N = 2, 8, 16, launches of 2^18..2^25 elements
// back to back): the smaller grid wins 1-3 % once every thread strides over at least
// kLongLaunchIters units, while shorter launches (the per-bucket launches of a DDP-style
// step) ramp up faster on the full grid and lose 2-4 % on the small one.
constexpr uint64_t kLongLaunchIters = 32;
inline unsigned int grid_streaming(uint64_t units, unsigned int tuned_blocks_per_sm) {
  const uint64_t threads = static_cast<uint64_t>(num_sms()) * tuned_blocks_per_sm * kThreads;
  return grid_for(units, units >= kLongLaunchIters * threads ? tuned_blocks_per_sm : 16u);
}

// Rank counts 1..16 get their own instantiation (every rank's load issued from a constant
// pointer slot, all in flight together); larger N takes the generic groups of 8. Measured on
// GB300 (fused step, 124M parameters, one launch): the generic path held 0.87 / 0.91 / 0.93
// / 0.95 / 0.94 of the copy peak at N = 3 / 5 / 6 / 7 / 12, the dedicated kernels 0.97-1.00,
// bit for bit the same; from N = 24 up the generic path holds 1.0 already.
template <typename F>
inline cudaError_t dispatch_nr(int n, F&& f) {
  switch (n) {
    case 1: return f(std::integral_constant<int, 1>{});
    case 2: return f(std::integral_constant<int, 2>{});
    case 3: return f(std::integral_constant<int, 3>{});
    case 4: return f(std::integral_constant<int, 4>{});
    case 5: return f(std::integral_constant<int, 5>{});
    case 6: return f(std::integral_constant<int, 6>{});
    case 7: return f(std::integral_constant<int, 7>{});
    case 8: return f(std::integral_constant<int, 8>{});
    case 9: return f(std::integral_constant<int, 9>{});
    case 10: return f(std::integral_constant<int, 10>{});
    case 11: return f(std::integral_constant<int, 11>{});
    case 12: return f(std::integral_constant<int, 12>{});
    case 13: return f(std::integral_constant<int, 13>{});
    case 14: return f(std::integral_constant<int, 14>{});
    case 15: return f(std::integral_constant<int, 15>{});
    case 16: return f(std::integral_constant<int, 16>{});
    default: return f(std::integral_constant<int, 0>{});
  }
}


}  // namespace
}  // namespace zgb
