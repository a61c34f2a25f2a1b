// Memory-bound kernels besides the fused step (fused_step.cu): the standalone
// reduce-scatter / DDP all-reduce, Adam, the parameter all-gather, the FSDP row gather,
// the FSDP backward's transpose-and-concatenate, and the bounded-wait self-test.
//
// All are HBM-bandwidth bound. The elementwise ones run over a Domain (see internal.h) in
// 4-element units per thread-iteration, so every global access of a warp is one
// contiguous run: reduce-scatter 2N + 4 bytes per parameter, Adam 28 (+2 with the cast),
// all-gather 6, row gather 4 per weight element, transpose 4 per element.
#include <string.h>

#include <algorithm>
#include <type_traits>

#include "step_common.cuh"

namespace zgb {

ZGB_DECLARE_ERROR_WORD();

namespace {

constexpr unsigned int kErrSelftest = (3u << 8) | 1u;  // the bounded-wait self-test

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
// Vector path: each thread keeps kAgInFlight 16-byte master loads in flight (4-element
// units one grid stride apart) on a grid of kAgBlocksPerSm CTAs per SM. Measured on GB300
// (N = 2..64, 0.24-9.6 GB moved): 4 x 4 held 0.93-0.98 of the copy bandwidth, against
// 0.86-0.93 for one load per thread on the full grid; 6 or 8 in flight, or 2-3 CTAs per
// SM, lost 5-25 %.
constexpr int kAgInFlight = 4;
constexpr unsigned int kAgBlocksPerSm = 4;
__global__ void __launch_bounds__(kThreads) allgather_kernel(MasterPtrs mp, int n, uint64_t shard,
                                                             uint16_t* __restrict__ full, int vec) {
  if (vec) {  // shard % 4 == 0 and aligned: a 4-element unit never straddles two ranks
    const uint64_t upr = shard / 4, total = upr * static_cast<uint64_t>(n);
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    for (uint64_t u0 = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u0 < total; u0 += kAgInFlight * stride) {
      float4 w[kAgInFlight];
      uint64_t dst[kAgInFlight];
#pragma unroll
      for (int k = 0; k < kAgInFlight; ++k) {
        const uint64_t u = u0 + k * stride;
        if (u < total) {
          const uint64_t r = u / upr, i = (u - r * upr) * 4;
          w[k] = __ldcs(reinterpret_cast<const float4*>(mp.p[r] + i));
          dst[k] = r * shard + i;
        }
      }
#pragma unroll
      for (int k = 0; k < kAgInFlight; ++k)
        if (u0 + k * stride < total)
          __stcs(reinterpret_cast<uint2*>(full + dst[k]),
                 make_uint2(pack_bf16x2(w[k].x, w[k].y), pack_bf16x2(w[k].z, w[k].w)));
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
  if (vec) {  // shard_elems % 8 == 0 and 16-byte aligned: 16-byte units, 4 in flight per thread
    const uint64_t upr = shard_elems / 8, total = upr * static_cast<uint64_t>(n);
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    for (uint64_t u0 = blockIdx.x * (uint64_t)kThreads + threadIdx.x; u0 < total; u0 += 4 * stride) {
      uint4 x[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t u = u0 + k * stride;
        if (u < total) {
          const uint64_t r = u / upr, i = (u - r * upr) * 8;
          x[k] = __ldcs(reinterpret_cast<const uint4*>(shards.p[r] + i));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t u = u0 + k * stride;
        if (u < total) {
          const uint64_t r = u / upr, i = (u - r * upr) * 8;
          __stcs(reinterpret_cast<uint4*>(full + r * shard_elems + i), x[k]);
        }
      }
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
// tiles through shared memory. The kernel below serves unaligned shapes (element
// accesses where needed); aligned ones take transpose_cat_pipe_kernel after it.
// ------------------------------------------------------------------------------------
#ifndef ZGB_TT_R
#define ZGB_TT_R 64
#endif
#ifndef ZGB_TT_C
#define ZGB_TT_C 64
#endif
constexpr int kTR = ZGB_TT_R;  // tile rows (source rows = output columns)
constexpr int kTC = ZGB_TT_C;  // tile columns (source columns = output rows)
static_assert(kTR % 8 == 0 && kTC % 16 == 0, "tile shape");

__global__ void __launch_bounds__(256) transpose_cat_kernel(GradPtrs srcs, int64_t rows, int64_t cols,
                                                            int64_t total_rows, uint16_t* __restrict__ dst, int vec) {
  __shared__ uint16_t tile[kTR][kTC + 2];
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTC;
  const int t = threadIdx.x;
  const int64_t row_tiles = (total_rows + kTR - 1) / kTR;
  for (int64_t ty = blockIdx.y; ty < row_tiles; ty += gridDim.y) {
    const int64_t r0 = ty * kTR;
    __syncthreads();  // the previous row tile's reads of `tile` are done
    // load: kTR rows of kTC columns, 16 bytes per thread-iteration
#pragma unroll
    for (int v = t; v < kTR * kTC / 8; v += 256) {
      const int rr = v / (kTC / 8), cv = (v % (kTC / 8)) * 8;
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
    // store: each thread-iteration builds two output rows (source columns cc, cc+1) x 8
    // output columns (source rows rv..rv+7) from eight 32-bit reads of (tile[row][cc],
    // tile[row][cc+1]), split into the two rows with byte permutes
#pragma unroll
    for (int u = t; u < kTR * kTC / 16; u += 256) {
      const int cc = (u / (kTR / 8)) * 2, rv = (u % (kTR / 8)) * 8;
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = *reinterpret_cast<const uint32_t*>(&tile[rv + j][cc]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t dc = c0 + cc + h;
        if (dc >= cols) continue;
        uint16_t* out = dst + dc * total_rows + r0 + rv;
        const uint32_t sel = h ? 0x7632u : 0x5410u;  // high or low halves of two words
        if (vec && r0 + rv + 8 <= total_rows) {
          __stcs(reinterpret_cast<uint4*>(out),
                 make_uint4(__byte_perm(w[0], w[1], sel), __byte_perm(w[2], w[3], sel), __byte_perm(w[4], w[5], sel),
                            __byte_perm(w[6], w[7], sel)));
        } else {
          for (int j = 0; j < 8; ++j)
            if (r0 + rv + j < total_rows) out[j] = static_cast<uint16_t>(h ? (w[j] >> 16) : (w[j] & 0xffffu));
        }
      }
    }
  }
}

// The aligned path (16-byte rows and buffers): persistent CTAs walk the 64 x 64 tiles
// through a ring of kPipeStages shared-memory tiles filled by cp.async, so the next tiles'
// loads are in flight while the current one is read out transposed. No padding (cp.async
// needs 16-byte-aligned destinations): 16-byte chunk c of tile row r sits at chunk
// c ^ ((r >> 3) & 7), which spreads one warp's column reads (eight rows 8 apart, four
// column pairs) over 32 banks. Measured on GB300 against the one-tile-per-CTA kernel above:
// W_up's shards 58 -> 44 us, X^T of 8 x 2048 tokens 66 -> 50 us, dY^T 215 -> 175 us
// (0.60-0.64 -> 0.79-0.80 of the copy bandwidth); 2 stages or 4 CTAs per SM were slower.
constexpr int kPipeStages = 3;
constexpr unsigned int kPipeBlocksPerSm = 8;

__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
  // src_bytes = 0 fills the 16 bytes with zeros and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One transpose-and-concatenate problem of the pipelined kernel. Requires cols % 8 == 0,
// total_rows % 8 == 0 and 16-byte-aligned sources and destination.
struct TransposeJob {
  GradPtrs srcs;
  int64_t rows, cols, total_rows, col_tiles, ntiles;
  uint16_t* dst;
};
// Up to two independent problems in one launch: tiles [0, j[0].ntiles) belong to the
// first, the rest to the second (launch_transpose_cat passes one, the second empty).
struct TransposeJobs {
  TransposeJob j[2];
};

__global__ void __launch_bounds__(256) transpose_cat_pipe_kernel(const __grid_constant__ TransposeJobs jobs) {
  __shared__ __align__(128) uint16_t ring[kPipeStages][64 * 64];
  const int t = threadIdx.x;
  const int64_t nt0 = jobs.j[0].ntiles, ntiles = nt0 + jobs.j[1].ntiles;
  // issue the copies of tile idx into ring slot `slot` (one commit group per call, empty
  // when idx is past the end, so every thread's group count stays in step)
  auto issue = [&](int64_t idx, int slot) {
    if (idx < ntiles) {
      const TransposeJob& J = jobs.j[idx < nt0 ? 0 : 1];
      const int64_t li = idx < nt0 ? idx : idx - nt0;
      const int64_t c0 = (li % J.col_tiles) * 64, r0 = (li / J.col_tiles) * 64;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int v = t + 256 * k, rr = v >> 3, ch = v & 7;  // 64 rows x 8 chunks of 16 B
        const int64_t gr = r0 + rr, gc = c0 + ch * 8;
        const bool in = gr < J.total_rows && gc < J.cols;
        const uint16_t* src = J.srcs.p[0];
        if (in) {
          const int64_t q = gr / J.rows, lr = gr - q * J.rows;
          src = J.srcs.p[q] + lr * J.cols + gc;
        }
        cp_async16(smem_u32(&ring[slot][rr * 64 + ((ch ^ ((rr >> 3) & 7)) * 8)]), src, in ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  int64_t idx = blockIdx.x;
#pragma unroll
  for (int s = 0; s < kPipeStages - 1; ++s) issue(idx + static_cast<int64_t>(s) * gridDim.x, s);
  for (int i = 0; idx < ntiles; ++i, idx += gridDim.x) {
    issue(idx + static_cast<int64_t>(kPipeStages - 1) * gridDim.x, (i + kPipeStages - 1) % kPipeStages);
    cp_async_wait<kPipeStages - 1>();  // this thread's copies of tile idx have landed
    __syncthreads();                    // and everyone else's
    const uint16_t* T = ring[i % kPipeStages];
    const TransposeJob& J = jobs.j[idx < nt0 ? 0 : 1];
    const int64_t li = idx < nt0 ? idx : idx - nt0;
    const int64_t c0 = (li % J.col_tiles) * 64, r0 = (li / J.col_tiles) * 64;
    // two output rows (source columns cc, cc + 1) x 8 output columns (source rows rv..rv+7)
    const int cc = (t >> 3) * 2, rv = (t & 7) * 8;
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = rv + j;
      w[j] = *reinterpret_cast<const uint32_t*>(&T[r * 64 + (((cc >> 3) ^ ((r >> 3) & 7)) * 8) + (cc & 7)]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t dc = c0 + cc + h;
      if (dc < J.cols && r0 + rv < J.total_rows) {  // total_rows % 8 == 0: all 8 in range
        const uint32_t sel = h ? 0x7632u : 0x5410u;
        __stcs(reinterpret_cast<uint4*>(J.dst + dc * J.total_rows + r0 + rv),
               make_uint4(__byte_perm(w[0], w[1], sel), __byte_perm(w[2], w[3], sel), __byte_perm(w[4], w[5], sel),
                          __byte_perm(w[6], w[7], sel)));
      }
    }
    __syncthreads();  // slot i % kPipeStages is refilled by the next iteration's issue
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------
// SiLU-gate backward of the MLP unit H = silu(G) * U: with s = 1 / (1 + exp(-g)),
//   silu(g) = g s,   silu'(g) = s (1 + g (1 - s)),
//   dU = dH silu(G),  dG = dH U silu'(G),
// from the bf16 activations the forward saved (G | U in one [rows, 2 d_ff] buffer) and the
// bf16 dH, in fp32 with one IEEE rounding per operation in the order written, stored as
// bf16 dG | dU [rows, 2 d_ff]. 10 bytes of HBM traffic per element.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void silu_gate_grad(float dh, float g, float u, float& dg, float& du) {
  const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)));
  const float silu = __fmul_rn(g, s);
  const float dsilu = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, s))));
  du = __fmul_rn(dh, silu);
  dg = __fmul_rn(__fmul_rn(dh, u), dsilu);
}

// vec: 8 elements per thread-iteration with 16-byte accesses (d_ff % 8 == 0, aligned
// buffers); otherwise one element
__global__ void __launch_bounds__(kThreads) silu_gate_backward_kernel(const uint16_t* __restrict__ dh,
                                                                      const uint16_t* __restrict__ gu,
                                                                      uint16_t* __restrict__ dgu, int64_t rows,
                                                                      int64_t d_ff, int vec) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (vec) {
    const int64_t per_row = d_ff / 8, units = rows * per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < units; i += stride) {
      const int64_t r = i / per_row, c = (i - r * per_row) * 8;
      const uint4 h = __ldcs(reinterpret_cast<const uint4*>(dh + r * d_ff + c));
      const uint4 g = __ldcs(reinterpret_cast<const uint4*>(gu + r * 2 * d_ff + c));
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(gu + r * 2 * d_ff + d_ff + c));
      const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
      uint32_t og[4], ou[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float g0, u0, g1, u1;
        silu_gate_grad(bf16_lo(hw[j]), bf16_lo(gw[j]), bf16_lo(uw[j]), g0, u0);
        silu_gate_grad(bf16_hi(hw[j]), bf16_hi(gw[j]), bf16_hi(uw[j]), g1, u1);
        og[j] = pack_bf16x2(g0, g1);
        ou[j] = pack_bf16x2(u0, u1);
      }
      __stcs(reinterpret_cast<uint4*>(dgu + r * 2 * d_ff + c), make_uint4(og[0], og[1], og[2], og[3]));
      __stcs(reinterpret_cast<uint4*>(dgu + r * 2 * d_ff + d_ff + c), make_uint4(ou[0], ou[1], ou[2], ou[3]));
    }
    return;
  }
  const int64_t total = rows * d_ff;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t r = i / d_ff, c = i - r * d_ff;
    float dg, du;
    silu_gate_grad(bf16_bits_to_f32(dh[i]), bf16_bits_to_f32(gu[r * 2 * d_ff + c]),
                   bf16_bits_to_f32(gu[r * 2 * d_ff + d_ff + c]), dg, du);
    dgu[r * 2 * d_ff + c] = f32_to_bf16_bits(dg);
    dgu[r * 2 * d_ff + d_ff + c] = f32_to_bf16_bits(du);
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

// Blocks per SM of the vector reduce and Adam grids on long launches, measured on GB300. A thread of the
// reduce keeps 8 B of gradient loads per rank in flight (all N ranks for N <= 16, eight
// at a time above): from 64 B (N >= 8) four blocks per SM held 0.96-1.00
// of the copy bandwidth where the full grid held 0.89-0.96; at N = 4 (32 B) six did
// best; with less in flight the full grid is needed to cover the latency. Adam keeps
// 64 B in flight per thread: four per SM.
inline unsigned int reduce_blocks_per_sm(int n) { return n >= 8 ? 4u : n >= 4 ? 6u : 16u; }
constexpr unsigned int kAdamBlocksPerSm = 4;

}  // namespace

cudaError_t launch_reduce(const GradPtrs& gp, int n, float* out, const Domain& d, float inv_n, bool vec,
                          cudaStream_t st) {
  const uint64_t total = d.seg_len * d.n_seg;
  if (total == 0) return cudaSuccess;
  if (!vec) {
    reduce_scalar_kernel<<<grid_for(total), kThreads, 0, st>>>(gp, n, out, d, inv_n);
    return cudaGetLastError();
  }
  const unsigned int grid = grid_streaming((d.seg_len + 3) / 4 * d.n_seg, reduce_blocks_per_sm(n));
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
    adam_vec_kernel<<<grid_streaming((d.seg_len + 3) / 4 * d.n_seg, kAdamBlocksPerSm), kThreads, 0, st>>>(
        g, master, m, v, param, d, sc);
  else
    adam_scalar_kernel<<<grid_for(total), kThreads, 0, st>>>(g, master, m, v, param, d, sc);
  return cudaGetLastError();
}

cudaError_t launch_allgather(const MasterPtrs& mp, int n, uint64_t shard, uint16_t* full, bool vec,
                             cudaStream_t st) {
  const uint64_t total = shard * static_cast<uint64_t>(n);
  if (total == 0) return cudaSuccess;
  allgather_kernel<<<vec ? grid_for(total / 4, kAgBlocksPerSm) : grid_for(total), kThreads, 0, st>>>(mp, n, shard, full,
                                                                                               vec ? 1 : 0);
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

namespace {

// the pipelined kernel's job for one problem, or false when its shapes or buffers are not
// aligned for it
bool pipe_job(const GradPtrs& srcs, int n, int64_t rows, int64_t cols, uint16_t* dst, TransposeJob* j) {
  const int64_t total_rows = rows * n;
  bool vec = cols % 8 == 0 && total_rows % 8 == 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
  for (int q = 0; q < n; ++q) vec = vec && (reinterpret_cast<uintptr_t>(srcs.p[q]) & 15) == 0;
  if (!vec) return false;
  j->srcs = srcs;
  j->rows = rows;
  j->cols = cols;
  j->total_rows = total_rows;
  j->col_tiles = (cols + 63) / 64;
  j->ntiles = j->col_tiles * ((total_rows + 63) / 64);
  j->dst = dst;
  return true;
}

cudaError_t launch_pipe(const TransposeJobs& jobs, cudaStream_t st) {
  const int64_t ntiles = jobs.j[0].ntiles + jobs.j[1].ntiles;
  if (ntiles == 0) return cudaSuccess;
  const unsigned int grid =
      static_cast<unsigned int>(std::min<int64_t>(ntiles, static_cast<int64_t>(num_sms()) * kPipeBlocksPerSm));
  transpose_cat_pipe_kernel<<<grid, 256, 0, st>>>(jobs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_transpose_cat(const GradPtrs& srcs, int n, int64_t rows, int64_t cols, uint16_t* dst,
                                 cudaStream_t st) {
  const int64_t total_rows = rows * n;
  if (total_rows == 0 || cols == 0) return cudaSuccess;
  TransposeJobs jobs;
  memset(&jobs, 0, sizeof(jobs));
  if (pipe_job(srcs, n, rows, cols, dst, &jobs.j[0])) return launch_pipe(jobs, st);
  const int64_t gy = std::min<int64_t>((total_rows + kTR - 1) / kTR, 65535), gx = (cols + kTC - 1) / kTC;
  if (gx > 0x7fffffff) return cudaErrorInvalidConfiguration;
  transpose_cat_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0, st>>>(
      srcs, rows, cols, total_rows, dst, 0);
  return cudaGetLastError();
}

cudaError_t launch_silu_gate_backward(const uint16_t* dh, const uint16_t* gu, uint16_t* dgu, int64_t rows, int64_t d_ff,
                                      cudaStream_t st) {
  if (rows <= 0 || d_ff <= 0) return cudaSuccess;
  const bool vec = d_ff % 8 == 0 && ((reinterpret_cast<uintptr_t>(dh) | reinterpret_cast<uintptr_t>(gu) |
                                       reinterpret_cast<uintptr_t>(dgu)) & 15) == 0;
  const uint64_t units = static_cast<uint64_t>(rows) * static_cast<uint64_t>(vec ? d_ff / 8 : d_ff);
  silu_gate_backward_kernel<<<grid_streaming(units, 4), kThreads, 0, st>>>(dh, gu, dgu, rows, d_ff, vec ? 1 : 0);
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
