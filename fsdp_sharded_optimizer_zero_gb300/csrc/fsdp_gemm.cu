// FSDP unit GEMM on the 5th-generation tensor cores: Y[M, R] = A[M, K] * W^T, where W
// [R, K] (the [out, in] layout of a linear layer) is held as N dim-0 row shards.
//
// The all-gather of W is fused into the operand loads: each W tile (or each CTA's half of
// one) lies inside one shard, so the TMA producer picks that shard's tensor map and loads
// the tile straight from the shard; the full W is never assembled. (With a caller scratch
// buffer the host instead gathers W first and passes one map.)
//
// Two kernels compute the same sums in the same order (bit-identical results):
//   fsdp_gemm_pair_kernel  a cluster of two CTAs per 256-row tile, tcgen05.mma.cta_group::2
//                          (M = 256, N = 256) over both CTAs' shared memory: each CTA loads
//                          half of A and half of B, a third fewer operand bytes per flop.
//                          The default, for every operand layout.
//   fsdp_gemm_kernel       one CTA per 128 x 256 tile, tcgen05.mma.cta_group::1
//                          (zero_set_gemm_kernel(1)).
// Both are compiled per operand layout (template parameter LAYOUT: A and / or B stored
// MN-major), so the producer and MMA threads carry no per-step layout logic.
// One-CTA kernel structure (one CTA per SM, persistent over its output tiles):
//   warp 0        TMA producer: A tile 128x64 and W tile 256x64 (bf16, 128-byte swizzle)
//                 per 64-wide K block into a 4-stage shared-memory ring;
//   warp 1        allocates 512 TMEM columns, then one lane issues tcgen05.mma
//                 (M=128, N=256, K=16; fp32 accumulators in TMEM, two 256-column buffers)
//                 and tcgen05.commit frees each stage and publishes each finished tile;
//   warps 2-5     epilogue (epilogue_tile, shared with the pair kernel): tcgen05.ld 32
//                 columns at a time into registers, each warp's 32 x 32 fp32 chunks staged
//                 in shared memory (128-byte swizzle) and written by TMA stores (64-column
//                 bf16 chunks when only a bf16 Y is asked for), then the accumulator buffer
//                 is released, so the epilogue of tile i overlaps the main loop of tile i+1.
// Other modes of both kernels: gate-up (two B operands, one N = 256 MMA per K step,
// SiLU-gate epilogue writing bf16 H), A split by rows into pieces with matching Y pieces
// (the backward's dX for all ranks in one launch), MN-major A / B operands split along
// K (the backward reading W and dY in place; see GemmParams), and the fused optimizer
// (template parameter ADAM): the weight-gradient GEMM's epilogue runs each rank's Adam on
// its rows of the reduce-scattered result (adam_chunk_rows) instead of storing it.
// Every mbarrier wait is bounded (error word + CTA abort flag, no trap); after an abort
// the producer drains its copies and the MMA warp its MMAs before TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace zgb {

ZGB_DECLARE_ERROR_WORD();

namespace {

#ifndef ZGB_GEMM_BN
#define ZGB_GEMM_BN 256
#endif
#ifndef ZGB_GEMM_STAGES
#define ZGB_GEMM_STAGES 4
#endif
constexpr int BM = 128, BN = ZGB_GEMM_BN, BK = 64, STAGES = ZGB_GEMM_STAGES;
constexpr int kMaxShards = kGemmMaxPieces;
constexpr int kThreads = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;

// per mode: output tile columns, bytes of one B tile, bytes of one stage (A + one or two B
// tiles), TMEM columns of one accumulator buffer (two buffers are allocated)
template <bool GATE_UP> struct Mode {
  static constexpr int TN = GATE_UP ? 128 : BN;
  static constexpr uint32_t BT_BYTES = TN * BK * 2;
  static constexpr uint32_t STAGE = A_BYTES + (GATE_UP ? 2u : 1u) * BT_BYTES;
  static constexpr uint32_t ACC = GATE_UP ? 2 * TN : TN;
  static constexpr uint32_t TMEM_COLS = 2 * ACC <= 32 ? 32 : (2 * ACC <= 64 ? 64 : (2 * ACC <= 128 ? 128 : (2 * ACC <= 256 ? 256 : 512)));
  // plain mode: each epilogue warp stages 32 x 32 fp32 output chunks in two 4 KiB buffers
  // for the TMA store (4 warps x 2 x 4 KiB)
  static constexpr uint32_t EPI = GATE_UP ? 0u : 4u * 2u * 4096u;
  static constexpr uint32_t SMEM = STAGES * STAGE + EPI + 1024;  // + alignment slack
};

constexpr unsigned int kErrEmpty = (2u << 8) | 1u;  // producer waiting for a free stage
constexpr unsigned int kErrFull = (2u << 8) | 2u;   // MMA waiting for a loaded stage
constexpr unsigned int kErrAccE = (2u << 8) | 3u;   // MMA waiting for a drained accumulator
constexpr unsigned int kErrAccF = (2u << 8) | 4u;   // epilogue waiting for a finished tile
constexpr unsigned int kErrDrain = (2u << 8) | 5u;  // draining after an abort

// Operand layouts. K-major (the default): A is [M, K] and B is [R, K] row-major, A split
// by rows into a_shards pieces of a_shard_rows rows (Y split the same way), B into
// n_shards row shards of shard_rows rows. MN-major (a_mn / b_mn): the operand is stored
// as [K, M] (A) or [K, R] (B) row-major with M (R) a multiple of 64, split along K into
// pieces of a_shard_rows / shard_rows K rows (multiples of BK); the MMA reads it
// transposed, so A^T or B^T never has to be materialised. Its tensor map is 3-D, {64
// columns, K rows, column chunks of 64} with a 128-byte chunk stride, so ONE box of
// 64 x BK x (BM or TN)/64 lands a whole stage operand as 64-column chunks of BK rows x
// 128 B, 8 KiB apart: the layout the MN-major descriptor reads. (One 2-D box per chunk
// took 5-6 TMA operations per stage and left the tensor pipe waiting: 15-46 % slower.)
struct GemmParams {
  CUtensorMap a[kMaxShards];     // A piece s: K-major [a_shard_rows, K] box 64 x 128; MN-major [a_shard_rows, M] box 64 x 64
  CUtensorMap w[kMaxShards];     // B piece s: K-major [shard_rows, K] box 64 x (256, or 128 in gate-up mode); MN-major [shard_rows, R] box 64 x 64
  CUtensorMap w2[kMaxShards];    // gate-up mode: the up projection's shards (w holds the gate's)
  float* y;                      // [M, R] fp32
  uint16_t* yb;                  // [M, R] bf16 or null (gate-up mode: H = silu(gate) * up)
  uint16_t* gu;                  // gate-up mode, nullable: [M, 2R] bf16, the gate and up projections G | U
  CUtensorMap ymap[kMaxShards];  // Y row piece s [y_shard_rows, R] fp32, box 32 x 32, 128B swizzle (y_tma)
  float alpha;                   // output scale (1: none)
  int m, r, k, shard_rows, n_shards;
  int a_shard_rows, a_shards;    // pieces of A (rows for K-major, K rows for MN-major)
  int y_shard_rows;              // Y split by rows into pieces of y_shard_rows rows
  int a_mn, b_mn;                // operand stored MN-major
  int y_tma;                     // write Y through shared memory and TMA stores
  CUtensorMap ybmap;             // bf16-only output: Y_bf16 [M, R], box 64 x 32, 128B swizzle (yb_tma)
  int yb_tma;                    // no fp32 Y: write bf16 Y through shared memory and TMA stores
  AdamFuse adam;                 // plain mode with the fused optimizer: the state the output indexes
};
constexpr uint32_t kMnChunk = 64 * BK * 2;  // one 64-column chunk of an MN-major stage operand: 8 KiB

// Output tile order of the persistent walk: bands of GROUP_M row blocks; inside a band the
// walk goes down the rows of one column of tiles, then to the next column. The 152 tiles
// in flight then touch ~24 A tiles and ~6 W tile columns instead of every A tile, which
// keeps the operands L2-resident next to the streaming fp32 output (Mistral MLP shapes:
// W_up 1508 -> 1695 TFLOP/s, W_down 1567 -> 1654 against whole-column order; 16, 32 and
// 48 measured no better). GROUP_M = 0 walks whole columns.
#ifndef ZGB_GEMM_GROUP_M
#define ZGB_GEMM_GROUP_M 24
#endif
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& mb, int& nb) {
  const int g = ZGB_GEMM_GROUP_M > 0 && ZGB_GEMM_GROUP_M < num_m ? ZGB_GEMM_GROUP_M : num_m;
  const int band = tile / (g * num_n), in_band = tile - band * g * num_n;
  const int rows = min(g, num_m - band * g);
  mb = band * g + in_band % rows;
  nb = in_band / rows;
}

// Warp-uniform bounded wait of the epilogue warps for a finished tile: lane 0 polls, the
// whole warp gets the result. The wait spans a tile's whole main loop, so between polls
// lane 0 sleeps (128 ns, doubling up to ZGB_EPI_POLL_NS): four warps spinning on the
// barrier took issue slots and power from the producer and MMA warps (Mistral backward
// GEMMs 2.5-3 % faster with a 2 us poll). 0 = poll without sleeping.
#ifndef ZGB_EPI_POLL_NS
#define ZGB_EPI_POLL_NS 2048
#endif
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int code) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) {
    if (ZGB_EPI_POLL_NS == 0) {
      ok = mbar_wait_bounded(bar, parity, abort, &g_zgb_dev_error, code) ? 1 : 0;
    } else if (mbar_try_wait(bar, parity)) {
      ok = 1;
    } else {
      const unsigned long long t0 = globaltimer_ns();
      for (unsigned int ns = 128;;) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity)) {
          ok = 1;
          break;
        }
        if (*abort) break;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
          atomicCAS(&g_zgb_dev_error, 0u, code);
          *abort = 1;
          break;
        }
        if (ns < ZGB_EPI_POLL_NS) ns *= 2;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// direct per-thread stores of one row's 32-column chunk (fp32 unless skipped, bf16 if asked)
__device__ __forceinline__ void store_row_chunk(const GemmParams& p, int row, int col0, const uint32_t (&r)[32],
                                                bool write_f32) {
  float* yrow = p.y + static_cast<size_t>(row) * p.r;
  const bool full = col0 + 32 <= p.r;
  if (!write_f32) {
  } else if (full && (p.r & 3) == 0) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      __stcs(reinterpret_cast<float4*>(yrow + col0 + j),
             make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                         __uint_as_float(r[j + 3])));
  } else {
    for (int j = 0; j < 32; ++j)
      if (col0 + j < p.r) yrow[col0 + j] = __uint_as_float(r[j]);
  }
  if (p.yb) {
    uint16_t* brow = p.yb + static_cast<size_t>(row) * p.r;
    if (full && (p.r & 7) == 0) {
#pragma unroll
      for (int j = 0; j < 32; j += 8)
        __stcs(reinterpret_cast<uint4*>(brow + col0 + j),
               make_uint4(pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                          pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                          pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5])),
                          pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]))));
    } else {
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.r) brow[col0 + j] = f32_to_bf16_bits(__uint_as_float(r[j]));
    }
  }
}

// Fused optimizer. Measured on GB300 (the ZeRO-3 steps): per-lane row loads of the state
// ran 6-14 % slower than the walk below, whatever their order; with the walk, 32 rows in
// flight on the one-CTA kernel's 4 epilogue warps and 8 to 16 on the pair kernel's 8 are
// best (fewer leave too few loads in flight, more spill); L2 prefetches two chunks ahead,
// -3 to +1 %. On the pair kernel the epilogue runs about as long as the main loop beside
// it, and its parts weigh a few per cent of the step each: the update's arithmetic (the
// correctly rounded divisions and square root about half of that), the state's DRAM
// traffic, and the state's stores.
//
// fused optimizer on one 32 x 32 chunk of the fp32 result, staged in shared memory (buf,
// 128-byte rows, 16-byte piece j of row i at slot j ^ (i % 8)): result (i, c) is the
// reduced gradient of parameter (row0 + i - split) * R + col0 + c of the weight set the
// chunk's rows belong to (a chunk's 32 rows never straddle the split: it is a multiple of
// 128). The warp walks the chunk's rows with one column per lane, so every state access
// is one contiguous 128-byte line; ROWS rows' loads are in flight before their arithmetic.
// adam_elem: the same operations as the Adam kernels (same bits).
constexpr int kAdamRows = 32;  // rows of a staged chunk whose state loads are in flight together (one-CTA kernel)
// L2 prefetch of the optimizer state the chunk at columns col0 .. col0 + 31 of rows
// row0 .. row0 + 31 will read: lane i takes row row0 + i, one 128-byte line per array
__device__ __forceinline__ void adam_prefetch_chunk(const GemmParams& p, int row0, int col0, int lane) {
  const int row = row0 + lane;
  if (col0 >= p.r || row >= p.m) return;
  const int set = row0 >= p.adam.split ? 1 : 0;
  const size_t idx = static_cast<size_t>(row - (set ? p.adam.split : 0)) * p.r + col0;
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p.adam.master[set] + idx));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p.adam.m[set] + idx));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p.adam.v[set] + idx));
}
template <int ROWS = kAdamRows>
__device__ __forceinline__ void adam_chunk_rows(const GemmParams& p, const uint8_t* buf, int row0, int col0,
                                                int lane) {
  const int col = col0 + lane;
  if (col >= p.r || row0 >= p.m) return;
  const int set = row0 >= p.adam.split ? 1 : 0;
  const size_t first = static_cast<size_t>(row0 - (set ? p.adam.split : 0)) * p.r + col;
  float* W = p.adam.master[set] + first;
  float* M = p.adam.m[set] + first;
  float* V = p.adam.v[set] + first;
  uint16_t* P = p.adam.w[set] + first;
  const size_t R = static_cast<size_t>(p.r);
  const int rows = min(32, p.m - row0);
  const uint32_t piece = static_cast<uint32_t>(lane) >> 2, word = static_cast<uint32_t>(lane) & 3u;
#pragma unroll 1
  for (int i0 = 0; i0 < rows; i0 += ROWS) {
    float w[ROWS], m[ROWS], v[ROWS];
#pragma unroll
    for (int k = 0; k < ROWS; ++k) {
      const int i = i0 + k;
      if (i < rows) {
        w[k] = __ldcs(W + i * R);
        m[k] = __ldcs(M + i * R);
        v[k] = __ldcs(V + i * R);
      }
    }
#pragma unroll
    for (int k = 0; k < ROWS; ++k) {
      const int i = i0 + k;
      if (i < rows) {
        // the gradient from the staged chunk when it is used: no register held across the loads
        const float g = *reinterpret_cast<const float*>(buf + i * 128 +
                                                        ((piece ^ (static_cast<uint32_t>(i) & 7u)) * 16) + word * 4);
        adam_elem(g, w[k], m[k], v[k], p.adam.sc);
        __stcs(W + i * R, w[k]);
        __stcs(M + i * R, m[k]);
        __stcs(V + i * R, v[k]);
        P[i * R] = f32_to_bf16_bits(w[k]);
      }
    }
  }
}

// gate-up epilogue: h = silu(g) * u = g / (1 + exp(-g)) * u in fp32, stored as bf16 (RNE)
__device__ __forceinline__ void store_gate_up_chunk(const GemmParams& p, int row, int col0, const uint32_t (&g)[32],
                                                    const uint32_t (&u)[32]) {
  float h[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float gj = __uint_as_float(g[j]);
    const float silu = __fdiv_rn(gj, __fadd_rn(1.0f, expf(-gj)));
    h[j] = __fmul_rn(silu, __uint_as_float(u[j]));
  }
  uint16_t* brow = p.yb + static_cast<size_t>(row) * p.r;
  if (col0 + 32 <= p.r && (p.r & 7) == 0) {
#pragma unroll
    for (int j = 0; j < 32; j += 8)
      __stcs(reinterpret_cast<uint4*>(brow + col0 + j),
             make_uint4(pack_bf16x2(h[j], h[j + 1]), pack_bf16x2(h[j + 2], h[j + 3]), pack_bf16x2(h[j + 4], h[j + 5]),
                        pack_bf16x2(h[j + 6], h[j + 7])));
  } else {
    for (int j = 0; j < 32; ++j)
      if (col0 + j < p.r) brow[col0 + j] = f32_to_bf16_bits(h[j]);
  }
  if (p.gu) {  // the saved activations of the backward: bf16 G at column c, U at column R + c
    uint16_t* grow = p.gu + static_cast<size_t>(row) * 2 * p.r;
    if (col0 + 32 <= p.r && (p.r & 7) == 0) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        __stcs(reinterpret_cast<uint4*>(grow + col0 + j),
               make_uint4(pack_bf16x2(__uint_as_float(g[j]), __uint_as_float(g[j + 1])),
                          pack_bf16x2(__uint_as_float(g[j + 2]), __uint_as_float(g[j + 3])),
                          pack_bf16x2(__uint_as_float(g[j + 4]), __uint_as_float(g[j + 5])),
                          pack_bf16x2(__uint_as_float(g[j + 6]), __uint_as_float(g[j + 7]))));
        __stcs(reinterpret_cast<uint4*>(grow + p.r + col0 + j),
               make_uint4(pack_bf16x2(__uint_as_float(u[j]), __uint_as_float(u[j + 1])),
                          pack_bf16x2(__uint_as_float(u[j + 2]), __uint_as_float(u[j + 3])),
                          pack_bf16x2(__uint_as_float(u[j + 4]), __uint_as_float(u[j + 5])),
                          pack_bf16x2(__uint_as_float(u[j + 6]), __uint_as_float(u[j + 7]))));
      }
    } else {
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.r) {
          grow[col0 + j] = f32_to_bf16_bits(__uint_as_float(g[j]));
          grow[p.r + col0 + j] = f32_to_bf16_bits(__uint_as_float(u[j]));
        }
    }
  }
}

// Epilogue of one output tile, run by the epilogue warps after the tile's accumulator is
// complete: a warp of quarter q reads TMEM lanes [32q, 32q + 32) (tile rows 32q + lane) at
// taddr, stages its chunks in its 8 KiB of shared memory at epi for TMA stores, and writes
// rows m0 + 32q + lane, columns n0 .. n0 + TN of Y (row piece ash, local row ml) or of H.
// With PARTS warps per quarter (the fused optimizer on the CTA pair), warp `part` of the
// quarter takes the 32-column chunks part, part + PARTS, ...
template <bool GATE_UP, bool ADAM = false, int PARTS = 1>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t taddr, uint8_t* epi, uint32_t& epi_chunk,
                                              int m0, int n0, int ash, int ml, int q, int lane, int part = 0) {
  static_assert(PARTS == 1 || (ADAM && !GATE_UP), "columns are split between warps for the fused optimizer only");
  constexpr int TN = Mode<GATE_UP>::TN;
#ifndef ZGB_PAIR_ADAM_ROWS
#define ZGB_PAIR_ADAM_ROWS 16
#endif
  constexpr int kAdamInFlight = PARTS == 1 ? kAdamRows : ZGB_PAIR_ADAM_ROWS;  // registers: 320 threads with PARTS = 2
  const int row = m0 + q * 32 + lane;
  if constexpr (GATE_UP) {
#pragma unroll 1
    for (int c = 0; c < TN; c += 32) {
      uint32_t g[32], u[32];
      tmem_ld_32cols(taddr + c, g);
      tmem_ld_32cols(taddr + TN + c, u);
      if (row < p.m && n0 + c < p.r) store_gate_up_chunk(p, row, n0 + c, g, u);
    }
  } else if (p.yb_tma) {
    // bf16-only output: 64 columns per chunk (two 32-column TMEM loads), each row packed
    // to 128 B of bf16 and placed with the 128-byte swizzle as in the fp32 path below
#pragma unroll 1
    for (int c = 0; c < TN; c += 64) {
      uint32_t r0[32], r1[32];
      tmem_ld_32cols(taddr + c, r0);
      tmem_ld_32cols(taddr + c + 32, r1);
      if (n0 + c >= p.r) continue;  // warp-uniform
      uint32_t w[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float a0 = __uint_as_float(r0[2 * j]), a1 = __uint_as_float(r0[2 * j + 1]);
        float b0 = __uint_as_float(r1[2 * j]), b1 = __uint_as_float(r1[2 * j + 1]);
        if (p.alpha != 1.0f) {
          a0 = __fmul_rn(a0, p.alpha);
          a1 = __fmul_rn(a1, p.alpha);
          b0 = __fmul_rn(b0, p.alpha);
          b1 = __fmul_rn(b1, p.alpha);
        }
        w[j] = pack_bf16x2(a0, a1);
        w[16 + j] = pack_bf16x2(b0, b1);
      }
      uint8_t* buf = epi + (epi_chunk & 1u) * 4096u;
      if (lane == 0 && epi_chunk >= 2) bulk_wait_group_read<1>();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) * 16)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.ybmap, n0 + c, m0 + q * 32, smem_u32(buf));
        bulk_commit_group();
      }
      ++epi_chunk;
    }
  } else {
    if constexpr (ADAM) {  // the first two chunks' state on its way to L2
      adam_prefetch_chunk(p, m0 + q * 32, n0 + 32 * part, lane);
      adam_prefetch_chunk(p, m0 + q * 32, n0 + 32 * (part + PARTS), lane);
    }
#pragma unroll 1
    for (int c = 32 * part; c < TN; c += 32 * PARTS) {
      uint32_t r[32];
      tmem_ld_32cols(taddr + c, r);
      if (n0 + c >= p.r) continue;  // warp-uniform
      if constexpr (ADAM) {
        if (c + 64 * PARTS < TN) adam_prefetch_chunk(p, m0 + q * 32, n0 + c + 64 * PARTS, lane);
      }
      if (p.alpha != 1.0f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fmul_rn(__uint_as_float(r[j]), p.alpha));
      }
      if constexpr (ADAM) {
        // stage the chunk as the fp32 TMA-store path does, optionally store it as Y, then
        // run the optimizer over it row by row
        uint8_t* buf = epi + (epi_chunk & 1u) * 4096u;
        if (lane == 0 && epi_chunk >= 2) bulk_wait_group_read<1>();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) * 16)) =
              make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (p.y_tma && lane == 0) {
          tma_store_2d(&p.ymap[ash], n0 + c, ml + q * 32, smem_u32(buf));
          bulk_commit_group();
        }
        ++epi_chunk;
        adam_chunk_rows<kAdamInFlight>(p, buf, m0 + q * 32, n0 + c, lane);
        continue;
      }
      if (p.y_tma) {
        // lane = row of a 32 x 32 chunk: 128-byte rows, 16-byte pieces placed with the
        // 128-byte swizzle (piece j of row i at slot j ^ (i % 8)): conflict-free writes,
        // and the layout the tensor map's swizzle reads back in order
        uint8_t* buf = epi + (epi_chunk & 1u) * 4096u;
        if (lane == 0 && epi_chunk >= 2) bulk_wait_group_read<1>();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) * 16)) =
              make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.ymap[ash], n0 + c, ml + q * 32, smem_u32(buf));
          bulk_commit_group();
        }
        ++epi_chunk;
        if (p.yb && row < p.m) store_row_chunk(p, row, n0 + c, r, false);
      } else if (row < p.m && (p.y || p.yb)) {
        store_row_chunk(p, row, n0 + c, r, p.y != nullptr);
      }
    }
  }
}

// GATE_UP = false: Y = alpha A W^T with 128 x 256 output tiles.
// GATE_UP = true: two B operands (gate and up shards, 128-row tiles each, back to back in
// the stage) share every A tile through one N = 256 MMA per K step; their two 128-column
// accumulators sit side by side in one 256-column TMEM buffer and the epilogue writes
// H = silu(gate) * up for a 128 x 128 tile.
// LAYOUT: bit 0 set = A MN-major, bit 1 = B MN-major (p.a_mn / p.b_mn, fixed at compile
// time: with the layout a run-time flag, the single producer thread's per-K-step work grew
// long enough to starve the tensor pipe of MN-major GEMMs by 10-30 %).
template <bool GATE_UP, bool ADAM = false, int LAYOUT = 0>
__global__ void __launch_bounds__(kThreads, 1) fsdp_gemm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!GATE_UP || LAYOUT == 0, "gate-up mode is K-major only");
  constexpr bool A_MN = (LAYOUT & 1) != 0, B_MN = (LAYOUT & 2) != 0;
  constexpr int TN = Mode<GATE_UP>::TN;                      // output tile columns
  constexpr uint32_t BT_BYTES = Mode<GATE_UP>::BT_BYTES;    // one B tile (two in gate-up mode)
  constexpr uint32_t STAGE_BYTES = Mode<GATE_UP>::STAGE;
  constexpr uint32_t ACC = Mode<GATE_UP>::ACC;
  constexpr uint32_t kTmemCols = Mode<GATE_UP>::TMEM_COLS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (p.m + BM - 1) / BM;
  const int num_n = (p.r + TN - 1) / TN;
  const int num_k = (p.k + BK - 1) / BK;
  const int tiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&accf_bar[a]), 1);
      mbar_init(smem_u32(&acce_bar[a]), 128);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.a_shards; ++s) prefetch_tmap(&p.a[s]);
    for (int s = 0; s < p.n_shards; ++s) {
      prefetch_tmap(&p.w[s]);
      if (GATE_UP) prefetch_tmap(&p.w2[s]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int64_t last_issue[STAGES];
      for (int s = 0; s < STAGES; ++s) last_issue[s] = -1;
      uint32_t it = 0, s = 0, ph = 0;  // K steps issued; their stage and its phase parity
      bool stop = false;
      for (int tile = blockIdx.x; tile < tiles && !stop; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, mb, nb);
        const int m0 = mb * BM;
        const int n0 = nb * TN;
        const int shard = B_MN ? 0 : n0 / p.shard_rows;
        const int nl = n0 - shard * p.shard_rows;
        const void* wmap = &p.w[shard];
        const int ash = A_MN ? 0 : m0 / p.a_shard_rows;  // the A row shard holding this tile's rows
        const int ml = m0 - ash * p.a_shard_rows;
        // MN-major operands: the K piece holding K block kb and the block's first row in it,
        // advanced one block at a time (pieces are whole K blocks when there are several)
        int aks = 0, akl = 0, bks = 0, bkl = 0;
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          if (it >= STAGES &&
              !mbar_wait_bounded(smem_u32(&empty_bar[s]), ph ^ 1u, abort, &g_zgb_dev_error, kErrEmpty)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[s]);
          uint8_t* sa = smem + s * STAGE_BYTES;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          if constexpr (A_MN) {  // K rows kb*BK.. of the piece holding them, BM / 64 M chunks
            tma_load_3d(smem_u32(sa), &p.a[aks], 0, akl, m0 / 64, fb);
            if ((akl += BK) == p.a_shard_rows) akl = 0, ++aks;
          } else {
            tma_load_2d(smem_u32(sa), &p.a[ash], kb * BK, ml, fb);
          }
          if constexpr (B_MN) {  // the same for B: TN / 64 chunks of 64 columns
            tma_load_3d(smem_u32(sa + A_BYTES), &p.w[bks], 0, bkl, n0 / 64, fb);
            if ((bkl += BK) == p.shard_rows) bkl = 0, ++bks;
          } else {
            tma_load_2d(smem_u32(sa + A_BYTES), wmap, kb * BK, nl, fb);
          }
          if (GATE_UP) tma_load_2d(smem_u32(sa + A_BYTES + BT_BYTES), &p.w2[shard], kb * BK, nl, fb);
          last_issue[s] = it;
          if (++s == STAGES) s = 0, ph ^= 1u;
        }
      }
      if (*abort) {
        int never = 0;
        for (int s = 0; s < STAGES; ++s)
          if (last_issue[s] >= 0)
            mbar_wait_bounded(smem_u32(&full_bar[s]), static_cast<uint32_t>(last_issue[s] / STAGES) & 1u, &never,
                              &g_zgb_dev_error, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // K-major: the next 16 K columns start 32 bytes further (+2 in the address field);
      // MN-major: 16 K rows = two 8-row groups further, 2048 bytes (+128)
      constexpr uint32_t a_step = A_MN ? 128u : 2u, b_step = B_MN ? 128u : 2u;
      // gate-up mode: the gate and up tiles sit back to back in the stage (128 rows each, the
      // same 128-byte row pitch), so ONE N = 256 MMA over both reads the A tile once and
      // fills the two side-by-side 128-column accumulators (gate, then up)
      constexpr uint32_t idesc = idesc_bf16_f32(BM, GATE_UP ? 2 * TN : TN, A_MN, B_MN);
      uint32_t i = 0, s = 0, ph = 0;
      bool stop = false, issued = false;
      for (int tile = blockIdx.x; tile < tiles && !stop; tile += gridDim.x, ++i) {
        const uint32_t a = i & 1u, u = i >> 1;
        if (u >= 1 && !mbar_wait_bounded(smem_u32(&acce_bar[a]), (u - 1) & 1u, abort, &g_zgb_dev_error, kErrAccE))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * ACC;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full_bar[s]), ph, abort, &g_zgb_dev_error, kErrFull)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
          const uint64_t ad = A_MN ? sw128_mnmajor_desc(sa, kMnChunk) : sw128_kmajor_desc(sa);
          const uint64_t bd = B_MN ? sw128_mnmajor_desc(sa + A_BYTES, kMnChunk) : sw128_kmajor_desc(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // K = 16 per MMA
            umma_bf16(d, ad + a_step * k, bd + b_step * k, idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty_bar[s]));
          issued = true;
          if (++s == STAGES) s = 0, ph ^= 1u;
        }
        if (!stop) umma_commit(smem_u32(&accf_bar[a]));
      }
      if (*abort && issued) {
        int never = 0;
        umma_commit(smem_u32(&drain_bar));
        mbar_wait_bounded(smem_u32(&drain_bar), 0, &never, &g_zgb_dev_error, kErrDrain);
      }
    }
  } else {
    // ---------------- epilogue (warps 2-5) ----------------
    const int q = warp & 3;  // a warp reads TMEM lanes [32q, 32q+32)
    uint32_t i = 0, epi_chunk = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++i) {
      const uint32_t a = i & 1u, u = i >> 1;
      if (!warp_wait(smem_u32(&accf_bar[a]), u & 1u, abort, kErrAccF)) break;
      tc_fence_after();
      int mb, nb;
      tile_coords(tile, num_m, num_n, mb, nb);
      const int m0 = mb * BM;
      const int n0 = nb * TN;
      const int ash = m0 / p.y_shard_rows;  // the Y row piece holding this tile's rows
      const int ml = m0 - ash * p.y_shard_rows;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * ACC;
      uint8_t* epi = smem + STAGES * STAGE_BYTES + static_cast<uint32_t>(q) * 2u * 4096u;
      epilogue_tile<GATE_UP, ADAM>(p, taddr, epi, epi_chunk, m0, n0, ash, ml, q, lane);
      tc_fence_before();
      mbar_arrive(smem_u32(&acce_bar[a]));
    }
    if (lane == 0) bulk_wait_group_all();  // no store may still read this CTA's shared memory
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---- CTA-pair form ----
// The same GEMM on the two-CTA tensor-core form: a cluster of two CTAs on two SMs computes
// a 256-row output tile with tcgen05.mma.cta_group::2 (M = 256, N = 256). Each CTA loads
// only its 128 A rows and 128 of the 256 B rows, and the MMA reads both CTAs' shared
// memory, so every SM moves a third fewer operand bytes per flop than in the one-CTA form
// (Mistral MLP GEMMs, live: 1.63-1.68 -> 1.74-1.79 PFLOP/s). Plain mode: CTA r loads W rows
// n0 + 128 r of a 256-column tile. Gate-up mode: the B operand of the N = 256 MMA is the
// gate tile followed by the up tile, so the even CTA loads the gate's 128 rows and the odd
// CTA the up projection's, and the accumulator holds gate | up exactly as in the one-CTA
// kernel. The other modes carry over: A and Y row pieces (each CTA's 128 rows lie in one
// piece, as pieces are multiples of 128 rows) and MN-major operands (each CTA's half is two
// 64-column chunks, one 3-D box).
//   both CTAs  warp 0: TMA producer; its copies complete on the EVEN CTA's full barrier,
//              which expects the stage bytes of both;
//   even CTA   warp 1: issues the MMAs; tcgen05.commit multicasts to both CTAs' empty
//              barriers (a stage is free in both) and accumulator barriers;
//   both CTAs  warps 2-5 (2-9 with the fused optimizer): epilogue of the CTA's own 128 rows
//              from its own TMEM; each warp then arrives on the even CTA's
//              accumulator-empty barrier (8 arrivals, 16).
// Before leaving, each producer waits until the MMAs released every stage it filled, and
// the two CTAs meet at a cluster barrier, so neither CTA's shared memory or barriers are
// still targeted by the other; every mbarrier wait is bounded as in the one-CTA kernel.
constexpr uint32_t PAIR_HALF = 128 * BK * 2;      // one CTA's 128 A rows, and its 128 B rows
constexpr uint32_t PAIR_STAGE = 2 * PAIR_HALF;
constexpr uint32_t PAIR_ACC = 256;                // TMEM columns of one accumulator (N = 256)
// Per variant: with the fused optimizer the epilogue does most of the kernel's instruction
// issue (the Adam arithmetic of a 128 x 256 tile per CTA) and its state loads' latency, so
// it runs 8 warps, two per TMEM lane quarter splitting the columns, with 16 rows of state
// loads in flight each (168 registers at 320 threads, no spills); their staging buffers
// take one operand stage (5 instead of 6; 5 measured within 1 % of 6 on the plain GEMMs).
template <bool ADAM> struct PairCfg {
  static constexpr int EPI_WARPS = ADAM ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int STAGES = ADAM ? 5 : 6;
  static constexpr uint32_t EPI = EPI_WARPS * 2u * 4096u;
  static constexpr uint32_t SMEM = STAGES * PAIR_STAGE + EPI + 1024;
};

constexpr unsigned int kErrPairEmpty = (4u << 8) | 1u;  // producer waiting for a free stage
constexpr unsigned int kErrPairFull = (4u << 8) | 2u;   // MMA waiting for both CTAs' copies
constexpr unsigned int kErrPairAccE = (4u << 8) | 3u;   // MMA waiting for both CTAs' epilogues
constexpr unsigned int kErrPairAccF = (4u << 8) | 4u;   // epilogue waiting for a finished tile
constexpr unsigned int kErrPairDrain = (4u << 8) | 5u;  // releasing stages / draining after an abort

// the walk of tile_coords over 256-row blocks (bands of 12 = the one-CTA kernel's 24 x 128 rows)
__device__ __forceinline__ void pair_tile_coords(int tile, int num_m, int num_n, int& mb, int& nb) {
  const int g = ZGB_GEMM_GROUP_M > 0 ? (ZGB_GEMM_GROUP_M + 1) / 2 : 0;
  const int band_rows = g > 0 && g < num_m ? g : num_m;
  const int band = tile / (band_rows * num_n), in_band = tile - band * band_rows * num_n;
  const int rows = min(band_rows, num_m - band * band_rows);
  mb = band * band_rows + in_band % rows;
  nb = in_band / rows;
}

template <bool GATE_UP, bool ADAM = false, int LAYOUT = 0>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<ADAM>::THREADS, 1)
    fsdp_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!GATE_UP || LAYOUT == 0, "gate-up mode is K-major only");
  constexpr int PAIR_STAGES = PairCfg<ADAM>::STAGES;
  constexpr int EPI_WARPS = PairCfg<ADAM>::EPI_WARPS;
  constexpr bool A_MN = (LAYOUT & 1) != 0, B_MN = (LAYOUT & 2) != 0;  // as in fsdp_gemm_kernel
  constexpr int TN = Mode<GATE_UP>::TN;  // output tile columns: 256, or 128 of H in gate-up mode
  static_assert(TN == (GATE_UP ? 128 : 256), "the pair MMA is N = 256: 256-column tiles, or gate | up halves");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[PAIR_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[PAIR_STAGES];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the even CTA, which issues the MMAs
  const int pair = static_cast<int>(blockIdx.x >> 1), pairs = static_cast<int>(gridDim.x >> 1);
  const int num_m = (p.m + 255) / 256;
  const int num_n = (p.r + TN - 1) / TN;
  const int num_k = (p.k + BK - 1) / BK;
  const int tiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&accf_bar[a]), 1);
      mbar_init(smem_u32(&acce_bar[a]), 2 * EPI_WARPS);  // every epilogue warp of both CTAs
    }
    mbar_init(smem_u32(&drain_bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.a_shards; ++s) prefetch_tmap(&p.a[s]);
    for (int s = 0; s < p.n_shards; ++s) prefetch_tmap(GATE_UP && rank ? &p.w2[s] : &p.w[s]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_base_sh), 2 * PAIR_ACC);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated before any copy
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      uint32_t it = 0, s = 0, ph = 0;  // K steps issued; their stage and its phase parity
      bool stop = false;
      for (int tile = pair; tile < tiles && !stop; tile += pairs) {
        int mb, nb;
        pair_tile_coords(tile, num_m, num_n, mb, nb);
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int nrow = nb * TN + (GATE_UP ? 0 : static_cast<int>(rank) * 128);
        // K-major pieces holding this CTA's rows; a half past the last row (M or R % 256 ==
        // 128) starts beyond the last piece and reads zeros
        const int ash = A_MN ? 0 : min(m0 / p.a_shard_rows, p.a_shards - 1);
        const int ml = m0 - ash * p.a_shard_rows;
        const int shard = B_MN ? 0 : min(nrow / p.shard_rows, p.n_shards - 1);
        const int nl = nrow - shard * p.shard_rows;
        const void* bmap = GATE_UP && rank ? &p.w2[shard] : &p.w[shard];
        int aks = 0, akl = 0, bks = 0, bkl = 0;  // MN-major: K piece and row of K block kb
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          if (it >= PAIR_STAGES &&
              !mbar_wait_bounded(smem_u32(&empty_bar[s]), ph ^ 1u, abort, &g_zgb_dev_error, kErrPairEmpty)) {
            stop = true;
            break;
          }
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * PAIR_STAGE);
          uint8_t* sa = smem + s * PAIR_STAGE;
          if constexpr (A_MN) {  // K rows kb*BK.. of the piece holding them, this CTA's two M chunks
            tma_load_3d_pair(smem_u32(sa), &p.a[aks], 0, akl, m0 / 64, fb);
            if ((akl += BK) == p.a_shard_rows) akl = 0, ++aks;
          } else {
            tma_load_2d_pair(smem_u32(sa), &p.a[ash], kb * BK, ml, fb);
          }
          if constexpr (B_MN) {  // the same for B: this CTA's two chunks of 64 columns
            tma_load_3d_pair(smem_u32(sa + PAIR_HALF), &p.w[bks], 0, bkl, nrow / 64, fb);
            if ((bkl += BK) == p.shard_rows) bkl = 0, ++bks;
          } else {
            tma_load_2d_pair(smem_u32(sa + PAIR_HALF), bmap, kb * BK, nl, fb);
          }
          if (++s == PAIR_STAGES) s = 0, ph ^= 1u;
        }
      }
      // every stage this CTA filled is read by the even CTA's MMAs: wait until they released it
      int never = 0;
      const uint32_t first = it > static_cast<uint32_t>(PAIR_STAGES) ? it - PAIR_STAGES : 0u;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_bounded(smem_u32(&empty_bar[j % PAIR_STAGES]), (j / PAIR_STAGES) & 1u, &never, &g_zgb_dev_error,
                          kErrPairDrain);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA) ----------------
    if (rank == 0 && lane == 0) {
      // K steps of 16 as in the one-CTA kernel: +32 B (K-major) or +2048 B (MN-major)
      constexpr uint32_t a_step = A_MN ? 128u : 2u, b_step = B_MN ? 128u : 2u;
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256, A_MN, B_MN);
      uint32_t i = 0, s = 0, ph = 0;
      bool stop = false, issued = false;
      for (int tile = pair; tile < tiles && !stop; tile += pairs, ++i) {
        const uint32_t a = i & 1u, u = i >> 1;
        if (u >= 1 && !mbar_wait_cluster_bounded(smem_u32(&acce_bar[a]), (u - 1) & 1u, abort, &g_zgb_dev_error,
                                                 kErrPairAccE))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * PAIR_ACC;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full_bar[s]), ph, abort, &g_zgb_dev_error, kErrPairFull)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * PAIR_STAGE);
          const uint64_t ad = A_MN ? sw128_mnmajor_desc(sa, kMnChunk) : sw128_kmajor_desc(sa);
          const uint64_t bd = B_MN ? sw128_mnmajor_desc(sa + PAIR_HALF, kMnChunk) : sw128_kmajor_desc(sa + PAIR_HALF);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16_pair(d, ad + a_step * k, bd + b_step * k, idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(smem_u32(&empty_bar[s]), 0x3);
          issued = true;
          if (++s == PAIR_STAGES) s = 0, ph ^= 1u;
        }
        if (!stop) umma_commit_pair(smem_u32(&accf_bar[a]), 0x3);
      }
      if (*abort && issued) {
        int never = 0;
        umma_commit_pair(smem_u32(&drain_bar), 0x1);
        mbar_wait_bounded(smem_u32(&drain_bar), 0, &never, &g_zgb_dev_error, kErrPairDrain);
      }
    }
  } else {
    // ---------------- epilogue (warps 2 .. 2 + EPI_WARPS - 1, both CTAs) ----------------
    const int q = warp & 3;                 // the TMEM lane quarter this warp may read
    const int part = (warp - 2) >> 2;       // which of the quarter's warps (column split)
    const int y_pieces = p.m / p.y_shard_rows;
    uint32_t i = 0, epi_chunk = 0;
    for (int tile = pair; tile < tiles; tile += pairs, ++i) {
      const uint32_t a = i & 1u, u = i >> 1;
      if (!warp_wait(smem_u32(&accf_bar[a]), u & 1u, abort, kErrPairAccF)) break;
      tc_fence_after();
      int mb, nb;
      pair_tile_coords(tile, num_m, num_n, mb, nb);
      const int m0 = mb * 256 + static_cast<int>(rank) * 128;
      const int ash = min(m0 / p.y_shard_rows, y_pieces - 1);  // the Y row piece (rows past M: clipped)
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * PAIR_ACC;
      uint8_t* epi = smem + PAIR_STAGES * PAIR_STAGE + static_cast<uint32_t>(warp - 2) * 2u * 4096u;
      epilogue_tile<GATE_UP, ADAM, EPI_WARPS / 4>(p, taddr, epi, epi_chunk, m0, nb * TN, ash,
                                                  m0 - ash * p.y_shard_rows, q, lane, part);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acce_bar[a]), 0));
    }
    if (lane == 0) bulk_wait_group_all();
  }

  tc_fence_before();
  cluster_sync_all();  // neither CTA's copies, MMAs or arrivals still target the other
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, 2 * PAIR_ACC);
  }
}

// ---- host side ----
// 0 (default) and 2: the CTA-pair kernel for every GEMM; 1: the one-CTA kernel everywhere
std::atomic<int> g_gemm_kernel{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
OncePerDevice g_attr_once[16];  // per kernel variant: gate-up, fused optimizer, operand layout

int get_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? ZERO_OK : set_error(ZERO_ERR_CUDA, "fsdp_unit_forward: cuTensorMapEncodeTiled unavailable");
}

int encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
              uint32_t box_rows, bool fp32 = false) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (fp32 ? 4 : 2)};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(ZERO_ERR_CUDA, "fsdp_unit_forward: cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ZERO_OK;
}

// MN-major operand [rows, cols] bf16 row-major (cols % 64 == 0) as the 3-D tensor
// {64, rows, cols / 64}: element (x, y, z) at base + 2 x + y * 2 cols + z * 128 B; box
// {64, BK, chunks}
int encode_mn(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t chunks) {
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BK), chunks};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(ZERO_ERR_CUDA, "fsdp_unit_backward: cuTensorMapEncodeTiled (MN-major) failed (%d)", (int)r);
  return ZERO_OK;
}

}  // namespace

namespace {

// One GEMM operand given as pieces: K-major pieces split the M (A) or R (B) rows; MN-major
// pieces ([K rows, M or R columns] row-major) split the K rows. piece_rows: rows of one
// piece (every piece the same).
struct Operand {
  int pieces;
  const uint16_t* const* ptr;
  bool mn;
  int64_t piece_rows;
};

// One of the kernels: gate-up or plain, plain with the fused optimizer (ADAM), for one
// operand layout, on CTA pairs or one CTA per tile.
template <bool GATE_UP, bool ADAM, int LAYOUT>
int launch_variant(const GemmParams& p, bool pair, int64_t m_tokens, int64_t rows_out, cudaStream_t st,
                   const char* who) {
  constexpr int TN = GATE_UP ? 128 : BN;
  constexpr int V = (GATE_UP ? 1 : 0) + (ADAM ? 2 : 0) + 4 * LAYOUT;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
  const cudaError_t attr = g_attr_once[V].run(dev, [] {
    cudaError_t a = cudaFuncSetAttribute(fsdp_gemm_kernel<GATE_UP, ADAM, LAYOUT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Mode<GATE_UP>::SMEM);
    if (a == cudaSuccess)
      a = cudaFuncSetAttribute(fsdp_gemm_pair_kernel<GATE_UP, ADAM, LAYOUT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg<ADAM>::SMEM);
    return a;
  });
  if (attr != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: %s", who, cudaGetErrorString(attr));
  if (pair) {
    // one 256-row tile per CTA pair at a time, as many pairs as can be resident at once: a
    // persistent grid larger than that runs its last clusters as a second wave (a 4-CTA
    // variant with 38 clusters where 36 fit ran at half speed). On GB300 all 76 pairs fit.
    static int max_pairs[16][64];
    static std::once_flag pairs_once[16][64];
    std::call_once(pairs_once[V][dev & 63], [&] {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * std::max(1, num_sms() / 2), 1, 1);
      cfg.blockDim = dim3(PairCfg<ADAM>::THREADS, 1, 1);
      cfg.dynamicSmemBytes = PairCfg<ADAM>::SMEM;
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, fsdp_gemm_pair_kernel<GATE_UP, ADAM, LAYOUT>, &cfg) != cudaSuccess ||
          nc < 1) {
        (void)cudaGetLastError();
        nc = std::max(1, num_sms() / 2);
      }
      max_pairs[V][dev & 63] = std::min(nc, std::max(1, num_sms() / 2));
    });
    const int64_t tiles = ((m_tokens + 255) / 256) * ((rows_out + TN - 1) / TN);
    const unsigned int pairs = static_cast<unsigned int>(std::min<int64_t>(tiles, max_pairs[V][dev & 63]));
    fsdp_gemm_pair_kernel<GATE_UP, ADAM, LAYOUT>
        <<<2 * pairs, PairCfg<ADAM>::THREADS, PairCfg<ADAM>::SMEM, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
    return ZERO_OK;
  }
  const int64_t tiles = ((m_tokens + BM - 1) / BM) * ((rows_out + TN - 1) / TN);
  const unsigned int grid = static_cast<unsigned int>(std::min<int64_t>(tiles, num_sms()));
  fsdp_gemm_kernel<GATE_UP, ADAM, LAYOUT><<<grid, kThreads, Mode<GATE_UP>::SMEM, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(ZERO_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return ZERO_OK;
}

// Y (y_pieces row pieces) = alpha * A * B^T, M x R, inner dimension K. GATE_UP: B and B2
// are the gate and up shards (K-major) and Y_bf16 receives H = silu(gate) * up.
template <bool GATE_UP>
int launch_gemm(const Operand& A, const Operand& B, const uint16_t* const* B2, int64_t m_tokens, int64_t rows_out,
                int64_t k_in, float* const* Y, int y_pieces, uint16_t* Y_bf16, float alpha, cudaStream_t st,
                const char* who, uint16_t* GU = nullptr, const AdamFuse* adam = nullptr) {
  constexpr int TN = GATE_UP ? 128 : BN;
  if (m_tokens > INT32_MAX / 2 || rows_out > INT32_MAX / 2 || k_in > INT32_MAX / 2)
    return set_error(ZERO_ERR_INVALID_ARG, "%s: sizes must be below 2^30", who);
  if (A.pieces < 1 || A.pieces > kMaxShards || B.pieces < 1 || B.pieces > kMaxShards || y_pieces < 1 ||
      y_pieces > kMaxShards)
    return set_error(ZERO_ERR_UNSUPPORTED, "%s: at most %d pieces per operand", who, kMaxShards);
  if (GATE_UP && (A.mn || B.mn)) return set_error(ZERO_ERR_UNSUPPORTED, "%s: gate-up mode is K-major only", who);
  // Kernel choice: the CTA-pair kernel unless the one-CTA kernel is asked for. With the
  // operand layout a template parameter, an MN-major operand costs the pair kernel 0-3 %
  // (Mistral W_up backward GEMMs: 1.013-1.050 ms for every layout), while the one-CTA
  // kernel runs 7-15 % behind it. Pair CTAs load 128-row halves of a K-major B, so B
  // pieces need a multiple of 128 rows; the one-CTA kernel loads whole TN-row tiles.
  const bool pair = g_gemm_kernel.load() != 1;
  // A and Y pieces
  if (A.mn) {
    if (A.piece_rows * A.pieces != k_in || (A.pieces > 1 && A.piece_rows % BK) || m_tokens % 64 || y_pieces != 1)
      return set_error(ZERO_ERR_UNSUPPORTED, "%s: unsupported split of the MN-major A operand", who);
  } else {
    if (A.piece_rows * A.pieces != m_tokens || y_pieces != A.pieces ||
        (A.pieces > 1 && (A.piece_rows % BM || GATE_UP || Y_bf16 || rows_out % 4)))
      return set_error(ZERO_ERR_UNSUPPORTED, "%s: unsupported row split of A / Y into %d pieces", who, A.pieces);
  }
  if (B.mn) {
    if (B.piece_rows * B.pieces != k_in || (B.pieces > 1 && B.piece_rows % BK) || rows_out % 64)
      return set_error(ZERO_ERR_UNSUPPORTED, "%s: unsupported split of the MN-major B operand", who);
  } else if (B.piece_rows * B.pieces != rows_out || (B.pieces > 1 && B.piece_rows % (pair ? 128 : TN) != 0)) {
    return set_error(ZERO_ERR_UNSUPPORTED,
                     "%s: the fused gather needs rows/n_ranks (%lld) to be a multiple of %d and n_ranks <= %d; "
                     "pass a scratch buffer to gather first",
                     who, (long long)B.piece_rows, pair ? 128 : TN, kMaxShards);
  }
  int rc = get_encode();
  if (rc) return rc;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  for (int s = 0; s < A.pieces; ++s) {
    rc = A.mn ? encode_mn(&p.a[s], A.ptr[s], m_tokens, A.piece_rows, BM / 64)
              : encode_2d(&p.a[s], A.ptr[s], k_in, A.piece_rows, BK, BM);
    if (rc) return rc;
  }
  for (int s = 0; s < B.pieces; ++s) {
    rc = B.mn ? encode_mn(&p.w[s], B.ptr[s], rows_out, B.piece_rows, pair ? 2 : TN / 64)
              : encode_2d(&p.w[s], B.ptr[s], k_in, B.piece_rows, BK, pair ? 128 : TN);
    if (rc) return rc;
    if (GATE_UP && (rc = encode_2d(&p.w2[s], B2[s], k_in, B.piece_rows, BK, TN))) return rc;
  }
  const int64_t y_rows = m_tokens / y_pieces;
  const bool no_f32 = Y == nullptr || Y[0] == nullptr;
  if (adam) {
    // the fused optimizer consumes the fp32 result in the epilogue; Y (fp32) may still be
    // written beside it, a bf16-only output may not
    bool ok = !GATE_UP && y_pieces == 1 && !Y_bf16 && rows_out % 8 == 0;
    for (int s = 0; ok && s < 2; ++s)
      ok = (reinterpret_cast<uintptr_t>(adam->master[s]) | reinterpret_cast<uintptr_t>(adam->m[s]) |
            reinterpret_cast<uintptr_t>(adam->v[s]) | reinterpret_cast<uintptr_t>(adam->w[s])) % 16 == 0 &&
           adam->master[s] && adam->m[s] && adam->v[s] && adam->w[s];
    if (!ok)
      return set_error(ZERO_ERR_UNSUPPORTED,
                       "%s: the fused optimizer needs one fp32 output piece, rows of a multiple of 8 and 16-byte-"
                       "aligned state",
                       who);
  } else if (!GATE_UP && no_f32) {  // bf16-only output through TMA stores
    if (!Y_bf16 || y_pieces != 1 || rows_out % 8 || (reinterpret_cast<uintptr_t>(Y_bf16) & 15))
      return set_error(ZERO_ERR_UNSUPPORTED,
                       "%s: a bf16-only output needs one 16-byte-aligned Y_bf16 with rows_out %% 8 == 0", who);
    if ((rc = encode_2d(&p.ybmap, Y_bf16, rows_out, m_tokens, 64, 32))) return rc;
    p.yb_tma = 1;
  }
  // fp32 output through TMA stores when its rows are 16-byte multiples (R % 4 == 0)
  bool y_aligned = !GATE_UP && !no_f32 && rows_out % 4 == 0;
  for (int s = 0; y_aligned && s < y_pieces; ++s) y_aligned = (reinterpret_cast<uintptr_t>(Y[s]) & 15) == 0;
  if (y_aligned) {
    for (int s = 0; s < y_pieces; ++s)
      if ((rc = encode_2d(&p.ymap[s], Y[s], rows_out, y_rows, 32, 32, true))) return rc;
    p.y_tma = 1;
  } else if (y_pieces > 1) {
    return set_error(ZERO_ERR_UNSUPPORTED, "%s: row-split outputs must be 16-byte aligned", who);
  }
  p.y = Y ? Y[0] : nullptr;
  p.a_shard_rows = static_cast<int>(A.piece_rows);
  p.a_shards = A.pieces;
  p.y_shard_rows = static_cast<int>(y_rows);
  p.a_mn = A.mn ? 1 : 0;
  p.b_mn = B.mn ? 1 : 0;
  p.yb = Y_bf16;
  p.gu = GATE_UP ? GU : nullptr;
  if (adam) p.adam = *adam;
  p.alpha = alpha;
  p.m = static_cast<int>(m_tokens);
  p.r = static_cast<int>(rows_out);
  p.k = static_cast<int>(k_in);
  p.shard_rows = static_cast<int>(B.piece_rows);
  p.n_shards = B.pieces;

  if constexpr (GATE_UP) {
    return launch_variant<true, false, 0>(p, pair, m_tokens, rows_out, st, who);
  } else {
    const int layout = (A.mn ? 1 : 0) | (B.mn ? 2 : 0);
    if (adam) {
      switch (layout) {
        case 0: return launch_variant<false, true, 0>(p, pair, m_tokens, rows_out, st, who);
        case 1: return launch_variant<false, true, 1>(p, pair, m_tokens, rows_out, st, who);
        case 2: return launch_variant<false, true, 2>(p, pair, m_tokens, rows_out, st, who);
        default: return launch_variant<false, true, 3>(p, pair, m_tokens, rows_out, st, who);
      }
    }
    switch (layout) {
      case 0: return launch_variant<false, false, 0>(p, pair, m_tokens, rows_out, st, who);
      case 1: return launch_variant<false, false, 1>(p, pair, m_tokens, rows_out, st, who);
      case 2: return launch_variant<false, false, 2>(p, pair, m_tokens, rows_out, st, who);
      default: return launch_variant<false, false, 3>(p, pair, m_tokens, rows_out, st, who);
    }
  }
}

}  // namespace

int launch_fsdp_gemm(int n_shards, const uint16_t* const* w_shards, int64_t rows_out, int64_t k_in,
                     const uint16_t* A, int64_t m_tokens, float* Y, uint16_t* Y_bf16, float alpha, cudaStream_t st) {
  const uint16_t* a1[1] = {A};
  float* y1[1] = {Y};
  return launch_gemm<false>({1, a1, false, m_tokens}, {n_shards, w_shards, false, rows_out / n_shards}, nullptr,
                            m_tokens, rows_out, k_in, y1, 1, Y_bf16, alpha, st, "fsdp_unit_forward");
}

int launch_fsdp_gemm_row_split(int a_shards, const uint16_t* const* A, float* const* Y, int64_t rows_per_shard,
                               const uint16_t* W, int64_t rows_out, int64_t k_in, float alpha, cudaStream_t st) {
  const uint16_t* w1[1] = {W};
  return launch_gemm<false>({a_shards, A, false, rows_per_shard}, {1, w1, false, rows_out}, nullptr,
                            rows_per_shard * a_shards, rows_out, k_in, Y, a_shards, nullptr, alpha, st,
                            "fsdp_unit_backward");
}

int launch_fsdp_gate_up(int n_shards, const uint16_t* const* gate_shards, const uint16_t* const* up_shards,
                        int64_t d_ff, int64_t d_model, const uint16_t* X, int64_t m_tokens, uint16_t* H,
                        cudaStream_t st, uint16_t* GU) {
  const uint16_t* a1[1] = {X};
  return launch_gemm<true>({1, a1, false, m_tokens}, {n_shards, gate_shards, false, d_ff / n_shards}, up_shards,
                           m_tokens, d_ff, d_model, nullptr, 1, H, 1.0f, st, "fsdp_mlp_forward", GU);
}

int launch_fsdp_bwd_dx(int n_ranks, const uint16_t* const* dY, int64_t dy_pieces_rows, int dy_pieces,
                       const uint16_t* const* w_shards, int64_t rows_out, int64_t k_in, float* const* dX,
                       cudaStream_t st) {
  return launch_gemm<false>({dy_pieces, dY, false, dy_pieces_rows}, {n_ranks, w_shards, true, rows_out / n_ranks},
                            nullptr, dy_pieces_rows * dy_pieces, k_in, rows_out, dX, dy_pieces, nullptr, 1.0f, st,
                            "fsdp_unit_backward");
}

int launch_fsdp_gemm_w_mn(int w_pieces, const uint16_t* const* W, int64_t w_piece_rows, int64_t n_out,
                          const uint16_t* A, int64_t m, float* Y, uint16_t* Y_bf16, float alpha, cudaStream_t st,
                          const char* who) {
  const uint16_t* a1[1] = {A};
  float* y1[1] = {Y};
  return launch_gemm<false>({1, a1, false, m}, {w_pieces, W, true, w_piece_rows}, nullptr, m, n_out,
                            w_piece_rows * w_pieces, y1, 1, Y_bf16, alpha, st, who);
}

int launch_fsdp_bwd_dw_in_place(int pieces, const uint16_t* const* dY, const uint16_t* const* X, int64_t piece_rows,
                                int64_t rows_out, int64_t k_in, float* dW, float alpha, cudaStream_t st,
                                const AdamFuse* adam, const char* who) {
  float* y1[1] = {dW};
  return launch_gemm<false>({pieces, dY, true, piece_rows}, {pieces, X, true, piece_rows}, nullptr, rows_out, k_in,
                            piece_rows * pieces, y1, 1, nullptr, alpha, st, who, nullptr, adam);
}

bool fsdp_fused_gather_ok(int n_ranks, int64_t rows_out) {
  if (n_ranks < 1 || n_ranks > kMaxShards || rows_out < 1 || rows_out % n_ranks) return false;
  // K-major forward: the pair kernel loads 128-row halves of each W tile, the one-CTA
  // kernel whole TN-row tiles, and each load must lie inside one shard
  return n_ranks == 1 || (rows_out / n_ranks) % (g_gemm_kernel.load() == 1 ? BN : 128) == 0;
}

int set_gemm_kernel(int which) {
  if (which < 0 || which > 2) return -1;
  g_gemm_kernel.store(which);
  return 0;
}

unsigned int fsdp_gemm_read_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_zgb_dev_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v) cudaMemcpyToSymbol(g_zgb_dev_error, &zero, sizeof(zero));
  return v;
}

}  // namespace zgb
