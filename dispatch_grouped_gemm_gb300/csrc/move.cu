// move.cu -- the bandwidth-bound steps: Dispatch (permute token rows into
// expert-contiguous padded order) and Combine (gather each token's K expert
// rows back and merge them), forward and backward.
//
// [HyperMegaMoE §2.1] Dispatch -> ... -> Combine; on one GPU these are a
// device-side permute and unpermute.  [MoE overlap explainer §6] the combine
// merges the top-k branches of a token weighted by their gates; here it is a
// deterministic gather: one warp per token, fp32 sums in fixed k order, a
// single bf16 rounding, no atomics.
//
// All row traffic uses 16-byte vectors (H is a multiple of 8 bf16).
#include <cuda_bf16.h>

#include <algorithm>

#include "hmm_internal.h"
#include "ptx.cuh"

namespace hmm {

namespace {

__device__ __forceinline__ float ld_weight(const void* w, int64_t i, int dtype) {
  if (dtype == HMM_DTYPE_F32) return static_cast<const float*>(w)[i];
  const uint16_t b = static_cast<const uint16_t*>(w)[i];
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void st_weight(void* w, int64_t i, int dtype, float v) {
  if (dtype == HMM_DTYPE_F32) {
    static_cast<float*>(w)[i] = v;
  } else {
    static_cast<__nv_bfloat16*>(w)[i] = __float2bfloat16_rn(v);
  }
}

__device__ __forceinline__ void acc8(float (&acc)[8], const uint4& v, float s) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc[2 * j] = fmaf(s, __uint_as_float(u[j] << 16), acc[2 * j]);
    acc[2 * j + 1] = fmaf(s, __uint_as_float(u[j] & 0xFFFF0000u), acc[2 * j + 1]);
  }
}

// Eight bf16 values to eight fp8 values (e5m2 or e4m3, saturating).
template <bool E5M2>
__device__ __forceinline__ uint2 bf16x8_to_fp8(const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(u[j] << 16);
    f[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
  }
  return pack_fp8x8<E5M2>(f);
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint4 r;
  uint32_t* u = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    u[j] = *reinterpret_cast<uint32_t*>(&p);
  }
  return r;
}

constexpr int MOVE_THREADS = 256;
constexpr int MOVE_WARPS = MOVE_THREADS / 32;
constexpr int UNROLL = 4;           // combine: 16-byte groups per lane per pass (x K rows)
constexpr int DISPATCH_UNROLL = 8;  // dispatch: a whole 2048-wide row per pass

}  // namespace

// Dispatch: token t's row of src goes to the padded rows of its K slots and,
// with the shared expert (E < Ex), to the shared expert's row poff[E] + t.
// The warps past T (launched when training) zero each expert's padding rows up
// to the first multiple of TROWS = 64 at or past its last row: the GEMMs'
// token blocks and the weight gradients' K blocks end there, so those rows
// are read and must be zero (the weight gradients sum over them), while the
// rows past it are never read.  In inference no padding row is written: the
// forward GEMMs compute outputs for the padding rows of a block, which no
// one reads.  Optionally also scatters the routing weight
// of every slot to its padded row (wperm: 1 on the shared rows, 0 on padding
// rows), and writes an fp8 copy of every row (dst8, ld8 8-byte groups per
// row; E5M2: e5m2, else e4m3), the weight-gradient GEMMs' operand for the
// low parts of their split operand.
//   spw: slots per warp.  A warp copies the row of one token to spw of its
// slots (K, plus the shared expert's row): with all of them (large T) the row
// is read once; with one (few tokens, e.g. decode) K times as many warps share
// the writes, the repeated reads hit L2.
template <bool E5M2>
__global__ void __launch_bounds__(MOVE_THREADS) dispatch_rows_kernel(
    const uint4* __restrict__ src, int64_t T, int64_t K, int64_t H8, MetaPtrs m, int E, int Ex,
    uint4* __restrict__ dst, uint2* __restrict__ dst8, int64_t ld8, const void* w, int w_dtype,
    float* wperm, int32_t* zero_ptr, int64_t zero_count, int spw) {
  const int lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * MOVE_WARPS + (threadIdx.x >> 5);
  grid_dep_wait();
  grid_dep_launch();
  if (zero_ptr) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * MOVE_THREADS + threadIdx.x;
         i < zero_count; i += static_cast<int64_t>(gridDim.x) * MOVE_THREADS)
      zero_ptr[i] = 0;
  }
  const int64_t KS = K + (E < Ex ? 1 : 0);
  const int64_t G = (KS + spw - 1) / spw;  // warps per token
  if (g < T * G) {
    const int64_t t = g / G;
    const int k0 = static_cast<int>(g % G) * spw;
    const int k1 = min(static_cast<int>(KS), k0 + spw);
    const bool mine = lane >= k0 && lane < k1;
    int32_t prow_l = -1;
    if (mine && lane < K) prow_l = m.slot2prow[t * K + lane];
    if (wperm && mine && lane < K && prow_l >= 0)
      wperm[prow_l] = ld_weight(w, t * K + lane, w_dtype);
    // the shared expert's row of this token, handled as slot K
    if (E < Ex && lane == K && mine) {
      prow_l = m.poff[E] + static_cast<int32_t>(t);
      if (wperm) wperm[prow_l] = 1.0f;
    }
    const uint4* s = src + t * H8;
    // every lane runs every iteration (the shuffles below read other lanes'
    // slots); only the loads and stores are guarded
    for (int64_t c0 = lane; c0 - lane < H8; c0 += 32 * DISPATCH_UNROLL) {
      uint4 v[DISPATCH_UNROLL];
#pragma unroll
      for (int u = 0; u < DISPATCH_UNROLL; ++u) {
        const int64_t c = c0 + 32 * u;
        if (c < H8) v[u] = s[c];
      }
      for (int k = k0; k < k1; ++k) {
        const int32_t prow = __shfl_sync(0xffffffffu, prow_l, k);
        if (prow < 0) continue;
        uint4* d = dst + static_cast<int64_t>(prow) * H8;
#pragma unroll
        for (int u = 0; u < DISPATCH_UNROLL; ++u) {
          const int64_t c = c0 + 32 * u;
          if (c < H8) d[c] = v[u];
        }
        if (dst8) {
          uint2* d8 = dst8 + static_cast<int64_t>(prow) * ld8;
#pragma unroll
          for (int u = 0; u < DISPATCH_UNROLL; ++u) {
            const int64_t c = c0 + 32 * u;
            if (c < H8) d8[c] = bf16x8_to_fp8<E5M2>(v[u]);
          }
        }
      }
    }
  } else {
    const int64_t q = g - T * G;
    const int64_t e = q / TROWS;
    if (e >= Ex) return;
    const int32_t cnt = m.counts[e];
    const int32_t pad = (cnt + TROWS - 1) / TROWS * TROWS - cnt;
    if (q % TROWS >= pad) return;
    const int32_t row = m.poff[e] + cnt + static_cast<int32_t>(q % TROWS);
    if (wperm && lane == 0) wperm[row] = 0.0f;
    uint4* d = dst + static_cast<int64_t>(row) * H8;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t c = lane; c < H8; c += 32) d[c] = z;
    if (dst8) {
      uint2* d8 = dst8 + static_cast<int64_t>(row) * ld8;
      for (int64_t c = lane; c < H8; c += 32) d8[c] = make_uint2(0, 0);
    }
  }
}

// Eight consecutive values (8-column group c) of row `row` of a bf16 or fp32
// row array with H8 groups per row, accumulated as acc += s * values.
template <bool F32>
__device__ __forceinline__ void acc_group(float (&acc)[8], const void* rows, int64_t row,
                                          int64_t c, int64_t H8, float s) {
  if constexpr (F32) {
    const float4* r = static_cast<const float4*>(rows) + (row * H8 + c) * 2;
    const float4 a = r[0], b = r[1];
    acc[0] = fmaf(s, a.x, acc[0]); acc[1] = fmaf(s, a.y, acc[1]);
    acc[2] = fmaf(s, a.z, acc[2]); acc[3] = fmaf(s, a.w, acc[3]);
    acc[4] = fmaf(s, b.x, acc[4]); acc[5] = fmaf(s, b.y, acc[5]);
    acc[6] = fmaf(s, b.z, acc[6]); acc[7] = fmaf(s, b.w, acc[7]);
  } else {
    acc8(acc, static_cast<const uint4*>(rows)[row * H8 + c], s);
  }
}

// Combine: out[t] = sum_k scale_k * rows[slot2prow[t*K+k]] (+ rows[*shared_row0
// + t], the shared expert's row, unit weight, when shared_row0 is given),
// fp32 in k order then the shared term, one bf16 rounding.  scale_k =
// topk_weights[t,k] (forward) or 1 (dX).  F32: the rows are fp32 (o and dX
// with the shared expert, whose unweighted term would otherwise carry a bf16
// rounding several times larger than the routed terms').
// With dwp != null (backward) lane k also writes
//   d_topk_weights[t,k] = sum over the act_grad N tiles of the per-row
//   partial dot products <G_s, a_s> (fixed order).
//   The grid's y dimension splits each token's row over several warps, each
// taking every gridDim.y-th group of 32 * UNROLL vectors (1 for large T;
// several for a few tokens, e.g. decode, so that enough rows are in flight).
template <bool WEIGHTED, bool F32>
__global__ void __launch_bounds__(MOVE_THREADS, F32 ? 2 : 4) combine_rows_kernel(
    const void* __restrict__ rows, const void* w, int w_dtype, int64_t T, int64_t K, int64_t H8,
    const int32_t* __restrict__ slot2prow, const int32_t* shared_row0, uint4* __restrict__ out,
    const float* dwp, int64_t dwp_ld, void* dw) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * MOVE_WARPS + (threadIdx.x >> 5);
  const int part = static_cast<int>(blockIdx.y);
  const int parts = static_cast<int>(gridDim.y);
  grid_dep_wait();
  grid_dep_launch();
  if (t >= T) return;
  int32_t prow_l = -1;
  float w_l = 0.0f;
  if (lane < K) {
    prow_l = slot2prow[t * K + lane];
    w_l = WEIGHTED ? ld_weight(w, t * K + lane, w_dtype) : 1.0f;
  }
  if (dwp && part == 0 && lane < K) {
    float d = 0.0f;
    if (prow_l >= 0)
      for (int64_t j = 0; j < dwp_ld; ++j) d += dwp[static_cast<int64_t>(prow_l) * dwp_ld + j];
    st_weight(dw, t * K + lane, w_dtype, d);
  }
  if (!out) return;
  const int64_t srow = shared_row0 ? *shared_row0 + t : -1;
  // every lane runs every iteration (the shuffles below read other lanes'
  // slots); only the loads and stores are guarded
  for (int64_t c0 = lane + static_cast<int64_t>(part) * 32 * UNROLL; c0 - lane < H8;
       c0 += static_cast<int64_t>(parts) * 32 * UNROLL) {
    float acc[UNROLL][8];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[u][j] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int32_t prow = __shfl_sync(0xffffffffu, prow_l, k);
      const float s = __shfl_sync(0xffffffffu, w_l, k);
      if (prow < 0) continue;
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int64_t c = c0 + 32 * u;
        if (c < H8) acc_group<F32>(acc[u], rows, prow, c, H8, s);
      }
    }
    if (srow >= 0) {
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int64_t c = c0 + 32 * u;
        if (c < H8) acc_group<F32>(acc[u], rows, srow, c, H8, 1.0f);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t c = c0 + 32 * u;
      if (c < H8) out[t * H8 + c] = pack8(acc[u]);
    }
  }
}

static int move_grid(int64_t warps) {
  return static_cast<int>((warps + MOVE_WARPS - 1) / MOVE_WARPS);
}

// Below this many tokens a warp per token leaves too few rows in flight to
// keep HBM busy: the dispatch gives each slot its own warp, the combine
// splits each token's row over several warps.
constexpr int64_t FEW_TOKENS = 1024;
static int dispatch_spw(const Plan& p) {
  return p.T >= FEW_TOKENS ? static_cast<int>(p.K + p.shared) : 1;
}
static int64_t dispatch_token_warps(const Plan& p) {
  const int64_t ks = p.K + p.shared, spw = dispatch_spw(p);
  return p.T * ((ks + spw - 1) / spw);
}
static int combine_parts(const Plan& p) {
  if (p.T >= FEW_TOKENS) return 1;
  const int64_t groups = (p.H / 8 + 32 * UNROLL - 1) / (32 * UNROLL);
  return static_cast<int>(std::min<int64_t>(groups, 8));
}

cudaError_t launch_dispatch_x(const Plan& p, const void* x, MetaPtrs m, void* x_perm, void* x8,
                              int32_t* zero_ptr, int64_t zero_count, cudaStream_t st, bool pdl) {
  // padding warps only when training (x8: the weight gradients will read them)
  const int64_t warps = dispatch_token_warps(p) + (x8 ? p.Ex * TROWS : 0);
  return launch_kernel(dispatch_rows_kernel<false>, move_grid(warps), MOVE_THREADS, 0, st, pdl, 1,
                       static_cast<const uint4*>(x), p.T, p.K, p.H / 8, m, static_cast<int>(p.E),
                       static_cast<int>(p.Ex), static_cast<uint4*>(x_perm),
                       static_cast<uint2*>(x8), p.ld8_h / 8, nullptr, 0, nullptr, zero_ptr,
                       zero_count, dispatch_spw(p));
}

cudaError_t launch_dispatch_dy(const Plan& p, const void* dy, const void* w, int w_dtype,
                               MetaPtrs m, CtrlPtrs c, void* dy_perm, void* dy8, float* wperm,
                               cudaStream_t st, bool pdl) {
  const int64_t warps = dispatch_token_warps(p) + p.Ex * TROWS;
  // also zero the backward launch counters (tickets and per-token-block ready
  // counters are contiguous in the control block)
  const int64_t nzero = p.ctrl_zero_count;
  return launch_kernel(dispatch_rows_kernel<true>, move_grid(warps), MOVE_THREADS, 0, st, pdl, 1,
                       static_cast<const uint4*>(dy), p.T, p.K, p.H / 8, m, static_cast<int>(p.E),
                       static_cast<int>(p.Ex), static_cast<uint4*>(dy_perm),
                       static_cast<uint2*>(dy8), p.ld8_h / 8, w, w_dtype, wperm, c.tickets, nzero,
                       dispatch_spw(p));
}

cudaError_t launch_combine_y(const Plan& p, const void* o, const void* w, int w_dtype, MetaPtrs m,
                             void* y, cudaStream_t st, bool pdl) {
  auto kern = p.shared ? combine_rows_kernel<true, true> : combine_rows_kernel<true, false>;
  const dim3 grid(move_grid(p.T), combine_parts(p));
  return launch_kernel(kern, grid, MOVE_THREADS, 0, st, pdl, 1, o, w, w_dtype,
                       p.T, p.K, p.H / 8, static_cast<const int32_t*>(m.slot2prow),
                       static_cast<const int32_t*>(p.shared ? m.poff + p.E : nullptr),
                       static_cast<uint4*>(y), static_cast<const float*>(nullptr), int64_t(0),
                       static_cast<void*>(nullptr));
}

cudaError_t launch_combine_dx(const Plan& p, const void* dx_perm, const float* dwp, MetaPtrs m,
                              void* dx, void* dw, int w_dtype, cudaStream_t st, bool pdl) {
  auto kern = p.shared ? combine_rows_kernel<false, true> : combine_rows_kernel<false, false>;
  const dim3 grid(move_grid(p.T), combine_parts(p));
  return launch_kernel(kern, grid, MOVE_THREADS, 0, st, pdl, 1, dx_perm,
                       static_cast<const void*>(nullptr), w_dtype, p.T, p.K, p.H / 8,
                       static_cast<const int32_t*>(m.slot2prow),
                       static_cast<const int32_t*>(p.shared ? m.poff + p.E : nullptr),
                       static_cast<uint4*>(dx), dw ? dwp : nullptr, p.dwp_ld, dw);
}

}  // namespace hmm
