// gmm.cu -- persistent grouped GEMM on sm_103a (TMA -> tcgen05.mma -> TMEM)
// with a per-expert tile scheduler and fused epilogues.
//
// The GEMMs of the fused MoE-FFN [HyperMegaMoE §2.1 GMM1/up_proj ->
// SwiGLU -> GMM2/down_proj; §2.2 act_grad, SwiGLUGrad, input-grad GMM,
// W2Grad, W1Grad] all run through one kernel template:
//
//   rows mode   out[rows of e] = A[rows of e] . B[e]       (A: permuted
//               activations, K-major; B: expert weights, MN- or K-major)
//   wgrad mode  out[e] = A[rows of e]^T . B[rows of e]     (contraction over
//               the expert's padded rows; A, B: activations, MN-major)
//
// One launch may hold two problems.  Tiles are handed out through a global
// atomic ticket, all tiles of problem 0 before those of problem 1.  A tile of
// problem 1 may wait on a per-M-tile ready counter that the epilogues of
// problem 0 release [HyperMegaMoE §2.1: tasks split by token/expert tile,
// event counts release downstream tasks, no global barrier].  Because every
// producer tile has a smaller ticket, it was already taken by a running CTA
// when its consumer spins, so the wait cannot deadlock; it is bounded anyway.
//
// CTA = 6 warps: warp 0 issues TMA loads (one thread), warp 1 allocates TMEM
// and issues tcgen05.mma (one thread), warps 2..5 drain the accumulators
// (each owns the 32 TMEM lanes of its warp id mod 4).  Two 128x256 fp32
// accumulators in TMEM (512 columns) let the epilogue of one tile overlap the
// MMAs of the next; a 4-stage ring of 48 KB smem stages feeds the MMAs.
#include <cuda_bf16.h>

#include <algorithm>

#include "ptx.cuh"

namespace hmm {

enum Epi : int { EPI_SWIGLU = 0, EPI_STORE = 1, EPI_DSWIGLU = 2 };

template <int EPI_, bool WGRAD_, bool B_MN_>
struct Cfg {
  static constexpr int EPI = EPI_;
  static constexpr bool WGRAD = WGRAD_;
  static constexpr bool A_MN = WGRAD_;  // activations transposed in the wgrad mode
  static constexpr bool B_MN = B_MN_;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
};

constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TI_DEPTH = 4;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 2 * BN;

struct Prob {
  int K;        // rows mode: contraction length
  int N;        // valid output columns (SwiGLU / SwiGLU grad: I)
  int M;        // wgrad: output rows per expert
  int n_tiles;  // tiles along N
  int m_tiles;  // wgrad: tiles along M
  int half;     // SwiGLU: I (offset of the up half in the 2I operand/outputs)
  void* out;
  int64_t ld_out;
  int64_t out_estride;  // wgrad: elements between experts' outputs
  void* out2;
  int64_t ld_out2;
  void* out3;
  int64_t ld_out3;
  void* out4;           // SwiGLU grad: low bf16 half of dH (same layout as out)
  void* out5;           // SwiGLU grad: low bf16 half of w*a (same layout as out2)
  int split;            // wgrad: 0 none, 1 A operand given as hi+lo, 2 B operand hi+lo
  const void* aux;
  int64_t ld_aux;
  const float* rowscale;
  int* signal;       // per-M-tile counters released after a tile's stores
  const int* wait;   // per-M-tile counters acquired before a tile's A loads
  int wait_target;
};

struct Params {
  Prob p[2];
  int nprob;
  const int32_t* poff;
  int E;
  int* ticket;
  unsigned* status;
  unsigned long long budget_ns;
};

struct TileInfo {
  int prob;   // -1: no more tiles
  int e;
  int m0;     // rows mode: first padded row; wgrad: first output row
  int n0;     // first output column
  int kb;     // K blocks (0: empty wgrad tile -> zeros)
  int krow0;  // wgrad: first padded row of the expert
};

// ----------------------------------------------------------------- scheduler
__device__ __forceinline__ int tiles_of(const Params& P, const Prob& pr, bool wgrad) {
  if (wgrad) return P.E * pr.m_tiles * pr.n_tiles;
  return (P.poff[P.E] / BM) * pr.n_tiles;
}

template <class C>
__device__ void decode_tile(const Params& P, const Prob& pr, int u, TileInfo& ti) {
  if constexpr (C::WGRAD) {
    const int per = pr.m_tiles * pr.n_tiles;
    const int e = u / per;
    const int r = u - e * per;
    ti.e = e;
    ti.m0 = (r / pr.n_tiles) * BM;
    ti.n0 = (r % pr.n_tiles) * BN;
    ti.krow0 = P.poff[e];
    ti.kb = (P.poff[e + 1] - P.poff[e]) / BK * (pr.split ? 2 : 1);
  } else {
    // largest e with n_tiles * poff[e]/BM <= u (empty experts own no tiles)
    int lo = 0, hi = P.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((P.poff[mid] / BM) * pr.n_tiles <= u)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int e = lo;
    const int mt0 = P.poff[e] / BM;
    const int nm = P.poff[e + 1] / BM - mt0;
    const int local = u - mt0 * pr.n_tiles;
    const int nb = local / nm;
    ti.e = e;
    ti.m0 = (mt0 + (local - nb * nm)) * BM;
    ti.n0 = nb * (C::EPI == EPI_SWIGLU ? BN / 2 : BN);
    ti.krow0 = 0;
    ti.kb = (pr.K + BK - 1) / BK;
  }
}

// ----------------------------------------------------------------- producer
template <class C>
__device__ __forceinline__ void load_stage(const Prob& pr, const TileInfo& ti, int kb,
                                           const CUtensorMap* tA, const CUtensorMap* tB,
                                           const CUtensorMap* tS, uint8_t* sA, uint8_t* sB,
                                           uint64_t* bar) {
  if constexpr (C::WGRAD) {
    // with a split operand the K loop runs twice over the expert's rows:
    // first against the high bf16 half, then against the low half
    const int nk = pr.split ? ti.kb / 2 : ti.kb;
    const bool lo = kb >= nk;
    const int k = ti.krow0 + (lo ? kb - nk : kb) * BK;
    const CUtensorMap* a = (pr.split == 1 && lo) ? tS : tA;
    const CUtensorMap* b = (pr.split == 2 && lo) ? tS : tB;
    tma_load_2d(sA, a, bar, ti.m0, k);
    tma_load_2d(sA + 8192, a, bar, ti.m0 + 64, k);
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * 8192, b, bar, ti.n0 + 64 * j, k);
  } else {
    (void)tS;
    const int k = kb * BK;
    tma_load_2d(sA, tA, bar, k, ti.m0);
    if constexpr (C::B_MN) {
      if constexpr (C::EPI == EPI_SWIGLU) {
        tma_load_3d(sB, tB, bar, ti.n0, k, ti.e);
        tma_load_3d(sB + 8192, tB, bar, ti.n0 + 64, k, ti.e);
        tma_load_3d(sB + 16384, tB, bar, pr.half + ti.n0, k, ti.e);
        tma_load_3d(sB + 24576, tB, bar, pr.half + ti.n0 + 64, k, ti.e);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) tma_load_3d(sB + j * 8192, tB, bar, ti.n0 + 64 * j, k, ti.e);
      }
    } else {
      tma_load_3d(sB, tB, bar, k, ti.n0, ti.e);
    }
  }
}

// ---------------------------------------------------------------------- MMA
template <class C>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t a_base, uint32_t b_base,
                                          bool first) {
#pragma unroll
  for (int kk = 0; kk < BK / 16; ++kk) {
    const uint64_t ad = C::A_MN ? sw128_desc(a_base + kk * 2048, 8192, 1024)
                                : sw128_desc(a_base + kk * 32, 16, 1024);
    const uint64_t bd = C::B_MN ? sw128_desc(b_base + kk * 2048, 8192, 1024)
                                : sw128_desc(b_base + kk * 32, 16, 1024);
    umma_bf16(d_tmem, ad, bd, C::IDESC, (first && kk == 0) ? 0u : 1u);
  }
}

// ----------------------------------------------------------------- epilogue
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float g) { return 1.0f / (1.0f + __expf(-g)); }

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v, int valid) {
  // valid: number of the 32 columns inside the output (multiple of 8)
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < valid) {
      uint4 u;
      u.x = pack_bf16(v[q * 8 + 0], v[q * 8 + 1]);
      u.y = pack_bf16(v[q * 8 + 2], v[q * 8 + 3]);
      u.z = pack_bf16(v[q * 8 + 4], v[q * 8 + 5]);
      u.w = pack_bf16(v[q * 8 + 6], v[q * 8 + 7]);
      d[q] = u;
    }
  }
}

// v = hi + lo with hi = bf16(v), lo = bf16(v - hi): the pair carries about
// 16 significant bits, enough for the weight-gradient GEMMs that consume it.
__device__ __forceinline__ void store_bf16x32_split(__nv_bfloat16* hi, __nv_bfloat16* lo,
                                                    const float* v, int valid) {
  float h[32], l[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    h[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
    l[j] = v[j] - h[j];
  }
  store_bf16x32(hi, h, valid);
  store_bf16x32(lo, l, valid);
}

__device__ __forceinline__ void store_f32x32(float* dst, const float* v, int valid) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (q * 4 < valid) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void load_f32x32(const float* src, float* v, int valid) {
  const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q * 4 < valid) f = s[q];
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
}

// Drains the accumulator of one tile; taddr addresses this warp's lanes.
template <class C>
__device__ __forceinline__ void epilogue_tile(const Prob& pr, const TileInfo& ti, uint32_t taddr,
                                              int row_in_tile) {
  const int lane = threadIdx.x & 31;
  (void)lane;
  if constexpr (C::EPI == EPI_SWIGLU) {
    // cols [0,128): gate of n0..n0+127, [128,256): up of the same columns
    const int64_t row = ti.m0 + row_in_tile;
    __nv_bfloat16* a_row = static_cast<__nv_bfloat16*>(pr.out) + row * pr.ld_out;
    float* h_row = pr.out2 ? static_cast<float*>(pr.out2) + row * pr.ld_out2 : nullptr;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = ti.n0 + c * 32;
      if (col >= pr.N) break;
      const int valid = min(32, pr.N - col);
      uint32_t g[32], u[32];
      tmem_ld32(taddr + c * 32, g);
      tmem_ld32(taddr + 128 + c * 32, u);
      tmem_ld_wait();
      float av[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float gf = __uint_as_float(g[j]), uf = __uint_as_float(u[j]);
        av[j] = silu_f(gf) * uf;
      }
      store_bf16x32(a_row + col, av, valid);
      if (h_row) {
        store_f32x32(h_row + col, reinterpret_cast<const float*>(g), valid);
        store_f32x32(h_row + pr.half + col, reinterpret_cast<const float*>(u), valid);
      }
    }
  } else if constexpr (C::EPI == EPI_STORE) {
    int64_t row;
    __nv_bfloat16* base;
    if constexpr (C::WGRAD) {
      row = ti.m0 + row_in_tile;
      base = static_cast<__nv_bfloat16*>(pr.out) + static_cast<int64_t>(ti.e) * pr.out_estride;
    } else {
      row = ti.m0 + row_in_tile;
      base = static_cast<__nv_bfloat16*>(pr.out);
    }
    const bool row_ok = !C::WGRAD || row < pr.M;
    __nv_bfloat16* orow = base + row * pr.ld_out;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col = ti.n0 + c * 32;
      if (col >= pr.N) break;
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      if (row_ok) store_bf16x32(orow + col, reinterpret_cast<const float*>(r), min(32, pr.N - col));
    }
  } else {  // EPI_DSWIGLU
    // acc = G = dy_perm . W2^T for columns n0..n0+255 of I.  With the saved
    // fp32 pre-activations g, u and the slot's routing weight w:
    //   a = silu(g) u,  dA = w G,
    //   dgate = dA u s (1 + g (1 - s)),  dup = dA g s     (s = sigmoid(g))
    // writes dH = [dgate | dup] (bf16), wa = w a (bf16, the W2Grad operand)
    // and the partial d_w = sum_j G_j a_j of this column block (fp32).
    const int64_t row = ti.m0 + row_in_tile;
    const float* h_row = static_cast<const float*>(pr.aux) + row * pr.ld_aux;
    __nv_bfloat16* dh_row = static_cast<__nv_bfloat16*>(pr.out) + row * pr.ld_out;
    __nv_bfloat16* wa_row = static_cast<__nv_bfloat16*>(pr.out2) + row * pr.ld_out2;
    __nv_bfloat16* dh_lo = static_cast<__nv_bfloat16*>(pr.out4) + row * pr.ld_out;
    __nv_bfloat16* wa_lo = static_cast<__nv_bfloat16*>(pr.out5) + row * pr.ld_out2;
    const float w = pr.rowscale[row];
    float dwp = 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col = ti.n0 + c * 32;
      if (col >= pr.N) break;
      const int valid = min(32, pr.N - col);
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      float gv[32], uv[32];
      load_f32x32(h_row + col, gv, valid);
      load_f32x32(h_row + pr.half + col, uv, valid);
      tmem_ld_wait();
      float dg[32], du[32], wa[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float G = __uint_as_float(r[j]);
        const float g = gv[j], u = uv[j];
        const float s = sigmoid_f(g);
        const float a = g * s * u;
        dwp = fmaf(G, a, dwp);
        const float dA = w * G;
        dg[j] = dA * u * s * (1.0f + g * (1.0f - s));
        du[j] = dA * g * s;
        wa[j] = w * a;
      }
      store_bf16x32_split(dh_row + col, dh_lo + col, dg, valid);
      store_bf16x32_split(dh_row + pr.half + col, dh_lo + pr.half + col, du, valid);
      store_bf16x32_split(wa_row + col, wa_lo + col, wa, valid);
    }
    static_cast<float*>(pr.out3)[row * pr.ld_out3 + ti.n0 / BN] = dwp;
  }
}

template <class C>
__device__ __forceinline__ void epilogue_zero(const Prob& pr, const TileInfo& ti, int row_in_tile) {
  // wgrad tile of an expert with no rows: the gradient is exactly zero
  const int64_t row = ti.m0 + row_in_tile;
  if (row >= pr.M) return;
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(pr.out) +
                        static_cast<int64_t>(ti.e) * pr.out_estride + row * pr.ld_out;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int col = ti.n0; col < min(ti.n0 + BN, pr.N); col += 8)
    *reinterpret_cast<uint4*>(orow + col) = z;
}

// Bounded wait that ignores the abort flag (used only to drain in-flight
// copies / MMAs before the CTA exits).
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 31u) == 31u && globaltimer_ns() - t0 > budget_ns) return;
  }
}

// ------------------------------------------------------------------- kernel
template <class C0, class C1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gmm_kernel(const __grid_constant__ Params P, const __grid_constant__ CUtensorMap tA0,
               const __grid_constant__ CUtensorMap tB0, const __grid_constant__ CUtensorMap tS0,
               const __grid_constant__ CUtensorMap tA1, const __grid_constant__ CUtensorMap tB1,
               const __grid_constant__ CUtensorMap tS1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* ti_full = tempty + 2;
  uint64_t* ti_empty = ti_full + TI_DEPTH;
  uint64_t* mma_done = ti_empty + TI_DEPTH;
  TileInfo* s_ti = reinterpret_cast<TileInfo*>(mma_done + 1);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_ti + TI_DEPTH);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    for (int i = 0; i < TI_DEPTH; ++i) {
      mbar_init(&ti_full[i], 1);
      mbar_init(&ti_empty[i], 5);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const WaitCtl wc{s_abort, P.status, P.budget_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tA0);
      tma_prefetch_desc(&tB0);
      if (P.p[0].split) tma_prefetch_desc(&tS0);
      if (P.nprob > 1) {
        tma_prefetch_desc(&tA1);
        tma_prefetch_desc(&tB1);
        if (P.p[1].split) tma_prefetch_desc(&tS1);
      }
      const int T0 = tiles_of(P, P.p[0], C0::WGRAD);
      const int T1 = P.nprob > 1 ? tiles_of(P, P.p[1], C1::WGRAD) : 0;
      uint32_t stage = 0, sphase = 0;
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      uint32_t issued = 0;  // k-blocks issued by this CTA
      bool ok = true;
      for (;;) {
        const int t = atomicAdd(P.ticket, 1);
        TileInfo ti;
        ti.prob = -1;
        if (t < T0) {
          ti.prob = 0;
          decode_tile<C0>(P, P.p[0], t, ti);
        } else if (t < T0 + T1) {
          ti.prob = 1;
          decode_tile<C1>(P, P.p[1], t - T0, ti);
        }
        if (!mbar_wait(&ti_empty[ti_slot], ti_phase ^ 1u, wc)) {
          ok = false;
          break;
        }
        s_ti[ti_slot] = ti;
        mbar_arrive(&ti_full[ti_slot]);
        if (++ti_slot == TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (ti.prob < 0) break;
        const Prob& pr = P.p[ti.prob];
        if (pr.wait) {
          if (!counter_wait(&pr.wait[ti.m0 / BM], pr.wait_target, wc)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!mbar_wait(&empty[stage], sphase ^ 1u, wc)) {
            ok = false;
            break;
          }
          uint8_t* sA = stages + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          if (ti.prob == 0)
            load_stage<C0>(pr, ti, kb, &tA0, &tB0, &tS0, sA, sB, &full[stage]);
          else
            load_stage<C1>(pr, ti, kb, &tA1, &tB1, &tS1, sA, sB, &full[stage]);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        // wait (bounded) for the copies still in flight before leaving
        for (uint32_t s = 0; s < STAGES; ++s)
          if (issued > s) drain_wait(&full[s], ((issued - 1 - s) / STAGES) & 1u, P.budget_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issue
      uint32_t stage = 0, sphase = 0;
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      for (;;) {
        if (!mbar_wait(&ti_full[ti_slot], ti_phase, wc)) break;
        const TileInfo ti = s_ti[ti_slot];
        mbar_arrive(&ti_empty[ti_slot]);
        if (++ti_slot == TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (ti.prob < 0) break;
        if (ti.kb == 0) continue;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!mbar_wait(&full[stage], sphase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b_base = a_base + A_BYTES;
          if (ti.prob == 0)
            mma_stage<C0>(d_tmem, a_base, b_base, kb == 0);
          else
            mma_stage<C1>(d_tmem, a_base, b_base, kb == 0);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(mma_done);
      drain_wait(mma_done, 0, P.budget_ns);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int ti_slot = 0;
    uint32_t ti_phase = 0;
    uint32_t acc = 0, acc_phase = 0;
    for (;;) {
      bool got = false;
      if (lane == 0) got = mbar_wait(&ti_full[ti_slot], ti_phase, wc);
      __syncwarp();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      const TileInfo ti = s_ti[ti_slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ti_empty[ti_slot]);
      if (++ti_slot == TI_DEPTH) {
        ti_slot = 0;
        ti_phase ^= 1u;
      }
      if (ti.prob < 0) break;
      const Prob& pr = P.p[ti.prob];
      if (ti.kb == 0) {
        if (ti.prob == 0)
          epilogue_zero<C0>(pr, ti, row_in_tile);
        else
          epilogue_zero<C1>(pr, ti, row_in_tile);
        continue;
      }
      if (lane == 0) got = mbar_wait(&tfull[acc], acc_phase, wc);
      __syncwarp();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (ti.prob == 0)
        epilogue_tile<C0>(pr, ti, taddr, row_in_tile);
      else
        epilogue_tile<C1>(pr, ti, taddr, row_in_tile);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (pr.signal) {
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) red_release_add(&pr.signal[ti.m0 / BM], 1);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ====================================================================== host
namespace {

int encode(const GemmEnv& env, CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
           const uint64_t* strides_bytes, const uint32_t* box) {
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = env.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd,
                          gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HMM_OK : HMM_ERR_CUDA;
}

// activations [rows, cols] row-major: box {64 cols, box_rows rows}
int map_act(const GemmEnv& env, CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
            uint32_t box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t str[1] = {static_cast<uint64_t>(cols) * 2};
  const uint32_t box[2] = {64, box_rows};
  return encode(env, m, base, 2, dims, str, box);
}

// expert weights [E, d1, d0] row-major: box {64, box1, 1}
int map_w(const GemmEnv& env, CUtensorMap* m, const void* base, int64_t E, int64_t d1, int64_t d0,
          uint32_t box1) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d0), static_cast<uint64_t>(d1),
                            static_cast<uint64_t>(E)};
  const uint64_t str[2] = {static_cast<uint64_t>(d0) * 2, static_cast<uint64_t>(d0 * d1) * 2};
  const uint32_t box[3] = {64, box1, 1};
  return encode(env, m, base, 3, dims, str, box);
}

template <class C0, class C1>
int launch(const GemmEnv& env, Params& P, const CUtensorMap& a0, const CUtensorMap& b0,
           const CUtensorMap& s0, const CUtensorMap& a1, const CUtensorMap& b1,
           const CUtensorMap& s1, int64_t max_tiles) {
  if (max_tiles <= 0) return HMM_OK;
  auto kern = gmm_kernel<C0, C1>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return HMM_ERR_CUDA;
  const int grid = static_cast<int>(std::min<int64_t>(env.num_sms, max_tiles));
  P.status = env.status;
  P.budget_ns = env.budget_ns;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, env.stream>>>(P, a0, b0, s0, a1, b1, s1);
  return cudaGetLastError() == cudaSuccess ? HMM_OK : HMM_ERR_CUDA;
}

}  // namespace

using CfgGmm1 = Cfg<EPI_SWIGLU, false, true>;
using CfgGmm2 = Cfg<EPI_STORE, false, true>;
using CfgActGrad = Cfg<EPI_DSWIGLU, false, false>;
using CfgInGrad = Cfg<EPI_STORE, false, false>;
using CfgWGrad = Cfg<EPI_STORE, true, true>;

int launch_forward_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                         const void* x_perm, const void* W1, const void* W2, void* a, float* h32,
                         void* o, bool skip_ready_release) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  CUtensorMap tA0, tB0, tA1, tB1;
  int rc = HMM_OK;
  rc |= map_act(env, &tA0, x_perm, R, H, BM);        // x_perm [R, H], K = H
  rc |= map_w(env, &tB0, W1, E, H, 2 * I, 64);       // W1 [E, H, 2I]: MN-major B
  rc |= map_act(env, &tA1, a, R, I, BM);             // a [R, I], K = I
  rc |= map_w(env, &tB1, W2, E, I, H, 64);           // W2 [E, I, H]: MN-major B
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  Params P{};
  P.nprob = 2;
  P.poff = m.poff;
  P.E = static_cast<int>(E);
  P.ticket = c.tickets + 0;
  Prob& g1 = P.p[0];
  g1.K = static_cast<int>(H);
  g1.N = static_cast<int>(I);
  g1.half = static_cast<int>(I);
  g1.n_tiles = static_cast<int>((I + BN / 2 - 1) / (BN / 2));
  g1.out = a;
  g1.ld_out = I;
  g1.out2 = h32;
  g1.ld_out2 = 2 * I;
  g1.signal = skip_ready_release ? nullptr : c.ready;
  Prob& g2 = P.p[1];
  g2.K = static_cast<int>(I);
  g2.N = static_cast<int>(H);
  g2.n_tiles = static_cast<int>((H + BN - 1) / BN);
  g2.out = o;
  g2.ld_out = H;
  g2.wait = c.ready;
  g2.wait_target = 4 * g1.n_tiles;
  const int64_t max_tiles = p.max_mtiles * (g1.n_tiles + g2.n_tiles);
  return launch<CfgGmm1, CfgGmm2>(env, P, tA0, tB0, tA0, tA1, tB1, tA1, max_tiles);
}

int launch_backward_data_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                               const void* dy_perm, const float* wperm, const float* h32,
                               const void* W1, const void* W2, void* dH, void* dH_lo, void* wa,
                               void* wa_lo, float* dwp, void* dx_perm) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  CUtensorMap tA0, tB0, tA1, tB1;
  int rc = HMM_OK;
  rc |= map_act(env, &tA0, dy_perm, R, H, BM);       // dy_perm [R, H], K = H
  rc |= map_w(env, &tB0, W2, E, I, H, BN);           // W2 [E, I, H] = (W2^T) K-major, N = I
  rc |= map_act(env, &tA1, dH, R, 2 * I, BM);        // dH [R, 2I] (high half), K = 2I
  rc |= map_w(env, &tB1, W1, E, H, 2 * I, BN);       // W1 [E, H, 2I] = (W1^T) K-major, N = H
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  Params P{};
  P.nprob = 2;
  P.poff = m.poff;
  P.E = static_cast<int>(E);
  P.ticket = c.tickets + 1;
  Prob& ag = P.p[0];
  ag.K = static_cast<int>(H);
  ag.N = static_cast<int>(I);
  ag.half = static_cast<int>(I);
  ag.n_tiles = static_cast<int>(p.nt_dswiglu);
  ag.out = dH;
  ag.ld_out = 2 * I;
  ag.out2 = wa;
  ag.ld_out2 = I;
  ag.out3 = dwp;
  ag.ld_out3 = p.nt_dswiglu;
  ag.out4 = dH_lo;
  ag.out5 = wa_lo;
  ag.aux = h32;
  ag.ld_aux = 2 * I;
  ag.rowscale = wperm;
  ag.signal = c.ready;
  Prob& ig = P.p[1];
  ig.K = static_cast<int>(2 * I);
  ig.N = static_cast<int>(H);
  ig.n_tiles = static_cast<int>((H + BN - 1) / BN);
  ig.out = dx_perm;
  ig.ld_out = H;
  ig.wait = c.ready;
  ig.wait_target = 4 * ag.n_tiles;
  const int64_t max_tiles = p.max_mtiles * (ag.n_tiles + ig.n_tiles);
  return launch<CfgActGrad, CfgInGrad>(env, P, tA0, tB0, tA0, tA1, tB1, tA1, max_tiles);
}

int launch_backward_weight_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                                 const void* x_perm, const void* dy_perm, const void* dH,
                                 const void* dH_lo, const void* wa, const void* wa_lo, void* dW1,
                                 void* dW2) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  // dW2[e] = (wa_hi + wa_lo)^T . dy_perm : [I, rows] x [rows, H]
  // dW1[e] = x_perm^T . (dH_hi + dH_lo)  : [H, rows] x [rows, 2I]
  CUtensorMap w2A, w2B, w2S, w1A, w1B, w1S;
  int rc = HMM_OK;
  rc |= map_act(env, &w2A, wa, R, I, 64);
  rc |= map_act(env, &w2B, dy_perm, R, H, 64);
  rc |= map_act(env, &w2S, wa_lo, R, I, 64);
  rc |= map_act(env, &w1A, x_perm, R, H, 64);
  rc |= map_act(env, &w1B, dH, R, 2 * I, 64);
  rc |= map_act(env, &w1S, dH_lo, R, 2 * I, 64);
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  Prob w2{}, w1{};
  w2.M = static_cast<int>(I);
  w2.N = static_cast<int>(H);
  w2.m_tiles = static_cast<int>((I + BM - 1) / BM);
  w2.n_tiles = static_cast<int>((H + BN - 1) / BN);
  w2.out = dW2;
  w2.ld_out = H;
  w2.out_estride = I * H;
  w2.split = 1;
  w1.M = static_cast<int>(H);
  w1.N = static_cast<int>(2 * I);
  w1.m_tiles = static_cast<int>((H + BM - 1) / BM);
  w1.n_tiles = static_cast<int>((2 * I + BN - 1) / BN);
  w1.out = dW1;
  w1.ld_out = 2 * I;
  w1.out_estride = H * 2 * I;
  w1.split = 2;
  Params P{};
  P.poff = m.poff;
  P.E = static_cast<int>(E);
  P.ticket = c.tickets + 2;
  if (dW2 && dW1) {
    // dW1 first: its tiles are the larger share, dW2 tiles fill the tail
    P.nprob = 2;
    P.p[0] = w1;
    P.p[1] = w2;
    const int64_t max_tiles = E * (w1.m_tiles * w1.n_tiles + w2.m_tiles * w2.n_tiles);
    return launch<CfgWGrad, CfgWGrad>(env, P, w1A, w1B, w1S, w2A, w2B, w2S, max_tiles);
  }
  if (dW1) {
    P.nprob = 1;
    P.p[0] = w1;
    return launch<CfgWGrad, CfgWGrad>(env, P, w1A, w1B, w1S, w1A, w1B, w1S,
                                      E * w1.m_tiles * w1.n_tiles);
  }
  if (dW2) {
    P.nprob = 1;
    P.p[0] = w2;
    return launch<CfgWGrad, CfgWGrad>(env, P, w2A, w2B, w2S, w2A, w2B, w2S,
                                      E * w2.m_tiles * w2.n_tiles);
  }
  return HMM_OK;
}

}  // namespace hmm
