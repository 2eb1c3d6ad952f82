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
// One launch holds up to four problems.  Tiles are handed out through a global
// atomic ticket in "schedule steps": step j holds, for every problem p, the
// tiles of expert j - lag_p.  A consumer problem runs a few experts behind its
// producer and waits on a ready counter (per M-tile, or per expert for the
// weight gradients) that the producer's epilogues release [HyperMegaMoE §2.1:
// tasks split by token/expert tile, event counts release downstream tasks, no
// global barrier; §2.2 / §5.2: W2Grad interleaved with the act_grad branch,
// W1Grad overlapped with the input gradient].  Interleaving experts mixes
// memory-bound and tensor-bound tiles in flight.  Every producer tile has a
// smaller ticket than its consumers, so it was already taken by a running CTA
// when a consumer spins: the wait cannot deadlock (and is bounded anyway).
//
// CTA = 7 warps: warp 6 schedules tiles (tickets, decoding, dependency waits,
// about one tile ahead), warp 0 issues TMA loads (one thread), warp 1
// allocates TMEM and issues tcgen05.mma (one thread), warps 2..5 drain the
// accumulators (each owns the 32 TMEM lanes of its warp id mod 4).  Two 128x256 fp32
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
constexpr int TI_DEPTH = 3;
// Warp roles: 0 TMA producer, 1 MMA issuer, 2..5 epilogue (one per TMEM lane
// quarter), 6 tile scheduler.  (Eight epilogue warps, two per quarter on
// alternate column chunks, were measured slower: more scattered epilogue
// traffic in flight slows the TMA operand feed of the same SM.)
constexpr int EPI_WARPS = 4;
constexpr int CH_SPLIT = EPI_WARPS / 4;  // warps sharing a lane quarter
constexpr int SCHED_WARP = 2 + EPI_WARPS;
constexpr int NUM_THREADS = 32 * (SCHED_WARP + 1);  // 11 warps
// alignment slack + stages + barriers, tile-info ring and schedule prefix table
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 512 + 4 * (3 * MAX_E + 8 + 1) + 256;
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
  int wgrad;            // 1: contraction over the expert's rows (tile count fixed per expert)
  int lag;              // the tiles of expert e are issued at schedule step e + lag
  int group;            // CTA group whose ticket queue holds this problem's tiles
  const void* aux;
  int64_t ld_aux;
  const float* rowscale;
  int* signal_m;        // per-M-tile counters released after a tile's stores
  int* signal_e;        // per-expert counters released after a tile's stores
  const int* wait_m;    // per-M-tile counter acquired before a tile's loads
  const int* wait_e;    // per-expert counter acquired before a tile's loads
  int wait_unit;        // target: wait_unit (per M-tile) or wait_unit * M-tiles of e
};

constexpr int MAX_PROB = 4;
constexpr int MAX_STEPS = 3 * MAX_E + 8;

struct Params {
  Prob p[MAX_PROB];
  int nprob;
  int steps[2];         // per CTA group: E + largest lag of its problems
  int group_split;      // CTAs [0, group_split) serve group 0, the rest group 1
                        // (0: one group)
  const int32_t* poff;
  const int32_t* counts;
  int E;
  int* ticket;
  unsigned* status;
  unsigned long long budget_ns;
  uint64_t* trace;      // per-tile timeline records (null: off)
  int trace_cap;
};

struct Maps {
  CUtensorMap m[MAX_PROB][3];  // A, B, and the low half of a split operand
};

struct TileInfo {
  int prob;   // -1: no more tiles
  int e;
  int m0;     // rows mode: first padded row; wgrad: first output row
  int n0;     // first output column
  int kb;     // K blocks (0: empty wgrad tile -> zeros)
  int krow0;  // wgrad: first padded row of the expert
};

// ------------------------------------------------------------------ tracing
__device__ __forceinline__ uint64_t* trace_rec(const Params& P, int lt) {
  if (P.trace == nullptr || lt >= P.trace_cap) return nullptr;
  return P.trace + (static_cast<int64_t>(blockIdx.x) * P.trace_cap + lt) * 8;
}
__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

// ----------------------------------------------------------------- scheduler
__device__ __forceinline__ int mtiles_of(const Params& P, int e) {
  return (P.poff[e + 1] - P.poff[e]) / BM;
}

__device__ __forceinline__ int tiles_of(const Params& P, const Prob& pr, int e) {
  if (e < 0 || e >= P.E) return 0;
  if (pr.wgrad) return pr.m_tiles * pr.n_tiles;
  return mtiles_of(P, e) * pr.n_tiles;
}

// Prefix sums of the tile counts of group g's schedule steps (one warp, into
// smem).
__device__ void build_schedule(const Params& P, int g, int* pref) {
  const int lane = threadIdx.x & 31;
  const int steps = P.steps[g];
  int carry = 0;
  if (lane == 0) pref[0] = 0;
  for (int base = 0; base < steps; base += 32) {
    const int j = base + lane;
    int v = 0;
    if (j < steps)
      for (int q = 0; q < P.nprob; ++q)
        if (P.p[q].group == g) v += tiles_of(P, P.p[q], j - P.p[q].lag);
    int inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += n;
    }
    if (j < steps) pref[j + 1] = carry + inc;
    carry += __shfl_sync(0xffffffffu, inc, 31);
  }
  __syncwarp();
}

// Ticket t of group g -> (problem, expert, local tile index).  Returns false
// past the end.
__device__ bool locate_tile(const Params& P, int g, const int* pref, int t, int& prob, int& e,
                            int& r) {
  const int steps = P.steps[g];
  if (t >= pref[steps]) return false;
  int lo = 0, hi = steps - 1;  // largest step j with pref[j] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  r = t - pref[lo];
  for (int q = 0; q < P.nprob; ++q) {
    if (P.p[q].group != g) continue;
    const int eq = lo - P.p[q].lag;
    const int c = tiles_of(P, P.p[q], eq);
    if (r < c) {
      prob = q;
      e = eq;
      return true;
    }
    r -= c;
  }
  return false;  // not reached
}

template <class C>
__device__ void decode_tile(const Params& P, const Prob& pr, int e, int r, TileInfo& ti) {
  ti.e = e;
  if constexpr (C::WGRAD) {
    ti.m0 = (r / pr.n_tiles) * BM;
    ti.n0 = (r % pr.n_tiles) * BN;
    ti.krow0 = P.poff[e];
    // rows past counts[e] are zero padding: skip whole zero K blocks
    ti.kb = (P.counts[e] + BK - 1) / BK * (pr.split ? 2 : 1);
  } else {
    const int nm = mtiles_of(P, e);
    const int nb = r / nm;  // M tiles innermost: a weight tile is reused from L2
    ti.m0 = P.poff[e] + (r - nb * nm) * BM;
    ti.n0 = nb * (C::EPI == EPI_SWIGLU ? BN / 2 : BN);
    ti.krow0 = 0;
    ti.kb = (pr.K + BK - 1) / BK;
  }
}

// ----------------------------------------------------------------- producer
// Loads the operand boxes of K block kb of a tile into one smem stage.  Every
// box starts at an inner coordinate that is a multiple of 8 elements (16 bytes).
template <class C>
__device__ __forceinline__ void stage_boxes(const Prob& pr, const TileInfo& ti, int kb,
                                            const CUtensorMap* tA, const CUtensorMap* tB,
                                            const CUtensorMap* tS, uint8_t* sA, uint8_t* sB,
                                            uint64_t* bar) {
  auto ld2 = [&](void* dst, const CUtensorMap* m, int c0, int c1) {
    tma_load_2d(dst, m, bar, c0, c1);
  };
  auto ld3 = [&](void* dst, const CUtensorMap* m, int c0, int c1, int c2) {
    tma_load_3d(dst, m, bar, c0, c1, c2);
  };

  if constexpr (C::WGRAD) {
    // with a split operand the K loop runs twice over the expert's rows:
    // first against the high bf16 half, then against the low half
    const int nk = pr.split ? ti.kb / 2 : ti.kb;
    const bool lo = kb >= nk;
    const int k = ti.krow0 + (lo ? kb - nk : kb) * BK;
    const CUtensorMap* a = (pr.split == 1 && lo) ? tS : tA;
    const CUtensorMap* b = (pr.split == 2 && lo) ? tS : tB;
    ld2(sA, a, ti.m0, k);
    ld2(sA + 8192, a, ti.m0 + 64, k);
#pragma unroll
    for (int j = 0; j < 4; ++j) ld2(sB + j * 8192, b, ti.n0 + 64 * j, k);
  } else {
    (void)tS;
    const int k = kb * BK;
    ld2(sA, tA, k, ti.m0);
    if constexpr (C::B_MN) {
      if constexpr (C::EPI == EPI_SWIGLU) {
        ld3(sB, tB, ti.n0, k, ti.e);
        ld3(sB + 8192, tB, ti.n0 + 64, k, ti.e);
        ld3(sB + 16384, tB, pr.half + ti.n0, k, ti.e);
        ld3(sB + 24576, tB, pr.half + ti.n0 + 64, k, ti.e);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) ld3(sB + j * 8192, tB, ti.n0 + 64 * j, k, ti.e);
      }
    } else {
      ld3(sB, tB, k, ti.n0, ti.e);
    }
  }
}

template <class C>
__device__ __forceinline__ void load_stage(const Prob& pr, const TileInfo& ti, int kb,
                                           const CUtensorMap* tA, const CUtensorMap* tB,
                                           const CUtensorMap* tS, uint8_t* sA, uint8_t* sB,
                                           uint64_t* bar) {
  stage_boxes<C>(pr, ti, kb, tA, tB, tS, sA, sB, bar);
}

// ---------------------------------------------------------------------- MMA
template <class C>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t a_base, uint32_t b_base,
                                          bool first) {
#pragma unroll
  for (int kk = 0; kk < BK / 16; ++kk) {
    const uint64_t ad = C::A_MN ? smem_desc(a_base + kk * 2048, 8192, 1024, LAYOUT_SW128)
                                : smem_desc(a_base + kk * 32, 16, 1024, LAYOUT_SW128);
    const uint64_t bd = C::B_MN ? smem_desc(b_base + kk * 2048, 8192, 1024, LAYOUT_SW128)
                                : smem_desc(b_base + kk * 32, 16, 1024, LAYOUT_SW128);
    umma_bf16(d_tmem, ad, bd, C::IDESC, (first && kk == 0) ? 0u : 1u);
  }
}

// ----------------------------------------------------------------- epilogue
// sigma(g) = 1 / (1 + exp(-g)) with the fast exponential and division
// intrinsics (a few ulp in fp32, far inside the bf16 output rounding).
// For g -> -inf the denominator overflows to inf and the quotient is 0.
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_f(float g) { return g * sigmoid_f(g); }

// 16-byte groups of one row segment: group q of the 32 columns at p + q * gs
// bytes (gs = 16: contiguous).
__device__ __forceinline__ void store_bf16x32(void* dst, int64_t gs, const float* v, int valid) {
  // valid: number of the 32 columns inside the output (multiple of 8)
  char* d = static_cast<char*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < valid) {
      uint4 u;
      u.x = pack_bf16(v[q * 8 + 0], v[q * 8 + 1]);
      u.y = pack_bf16(v[q * 8 + 2], v[q * 8 + 3]);
      u.z = pack_bf16(v[q * 8 + 4], v[q * 8 + 5]);
      u.w = pack_bf16(v[q * 8 + 6], v[q * 8 + 7]);
      *reinterpret_cast<uint4*>(d + q * gs) = u;
    }
  }
}

// v = hi + lo with hi = bf16(v), lo = bf16(v - hi): the pair carries about
// 16 significant bits, enough for the weight-gradient GEMMs that consume it.
__device__ __forceinline__ void store_bf16x32_split(void* hi, void* lo, int64_t gs,
                                                    const float* v, int valid) {
  float h[32], l[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    h[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
    l[j] = v[j] - h[j];
  }
  store_bf16x32(hi, gs, h, valid);
  store_bf16x32(lo, gs, l, valid);
}

__device__ __forceinline__ void store_bf16x8_split(__nv_bfloat16* hi, __nv_bfloat16* lo,
                                                   const float* v) {
  uint4 h, l;
  uint32_t* hp = reinterpret_cast<uint32_t*>(&h);
  uint32_t* lp = reinterpret_cast<uint32_t*>(&l);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float h0 = __bfloat162float(__float2bfloat16_rn(v[2 * j]));
    const float h1 = __bfloat162float(__float2bfloat16_rn(v[2 * j + 1]));
    hp[j] = pack_bf16(h0, h1);
    lp[j] = pack_bf16(v[2 * j] - h0, v[2 * j + 1] - h1);
  }
  *reinterpret_cast<uint4*>(hi) = h;
  *reinterpret_cast<uint4*>(lo) = l;
}

__device__ __forceinline__ void store_f32x32(void* dst, int64_t gs, const float* v, int valid) {
  char* d = static_cast<char*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (q * 4 < valid)
      *reinterpret_cast<float4*>(d + q * gs) =
          make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void load_f32x32(const void* src, int64_t gs, float* v, int valid) {
  const char* s = static_cast<const char*>(src);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q * 4 < valid) f = *reinterpret_cast<const float4*>(s + q * gs);
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
}

// Drains the accumulator of one tile; taddr addresses this warp's lanes.
// ch: which warp of the lane quarter (chunks ch, ch + CH_SPLIT, ...).
template <class C>
__device__ __forceinline__ void epilogue_tile(const Prob& pr, const TileInfo& ti, uint32_t taddr,
                                              int row_in_tile, int ch) {
  if constexpr (C::EPI == EPI_SWIGLU) {
    // cols [0,128): gate of n0..n0+127, [128,256): up of the same columns
    const int64_t row = ti.m0 + row_in_tile;
    __nv_bfloat16* a_row = static_cast<__nv_bfloat16*>(pr.out) + row * pr.ld_out;
    float* h_row = pr.out2 ? static_cast<float*>(pr.out2) + row * pr.ld_out2 : nullptr;
#pragma unroll 1
    for (int c = ch; c < 4; c += CH_SPLIT) {
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
      store_bf16x32(a_row + col, 16, av, valid);
      if (h_row) {
        store_f32x32(h_row + col, 16, reinterpret_cast<const float*>(g), valid);
        store_f32x32(h_row + pr.half + col, 16, reinterpret_cast<const float*>(u), valid);
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
    for (int c = ch; c < BN / 32; c += CH_SPLIT) {
      const int col = ti.n0 + c * 32;
      if (col >= pr.N) break;
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      if (row_ok)
        store_bf16x32(orow + col, 16, reinterpret_cast<const float*>(r), min(32, pr.N - col));
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
    for (int c = ch; c < BN / 32; c += CH_SPLIT) {
      const int col = ti.n0 + c * 32;
      if (col >= pr.N) break;
      const int valid = min(32, pr.N - col);
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      float gv[32], uv[32];
      load_f32x32(h_row + col, 16, gv, valid);
      load_f32x32(h_row + pr.half + col, 16, uv, valid);
      tmem_ld_wait();
      // eight columns at a time: compute, split into bf16 hi + lo, store
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q * 8 < valid) {
          float dg[8], du[8], wa[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float G = __uint_as_float(r[q * 8 + j]);
            const float g = gv[q * 8 + j], u = uv[q * 8 + j];
            const float sg = sigmoid_f(g);
            const float a = g * sg * u;
            dwp = fmaf(G, a, dwp);
            const float dA = w * G;
            dg[j] = dA * u * sg * (1.0f + g * (1.0f - sg));
            du[j] = dA * g * sg;
            wa[j] = w * a;
          }
          const int cq = col + q * 8;
          store_bf16x8_split(dh_row + cq, dh_lo + cq, dg);
          store_bf16x8_split(dh_row + pr.half + cq, dh_lo + pr.half + cq, du);
          store_bf16x8_split(wa_row + cq, wa_lo + cq, wa);
        }
      }
    }
    // one partial per (column block, warp of the quarter); the combine sums
    // them in order
    static_cast<float*>(pr.out3)[row * pr.ld_out3 + (ti.n0 / BN) * CH_SPLIT + ch] = dwp;
  }
}

template <class C>
__device__ __forceinline__ void epilogue_zero(const Prob& pr, const TileInfo& ti, int row_in_tile,
                                              int ch) {
  // wgrad tile of an expert with no rows: the gradient is exactly zero
  const int64_t row = ti.m0 + row_in_tile;
  if (row >= pr.M) return;
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(pr.out) +
                        static_cast<int64_t>(ti.e) * pr.out_estride + row * pr.ld_out;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int c = ch; c < BN / 32; c += CH_SPLIT)
    for (int col = ti.n0 + c * 32; col < min(ti.n0 + c * 32 + 32, pr.N); col += 8)
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
#define HMM_BY_PROB(q, F, ...)       \
  switch (q) {                       \
    case 0: F<C0>(__VA_ARGS__); break; \
    case 1: F<C1>(__VA_ARGS__); break; \
    case 2: F<C2>(__VA_ARGS__); break; \
    default: F<C3>(__VA_ARGS__); break; \
  }

template <class C0, class C1, class C2, class C3>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gmm_kernel(const __grid_constant__ Params P, const __grid_constant__ Maps maps) {
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
  int* s_pref = reinterpret_cast<int*>(s_tmem + 2);  // [steps + 1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_WARPS);
    }
    for (int i = 0; i < TI_DEPTH; ++i) {
      mbar_init(&ti_full[i], 1);
      mbar_init(&ti_empty[i], 2 + EPI_WARPS);  // TMA producer, MMA issuer, epilogue warps
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

  const int group = (P.group_split > 0 && static_cast<int>(blockIdx.x) >= P.group_split) ? 1 : 0;
  if (warp == SCHED_WARP) {
    // --------------------------------------------------------- tile scheduler
    // Fetches tickets, decodes them and waits for each tile's dependencies
    // about one tile ahead of the TMA producer, so neither the ticket atomic
    // nor a ready-counter poll sits on the load path.  (A deeper lookahead
    // spreads the M tiles that share a weight tile over time and costs L2
    // reuse of the weights.)  Lane 0 does the bookkeeping.
    build_schedule(P, group, s_pref);
    int ti_slot = 0;
    uint32_t ti_phase = 0;
    int lt = 0;  // tiles of this CTA so far (trace index)
    int t = 0;
    if (lane == 0) t = atomicAdd(P.ticket + group, 1);
    for (;;) {
      TileInfo ti;
      ti.prob = -1;
      ti.e = ti.m0 = ti.n0 = ti.kb = ti.krow0 = 0;
      bool ok = true;
      if (lane == 0) {
        int q = 0, e = 0, r = 0;
        if (locate_tile(P, group, s_pref, t, q, e, r)) {
          ti.prob = q;
          HMM_BY_PROB(q, decode_tile, P, P.p[q], e, r, ti);
          t = atomicAdd(P.ticket + group, 1);  // next ticket, early
          const Prob& pr = P.p[q];
          if (pr.wait_m || pr.wait_e)
            ok = pr.wait_m ? counter_wait(&pr.wait_m[ti.m0 / BM], pr.wait_unit, wc)
                           : counter_wait(&pr.wait_e[ti.e], pr.wait_unit * mtiles_of(P, ti.e),
                                          wc);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ti.prob = __shfl_sync(0xffffffffu, ti.prob, 0);
      ti.e = __shfl_sync(0xffffffffu, ti.e, 0);
      ti.m0 = __shfl_sync(0xffffffffu, ti.m0, 0);
      ti.n0 = __shfl_sync(0xffffffffu, ti.n0, 0);
      ti.kb = __shfl_sync(0xffffffffu, ti.kb, 0);
      ti.krow0 = __shfl_sync(0xffffffffu, ti.krow0, 0);
      bool got = false;
      if (lane == 0) got = mbar_wait(&ti_empty[ti_slot], ti_phase ^ 1u, wc);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      if (lane == 0) {
        if (ti.prob >= 0) {
          if (uint64_t* rec = trace_rec(P, lt)) {
            rec[0] = (static_cast<uint64_t>(sm_id()) << 48) |
                     (static_cast<uint64_t>(ti.prob) << 40) |
                     (static_cast<uint64_t>(ti.e & 0xFFFFF) << 20) |
                     static_cast<uint64_t>(ti.kb & 0xFFFFF);
            rec[1] = globaltimer_ns();
          }
        }
        s_ti[ti_slot] = ti;
        mbar_arrive(&ti_full[ti_slot]);
      }
      __syncwarp();
      ++lt;
      if (++ti_slot == TI_DEPTH) {
        ti_slot = 0;
        ti_phase ^= 1u;
      }
      if (ti.prob < 0) break;
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- TMA producer
      for (int q = 0; q < P.nprob; ++q) {
        tma_prefetch_desc(&maps.m[q][0]);
        tma_prefetch_desc(&maps.m[q][1]);
        if (P.p[q].split) tma_prefetch_desc(&maps.m[q][2]);
      }
      uint32_t stage = 0, sphase = 0;
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      uint32_t issued = 0;  // k-blocks issued by this CTA
      bool ok = true;
      int lt = 0;
      for (;;) {
        if (!mbar_wait(&ti_full[ti_slot], ti_phase, wc)) {
          ok = false;
          break;
        }
        const TileInfo ti = s_ti[ti_slot];
        mbar_arrive(&ti_empty[ti_slot]);
        if (++ti_slot == TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (ti.prob < 0) break;
        const Prob& pr = P.p[ti.prob];
        // the scheduler acquired this tile's ready counter (gpu scope) before
        // publishing it; order that with the async-proxy loads below
        if (pr.wait_m || pr.wait_e) fence_proxy_async_global();
        const CUtensorMap* mp = maps.m[ti.prob];
        uint64_t* rec = trace_rec(P, lt++);
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!mbar_wait(&empty[stage], sphase ^ 1u, wc)) {
            ok = false;
            break;
          }
          if (rec && kb == 0) rec[2] = globaltimer_ns();
          uint8_t* sA = stages + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          HMM_BY_PROB(ti.prob, load_stage, pr, ti, kb, &mp[0], &mp[1], &mp[2], sA, sB,
                      &full[stage]);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (rec && ok) rec[3] = globaltimer_ns();
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
      int lt = 0;
      for (;;) {
        if (!mbar_wait(&ti_full[ti_slot], ti_phase, wc)) break;
        const TileInfo ti = s_ti[ti_slot];
        mbar_arrive(&ti_empty[ti_slot]);
        if (++ti_slot == TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (ti.prob < 0) break;
        uint64_t* rec = trace_rec(P, lt++);
        if (ti.kb == 0) continue;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        if (rec) rec[4] = globaltimer_ns();
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
          HMM_BY_PROB(ti.prob, mma_stage, d_tmem, a_base, b_base, kb == 0);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (rec) rec[5] = globaltimer_ns();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(mma_done);
      drain_wait(mma_done, 0, P.budget_ns);
    }
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int ch = (warp - 2) / 4;  // which warp of the lane quarter
    const int row_in_tile = q * 32 + lane;
    int ti_slot = 0;
    uint32_t ti_phase = 0;
    uint32_t acc = 0, acc_phase = 0;
    int lt = 0;
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
      uint64_t* rec = (warp == 2 && lane == 0) ? trace_rec(P, lt) : nullptr;  // one warp reports
      ++lt;
      if (ti.kb == 0) {
        HMM_BY_PROB(ti.prob, epilogue_zero, pr, ti, row_in_tile, ch);
        continue;
      }
      if (lane == 0) got = mbar_wait(&tfull[acc], acc_phase, wc);
      __syncwarp();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      if (rec) rec[6] = globaltimer_ns();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      HMM_BY_PROB(ti.prob, epilogue_tile, pr, ti, taddr, row_in_tile, ch);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (rec) rec[7] = globaltimer_ns();
      if (pr.signal_m || pr.signal_e) {
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) {
          if (pr.signal_m) red_release_add(&pr.signal_m[ti.m0 / BM], 1);
          if (pr.signal_e) red_release_add(&pr.signal_e[ti.e], 1);
        }
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

template <class C0, class C1, class C2, class C3>
int launch(const GemmEnv& env, Params& P, const Maps& maps, int64_t max_tiles, int kind) {
  if (max_tiles <= 0 || P.nprob == 0) return HMM_OK;
  if (env.trace && env.trace_which == kind) {
    P.trace = env.trace;
    P.trace_cap = env.trace_cap;
  }
  auto kern = gmm_kernel<C0, C1, C2, C3>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return HMM_ERR_CUDA;
  int max_lag[2] = {-1, -1};
  for (int q = 0; q < P.nprob; ++q)
    max_lag[P.p[q].group] = std::max(max_lag[P.p[q].group], P.p[q].lag);
  for (int g = 0; g < 2; ++g) {
    P.steps[g] = max_lag[g] < 0 ? 0 : P.E + max_lag[g];
    if (P.steps[g] > MAX_STEPS) return HMM_ERR_SHAPE;
  }
  int grid = static_cast<int>(std::min<int64_t>(env.num_sms, max_tiles));
  if (max_lag[1] < 0) P.group_split = 0;
  if (P.group_split > 0) {
    // both groups need CTAs: the grid is every SM, the split inside it
    grid = env.num_sms;
    P.group_split = std::min(std::max(P.group_split, 1), grid - 1);
  }
  P.status = env.status;
  P.budget_ns = env.budget_ns;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, env.stream>>>(P, maps);
  return cudaGetLastError() == cudaSuccess ? HMM_OK : HMM_ERR_CUDA;
}

}  // namespace

using CfgGmm1 = Cfg<EPI_SWIGLU, false, true>;
using CfgGmm2 = Cfg<EPI_STORE, false, true>;
using CfgActGrad = Cfg<EPI_DSWIGLU, false, false>;
using CfgInGrad = Cfg<EPI_STORE, false, false>;
using CfgW2Grad = Cfg<EPI_STORE, true, true>;
using CfgW1Grad = Cfg<EPI_STORE, true, true>;

int launch_forward_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                         const void* x_perm, const void* W1, const void* W2, void* a, float* h32,
                         void* o, bool skip_ready_release) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  Maps maps;
  int rc = HMM_OK;
  rc |= map_act(env, &maps.m[0][0], x_perm, R, H, BM);   // x_perm [R, H], K = H
  rc |= map_w(env, &maps.m[0][1], W1, E, H, 2 * I, 64);  // W1 [E, H, 2I]: MN-major B
  rc |= map_act(env, &maps.m[1][0], a, R, I, BM);        // a [R, I], K = I
  rc |= map_w(env, &maps.m[1][1], W2, E, I, H, 64);      // W2 [E, I, H]: MN-major B
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  maps.m[0][2] = maps.m[0][0];
  maps.m[1][2] = maps.m[1][0];
  Params P{};
  P.nprob = 2;
  P.poff = m.poff;
  P.counts = m.counts;
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
  g1.signal_m = skip_ready_release ? nullptr : c.ready;
  Prob& g2 = P.p[1];
  g2.K = static_cast<int>(I);
  g2.N = static_cast<int>(H);
  g2.n_tiles = static_cast<int>((H + BN - 1) / BN);
  g2.out = o;
  g2.ld_out = H;
  // GMM2 after every GMM1 tile has been handed out: its ready waits then only
  // meet the last wave of GMM1 tiles
  g2.lag = static_cast<int>(E);
  g2.wait_m = c.ready;
  g2.wait_unit = EPI_WARPS * g1.n_tiles;  // every epilogue warp of every GMM1 tile of the M tile
  const int64_t max_tiles = p.max_mtiles * (g1.n_tiles + g2.n_tiles);
  return launch<CfgGmm1, CfgGmm2, CfgGmm2, CfgGmm2>(env, P, maps, max_tiles, 0);
}

int launch_backward_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                          const void* x_perm, const void* dy_perm, const float* wperm,
                          const float* h32, const void* W1, const void* W2, void* dH,
                          void* dH_lo, void* wa, void* wa_lo, float* dwp, void* dx_perm,
                          void* dW1, void* dW2) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  Maps maps;
  int rc = HMM_OK;
  // act_grad: G = dy_perm . W2^T   (B = W2 [E, I, H] read K-major, N = I)
  rc |= map_act(env, &maps.m[0][0], dy_perm, R, H, BM);
  rc |= map_w(env, &maps.m[0][1], W2, E, I, H, BN);
  // input-grad: dX_perm = dH . W1^T (B = W1 [E, H, 2I] read K-major, N = H)
  rc |= map_act(env, &maps.m[1][0], dH, R, 2 * I, BM);
  rc |= map_w(env, &maps.m[1][1], W1, E, H, 2 * I, BN);
  // W2Grad: dW2[e] = (wa_hi + wa_lo)^T . dy_perm    [I, rows] x [rows, H]
  rc |= map_act(env, &maps.m[2][0], wa, R, I, 64);
  rc |= map_act(env, &maps.m[2][1], dy_perm, R, H, 64);
  rc |= map_act(env, &maps.m[2][2], wa_lo, R, I, 64);
  // W1Grad: dW1[e] = x_perm^T . (dH_hi + dH_lo)     [H, rows] x [rows, 2I]
  rc |= map_act(env, &maps.m[3][0], x_perm, R, H, 64);
  rc |= map_act(env, &maps.m[3][1], dH, R, 2 * I, 64);
  rc |= map_act(env, &maps.m[3][2], dH_lo, R, 2 * I, 64);
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  const CUtensorMap map_w2[3] = {maps.m[2][0], maps.m[2][1], maps.m[2][2]};
  const CUtensorMap map_w1[3] = {maps.m[3][0], maps.m[3][1], maps.m[3][2]};
  maps.m[0][2] = maps.m[0][0];
  maps.m[1][2] = maps.m[1][0];
  Params P{};
  P.poff = m.poff;
  P.counts = m.counts;
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
  static_assert(CH_SPLIT == 1, "the d_w partial buffer holds one entry per act_grad N tile");
  ag.ld_out3 = p.dwp_ld;
  ag.out4 = dH_lo;
  ag.out5 = wa_lo;
  ag.aux = h32;
  ag.ld_aux = 2 * I;
  ag.rowscale = wperm;
  ag.signal_m = c.ready;
  ag.signal_e = c.eready;
  Prob& ig = P.p[1];
  ig.K = static_cast<int>(2 * I);
  ig.N = static_cast<int>(H);
  ig.n_tiles = static_cast<int>((H + BN - 1) / BN);
  ig.out = dx_perm;
  ig.ld_out = H;
  ig.wait_m = c.ready;
  ig.wait_unit = EPI_WARPS * ag.n_tiles;
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
  for (Prob* w : {&w2, &w1}) {
    w->wgrad = 1;
    w->wait_e = c.eready;
    w->wait_unit = EPI_WARPS * ag.n_tiles;  // every act_grad tile of every M tile of the expert
  }
  ig.lag = static_cast<int>(E);  // input-grad after every act_grad tile is handed out
  const int64_t data_tiles = p.max_mtiles * (ag.n_tiles + ig.n_tiles);
  const int64_t w_tiles = (dW2 ? E * w2.m_tiles * w2.n_tiles : 0) +
                          (dW1 ? E * w1.m_tiles * w1.n_tiles : 0);
  const int nw = (dW2 ? 1 : 0) + (dW1 ? 1 : 0);
  if (!dW2) w2.m_tiles = 0;  // fixed problem slots: W2Grad, then W1Grad
  if (!dW1) w1.m_tiles = 0;
  auto add_wgrad = [&](Params& Q, int first, int group) {
    Q.p[first] = w2;
    Q.p[first].group = group;
    Q.p[first + 1] = w1;
    Q.p[first + 1].group = group;
    for (int j = 0; j < 3; ++j) {
      maps.m[first][j] = map_w2[j];
      maps.m[first + 1][j] = map_w1[j];
    }
    Q.nprob = first + 2;
  };
  if (env.bwd_data_sms > 0 && nw > 0) {
    // Two CTA groups in one launch: env.bwd_data_sms SMs run act_grad and
    // input-grad, the others the weight gradients, trailing act_grad expert by
    // expert.
    add_wgrad(P, 2, 1);
    P.group_split = env.bwd_data_sms;
    return launch<CfgActGrad, CfgInGrad, CfgW2Grad, CfgW1Grad>(env, P, maps,
                                                              data_tiles + w_tiles, 1);
  }
  // Default: two launches.  The data gradients first; then the weight
  // gradients, whose per-expert waits are already satisfied: on CTA pairs
  // (2-SM MMAs) unless disabled, else on single CTAs.
  P.nprob = 2;
  rc = launch<CfgActGrad, CfgInGrad, CfgInGrad, CfgInGrad>(env, P, maps, data_tiles, 1);
  if (rc != HMM_OK || nw == 0) return rc;
  if (env.pair_wgrad)
    return launch_wgrad_pair(env, p, m, x_perm, dy_perm, dH, dH_lo, wa, wa_lo, dW1, dW2);
  Params W{};
  W.poff = m.poff;
  W.counts = m.counts;
  W.E = static_cast<int>(E);
  W.ticket = c.tickets + 3;
  add_wgrad(W, 0, 0);
  for (int q = 0; q < W.nprob; ++q) W.p[q].wait_e = nullptr;  // act_grad has completed
  return launch<CfgW2Grad, CfgW1Grad, CfgW1Grad, CfgW1Grad>(env, W, maps, w_tiles, 2);
}

}  // namespace hmm
