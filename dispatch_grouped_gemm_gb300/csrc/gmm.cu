// gmm.cu -- persistent grouped GEMM on sm_103a (TMA -> tcgen05.mma -> TMEM)
// with a per-expert tile scheduler and fused epilogues: the row-mode GEMMs of
// the fused MoE-FFN.
//
// [HyperMegaMoE §2.1 GMM1/up_proj -> SwiGLU -> GMM2/down_proj; §2.2 act_grad
// with SwiGLUGrad, input-grad GMM]:
//
//   out[rows of e] = T[rows of e] . W[e]
//
// T holds the expert's routed token rows in the padded row space (x_perm /
// dy_perm, written by the dispatch kernels, or a / dH, written by the GMM1 /
// act_grad epilogues); W is the expert's weight slab.  The MMA computes the
// transposed product, out^T = W^T . T^T: the weight columns sit on M (128 per
// CTA, the TMEM lanes) and the token rows on N (up to 256 per tile, the
// accumulator columns).  A tile's token block is cut at a multiple of 64 rows
// past the expert's last row, so an expert of 384 rows costs 256 + 128 rows of
// MMA work instead of four 128-row tiles.  (Gathering the token rows with TMA
// gather4 loads instead of a separate permute was measured about 3.5x slower
// per tile: 32 requests per K block.)  The weight gradients run in
// gmm_pair.cu.
//
// One launch holds up to four problems: a producer and a consumer problem for
// the routed experts [0, E) and, with the optional shared expert
// [HyperMegaMoE §6.1], the same pair for the shared expert, which is expert
// E of the padded row space (every token, routing weight 1) with its own
// weight slabs.  Tiles are handed out through a global atomic ticket in
// "schedule steps": step j holds, for every problem p, the tiles of expert
// j - lag_p (if it lies in p's expert range).  The consumer problems run
// behind every producer tile and wait on per-token-block ready counters that
// the producer's epilogues release [HyperMegaMoE §2.1: tasks split by
// token/expert tile, event counts release downstream tasks, no global
// barrier].  Every producer tile has a smaller ticket than its consumers, so
// it was already taken by a running CTA when a consumer spins: the wait
// cannot deadlock (and is bounded anyway).
//
// CTA = 7 warps: warp 6 schedules tiles (tickets, decoding, dependency waits,
// about one tile ahead), warp 0 issues TMA loads, warp 1 allocates TMEM and
// issues tcgen05.mma (one thread), warps 2..5 drain the accumulators (each
// owns the 32 TMEM lanes, i.e. weight columns, of its warp id mod 4).  Two
// 128 x 256 fp32 accumulators in TMEM (512 columns) let the epilogue of one
// tile overlap the MMAs of the next; 192 KB of shared-memory stages feed the
// MMAs.
//
// PAIR = true: clusters of two CTAs compute tiles of 256 weight columns with
// 2-SM MMAs (tcgen05.mma.cta_group::2): each CTA stages its own 128 weight
// columns and half of the token rows and drains its own 128 x N accumulator.
// Only the even CTA schedules; it writes each tile record into both CTAs'
// rings.
#include <cuda_bf16.h>

#include <algorithm>

#include "epilogue.cuh"
#include "ptx.cuh"

namespace hmm {

enum Epi : int { EPI_SWIGLU = 0, EPI_STORE = 1, EPI_DSWIGLU = 2 };

// Weight columns per CTA (the TMEM lanes), token rows per tile at most (the
// accumulator columns) and the granularity of a token block's end.
constexpr int BW = 128;
constexpr int NT = 256;

// EPI: epilogue; W_MN: weights MN-major (forward), else K-major (data
// gradients).  Token rows are K-major.  IDESC / IDESC2: instruction
// descriptors (1 CTA: M = 128; CTA pair: M = 256) without N, which each tile
// sets to its token rows.
template <int EPI_, bool W_MN_>
struct Cfg {
  static constexpr int EPI = EPI_;
  static constexpr bool W_MN = W_MN_;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BW, 0, W_MN ? 1 : 0, 0);
  static constexpr uint32_t IDESC2 = idesc_bf16_f32(2 * BW, 0, W_MN ? 1 : 0, 0);
  // output columns (SwiGLU: I columns, gate and up) of one CTA's 128 lanes
  static constexpr int WCOLS = EPI == EPI_SWIGLU ? BW / 2 : BW;
};
__host__ __device__ constexpr uint32_t idesc_n(int n) { return static_cast<uint32_t>(n >> 3) << 17; }

constexpr int STAGES = 4;
constexpr int W_BYTES = BW * BK * 2;  // 16 KB: 128 weight columns, 64 deep
constexpr int T_BYTES = NT * BK * 2;  // 32 KB: 256 token rows, 64 deep
constexpr int STAGE_BYTES = W_BYTES + T_BYTES;
// CTA pairs: each CTA stages its 128 weight columns and up to 128 of the
// token rows, 32 KB per K block, in six stages (the same 192 KB)
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_T_BYTES = (NT / 2) * BK * 2;  // 16 KB
constexpr int PAIR_STAGE_BYTES = W_BYTES + PAIR_T_BYTES;
// Small token blocks (routings of a few rows per expert, e.g. decode): single
// CTAs with blocks of at most 64 rows and eight 24 KB stages, so as many
// weight bytes are in flight per SM as with 256-row blocks (the weights are
// what such a launch streams).
constexpr int SMALL_NT = 64;
constexpr int SMALL_STAGES = 8;
constexpr int SMALL_T_BYTES = SMALL_NT * BK * 2;  // 8 KB
constexpr int SMALL_STAGE_BYTES = W_BYTES + SMALL_T_BYTES;
constexpr int MAX_STAGES = SMALL_STAGES;
static_assert(PAIR_STAGES * PAIR_STAGE_BYTES <= STAGES * STAGE_BYTES, "pair stages");
static_assert(SMALL_STAGES * SMALL_STAGE_BYTES <= STAGES * STAGE_BYTES, "small stages");
constexpr int TI_DEPTH = 3;
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 .. 1 + EW epilogue (EW = 4: one
// per TMEM lane quarter; EW = 8, the data-gradient launch: two per quarter,
// each with 16 rows of every chunk), 2 + EW tile scheduler.
constexpr int EPI_WARPS = 4;  // the four lane quarters (shared-memory buffers of all EW)
__host__ __device__ constexpr int gmm_threads(int ew) { return 32 * (ew + 3); }
constexpr int MAX_PROB = 4;
constexpr int MAX_STEPS = 2 * MAX_E + 8;
// alignment slack + stages + epilogue buffers + barriers, tile-info ring and
// schedule prefix table
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_WARPS * XBUF_BYTES + 512 +
                           4 * (MAX_STEPS + 1) + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 2 * NT;

struct Prob {
  int K;        // contraction length
  int N;        // valid output columns (SwiGLU / SwiGLU grad: I)
  int n_tiles;  // weight tiles along N (a CTA pair's tile spans both CTAs' columns)
  int half;     // SwiGLU: I (offset of the up half in the 2I operand/outputs)
  void* out;
  int64_t ld_out;
  void* out2;
  int64_t ld_out2;      // SwiGLU: column blocks of the blocked pre-activations
  void* out3;
  int64_t ld_out3;
  void* out4;           // SwiGLU grad: e5m2 low part of dH (ld_lo4 bytes per row)
  void* out5;           // SwiGLU grad: e5m2 low part of w*a (ld_lo5 bytes per row)
  int64_t ld_lo4, ld_lo5;
  int out_f32;          // STORE: fp32 outputs (else bf16)
  int lag;              // the tiles of expert e are issued at schedule step e + lag
  int e_lo, e_hi;       // experts of this problem; W holds experts e_lo .. e_hi - 1
  const void* aux;      // SwiGLU grad: the blocked fp32 pre-activations
  int64_t ld_aux;       // their column blocks per row block
  const float* rowscale;
  int* signal_m;        // per-token-block counters (index row0 / 64) released after a tile
  const int* wait_m;    // per-token-block counter acquired before a tile's loads
  int wait_unit;        // per-token-block target
  // the combine folded into this (GMM2) epilogue; cmb == null: a separate kernel
  int* cmb;                   // [T][cmb_nseg] rows counted per (token, 32-column segment)
  const int32_t* slot2prow;   // [T * K]
  const int32_t* prow2slot;   // [R]
  const int32_t* cmb_poff;    // padded offsets (the shared expert's rows start at [cmb_E])
  const void* cmb_w;          // topk_weights [T, K], bf16 or fp32 (cmb_w_f32)
  void* cmb_y;                // y [T, N] bf16
  int cmb_w_f32, cmb_K, cmb_KS, cmb_T, cmb_nseg, cmb_E;
};

struct Params {
  Prob p[MAX_PROB];
  int nprob;
  int pair;             // CTA pairs: a tile spans 256 weight columns
  int nt;               // token rows per block at most (256, or 64 in small mode)
  int steps;            // E + largest lag
  const int32_t* poff;
  const int32_t* counts;
  int E;
  int* ticket;
  unsigned* status;
  unsigned long long budget_ns;
  uint64_t* trace;      // per-tile timeline records (null: off)
  int trace_cap;
};

// Token-row maps by block size: t[q][i] loads the token rows of a block of
// 64 (i + 1) rows, in one box per CTA (pairs: the CTA's half, 32 (i + 1)
// rows; single CTAs: all of them; small blocks: i = 0 only).
constexpr int TOK_MAPS = NT / TROWS;
struct Maps {
  CUtensorMap w[MAX_PROB];            // weights
  CUtensorMap t[MAX_PROB][TOK_MAPS];  // token rows
};

struct TileInfo {
  int prob;   // -1: no more tiles
  int e;
  int row0;   // first padded row of the token block (a multiple of 64)
  int nrow;   // token rows of the block: 64 .. 256, a multiple of 64
  int w0;     // first output column of the tile (of the even CTA in a pair)
  int kb;     // K blocks
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
// Token blocks of expert e: 256 rows each, the last one ending at the first
// multiple of 64 rows at or past the expert's last row.
__device__ __forceinline__ int nblocks_of(const Params& P, int e) {
  return (P.counts[e] + P.nt - 1) / P.nt;
}

__device__ __forceinline__ int tiles_of(const Params& P, const Prob& pr, int e) {
  if (e < pr.e_lo || e >= pr.e_hi) return 0;
  return nblocks_of(P, e) * pr.n_tiles;
}

// Prefix sums of the tile counts of the schedule steps (one warp, into smem).
__device__ void build_schedule(const Params& P, int* pref) {
  const int lane = threadIdx.x & 31;
  const int steps = P.steps;
  int carry = 0;
  if (lane == 0) pref[0] = 0;
  for (int base = 0; base < steps; base += 32) {
    const int j = base + lane;
    int v = 0;
    if (j < steps)
      for (int q = 0; q < P.nprob; ++q) v += tiles_of(P, P.p[q], j - P.p[q].lag);
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

// Ticket t -> (problem, expert, local tile index).  Returns false past the end.
__device__ bool locate_tile(const Params& P, const int* pref, int t, int& prob, int& e, int& r) {
  const int steps = P.steps;
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
  const int nb = nblocks_of(P, e);
  const int wt = r / nb;  // token blocks innermost: a weight tile is reused from L2
  const int b = r - wt * nb;
  const int rows = (P.counts[e] + TROWS - 1) / TROWS * TROWS;
  // the expert's rows in nb blocks of equal size (a multiple of 64, the last
  // one shorter): 384 rows as 192 + 192, not 256 + 128.  A tile's MMAs take
  // about as long for any block size, its SwiGLU-grad epilogue in proportion
  // to the rows, so even blocks keep that epilogue under the MMAs.
  const int nt = (rows / nb + TROWS - 1) / TROWS * TROWS;
  ti.row0 = P.poff[e] + nt * b;
  ti.nrow = min(nt, rows - nt * b);
  ti.w0 = wt * C::WCOLS * (P.pair ? 2 : 1);
  ti.kb = (pr.K + BK - 1) / BK;
}

// ----------------------------------------------------------------- producer
// K block kb of a tile into one smem stage (one thread): this CTA's 128 weight
// columns (sW) and the tile's token rows (sT).  Every box starts at an inner
// coordinate that is a multiple of 8 elements (16 bytes).
//   PAIR: this CTA's share (its weight columns, its half of the token rows),
//   counted on the even CTA's full barrier (shared::cluster address bar_cl;
//   the even CTA arms it for both).  The token rows come in one box of exactly
//   the rows the MMA reads (tT: the map of this block size).  Returns the
//   bytes this CTA loads.
template <class C, bool PAIR, bool SMALL>
__device__ __forceinline__ uint32_t load_stage(const Prob& pr, const TileInfo& ti, int kb,
                                               const CUtensorMap* tT, const CUtensorMap* tW,
                                               uint8_t* sW, uint8_t* sT, uint64_t* bar,
                                               uint32_t bar_cl, uint32_t rank) {
  const int k = kb * BK;
  const int eb = ti.e - pr.e_lo;  // expert index inside this problem's weight slabs
  const int wc = ti.w0 + C::WCOLS * static_cast<int>(rank);  // this CTA's first column
  if constexpr (PAIR) {
    const uint32_t bytes = W_BYTES + (ti.nrow / 2) * BK * 2;
    if (rank == 0) mbar_arrive_expect_tx(bar, 2 * bytes);
    if constexpr (C::W_MN) {
      // SwiGLU: 64 gate columns, then the same 64 up columns
      const int c2 = C::EPI == EPI_SWIGLU ? pr.half + wc : wc + 64;
      tma_load_3d_pair(sW, tW, bar_cl, wc, k, eb);
      tma_load_3d_pair(sW + 8192, tW, bar_cl, c2, k, eb);
    } else {
      tma_load_3d_pair(sW, tW, bar_cl, k, wc, eb);
    }
    tma_load_2d_pair(sT, tT, bar_cl, k, ti.row0 + (ti.nrow / 2) * static_cast<int>(rank));
    return bytes;
  } else {
    // one box of the block's rows (small mode: 64)
    const uint32_t bytes = W_BYTES + ti.nrow * BK * 2;
    mbar_arrive_expect_tx(bar, bytes);
    if constexpr (C::W_MN) {
      const int c2 = C::EPI == EPI_SWIGLU ? pr.half + wc : wc + 64;
      tma_load_3d(sW, tW, bar, wc, k, eb);
      tma_load_3d(sW + 8192, tW, bar, c2, k, eb);
    } else {
      tma_load_3d(sW, tW, bar, k, wc, eb);
    }
    tma_load_2d(sT, tT, bar, k, ti.row0);
    return bytes;
  }
}

// ---------------------------------------------------------------------- MMA
// Weights: MN-major (two 64-column chunks 8 KB apart, 8-row groups 1 KB,
// 2 KB per 16-deep step) or K-major; token rows K-major.
template <class C, bool PAIR>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t w_base, uint32_t t_base,
                                          uint32_t idesc, bool first) {
#pragma unroll
  for (int kk = 0; kk < BK / 16; ++kk) {
    const uint64_t ad = C::W_MN ? smem_desc(w_base + kk * 2048, 8192, 1024, LAYOUT_SW128)
                                : smem_desc(w_base + kk * 32, 16, 1024, LAYOUT_SW128);
    const uint64_t bd = smem_desc(t_base + kk * 32, 16, 1024, LAYOUT_SW128);
    if constexpr (PAIR)
      umma_bf16_pair(d_tmem, ad, bd, idesc, (first && kk == 0) ? 0u : 1u);
    else
      umma_bf16(d_tmem, ad, bd, idesc, (first && kk == 0) ? 0u : 1u);
  }
}

// ----------------------------------------------------------------- epilogue
// sigma(g) = 1 / (1 + exp(-g)) with the fast exponential and division
// intrinsics (a few ulp in fp32, far inside the bf16 output rounding).
// For g -> -inf the denominator overflows to inf and the quotient is 0.
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_f(float g) { return g * sigmoid_f(g); }

// v ~ hi + lo with hi = bf16(v) and lo = e5m2(v - hi): the weight-gradient
// GEMMs take hi in a bf16 MMA and lo, at most 2^-9 |v| and needed only to a
// few bits, in an fp8 MMA against an fp8 copy of the other operand (e5m2
// keeps lo's small magnitudes in range).
__device__ __forceinline__ void store_bf16x8_split(__nv_bfloat16* hi, uint8_t* lo,
                                                   const float* v) {
  float h[8], l[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
    l[j] = v[j] - h[j];
  }
  *reinterpret_cast<uint4*>(hi) = pack_bf16x8(h);
  *reinterpret_cast<uint2*>(lo) = pack_fp8x8<true>(l);
}

// The fp32 pre-activations saved for the backward are stored in 32 x 32
// blocks: block (row / 32, col / 32) of the gate half followed by the same
// block of the up half, 8 KB contiguous, blocks ordered by row block, then
// column block (ncb = ceil(I / 32) per row block).  The forward epilogue
// writes, and the SwiGLU-grad epilogue reads, exactly these blocks (a 32-row
// TMEM lane quarter times a 32-column chunk), so both move 8 KB runs instead
// of 128-byte pieces of rows 2I floats apart.
__device__ __forceinline__ int64_t hblock_offset(int64_t row, int col, int64_t ncb) {
  return (((row >> 5) * ncb + (col >> 5)) << 11) + ((row & 31) << 5) + (col & 31);
}

__device__ __forceinline__ void store_f32x8(float* dst, const float* v) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// State an epilogue warp carries from tile to tile.  The SwiGLU epilogue
// pairs the gate lane quarter g (0, 1) with the up quarter g + 2: both stage
// their transposed 32 x 32 block in shared memory and each then reads both
// blocks for half of the rows; xfull / xfree (two arrivals each) order the
// exchange, one phase per chunk.
struct EpiState {
  int q;            // TMEM lane quarter of this warp
  int lane;
  int hoff;         // eight epilogue warps: the warp's 16 rows of each 32-row chunk (0, 16)
  float* own;       // this warp's transposition buffer
  float* xbufs;     // the four quarters' transposition buffers
  uint64_t* xfull;  // [2], per gate quarter
  uint64_t* xfree;  // [2]
  uint32_t nchunk;  // chunks exchanged so far (SwiGLU)
};

// lane 0 waits (bounded) on bar's phase `parity`; every lane gets the result
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane,
                                          const WaitCtl& wc) {
  bool ok = false;
  if (lane == 0) ok = mbar_wait(bar, parity, wc);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0);
}

// Drains the accumulator of one tile: TMEM lanes of quarter q are the output
// columns c0 .. c0 + 31 (c0 = first column of this CTA + 32 q; SwiGLU: the I
// columns of the gate / up quarter pair), TMEM columns 32 j .. 32 j + 31 the
// token rows row0 + 32 j .. of chunk j.  Each chunk goes through the
// transposition buffer, after which lane l holds columns 8 (l & 3) .. + 7 of
// the rows (l >> 2) + 8 k.  Column chunks are skipped per lane with plain
// conditionals, never an early exit: the next chunk's TMEM load is a
// warp-wide instruction.  ok turns false when a bounded wait gave up.
//   EW = 8 (two warps per lane quarter; STORE and SwiGLU grad only): each
// warp takes 16 rows of every chunk (es.hoff), through a 16-row buffer, and
// lane l holds columns 8 (l & 3) .. + 7 of the rows (l >> 2) + 8 k, k < 2.
template <class C, int EW>
__device__ __forceinline__ void epilogue_tile(const Prob& pr, const TileInfo& ti, uint32_t taddr,
                                              uint32_t rank, EpiState& es, const WaitCtl& wc,
                                              bool& ok) {
  static_assert(EW == 4 || (EW == 8 && C::EPI != EPI_SWIGLU), "epilogue warps");
  constexpr int KR = EW == 8 ? 2 : 4;  // rows per lane and chunk
  const int cta_col0 = ti.w0 + C::WCOLS * static_cast<int>(rank);
  const int lane = es.lane;
  const int q = es.q;
  const int hoff = EW == 8 ? es.hoff : 0;
  const int cg = (lane & 3) * 8;  // this lane's first column within a 32-column block
  const int nch = ti.nrow / 32;
  float* own = es.own;
  // this warp's rows of chunk j from TMEM, transposed: v[k] = row (l >> 2) + 8 k
  auto load_chunk = [&](int j, float (&v)[KR][8]) {
    if constexpr (EW == 8) {
      uint32_t r[16];
      tmem_ld16(taddr + j * 32 + hoff, r);
      tmem_ld_wait();
      xwrite_t16(own, lane, r);
      __syncwarp();
      xread16(own, lane, v);
    } else {
      uint32_t r[32];
      tmem_ld32(taddr + j * 32, r);
      tmem_ld_wait();
      xwrite_t(own, lane, r);
      __syncwarp();
      xread(own, lane, v);
    }
    __syncwarp();
  };
  if constexpr (C::EPI == EPI_SWIGLU) {
    // a = silu(gate) * up of I columns c .. c + 7; training also saves the
    // fp32 pre-activations (blocked layout)
    const int gq = q & 1;
    const float* gbuf = es.xbufs + gq * (XBUF_BYTES / 4);
    const float* ubuf = es.xbufs + (gq + 2) * (XBUF_BYTES / 4);
    const int kh = q < 2 ? 0 : 2;  // gate quarter: rows k = 0, 1 of a chunk; up quarter: 2, 3
    const int c = cta_col0 + 32 * gq + cg;
#pragma unroll 1
    for (int j = 0; j < nch; ++j) {
      uint32_t r[32];
      tmem_ld32(taddr + j * 32, r);
      tmem_ld_wait();
      const uint32_t ph = es.nchunk & 1u;
      // the partner has read the previous chunk out of this buffer
      if (!warp_wait(&es.xfree[gq], ph ^ 1u, lane, wc)) {
        ok = false;
        return;
      }
      xwrite_t(own, lane, r);
      __syncwarp();
      if (lane == 0) mbar_arrive(&es.xfull[gq]);
      if (!warp_wait(&es.xfull[gq], ph, lane, wc)) {
        ok = false;
        return;
      }
      const float* gs = gbuf + (lane >> 2) * XS + cg;
      const float* us = ubuf + (lane >> 2) * XS + cg;
      float gv[2][8], uv[2][8];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int o = (kh + kk) * 8 * XS;
        const float4 g0 = *reinterpret_cast<const float4*>(gs + o);
        const float4 g1 = *reinterpret_cast<const float4*>(gs + o + 4);
        const float4 u0 = *reinterpret_cast<const float4*>(us + o);
        const float4 u1 = *reinterpret_cast<const float4*>(us + o + 4);
        gv[kk][0] = g0.x; gv[kk][1] = g0.y; gv[kk][2] = g0.z; gv[kk][3] = g0.w;
        gv[kk][4] = g1.x; gv[kk][5] = g1.y; gv[kk][6] = g1.z; gv[kk][7] = g1.w;
        uv[kk][0] = u0.x; uv[kk][1] = u0.y; uv[kk][2] = u0.z; uv[kk][3] = u0.w;
        uv[kk][4] = u1.x; uv[kk][5] = u1.y; uv[kk][6] = u1.z; uv[kk][7] = u1.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&es.xfree[gq]);
      ++es.nchunk;
      if (c < pr.N) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int64_t row = ti.row0 + 32 * j + (lane >> 2) + 8 * (kh + kk);
          float av[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) av[i] = silu_f(gv[kk][i]) * uv[kk][i];
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(pr.out) + row * pr.ld_out + c) =
              pack_bf16x8(av);
          if (pr.out2) {
            float* hp = static_cast<float*>(pr.out2) + hblock_offset(row, c, pr.ld_out2);
            store_f32x8(hp, gv[kk]);
            store_f32x8(hp + 1024, uv[kk]);
          }
        }
      }
    }
  } else if constexpr (C::EPI == EPI_STORE) {
    const int c = cta_col0 + 32 * q + cg;
#pragma unroll 1
    for (int j = 0; j < nch; ++j) {
      float v[KR][8];
      load_chunk(j, v);
      if (c < pr.N) {
#pragma unroll
        for (int k = 0; k < KR; ++k) {
          const int64_t row = ti.row0 + 32 * j + hoff + (lane >> 2) + 8 * k;
          if (pr.out_f32)
            store_f32x8(static_cast<float*>(pr.out) + row * pr.ld_out + c, v[k]);
          else
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(pr.out) + row * pr.ld_out + c) =
                pack_bf16x8(v[k]);
        }
      }
    }
  } else {  // EPI_DSWIGLU
    // acc = G^T, G = dy_perm . W2^T for I columns c0 .. c0 + 31.  With the
    // saved fp32 pre-activations g, u and the slot's routing weight w:
    //   a = silu(g) u,  dA = w G,
    //   dgate = dA u s (1 + g (1 - s)),  dup = dA g s     (s = sigmoid(g))
    // writes dH = [dgate | dup] and wa = w a (the W2Grad operand), each as
    // a bf16 high part and an e5m2 low part, and the partial
    // d_w = sum_j G_j a_j over these 32 columns (fp32).  The pre-activations
    // and routing weights of the next chunk are loaded while the current one
    // is computed.
    const float* hb = static_cast<const float*>(pr.aux);
    const int c0 = cta_col0 + 32 * q;
    const int c = c0 + cg;
    const bool colok = c < pr.N;
    float4 gn[KR][2], un[KR][2];
    float wn[KR];
    auto load_h = [&](int j) {
#pragma unroll
      for (int k = 0; k < KR; ++k) {
        const int64_t row = ti.row0 + 32 * j + hoff + (lane >> 2) + 8 * k;
        const float4* p = reinterpret_cast<const float4*>(hb + hblock_offset(row, c, pr.ld_aux));
        const float4* pu = p + 256;  // the up block follows the gate block
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        gn[k][0] = colok ? __ldg(p) : z;
        gn[k][1] = colok ? __ldg(p + 1) : z;
        un[k][0] = colok ? __ldg(pu) : z;
        un[k][1] = colok ? __ldg(pu + 1) : z;
        wn[k] = __ldg(pr.rowscale + row);
      }
    };
    // the 8 KB block (gate, then up) of the chunk PF_H ahead into L2: two
    // 128-byte lines per lane, no registers held (the loads of the next
    // chunk are all the registers allow)
    auto prefetch_h = [&](int j) {
      const int64_t row = ti.row0 + 32 * j;
      const char* blk = reinterpret_cast<const char*>(hb + hblock_offset(row, c0, pr.ld_aux));
      if constexpr (EW == 8) {
        // this warp's 16 rows: lanes 0-15 the gate lines, 16-31 the up lines
        asm volatile("prefetch.global.L2 [%0];" ::"l"(blk + (lane >> 4) * 4096 +
                                                       (hoff + (lane & 15)) * 128));
      } else {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(blk + lane * 128));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(blk + 4096 + lane * 128));
      }
    };
    constexpr int PF_H = 2;
    load_h(0);
    if (c0 < pr.N)
      for (int j = 1; j < PF_H && j < nch; ++j) prefetch_h(j);
#pragma unroll 1
    for (int j = 0; j < nch; ++j) {
      if (j + PF_H < nch && c0 < pr.N) prefetch_h(j + PF_H);
      float gv[KR][8], uv[KR][8], w[KR];
#pragma unroll
      for (int k = 0; k < KR; ++k) {
        gv[k][0] = gn[k][0].x; gv[k][1] = gn[k][0].y; gv[k][2] = gn[k][0].z; gv[k][3] = gn[k][0].w;
        gv[k][4] = gn[k][1].x; gv[k][5] = gn[k][1].y; gv[k][6] = gn[k][1].z; gv[k][7] = gn[k][1].w;
        uv[k][0] = un[k][0].x; uv[k][1] = un[k][0].y; uv[k][2] = un[k][0].z; uv[k][3] = un[k][0].w;
        uv[k][4] = un[k][1].x; uv[k][5] = un[k][1].y; uv[k][6] = un[k][1].z; uv[k][7] = un[k][1].w;
        w[k] = wn[k];
      }
      if (j + 1 < nch) load_h(j + 1);
      float Gv[KR][8];
      load_chunk(j, Gv);
      float dwp[KR];
#pragma unroll
      for (int k = 0; k < KR; ++k) {
        const int64_t row = ti.row0 + 32 * j + hoff + (lane >> 2) + 8 * k;
        float dg[8], du[8], wa[8];
        dwp[k] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float G = Gv[k][i], g = gv[k][i], u = uv[k][i];
          const float sg = sigmoid_f(g);
          const float a = g * sg * u;
          dwp[k] = fmaf(G, a, dwp[k]);
          const float dA = w[k] * G;
          dg[i] = dA * u * sg * (1.0f + g * (1.0f - sg));
          du[i] = dA * g * sg;
          wa[i] = w[k] * a;
        }
        if (colok) {
          __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(pr.out) + row * pr.ld_out + c;
          uint8_t* dl = static_cast<uint8_t*>(pr.out4) + row * pr.ld_lo4 + c;
          store_bf16x8_split(dh, dl, dg);
          store_bf16x8_split(dh + pr.half, dl + pr.half, du);
          store_bf16x8_split(static_cast<__nv_bfloat16*>(pr.out2) + row * pr.ld_out2 + c,
                             static_cast<uint8_t*>(pr.out5) + row * pr.ld_lo5 + c, wa);
        }
      }
      // one partial per (row, 32-column block): the four lanes of a row add
      // theirs in a fixed tree, the combine sums the blocks in order
#pragma unroll
      for (int k = 0; k < KR; ++k) {
        dwp[k] += __shfl_xor_sync(0xffffffffu, dwp[k], 1);
        dwp[k] += __shfl_xor_sync(0xffffffffu, dwp[k], 2);
      }
      if (cg == 0 && c0 < pr.N) {
#pragma unroll
        for (int k = 0; k < KR; ++k) {
          const int64_t row = ti.row0 + 32 * j + hoff + (lane >> 2) + 8 * k;
          static_cast<float*>(pr.out3)[row * pr.ld_out3 + c0 / 32] = dwp[k];
        }
      }
    }
  }
}

// ------------------------------------------------------------ fused combine
// The combine folded into the GMM2 epilogue [HyperMegaMoE §6.2: unpermute and
// top-k weighted merge inside the fused operator; MoE overlap explainer §6:
// a token is published once all of its branches have arrived].  After a warp
// has stored its 32 columns (segment c0 / 32) of o for the token block of a
// tile, it counts each routed row on its token's counter of that segment;
// the count that completes the token's KS rows (K, plus the shared expert's
// row) makes this warp the owner of the token's segment, and it sums those
// rows and writes y.  The sum is the separate combine's, operation for
// operation: fp32 fmaf over k = 0 .. K-1 in order with the routing weight
// (slots with an invalid id skipped), then the shared row with weight 1, one
// bf16 rounding.  Every request is issued in batches (all rows' counts at
// once; per token, the rows of four slots at once): each step is one round
// trip to L2, not one per row.

// One token's segment: y[t][c0 .. c0 + 31] (columns below N).
template <bool F32>
__device__ __forceinline__ void finish_token(const Prob& pr, int t, int c0) {
  constexpr int VPR = F32 ? 8 : 4;  // 16-byte vectors per row of 32 columns
  constexpr int KB = F32 ? 2 : 4;   // slots whose rows are loaded together
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
  const int K = pr.cmb_K;
  const int ncv = min(32, pr.N - c0) / 8;  // 8-column groups inside N
  auto add_rows = [&](const int32_t (&pk)[KB], const float (&wk)[KB]) {
    uint4 v[KB][VPR];
#pragma unroll
    for (int j = 0; j < KB; ++j)
#pragma unroll
      for (int q = 0; q < VPR; ++q) {
        v[j][q] = make_uint4(0, 0, 0, 0);
        if (pk[j] >= 0 && q < (F32 ? 2 * ncv : ncv)) {
          const uint8_t* base = static_cast<const uint8_t*>(pr.out) +
                                (static_cast<int64_t>(pk[j]) * pr.ld_out + c0) * (F32 ? 4 : 2);
          v[j][q] = __ldcg(reinterpret_cast<const uint4*>(base) + q);
        }
      }
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      if (pk[j] < 0) continue;
      const float s = wk[j];
#pragma unroll
      for (int q = 0; q < VPR; ++q) {
        const uint32_t u[4] = {v[j][q].x, v[j][q].y, v[j][q].z, v[j][q].w};
        if constexpr (F32) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[4 * q + i] = fmaf(s, __uint_as_float(u[i]), acc[4 * q + i]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[8 * q + 2 * i] = fmaf(s, bf16_lo(u[i]), acc[8 * q + 2 * i]);
            acc[8 * q + 2 * i + 1] = fmaf(s, bf16_hi(u[i]), acc[8 * q + 2 * i + 1]);
          }
        }
      }
    }
  };
  for (int k0 = 0; k0 < K; k0 += KB) {
    int32_t pk[KB];
    float wk[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int k = k0 + j;
      pk[j] = -1;
      wk[j] = 0.0f;
      if (k < K) {
        const int64_t sk = static_cast<int64_t>(t) * K + k;
        pk[j] = pr.slot2prow[sk];
        wk[j] = pr.cmb_w_f32 ? static_cast<const float*>(pr.cmb_w)[sk]
                             : bf16_lo(static_cast<const uint16_t*>(pr.cmb_w)[sk]);
      }
    }
    add_rows(pk, wk);
  }
  if (pr.cmb_KS > K) {
    int32_t pk[KB];
    float wk[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      pk[j] = j == 0 ? pr.cmb_poff[pr.cmb_E] + t : -1;
      wk[j] = 1.0f;
    }
    add_rows(pk, wk);
  }
  __nv_bfloat16* yr = static_cast<__nv_bfloat16*>(pr.cmb_y) + static_cast<int64_t>(t) * pr.N + c0;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (q < ncv) reinterpret_cast<uint4*>(yr)[q] = pack_bf16x8(acc + 8 * q);
}

// list: this warp's shared-memory scratch (NT ints).
template <bool F32>
__device__ __noinline__ void combine_tile(const Prob& pr, const TileInfo& ti, int c0, int lane,
                                          int* list) {
  if (c0 >= pr.N) return;
  const int seg = c0 >> 5;
  const bool shared = ti.e == pr.cmb_E;
  const int64_t srow0 = shared ? pr.cmb_poff[pr.cmb_E] : 0;
  // this warp's stores of o are visible at gpu scope before its counts
  __threadfence();
  __syncwarp();
  // every row of the block at once (lane l: rows l, l + 32, ...)
  constexpr int MAXG = NT / 32;
  int tk[MAXG], old[MAXG];
#pragma unroll
  for (int i = 0; i < MAXG; ++i) {
    tk[i] = -1;
    if (32 * i < ti.nrow) {
      const int64_t prow = ti.row0 + 32 * i + lane;
      if (shared) {
        if (prow - srow0 < pr.cmb_T) tk[i] = static_cast<int>(prow - srow0);
      } else {
        const int32_t sl = pr.prow2slot[prow];
        if (sl >= 0) tk[i] = sl / pr.cmb_K;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < MAXG; ++i)
    old[i] = tk[i] >= 0 ? atomicAdd(&pr.cmb[static_cast<int64_t>(tk[i]) * pr.cmb_nseg + seg], 1)
                        : -1;
  // the tokens whose segment this warp completed, compacted
  int nfin = 0;
#pragma unroll
  for (int i = 0; i < MAXG; ++i) {
    const bool f = old[i] == pr.cmb_KS - 1;
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (f) list[nfin + __popc(m & ((1u << lane) - 1u))] = tk[i];
    nfin += __popc(m);
  }
  if (nfin == 0) return;
  __syncwarp();
  __threadfence();  // the other rows of the completed segments, written by other warps
  for (int b = 0; b < nfin; b += 32)
    if (b + lane < nfin) finish_token<F32>(pr, list[b + lane], c0);
  __syncwarp();
}

// ------------------------------------------------------------------- kernel
// Problems 0 and 2 share configuration C0 (producers: GMM1, act_grad),
// problems 1 and 3 C1 (consumers: GMM2, input-grad); 2 and 3 are the shared
// expert's.
#define HMM_BY_PROB(q, F, ...)   \
  if (((q) & 1) == 0) {          \
    F<C0>(__VA_ARGS__);          \
  } else {                       \
    F<C1>(__VA_ARGS__);          \
  }
#define HMM_BY_PROB_P(q, F, ...)  \
  if (((q) & 1) == 0) {           \
    F<C0, PAIR>(__VA_ARGS__);     \
  } else {                        \
    F<C1, PAIR>(__VA_ARGS__);     \
  }
template <bool PAIR, bool SMALL, int EW, class C0, class C1>
__global__ void __launch_bounds__(gmm_threads(EW), 1)
    gmm_kernel(const __grid_constant__ Params P, const __grid_constant__ Maps maps) {
  static_assert(!(PAIR && SMALL), "small token blocks run on single CTAs");
  static_assert(EW == 4 || EW == 8, "epilogue warps");
  static_assert(EW * XBUF_HALF <= EPI_WARPS * XBUF_BYTES, "transposition buffers");
  constexpr int SCHED_WARP = 2 + EW;
  constexpr int NST = PAIR ? PAIR_STAGES : (SMALL ? SMALL_STAGES : STAGES);
  constexpr int SBYTES = PAIR ? PAIR_STAGE_BYTES : (SMALL ? SMALL_STAGE_BYTES : STAGE_BYTES);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  float* xbufs = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + EPI_WARPS * XBUF_BYTES);
  uint64_t* full = bars;                    // [NST]; in a pair: the even CTA's counts both CTAs
  uint64_t* empty = bars + MAX_STAGES;      // [NST]
  uint64_t* tfull = bars + 2 * MAX_STAGES;  // [2]
  uint64_t* tempty = tfull + 2;             // [2]; in a pair: the even CTA's, both CTAs arrive
  uint64_t* ti_full = tempty + 2;
  uint64_t* ti_empty = ti_full + TI_DEPTH;  // in a pair: the even CTA's, both CTAs arrive
  uint64_t* mma_done = ti_empty + TI_DEPTH;
  uint64_t* xfull = mma_done + 1;           // [2] SwiGLU epilogue exchange
  uint64_t* xfree = xfull + 2;              // [2]
  TileInfo* s_ti = reinterpret_cast<TileInfo*>(xfree + 2);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_ti + TI_DEPTH);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 2;  // K blocks this CTA's producer issued
  uint32_t* s_sbytes = s_tmem + 3;  // [MAX_STAGES] bytes of this CTA's last loads per slot
  // [2 + MAX_STAGES] even CTA of a pair: the odd CTA's count, abort flag, bytes per slot
  uint32_t* s_peer = s_sbytes + MAX_STAGES;
  int* s_pref = reinterpret_cast<int*>(s_peer + 2 + MAX_STAGES);  // [steps + 1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 2 * EW : EW);
    }
    for (int i = 0; i < TI_DEPTH; ++i) {
      mbar_init(&ti_full[i], 1);
      // consumers: TMA producer, MMA issuer, epilogue warps (+ the odd CTA's
      // producer and epilogue warps in a pair)
      mbar_init(&ti_empty[i], PAIR ? 2 * (1 + EW) + 1 : 2 + EW);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xfull[i], 2);
      mbar_init(&xfree[i], 2);
    }
    *s_abort = 0;
    *s_issued = 0;
    for (int i = 0; i < 2 + MAX_STAGES; ++i) s_peer[i] = 0;
    for (int i = 0; i < MAX_STAGES; ++i) s_sbytes[i] = 0;
    fence_mbar_init();
  }
  if constexpr (PAIR) cluster_sync_all();  // barriers initialised before any remote arrive
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(s_tmem, TMEM_COLS);  // collective: one warp in each CTA of the pair
      tmem_relinquish_pair();
    } else {
      tmem_alloc(s_tmem, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  // set-up done: from here on global memory (routing metadata, operands,
  // counters) that the stream's previous kernel may still be writing.  (The
  // next kernel is let in only when this CTA's producer has issued its last
  // tile: its CTAs would otherwise wait beside this launch for all of it.)
  grid_dep_wait();
  const WaitCtl wc{s_abort, P.status, P.budget_ns};
  // in a pair the odd CTA's consumers release the even CTA's tile-info slots
  auto ti_release = [&](int slot) {
    if (!PAIR || leader)
      mbar_arrive(&ti_empty[slot]);
    else
      mbar_arrive_peer(mapa_shared(smem_u32(&ti_empty[slot]), 0));
  };

  if (warp == SCHED_WARP) {
    // --------------------------------------------------------- tile scheduler
    // Fetches tickets, decodes them and waits for each tile's dependencies
    // about one tile ahead of the TMA producer, so neither the ticket atomic
    // nor a ready-counter poll sits on the load path.  (A deeper lookahead
    // spreads the token blocks that share a weight tile over time and costs
    // L2 reuse of the weights.)  Lane 0 does the bookkeeping.  In a pair only
    // the even CTA schedules; it writes each tile into both CTAs' rings.
    if (!PAIR || leader) {
      build_schedule(P, s_pref);
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      int lt = 0;  // tiles of this CTA so far (trace index)
      int t = 0;
      if (lane == 0) t = atomicAdd(P.ticket, 1);
      for (;;) {
        TileInfo ti;
        ti.prob = -1;
        ti.e = ti.row0 = ti.nrow = ti.w0 = ti.kb = 0;
        bool ok = true;
        if (lane == 0) {
          int q = 0, e = 0, r = 0;
          if (locate_tile(P, s_pref, t, q, e, r)) {
            ti.prob = q;
            HMM_BY_PROB(q, decode_tile, P, P.p[q], e, r, ti);
            t = atomicAdd(P.ticket, 1);  // next ticket, early
            const Prob& pr = P.p[q];
            if (pr.wait_m) ok = counter_wait(&pr.wait_m[ti.row0 / TROWS], pr.wait_unit, wc);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        // every lane leaves the loop with lane 0 (end marker below)
        ti.prob = __shfl_sync(0xffffffffu, ti.prob, 0);
        bool got = false;
        if (lane == 0) got = mbar_wait<PAIR>(&ti_empty[ti_slot], ti_phase ^ 1u, wc);
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
          if constexpr (PAIR) {
            const uint32_t dst = mapa_shared(smem_u32(&s_ti[ti_slot]), 1);
            const int* src = reinterpret_cast<const int*>(&ti);
#pragma unroll
            for (int j = 0; j < static_cast<int>(sizeof(TileInfo) / 4); ++j)
              st_shared_cluster(dst + 4 * j, src[j]);
            mbar_arrive_cluster(mapa_shared(smem_u32(&ti_full[ti_slot]), 1));
          }
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
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- TMA producer
      for (int q = 0; q < P.nprob; ++q) tma_prefetch_desc(&maps.w[q]);
      uint32_t stage = 0, sphase = 0;
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      uint32_t issued = 0;  // k-blocks issued by this CTA
      bool ok = true;
      int lt = 0;
      for (;;) {
        if (!mbar_wait<PAIR>(&ti_full[ti_slot], ti_phase, wc)) {
          ok = false;
          break;
        }
        const TileInfo ti = s_ti[ti_slot];
        ti_release(ti_slot);
        if (++ti_slot == TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (ti.prob < 0) break;
        const Prob& pr = P.p[ti.prob];
        // the scheduler acquired this tile's ready counter (gpu scope) before
        // publishing it; order that with the async-proxy loads below
        if (pr.wait_m) fence_proxy_async_global();
        const CUtensorMap* tW = &maps.w[ti.prob];
        const CUtensorMap* tT = &maps.t[ti.prob][ti.nrow / TROWS - 1];
        uint64_t* rec = (!PAIR || leader) ? trace_rec(P, lt) : nullptr;
        ++lt;
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!mbar_wait(&empty[stage], sphase ^ 1u, wc)) {
            ok = false;
            break;
          }
          if (rec && kb == 0) rec[2] = globaltimer_ns();
          uint8_t* sW = stages + stage * SBYTES;
          const uint32_t full_cl = PAIR ? mapa_shared(smem_u32(&full[stage]), 0) : 0u;
          uint32_t bytes = 0;
          if ((ti.prob & 1) == 0)
            bytes = load_stage<C0, PAIR, SMALL>(pr, ti, kb, tT, tW, sW, sW + W_BYTES,
                                                &full[stage], full_cl, rank);
          else
            bytes = load_stage<C1, PAIR, SMALL>(pr, ti, kb, tT, tW, sW, sW + W_BYTES,
                                                &full[stage], full_cl, rank);
          s_sbytes[stage] = bytes;
          ++issued;
          if (++stage == NST) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (rec && ok) rec[3] = globaltimer_ns();
        if (!ok) break;
      }
      // wait (bounded) for the copies still in flight before leaving (CTA
      // pairs: both CTAs' copies, at teardown, see pair_teardown)
      if (!PAIR && !ok)
        for (uint32_t s = 0; s < NST; ++s)
          if (issued > s) drain_wait(&full[s], ((issued - 1 - s) / NST) & 1u, P.budget_ns);
      *s_issued = issued;
      grid_dep_launch();  // this CTA is in its last tile
    }
  } else if (warp == 1) {
    if (lane == 0 && (!PAIR || leader)) {
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
        if (!mbar_wait<PAIR>(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        if (rec) rec[4] = globaltimer_ns();
        const uint32_t d_tmem = tmem_base + acc * NT;
        uint32_t idesc = idesc_n(ti.nrow);  // N = the tile's token rows
        if (ti.prob & 1)
          idesc |= PAIR ? C1::IDESC2 : C1::IDESC;
        else
          idesc |= PAIR ? C0::IDESC2 : C0::IDESC;
        bool ok = true;
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!mbar_wait(&full[stage], sphase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w_base = smem_u32(stages + stage * SBYTES);
          const uint32_t t_base = w_base + W_BYTES;
          HMM_BY_PROB_P(ti.prob, mma_stage, d_tmem, w_base, t_base, idesc, kb == 0);
          if constexpr (PAIR)
            umma_commit_pair(&empty[stage], 0x3);
          else
            umma_commit(&empty[stage]);
          if (++stage == NST) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(&tfull[acc], 0x3);
        else
          umma_commit(&tfull[acc]);
        if (rec) rec[5] = globaltimer_ns();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by this thread completes before TMEM is released
      if constexpr (PAIR)
        umma_commit_pair(mma_done, 0x1);
      else
        umma_commit(mma_done);
      drain_wait(mma_done, 0, P.budget_ns);
    }
  } else if (warp >= 2 && warp < 2 + EW) {
    // ------------------------------------------------------------- epilogue
    EpiState es;
    es.q = warp & 3;
    es.lane = lane;
    es.hoff = EW == 8 ? 16 * ((warp - 2) >> 2) : 0;
    es.own = EW == 8 ? xbufs + (warp - 2) * (XBUF_HALF / 4) : xbufs + es.q * (XBUF_BYTES / 4);
    es.xbufs = xbufs;
    es.xfull = xfull;
    es.xfree = xfree;
    es.nchunk = 0;
    const uint32_t tempty_cl[2] = {PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u,
                                   PAIR ? mapa_shared(smem_u32(&tempty[1]), 0) : 0u};
    int ti_slot = 0;
    uint32_t ti_phase = 0;
    uint32_t acc = 0, acc_phase = 0;
    int lt = 0;
    for (;;) {
      bool got = false;
      if (lane == 0) got = mbar_wait<PAIR>(&ti_full[ti_slot], ti_phase, wc);
      __syncwarp();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      TileInfo ti = s_ti[ti_slot];
      __syncwarp();
      if (lane == 0) ti_release(ti_slot);
      if (++ti_slot == TI_DEPTH) {
        ti_slot = 0;
        ti_phase ^= 1u;
      }
      if (ti.prob < 0) break;
      const Prob& pr = P.p[ti.prob];
      // one warp of the (even) CTA reports
      uint64_t* rec = (warp == 2 && lane == 0 && leader) ? trace_rec(P, lt) : nullptr;
      ++lt;
      if (lane == 0) got = mbar_wait(&tfull[acc], acc_phase, wc);
      __syncwarp();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      if (rec) rec[6] = globaltimer_ns();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(es.q * 32) << 16) + acc * NT;
      bool eok = true;
      if ((ti.prob & 1) == 0)
        epilogue_tile<C0, EW>(pr, ti, taddr, rank, es, wc, eok);
      else
        epilogue_tile<C1, EW>(pr, ti, taddr, rank, es, wc, eok);
      if (!eok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (!PAIR || leader)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_peer(tempty_cl[acc]);
      }
      if (rec) rec[7] = globaltimer_ns();
      if (pr.signal_m) {
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) red_release_add(&pr.signal_m[ti.row0 / TROWS], 1);
      }
      if (pr.cmb) {
        // after the accumulator's release: this overlaps the next tile's MMAs
        const int c0 = ti.w0 + C1::WCOLS * static_cast<int>(rank) + 32 * es.q;
        int* list = reinterpret_cast<int*>(xbufs + es.q * (XBUF_BYTES / 4));
        if (pr.out_f32)
          combine_tile<true>(pr, ti, c0, lane, list);
        else
          combine_tile<false>(pr, ti, c0, lane, list);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  // no copy of either CTA in flight, no peer access to our smem or TMEM after this
  if constexpr (PAIR)
    pair_teardown<NST>(leader, *s_issued, *s_abort, s_peer, s_sbytes, full, P.budget_ns);
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
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

template <bool PAIR, bool SMALL, int EW, class C0, class C1>
int launch(const GemmEnv& env, Params& P, const Maps& maps, int64_t max_tiles, int kind) {
  if (max_tiles <= 0 || P.nprob == 0) return HMM_OK;
  if (env.trace && env.trace_which == kind) {
    P.trace = env.trace;
    P.trace_cap = env.trace_cap;
  }
  auto kern = gmm_kernel<PAIR, SMALL, EW, C0, C1>;
  constexpr int NUM_THREADS = gmm_threads(EW);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return HMM_ERR_CUDA;
  int max_lag = 0;
  for (int q = 0; q < P.nprob; ++q) max_lag = std::max(max_lag, P.p[q].lag);
  P.steps = P.E + max_lag;
  if (P.steps > MAX_STEPS) return HMM_ERR_SHAPE;
  P.status = env.status;
  P.budget_ns = env.budget_ns;
  P.pair = PAIR ? 1 : 0;
  P.nt = SMALL ? SMALL_NT : NT;
  if constexpr (PAIR) {
    // clusters of two CTAs, as many as can be resident at once (the tile
    // dependencies inside the launch need every CTA running)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = env.stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = env.num_sms / 2;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active <= 0)
      return HMM_ERR_CUDA;
    clusters = static_cast<int>(std::min<int64_t>(std::min(clusters, active), max_tiles));
    return launch_kernel(kern, 2 * clusters, NUM_THREADS, SMEM_BYTES, env.stream, env.pdl, 2, P,
                         maps) == cudaSuccess
               ? HMM_OK
               : HMM_ERR_CUDA;
  } else {
    const int grid = static_cast<int>(std::min<int64_t>(env.num_sms, max_tiles));
    return launch_kernel(kern, grid, NUM_THREADS, SMEM_BYTES, env.stream, env.pdl, 1, P, maps) ==
                   cudaSuccess
               ? HMM_OK
               : HMM_ERR_CUDA;
  }
}

}  // namespace

using CfgGmm1 = Cfg<EPI_SWIGLU, true>;     // tokens x_perm, weights W1 (MN-major)
using CfgGmm2 = Cfg<EPI_STORE, true>;      // tokens a, weights W2 (MN-major)
using CfgActGrad = Cfg<EPI_DSWIGLU, false>; // tokens dy_perm, weights W2 rows (K-major)
using CfgInGrad = Cfg<EPI_STORE, false>;   // tokens dH, weights W1 rows (K-major)
// epilogue warps of the data-gradient launch: two per TMEM lane quarter, so
// every SM sub-partition holds two SwiGLU-grad epilogue warps
constexpr int DATA_EW = 8;

namespace {

// Problems 2 and 3 (the shared expert, expert E of the padded rows) copy
// problems 0 and 1 with their own weight maps.
//   Tile counts and ready units: a tile spans WCOLS output columns per CTA;
// every epilogue warp of every CTA of a producer tile releases the tile's
// token block once.
void add_shared(Params& P, Maps& maps, int E, const CUtensorMap& B0, const CUtensorMap& B1) {
  for (int q = 0; q < 2; ++q) {
    P.p[2 + q] = P.p[q];
    P.p[2 + q].e_lo = E;
    P.p[2 + q].e_hi = E + 1;
    for (int i = 0; i < TOK_MAPS; ++i) maps.t[2 + q][i] = maps.t[q][i];
  }
  maps.w[2] = B0;
  maps.w[3] = B1;
  P.nprob = 4;
}

// The token-row maps of an activation [rows, cols] for the launch's mode:
// boxes of the rows one CTA loads for a block of 64 (i + 1) rows.
int map_tokens(const GemmEnv& env, CUtensorMap* t, const void* base, int64_t rows,
               int64_t cols) {
  int rc = HMM_OK;
  for (int i = 0; i < TOK_MAPS; ++i) {
    if (env.small_rows && i > 0) {
      t[i] = t[0];  // small token blocks are 64 rows
      continue;
    }
    const uint32_t box = env.pair_rows ? 32u * (i + 1) : 64u * (i + 1);
    rc |= map_act(env, &t[i], base, rows, cols, box);
  }
  return rc;
}

}  // namespace

int launch_forward_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                         const void* x_perm, const void* W1, const void* W2, const void* Ws1,
                         const void* Ws2, void* a, float* h32, void* o, bool skip_ready_release,
                         int* cmb, const void* w, int w_dtype, void* fused_y) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  Maps maps;
  int rc = HMM_OK;
  rc |= map_tokens(env, maps.t[0], x_perm, R, H);        // x_perm [R, H], K = H
  rc |= map_w(env, &maps.w[0], W1, E, H, 2 * I, 64);      // W1 [E, H, 2I]: MN-major
  rc |= map_tokens(env, maps.t[1], a, R, I);              // a [R, I], K = I
  rc |= map_w(env, &maps.w[1], W2, E, I, H, 64);          // W2 [E, I, H]: MN-major
  CUtensorMap s0, s1;
  if (p.shared) {
    rc |= map_w(env, &s0, Ws1, 1, H, 2 * I, 64);  // shared expert's [H, 2I], [I, H]
    rc |= map_w(env, &s1, Ws2, 1, I, H, 64);
  }
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  Params P{};
  P.nprob = 2;
  P.poff = m.poff;
  P.counts = m.counts;
  P.E = static_cast<int>(p.Ex);
  P.ticket = c.tickets + 0;
  Prob& g1 = P.p[0];
  g1.K = static_cast<int>(H);
  g1.N = static_cast<int>(I);
  g1.half = static_cast<int>(I);
  const int ncta = env.pair_rows ? 2 : 1;
  g1.n_tiles = static_cast<int>((I + CfgGmm1::WCOLS * ncta - 1) / (CfgGmm1::WCOLS * ncta));
  g1.out = a;
  g1.ld_out = I;
  g1.out2 = h32;
  g1.ld_out2 = (I + 31) / 32;  // column blocks of the blocked layout
  g1.e_lo = 0;
  g1.e_hi = static_cast<int>(E);
  g1.signal_m = skip_ready_release ? nullptr : c.ready;
  Prob& g2 = P.p[1];
  g2.K = static_cast<int>(I);
  g2.N = static_cast<int>(H);
  g2.n_tiles = static_cast<int>((H + CfgGmm2::WCOLS * ncta - 1) / (CfgGmm2::WCOLS * ncta));
  g2.out = o;
  g2.ld_out = H;
  g2.out_f32 = p.shared ? 1 : 0;  // fp32 rows for the y combine with the shared expert
  g2.e_lo = 0;
  g2.e_hi = static_cast<int>(E);
  // GMM2 after every GMM1 tile has been handed out: its ready waits then only
  // meet the last wave of GMM1 tiles
  g2.lag = static_cast<int>(p.Ex);
  g2.wait_m = c.ready;
  g2.wait_unit = EPI_WARPS * ncta * g1.n_tiles;  // every GMM1 tile of the token block
  if (fused_y) {
    g2.cmb = cmb;
    g2.slot2prow = m.slot2prow;
    g2.prow2slot = m.prow2slot;
    g2.cmb_poff = m.poff;
    g2.cmb_w = w;
    g2.cmb_y = fused_y;
    g2.cmb_w_f32 = w_dtype == HMM_DTYPE_F32 ? 1 : 0;
    g2.cmb_K = static_cast<int>(p.K);
    g2.cmb_KS = static_cast<int>(p.K + p.shared);
    g2.cmb_T = static_cast<int>(p.T);
    g2.cmb_nseg = static_cast<int>(p.cmb_nseg);
    g2.cmb_E = static_cast<int>(E);
  }
  if (p.shared) add_shared(P, maps, static_cast<int>(E), s0, s1);
  const int64_t max_tiles = (p.R / TROWS) * (g1.n_tiles + g2.n_tiles);
  if (env.pair_rows) return launch<true, false, 4, CfgGmm1, CfgGmm2>(env, P, maps, max_tiles, 0);
  if (env.small_rows) return launch<false, true, 4, CfgGmm1, CfgGmm2>(env, P, maps, max_tiles, 0);
  return launch<false, false, 4, CfgGmm1, CfgGmm2>(env, P, maps, max_tiles, 0);
}

int launch_data_grad_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                           const void* dy_perm, const float* wperm, const float* h32,
                           const void* W1, const void* W2, const void* Ws1, const void* Ws2,
                           void* dH, void* dH_lo, void* wa, void* wa_lo, float* dwp,
                           void* dx_perm, bool skip_ready_release) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  Maps maps;
  int rc = HMM_OK;
  // act_grad: G = dy_perm . W2^T   (weights: 128 rows of W2 [E, I, H] per CTA, N = I)
  rc |= map_tokens(env, maps.t[0], dy_perm, R, H);
  rc |= map_w(env, &maps.w[0], W2, E, I, H, BW);
  // input-grad: dX_perm = dH . W1^T (weights: 128 rows of W1 [E, H, 2I] per CTA, N = H)
  rc |= map_tokens(env, maps.t[1], dH, R, 2 * I);
  rc |= map_w(env, &maps.w[1], W1, E, H, 2 * I, BW);
  CUtensorMap s0, s1;
  if (p.shared) {
    rc |= map_w(env, &s0, Ws2, 1, I, H, BW);
    rc |= map_w(env, &s1, Ws1, 1, H, 2 * I, BW);
  }
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  Params P{};
  P.nprob = 2;
  P.poff = m.poff;
  P.counts = m.counts;
  P.E = static_cast<int>(p.Ex);
  P.ticket = c.tickets + 1;
  Prob& ag = P.p[0];
  ag.K = static_cast<int>(H);
  ag.N = static_cast<int>(I);
  ag.half = static_cast<int>(I);
  const int ncta = env.pair_rows ? 2 : 1;
  ag.n_tiles = static_cast<int>((I + CfgActGrad::WCOLS * ncta - 1) / (CfgActGrad::WCOLS * ncta));
  ag.out = dH;
  ag.ld_out = 2 * I;
  ag.out2 = wa;
  ag.ld_out2 = I;
  ag.out3 = dwp;
  ag.ld_out3 = p.dwp_ld;  // one d_w partial per row and 32-column block of I
  ag.out4 = dH_lo;
  ag.ld_lo4 = p.ld8_2i;
  ag.out5 = wa_lo;
  ag.ld_lo5 = p.ld8_i;
  ag.aux = h32;
  ag.ld_aux = (I + 31) / 32;
  ag.rowscale = wperm;
  ag.e_lo = 0;
  ag.e_hi = static_cast<int>(E);
  ag.signal_m = skip_ready_release ? nullptr : c.ready;
  Prob& ig = P.p[1];
  ig.K = static_cast<int>(2 * I);
  ig.N = static_cast<int>(H);
  ig.n_tiles = static_cast<int>((H + CfgInGrad::WCOLS * ncta - 1) / (CfgInGrad::WCOLS * ncta));
  ig.out = dx_perm;
  ig.ld_out = H;
  ig.out_f32 = p.shared ? 1 : 0;  // fp32 rows for the dX combine with the shared expert
  ig.e_lo = 0;
  ig.e_hi = static_cast<int>(E);
  ig.wait_m = c.ready;
  ig.wait_unit = DATA_EW * ncta * ag.n_tiles;  // every epilogue warp of every act_grad tile
  ig.lag = static_cast<int>(p.Ex);  // input-grad after every act_grad tile is handed out
  if (p.shared) add_shared(P, maps, static_cast<int>(E), s0, s1);
  const int64_t data_tiles = (p.R / TROWS) * (ag.n_tiles + ig.n_tiles);
  if (env.pair_rows)
    return launch<true, false, DATA_EW, CfgActGrad, CfgInGrad>(env, P, maps, data_tiles, 1);
  if (env.small_rows)
    return launch<false, true, DATA_EW, CfgActGrad, CfgInGrad>(env, P, maps, data_tiles, 1);
  return launch<false, false, DATA_EW, CfgActGrad, CfgInGrad>(env, P, maps, data_tiles, 1);
}

}  // namespace hmm
