// gmm_pair.cu -- the weight-gradient GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// [HyperMegaMoE §2.2 W2Grad, W1Grad]
//   dW2[e] = wa_hi^T . dy_perm + wa_lo^T . dy8      [I, rows of e] x [rows of e, H]
//   dW1[e] = x_perm^T . dH_hi + x8^T . dH_lo        [H, rows of e] x [rows of e, 2I]
// for the routed experts and, with the optional shared expert [HyperMegaMoE
// §6.1], for the shared expert (expert E of the padded rows, every token).
// The rounded operand comes as a bf16 high part and an e5m2 low part (the
// rest, at most 2^-9 of the value); the low part meets an fp8 copy of the
// other operand (x8 e4m3, dy8 e5m2) in an fp8 MMA at twice the bf16 rate,
// accumulating into the same fp32 TMEM tile.  Every 64-row K step stages the
// bf16 A and B and the two fp8 operands together (48 KB per CTA) and issues
// four bf16 and two fp8 MMAs.
//
// Two CTAs of a cluster compute one 256 x 256 output tile with 2-SM MMAs:
// each CTA loads its 128 rows of A and its 128 of the 256 columns of B, and
// each accumulates its 128 rows x 256 columns in its own TMEM (the fp8 MMAs
// add into the same accumulator).
//
// Roles per CTA: warp 0 issues TMA (both CTAs, one thread), warp 1 issues the
// MMAs (even CTA only), warps 2..5 drain TMEM (both CTAs), warp 6 schedules
// (even CTA only).  The even CTA's
// full barriers count the bytes of both CTAs; the MMA commits arrive on the
// empty / accumulator-full barriers of both CTAs; both CTAs' epilogues release
// the even CTA's accumulator-empty barrier.
//
// Schedule: a tile's cost is its expert's K blocks (rows / 64), so with a hot
// expert a few tiles cost ten times the others.  Tiles are therefore handed
// out longest first: the experts sorted by routed rows (descending, ties by
// id; empty experts last), all tiles of one expert together, through a global
// ticket.  The even CTA's scheduler warp takes the tickets (each one a tile
// ahead of its use, so the atomic's latency stays off every other role) and
// publishes the tiles in a shared-memory ring of both CTAs, up to
// P_TI_DEPTH tiles ahead of the slowest reader.  The last cluster to finish
// resets the ticket for the next launch.  Every wait is bounded.
#include <cuda_bf16.h>

#include <algorithm>

#include "epilogue.cuh"
#include "ptx.cuh"

namespace hmm {

namespace {

// Expert rows per K step (a multiple of 32) and stages (192 KB in all).  Eight
// 24 KB stages of 32 rows made the launch 23 % slower than four of 64: more,
// smaller copies and barrier round trips per byte.
constexpr int PK = 64;
static_assert(PK == TROWS, "K blocks end where the zeroed padding rows end");
constexpr int PSTAGES = 4 * 64 / PK;
constexpr int PA_BYTES = 128 * PK * 2;  // this CTA's 128 rows of A, PK deep (bf16)
constexpr int PB_BYTES = 128 * PK * 2;  // this CTA's 128 columns of B, PK deep (bf16)
constexpr int PL_BYTES = 128 * PK;      // the low part of the split one of them (e5m2)
constexpr int PO_BYTES = 128 * PK;      // the fp8 copy of the other one
constexpr int PSTAGE = PA_BYTES + PB_BYTES + PL_BYTES + PO_BYTES;
constexpr int P_EPI_WARPS = 4;
constexpr int P_SCHED_WARP = 2 + P_EPI_WARPS;
constexpr int P_THREADS = 32 * (P_SCHED_WARP + 1);  // 7 warps
constexpr int P_TI_DEPTH = 8;  // tile ring: the producer runs up to a few small tiles ahead
// the routed rows of every expert, the sorted expert order and the tile
// prefix over it (experts 0 .. MAX_E, the last one the optional shared expert)
constexpr int P_ORD_BYTES = 4 * (MAX_E + 1) + 4 * (MAX_E + 1) + 4 * (MAX_E + 2);
constexpr int P_SMEM = 1024 + PSTAGES * PSTAGE + P_EPI_WARPS * XBUF_BYTES + 1024 + P_ORD_BYTES;
static_assert(P_SMEM <= 232448, "shared memory per CTA");
constexpr uint32_t P_TMEM_COLS = 512;
constexpr uint32_t IDESC_PAIR = idesc_bf16_f32(256, 256, 1, 1);  // both MN-major
// fp8 MMAs on the low part: W1Grad x8 (e4m3) . dH_lo (e5m2); W2Grad wa_lo (e5m2) . dy8 (e5m2)
constexpr uint32_t IDESC_LO_B = idesc_f8_f32(256, 256, F8_E4M3, F8_E5M2, 1, 1);
constexpr uint32_t IDESC_LO_A = idesc_f8_f32(256, 256, F8_E5M2, F8_E5M2, 1, 1);

struct PairProb {
  int e_lo, n_e; // experts e_lo .. e_lo + n_e - 1 of the padded rows
  int M, N;      // output [M, N] per expert
  int mpairs;    // 256-row tile pairs along M
  int n_tiles;   // 256-column tiles along N
  int split;     // the operand given as bf16 high + e5m2 low parts: 1 A, 2 B
  __nv_bfloat16* out;
  int64_t ld_out;
  int64_t out_estride;
};

struct PairParams {
  PairProb p[4];
  int nprob;
  const int32_t* poff;
  const int32_t* counts;
  int Ex;           // experts of the padded rows (E, plus the shared expert)
  int* ticket;      // [2] tile ticket and finished-cluster count, zero at launch
  unsigned* status;
  unsigned long long budget_ns;
  uint64_t* trace;  // per-tile timeline records of the even CTA (null: off)
  int trace_cap;
};

struct PairMaps {
  CUtensorMap m[4][4];  // A, B (bf16), low part of the split one, fp8 copy of the other
  CUtensorMap out[4];   // the output [experts][M][N] (bf16), stored in 32 x 32 boxes
};

// One tile of the ring (prob < 0: no more tiles).
struct PairTile {
  int prob, e, m0, n0, kb, krow0;
};

// Tiles of expert x over all problems that include it.
__device__ __forceinline__ int expert_tiles(const PairParams& P, int x) {
  int n = 0;
  for (int q = 0; q < P.nprob; ++q)
    if (x >= P.p[q].e_lo && x < P.p[q].e_lo + P.p[q].n_e) n += P.p[q].mpairs * P.p[q].n_tiles;
  return n;
}

// Longest first: ord[i] = the expert of rank i (routed rows descending, ties
// by id), pre[i] = tiles of the experts of rank < i.  One CTA's threads; cnt
// is scratch for the routed rows.
__device__ void build_order(const PairParams& P, int* cnt, int* ord, int* pre) {
  const int Ex = P.Ex;
  for (int x = threadIdx.x; x < Ex; x += blockDim.x) cnt[x] = P.counts[x];
  __syncthreads();
  for (int x = threadIdx.x; x < Ex; x += blockDim.x) {
    const int cx = cnt[x];
    int r = 0;
    for (int y = 0; y < Ex; ++y) {
      const int cy = cnt[y];
      r += (cy > cx || (cy == cx && y < x)) ? 1 : 0;
    }
    ord[r] = x;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) pre[0] = 0;
    for (int base = 0; base < Ex; base += 32) {
      const int i = base + lane;
      int v = i < Ex ? expert_tiles(P, ord[i]) : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += n;
      }
      if (i < Ex) pre[i + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
}

// Ticket u (< pre[Ex]) -> tile.
__device__ void pair_decode(const PairParams& P, const int* ord, const int* pre, int u,
                            PairTile& t) {
  int lo = 0, hi = P.Ex - 1;  // largest rank i with pre[i] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int x = ord[lo];
  int r = u - pre[lo];
  int q = 0;
  for (; q < P.nprob; ++q) {
    const PairProb& pr = P.p[q];
    if (x < pr.e_lo || x >= pr.e_lo + pr.n_e) continue;
    const int per = pr.mpairs * pr.n_tiles;
    if (r < per) break;
    r -= per;
  }
  const PairProb& pr = P.p[q];
  t.prob = q;
  t.e = x;
  t.m0 = (r / pr.n_tiles) * 256;
  t.n0 = (r % pr.n_tiles) * 256;
  t.krow0 = P.poff[x];
  // rows past counts[e] are zero padding: skip whole zero K blocks
  t.kb = (P.counts[x] + PK - 1) / PK;
}

// Timeline record of this CTA's lt-th tile (even CTA of the pair only).
__device__ __forceinline__ uint64_t* pair_rec(const PairParams& P, bool leader, int lt) {
  if (!leader || P.trace == nullptr || lt >= P.trace_cap) return nullptr;
  return P.trace + (static_cast<int64_t>(blockIdx.x) * P.trace_cap + lt) * 8;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    wgrad_pair_kernel(const __grid_constant__ PairParams P, const __grid_constant__ PairMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  float* xbufs = reinterpret_cast<float*>(smem + PSTAGES * PSTAGE);
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + PSTAGES * PSTAGE + P_EPI_WARPS * XBUF_BYTES);
  uint64_t* full = bars;                    // used in the even CTA
  uint64_t* empty = bars + PSTAGES;         // both CTAs
  uint64_t* tfull = empty + PSTAGES;        // both CTAs
  uint64_t* tempty = tfull + 2;             // even CTA
  uint64_t* mma_done = tempty + 2;          // even CTA
  uint64_t* ti_full = mma_done + 1;         // [P_TI_DEPTH] both CTAs
  uint64_t* ti_empty = ti_full + P_TI_DEPTH;  // [P_TI_DEPTH] even CTA: every reader arrives
  PairTile* s_ti = reinterpret_cast<PairTile*>(ti_empty + P_TI_DEPTH);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_ti + P_TI_DEPTH);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 2;  // K blocks this CTA's producer issued
  uint32_t* s_sbytes = s_tmem + 3;  // [PSTAGES] bytes of this CTA's loads per slot (fixed)
  uint32_t* s_peer = s_sbytes + PSTAGES;  // [2 + PSTAGES] even CTA: the odd CTA's count, flag, bytes
  int* s_cnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + 1024);
  int* s_ord = s_cnt + (MAX_E + 1);
  int* s_pre = s_ord + (MAX_E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < P_TI_DEPTH; ++i) {
      mbar_init(&ti_full[i], 1);
      // readers: both CTAs' producers and epilogue warps, the even CTA's MMA
      // issuer
      mbar_init(&ti_empty[i], 3 + 2 * P_EPI_WARPS);
    }
    *s_abort = 0;
    *s_issued = 0;
    for (int i = 0; i < PSTAGES; ++i) s_sbytes[i] = PSTAGE;
    for (int i = 0; i < 2 + PSTAGES; ++i) s_peer[i] = 0;
    fence_mbar_init();
  }
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, P_TMEM_COLS);  // collective: one warp in each CTA of the pair
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  // set-up done: from here on global memory the stream's previous kernel may
  // still be writing.  (The next kernel is let in only when this CTA's
  // producer has issued its last tile.)
  grid_dep_wait();
  const WaitCtl wc{s_abort, P.status, P.budget_ns};
  if (leader) build_order(P, s_cnt, s_ord, s_pre);  // only the even CTA decodes tickets
  // readers of the ring: the odd CTA's release the even CTA's slots
  const auto ti_release = [&](int slot) {
    if (leader)
      mbar_arrive(&ti_empty[slot]);
    else
      mbar_arrive_peer(mapa_shared(smem_u32(&ti_empty[slot]), 0));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- TMA producer
      for (int q = 0; q < P.nprob; ++q)
        for (int j = 0; j < 4; ++j) tma_prefetch_desc(&maps.m[q][j]);
      for (int q = 0; q < P.nprob; ++q) tma_prefetch_desc(&maps.out[q]);
      uint32_t stage = 0, sphase = 0;
      uint32_t issued = 0;
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      bool ok = true;
      int lt = 0;
      for (;;) {
        const bool got = leader ? mbar_wait(&ti_full[ti_slot], ti_phase, wc)
                                : mbar_wait<true>(&ti_full[ti_slot], ti_phase, wc);
        if (!got) {
          ok = false;
          break;
        }
        const PairTile t = s_ti[ti_slot];
        ti_release(ti_slot);
        if (++ti_slot == P_TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (t.prob < 0) break;
        const PairProb& pr = P.p[t.prob];
        const CUtensorMap* mp = maps.m[t.prob];
        uint64_t* rec = pair_rec(P, leader, lt++);
        if (rec) {
          uint32_t smid;
          asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
          rec[0] = (static_cast<uint64_t>(smid) << 48) | (static_cast<uint64_t>(t.prob) << 40) |
                   (static_cast<uint64_t>(t.e & 0xFFFFF) << 20) |
                   static_cast<uint64_t>(t.kb & 0xFFFFF);
          rec[1] = globaltimer_ns();
        }
        const int ma = t.m0 + 128 * static_cast<int>(rank);  // this CTA's rows of the output
        const int nbc = t.n0 + 128 * static_cast<int>(rank);  // this CTA's half of B's columns
        for (int kb = 0; kb < t.kb; ++kb) {
          if (!mbar_wait(&empty[stage], sphase ^ 1u, wc)) {
            ok = false;
            break;
          }
          if (rec && kb == 0) rec[2] = globaltimer_ns();
          const int k = t.krow0 + kb * PK;
          uint8_t* sA = stages + stage * PSTAGE;
          uint8_t* sB = sA + PA_BYTES;
          uint8_t* sL = sB + PB_BYTES;
          uint8_t* sO = sL + PL_BYTES;
          // the low part sits on the split side, the fp8 copy on the other
          const int lc = pr.split == 1 ? ma : nbc;
          const int oc = pr.split == 1 ? nbc : ma;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * PSTAGE);
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          tma_load_2d_pair(sA, &mp[0], bar, ma, k);
          tma_load_2d_pair(sA + PA_BYTES / 2, &mp[0], bar, ma + 64, k);
          tma_load_2d_pair(sB, &mp[1], bar, nbc, k);
          tma_load_2d_pair(sB + PB_BYTES / 2, &mp[1], bar, nbc + 64, k);
          tma_load_2d_pair(sL, &mp[2], bar, lc, k);  // 128 fp8 columns in one box
          tma_load_2d_pair(sO, &mp[3], bar, oc, k);
          ++issued;
          if (++stage == PSTAGES) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (rec && ok) rec[3] = globaltimer_ns();
        if (!ok) break;
      }
      // copies still in flight after an abort are drained at teardown
      // (pair_teardown: both CTAs' copies are counted on the even CTA)
      *s_issued = issued;
      grid_dep_launch();  // this CTA is in its last tile
    }
  } else if (warp == P_SCHED_WARP) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------- tile scheduler
      const int total = s_pre[P.Ex];
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      int u = atomicAdd(P.ticket, 1);
      for (;;) {
        PairTile t;
        t.prob = -1;
        t.e = t.m0 = t.n0 = t.kb = t.krow0 = 0;
        if (u < total) {
          pair_decode(P, s_ord, s_pre, u, t);
          u = atomicAdd(P.ticket, 1);  // the next ticket, used one tile later
        }
        if (!mbar_wait(&ti_empty[ti_slot], ti_phase ^ 1u, wc)) break;
        s_ti[ti_slot] = t;
        const uint32_t dst = mapa_shared(smem_u32(&s_ti[ti_slot]), 1);
        const int* src = reinterpret_cast<const int*>(&t);
#pragma unroll
        for (int j = 0; j < static_cast<int>(sizeof(PairTile) / 4); ++j)
          st_shared_cluster(dst + 4 * j, src[j]);
        mbar_arrive_cluster(mapa_shared(smem_u32(&ti_full[ti_slot]), 1));
        mbar_arrive(&ti_full[ti_slot]);
        if (++ti_slot == P_TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (t.prob < 0) break;
      }
      // the last cluster to finish resets the ticket for the next launch (no
      // ticket is taken after a cluster's increment of the count)
      __threadfence();
      if (atomicAdd(P.ticket + 1, 1) == static_cast<int>(ncluster_x()) - 1) {
        atomicExch(P.ticket, 0);
        atomicExch(P.ticket + 1, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issue
      uint32_t stage = 0, sphase = 0;
      uint32_t acc = 0, acc_phase = 0;
      int ti_slot = 0;
      uint32_t ti_phase = 0;
      bool ok = true;
      int lt = 0;
      for (;;) {
        if (!mbar_wait(&ti_full[ti_slot], ti_phase, wc)) break;
        const PairTile t = s_ti[ti_slot];
        mbar_arrive(&ti_empty[ti_slot]);
        if (++ti_slot == P_TI_DEPTH) {
          ti_slot = 0;
          ti_phase ^= 1u;
        }
        if (t.prob < 0) break;
        const int split = P.p[t.prob].split;
        uint64_t* rec = pair_rec(P, leader, lt++);
        if (t.kb == 0) continue;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        if (rec) rec[4] = globaltimer_ns();
        const uint32_t d_tmem = tmem_base + acc * 256;
        for (int kb = 0; kb < t.kb; ++kb) {
          if (!mbar_wait(&full[stage], sphase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(stages + stage * PSTAGE);
          const uint32_t b_base = a_base + PA_BYTES;
          const uint32_t l_base = b_base + PB_BYTES;
          const uint32_t o_base = l_base + PL_BYTES;
#pragma unroll
          for (int kk = 0; kk < PK / 16; ++kk) {
            // MN-major bf16: two 64-wide chunks PA_BYTES / 2 apart, 8-row groups 1 KB
            const uint64_t ad = smem_desc(a_base + kk * 2048, PA_BYTES / 2, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(b_base + kk * 2048, PB_BYTES / 2, 1024, LAYOUT_SW128);
            umma_bf16_pair(d_tmem, ad, bd, IDESC_PAIR, (kb == 0 && kk == 0) ? 0u : 1u);
          }
          // the low part against the fp8 copy: MN-major fp8, one 128-wide
          // chunk, 8-row groups 1 KB, 32 rows of K per MMA
          const uint32_t a2_base = split == 1 ? l_base : o_base;
          const uint32_t b2_base = split == 1 ? o_base : l_base;
#pragma unroll
          for (int kk = 0; kk < PK / 32; ++kk) {
            const uint64_t ad = smem_desc(a2_base + kk * 4096, 8192, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(b2_base + kk * 4096, 8192, 1024, LAYOUT_SW128);
            umma_f8_pair(d_tmem, ad, bd, split == 1 ? IDESC_LO_A : IDESC_LO_B, 1u);
          }
          umma_commit_pair(&empty[stage], 0x3);
          if (++stage == PSTAGES) {
            stage = 0;
            sphase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], 0x3);
        if (rec) rec[5] = globaltimer_ns();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit_pair(mma_done, 0x1);
      drain_wait(mma_done, 0, P.budget_ns);
    }
  } else if (warp >= 2 && warp < 2 + P_EPI_WARPS) {
    // ------------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int row_in_half = q4 * 32 + lane;
    // two 2 KB staging buffers of 32 rows x 32 bf16 columns, 64-byte swizzled
    // (16-byte unit u of row r at u ^ ((r >> 1) & 3)), one per chunk in turn
    uint8_t* obuf = reinterpret_cast<uint8_t*>(xbufs + (warp - 2) * (XBUF_BYTES / 4));
    uint32_t ck = 0;  // chunks this warp has stored
    uint32_t acc = 0, acc_phase = 0;
    int ti_slot = 0;
    uint32_t ti_phase = 0;
    const uint32_t tempty_cl[2] = {mapa_shared(smem_u32(&tempty[0]), 0),
                                   mapa_shared(smem_u32(&tempty[1]), 0)};
    int lt = 0;
    for (;;) {
      bool got = false;
      if (lane == 0)
        got = leader ? mbar_wait(&ti_full[ti_slot], ti_phase, wc)
                     : mbar_wait<true>(&ti_full[ti_slot], ti_phase, wc);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      const PairTile t = s_ti[ti_slot];
      __syncwarp();
      if (lane == 0) ti_release(ti_slot);
      if (++ti_slot == P_TI_DEPTH) {
        ti_slot = 0;
        ti_phase ^= 1u;
      }
      if (t.prob < 0) break;
      const PairProb& pr = P.p[t.prob];
      uint64_t* rec = (warp == 2 && lane == 0) ? pair_rec(P, leader, lt) : nullptr;
      ++lt;
      const int64_t row = t.m0 + 128 * static_cast<int>(rank) + row_in_half;
      __nv_bfloat16* orow =
          pr.out + static_cast<int64_t>(t.e - pr.e_lo) * pr.out_estride + row * pr.ld_out;
      if (t.kb == 0) {
        // an expert with no rows: its weight gradient is exactly zero
        if (row < pr.M)
          for (int col = t.n0; col < min(t.n0 + 256, pr.N); col += 8)
            *reinterpret_cast<uint4*>(orow + col) = make_uint4(0, 0, 0, 0);
        continue;
      }
      got = false;
      if (lane == 0) got = mbar_wait(&tfull[acc], acc_phase, wc);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      if (rec) rec[6] = globaltimer_ns();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + acc * 256;
      // rows of this warp's chunks (the store leaves out rows past M and
      // columns past N)
      const int row0 = t.m0 + 128 * static_cast<int>(rank) + q4 * 32;
      const CUtensorMap* omap = &maps.out[t.prob];
      // each chunk's TMEM load is issued before the previous chunk is
      // converted and stored, so its latency hides behind that work
      const int nch = min(8, (pr.N - t.n0 + 31) / 32);  // chunks inside the output
      uint32_t ra[32], rb[32];
      if (nch > 0) {
        tmem_ld32(taddr, ra);
        tmem_ld_wait_for(ra);
      }
      auto drain = [&](const uint32_t (&r)[32], int c) {
        uint8_t* sb = obuf + (ck & 1u) * 2048;
        if (lane == 0) bulk_wait_group_read<1>();  // chunk ck - 2's store has read sb
        __syncwarp();
        // lane = row: its 32 columns as four 16-byte units
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[8 * u + i]);
          *reinterpret_cast<uint4*>(sb + lane * 64 + 16 * (u ^ ((lane >> 1) & 3))) =
              pack_bf16x8(f);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(omap, sb, t.n0 + 32 * c, row0, t.e - pr.e_lo);
          bulk_commit_group();
        }
        ++ck;
      };
#pragma unroll
      for (int c = 0; c < 8; c += 2) {
        if (c < nch) {
          if (c + 1 < nch) tmem_ld32(taddr + (c + 1) * 32, rb);
          drain(ra, c);
          if (c + 1 < nch) {
            tmem_ld_wait_for(rb);
            if (c + 2 < nch) tmem_ld32(taddr + (c + 2) * 32, ra);
            drain(rb, c + 1);
            if (c + 2 < nch) tmem_ld_wait_for(ra);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_peer(tempty_cl[acc]);
      }
      if (rec) rec[7] = globaltimer_ns();
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group<0>();  // every store has landed
  }

  tc_fence_before();
  __syncthreads();
  // no copy of either CTA in flight, no peer access to our smem or TMEM after this
  pair_teardown<PSTAGES>(leader, *s_issued, *s_abort, s_peer, s_sbytes, full, P.budget_ns);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, P_TMEM_COLS);  // collective, like the allocation
  }
}

// fp8 rows (ld bytes apart): boxes of 128 columns x PK rows
int encode2d_u8(const GemmEnv& env, CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                int64_t ld) {
  const cuuint64_t gd[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gs[1] = {static_cast<cuuint64_t>(ld)};
  const cuuint32_t bx[2] = {128, PK};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = env.encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gd, gs,
                          bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HMM_OK : HMM_ERR_CUDA;
}

// the bf16 outputs [experts][rows][cols] (rows * cols per expert, cols per
// row): boxes of 32 columns x 32 rows of one expert, 64-byte swizzled
int encode_out(const GemmEnv& env, CUtensorMap* m, void* base, int64_t experts, int64_t rows,
               int64_t cols) {
  const cuuint64_t gd[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                            static_cast<cuuint64_t>(experts)};
  const cuuint64_t gs[2] = {static_cast<cuuint64_t>(cols) * 2,
                            static_cast<cuuint64_t>(rows * cols) * 2};
  const cuuint32_t bx[3] = {32, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = env.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, gd, gs, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HMM_OK : HMM_ERR_CUDA;
}

int encode2d(const GemmEnv& env, CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  const cuuint64_t gd[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gs[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t bx[2] = {64, PK};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = env.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gd, gs,
                          bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HMM_OK : HMM_ERR_CUDA;
}

}  // namespace

int launch_wgrad_pair(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                      const void* x_perm,
                      const void* x8, const void* dy_perm, const void* dy8, const void* dH,
                      const void* dH_lo8, const void* wa, const void* wa_lo8, void* dW1,
                      void* dW2, void* dWs1, void* dWs2) {
  const int64_t H = p.H, I = p.I, E = p.E, R = p.R;
  if (!dW1 && !dW2 && !dWs1 && !dWs2) return HMM_OK;
  PairMaps maps;
  PairParams P{};
  P.poff = m.poff;
  P.counts = m.counts;
  P.Ex = static_cast<int>(p.Ex);
  P.ticket = c.tickets + 2;  // [2]: ticket, finished clusters (zero; reset by the launch)
  P.status = env.status;
  P.budget_ns = env.budget_ns;
  if (env.trace && env.trace_which == 2) {
    P.trace = env.trace;
    P.trace_cap = env.trace_cap;
  }
  int rc = HMM_OK;
  int q = 0;
  // dW2 of experts [e_lo, e_lo + n_e): wa_hi^T . dy_perm + wa_lo^T . dy8
  auto add_w2 = [&](void* out, int e_lo, int n_e) {
    rc |= encode2d(env, &maps.m[q][0], wa, R, I);
    rc |= encode2d(env, &maps.m[q][1], dy_perm, R, H);
    rc |= encode2d_u8(env, &maps.m[q][2], wa_lo8, R, I, p.ld8_i);
    rc |= encode2d_u8(env, &maps.m[q][3], dy8, R, H, p.ld8_h);
    rc |= encode_out(env, &maps.out[q], out, n_e, I, H);
    PairProb& w = P.p[q++];
    w.e_lo = e_lo;
    w.n_e = n_e;
    w.M = static_cast<int>(I);
    w.N = static_cast<int>(H);
    w.mpairs = static_cast<int>((I + 255) / 256);
    w.n_tiles = static_cast<int>((H + 255) / 256);
    w.split = 1;
    w.out = static_cast<__nv_bfloat16*>(out);
    w.ld_out = H;
    w.out_estride = I * H;
  };
  // dW1 of experts [e_lo, e_lo + n_e): x_perm^T . dH_hi + x8^T . dH_lo
  auto add_w1 = [&](void* out, int e_lo, int n_e) {
    rc |= encode2d(env, &maps.m[q][0], x_perm, R, H);
    rc |= encode2d(env, &maps.m[q][1], dH, R, 2 * I);
    rc |= encode2d_u8(env, &maps.m[q][2], dH_lo8, R, 2 * I, p.ld8_2i);
    rc |= encode2d_u8(env, &maps.m[q][3], x8, R, H, p.ld8_h);
    rc |= encode_out(env, &maps.out[q], out, n_e, H, 2 * I);
    PairProb& w = P.p[q++];
    w.e_lo = e_lo;
    w.n_e = n_e;
    w.M = static_cast<int>(H);
    w.N = static_cast<int>(2 * I);
    w.mpairs = static_cast<int>((H + 255) / 256);
    w.n_tiles = static_cast<int>((2 * I + 255) / 256);
    w.split = 2;
    w.out = static_cast<__nv_bfloat16*>(out);
    w.ld_out = 2 * I;
    w.out_estride = H * 2 * I;
  };
  if (dW2) add_w2(dW2, 0, static_cast<int>(E));
  if (dW1) add_w1(dW1, 0, static_cast<int>(E));
  if (p.shared && dWs2) add_w2(dWs2, static_cast<int>(E), 1);
  if (p.shared && dWs1) add_w1(dWs1, static_cast<int>(E), 1);
  if (rc != HMM_OK) return HMM_ERR_CUDA;
  P.nprob = q;
  int64_t total = 0;
  for (int i = 0; i < q; ++i) total += int64_t(P.p[i].n_e) * P.p[i].mpairs * P.p[i].n_tiles;
  if (total <= 0) return HMM_OK;
  if (cudaFuncSetAttribute(wgrad_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           P_SMEM) != cudaSuccess)
    return HMM_ERR_CUDA;
  // as many pairs as can be resident at once (each takes tiles by ticket)
  int clusters = env.num_sms / 2;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = P_SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, wgrad_pair_kernel, &cfg) == cudaSuccess &&
        active > 0)
      clusters = std::min(clusters, active);
  }
  clusters = static_cast<int>(std::min<int64_t>(clusters, total));
  // (cluster shape from the kernel's __cluster_dims__)
  return launch_kernel(wgrad_pair_kernel, 2 * clusters, P_THREADS, P_SMEM, env.stream, env.pdl, 1,
                       P, maps) == cudaSuccess
             ? HMM_OK
             : HMM_ERR_CUDA;
}

}  // namespace hmm
