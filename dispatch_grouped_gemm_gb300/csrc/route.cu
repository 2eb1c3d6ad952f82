// route.cu -- routing metadata on the device, with no host round trip.
//
// [HyperMegaMoE §3.3] the operator manages "offset, size and group list"
// internally; [HyperMegaMoE §4.1] each token expands into K expert slots
// (slot s = t*K + k, global expert ids); [MoE overlap explainer §5] counts,
// prefix sums, offsets and the token permutation belong on the device.
//
// Output (bit-exact, deterministic):
//   counts[e]            slots routed to e
//   offsets[e]           exclusive prefix of counts
//   slot2row / row2slot  stable sort of slots by expert (ties by ascending s)
// plus the padded layout the GEMMs use: expert e owns padded rows
// [poff[e], poff[e+1]) with poff[e+1]-poff[e] = counts[e] rounded up to BM.
//
// Per-chunk histograms -> scan over chunks and experts -> per-chunk stable
// ranks.  A chunk (1024 slots) belongs to one block of 8 warps, 128 slots per
// warp: warp match_any groups equal ids inside each 32-slot step, so the order
// inside a warp follows s, and the warps' per-expert counts are prefix-summed
// in shared memory, so the order across warps follows s too.  Each warp loads
// its ids into registers before the first step, so the steps do not wait on
// global loads one after another.  When the chunk histograms are small
// (nchunks * E <= ROUTE_FUSE_MAX) every rank block redoes the scan from them
// (two launches); otherwise one block scans between the two (three).
#include "hmm_internal.h"

namespace hmm {

constexpr int WSLOTS = RCHUNK / RWARPS;  // slots per warp of a chunk
constexpr int RSTEPS = WSLOTS / 32;      // 32-slot steps per warp
// The rank blocks redo the scan themselves when every block reading the whole
// chunk-histogram matrix stays cheap (at most this many values, 128 KB) and
// their shared memory stays under 48 KB.
constexpr int64_t ROUTE_FUSE_MAX = 32768;
constexpr int ROUTE_FUSE_MAX_E = 512;

// ids of slots s0 + 32 j + lane, j < RSTEPS (-2 past s1: "no slot")
__device__ __forceinline__ void load_chunk_ids(const int32_t* __restrict__ ids, int64_t s0,
                                               int64_t s1, int lane, int (&v)[RSTEPS]) {
#pragma unroll
  for (int j = 0; j < RSTEPS; ++j) {
    const int64_t s = s0 + 32 * j + lane;
    v[j] = s < s1 ? __ldg(ids + s) : -2;
  }
}

__global__ void __launch_bounds__(RWARPS * 32) route_count_kernel(const int32_t* __restrict__ ids,
                                                                  int64_t TK, int E,
                                                                  int64_t nchunks,
                                                                  int32_t* __restrict__ chunk_cnt,
                                                                  unsigned* status) {
  extern __shared__ int32_t sh[];  // [E]: the chunk's histogram
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();
  const int64_t c0 = chunk * RCHUNK;
  const int64_t c1 = (c0 + RCHUNK < TK ? c0 + RCHUNK : TK);
  const int64_t s0 = c0 + static_cast<int64_t>(warp) * WSLOTS;
  int v[RSTEPS];
  load_chunk_ids(ids, s0, c1, lane, v);
  bool bad = false;
#pragma unroll
  for (int j = 0; j < RSTEPS; ++j) {
    const int e = v[j];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&sh[e], 1);
    else if (e != -2)
      bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, HMM_STATUS_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_cnt[chunk * E + e] = sh[e];
}

// Block-wide exclusive scan of one value per thread (blockDim.x a multiple of
// 32, at most 1024); *total gets the sum.
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_tot, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  int32_t inc = v;
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int32_t wv = lane < nwarps ? warp_tot[lane] : 0;
    int32_t winc = wv;
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, winc, d);
      if (lane >= d) winc += n;
    }
    if (lane < nwarps) warp_tot[lane] = winc - wv;
    if (lane == 31) *total = winc;
  }
  __syncthreads();
  const int32_t r = warp_tot[warp] + inc - v;
  __syncthreads();
  return r;
}

// Ex = E + shared experts; the shared expert (e == E, when present) owns all
// T tokens, in token order, after the routed experts.
__global__ void __launch_bounds__(1024) route_scan_kernel(int E, int Ex, int32_t T,
                                                          int64_t nchunks, MetaPtrs m,
                                                          CtrlPtrs c, int64_t zero_count) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t tot_cnt, tot_pad;
  const int e = threadIdx.x;
  grid_dep_wait();
  grid_dep_launch();
  // counts of expert e over the chunks, loaded eight chunks at a time
  constexpr int CB = 8;
  int32_t cnt = (e >= E && e < Ex) ? T : 0;
  if (e < E) {
    for (int64_t ch0 = 0; ch0 < nchunks; ch0 += CB) {
      int32_t v[CB];
#pragma unroll
      for (int j = 0; j < CB; ++j)
        v[j] = ch0 + j < nchunks ? c.chunk_base[(ch0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < CB; ++j) cnt += v[j];
    }
  }
  const int32_t padded = (cnt + BM - 1) / BM * BM;
  const int32_t off = block_exclusive_scan(cnt, warp_tot, &tot_cnt);
  const int32_t poff = block_exclusive_scan(padded, warp_tot, &tot_pad);
  if (e < Ex) {
    m.counts[e] = cnt;
    m.offsets[e] = off;
    m.poff[e] = poff;
    // chunk counts -> first row of each chunk's slots of e
    int32_t run = off;
    for (int64_t ch0 = 0; e < E && ch0 < nchunks; ch0 += CB) {
      int32_t v[CB];
#pragma unroll
      for (int j = 0; j < CB; ++j)
        v[j] = ch0 + j < nchunks ? c.chunk_base[(ch0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        if (ch0 + j < nchunks) c.chunk_base[(ch0 + j) * E + e] = run;
        run += v[j];
      }
    }
    for (int32_t r = poff + cnt; r < poff + padded; ++r) m.prow2slot[r] = -1;
  }
  if (e == 0) {
    m.offsets[Ex] = tot_cnt;
    m.poff[Ex] = tot_pad;
  }
  // tickets and per-token-block ready counters of this call
  for (int64_t i = e; i < zero_count; i += blockDim.x) c.tickets[i] = 0;
}

// Scan over chunks and experts inside a rank block (the fused form): from the
// chunk histograms, per expert e < Ex, its total (T for the shared expert),
// the slots of e in chunks before this one, and the exclusive prefixes over
// experts of the totals and of the totals padded to BM.  Block 0 publishes
// counts, offsets and poff; every block takes a share of the padding rows of
// prow2slot and of the counters to zero.
__device__ void route_scan_in_block(int E, int Ex, int32_t T, int64_t nchunks, int64_t chunk,
                                    const int32_t* __restrict__ chunk_cnt, MetaPtrs m,
                                    int32_t* tickets, int64_t zero_count, int32_t* s_tot,
                                    int32_t* s_bef, int32_t* s_off, int32_t* s_poff,
                                    int32_t* warp_tot) {
  const int tid = threadIdx.x;
  for (int e = tid; e < Ex; e += blockDim.x) {
    s_tot[e] = e < E ? 0 : T;
    s_bef[e] = 0;
  }
  __syncthreads();
  // column sums of the [nchunks, E] histograms, eight loads in flight per thread
  constexpr int U = 8;
  const int64_t n = nchunks * E;
  for (int64_t i0 = tid; i0 < n; i0 += static_cast<int64_t>(U) * blockDim.x) {
    int32_t v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + static_cast<int64_t>(u) * blockDim.x;
      v[u] = i < n ? chunk_cnt[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + static_cast<int64_t>(u) * blockDim.x;
      if (i < n) {
        const int e = static_cast<int>(i % E);
        atomicAdd(&s_tot[e], v[u]);
        if (i / E < chunk) atomicAdd(&s_bef[e], v[u]);
      }
    }
  }
  __syncthreads();
  // exclusive prefixes over experts: thread t takes experts [t*G, t*G + G)
  const int G = (Ex + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
  const int e0 = min(tid * G, Ex), e1 = min(e0 + G, Ex);
  int32_t c_loc = 0, p_loc = 0;
  for (int e = e0; e < e1; ++e) {
    c_loc += s_tot[e];
    p_loc += (s_tot[e] + BM - 1) / BM * BM;
  }
  int32_t* tot = warp_tot + 32;
  const int32_t c_base = block_exclusive_scan(c_loc, warp_tot, tot);
  const int32_t p_base = block_exclusive_scan(p_loc, warp_tot, tot + 1);
  int32_t cr = c_base, pr = p_base;
  for (int e = e0; e < e1; ++e) {
    s_off[e] = cr;
    s_poff[e] = pr;
    cr += s_tot[e];
    pr += (s_tot[e] + BM - 1) / BM * BM;
  }
  if (tid == 0) {
    s_off[Ex] = tot[0];
    s_poff[Ex] = tot[1];
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e <= Ex; e += blockDim.x) {
      if (e < Ex) m.counts[e] = s_tot[e];
      m.offsets[e] = s_off[e];
      m.poff[e] = s_poff[e];
    }
  }
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
  const int64_t gs = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = g0; g < static_cast<int64_t>(Ex) * BM; g += gs) {
    const int e = static_cast<int>(g / BM);
    const int32_t r = s_poff[e] + s_tot[e] + static_cast<int32_t>(g % BM);
    if (r < s_poff[e + 1]) m.prow2slot[r] = -1;
  }
  for (int64_t i = g0; i < zero_count; i += gs) tickets[i] = 0;
}

// FUSED: the scan above runs in every block (chunk_base holds the chunk
// histograms); else chunk_base holds each chunk's first row per expert and
// counts/offsets/poff come from route_scan_kernel.
template <bool FUSED>
__global__ void __launch_bounds__(RWARPS * 32) route_rank_kernel(
    const int32_t* __restrict__ ids, int64_t TK, int E, int Ex, int32_t T, int64_t nchunks,
    MetaPtrs m, CtrlPtrs c, int64_t zero_count, int32_t* slot2row, int32_t* row2slot) {
  // [RWARPS][E]: per-warp counts, then cursors; FUSED: then per expert its
  // total [Ex], earlier-chunk slots [Ex], offset [Ex + 1], padded offset [Ex + 1]
  extern __shared__ int32_t sh[];
  __shared__ int32_t warp_tot[34];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* cnt = sh + warp * E;
  int32_t* s_tot = sh + RWARPS * E;
  int32_t* s_bef = s_tot + Ex;
  int32_t* s_off = s_bef + Ex;
  int32_t* s_poff = s_off + Ex + 1;
  const int64_t chunk = blockIdx.x;
  const int64_t c0 = chunk * RCHUNK;
  const int64_t c1 = (c0 + RCHUNK < TK ? c0 + RCHUNK : TK);
  const int64_t s0 = c0 + static_cast<int64_t>(warp) * WSLOTS;
  grid_dep_wait();
  grid_dep_launch();
  int v[RSTEPS];
  load_chunk_ids(ids, s0, c1, lane, v);
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  // 1. this warp's slots per expert (one lane per group of equal ids adds)
#pragma unroll
  for (int j = 0; j < RSTEPS; ++j) {
    if (s0 + 32 * j < c1) {  // warp-uniform
      const int e = v[j];
      const bool ok = static_cast<unsigned>(e) < static_cast<unsigned>(E);
      const int key = ok ? e : -1 - lane;  // invalid lanes never group
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (ok && lane == 31 - __clz(peers)) cnt[e] += __popc(peers);
      __syncwarp();
    }
  }
  if constexpr (FUSED) {
    route_scan_in_block(E, Ex, T, nchunks, chunk, c.chunk_base, m, c.tickets, zero_count, s_tot,
                        s_bef, s_off, s_poff, warp_tot);
  }
  __syncthreads();
  // 2. cursor of warp w for expert e: the padded row of its first slot of e
  //    = the chunk's first row of e + the slots of e in warps 0 .. w-1
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = FUSED ? s_poff[e] + s_bef[e]
                        : c.chunk_base[chunk * E + e] + (m.poff[e] - m.offsets[e]);
#pragma unroll
    for (int w = 0; w < RWARPS; ++w) {
      const int32_t cw = sh[w * E + e];
      sh[w * E + e] = run;
      run += cw;
    }
  }
  __syncthreads();
  // 3. stable ranks inside the warp, rows from the cursors
#pragma unroll
  for (int j = 0; j < RSTEPS; ++j) {
    if (s0 + 32 * j < c1) {  // warp-uniform
      const int64_t s = s0 + 32 * j + lane;
      const bool in = s < c1;
      const int e = v[j];
      const bool ok = in && static_cast<unsigned>(e) < static_cast<unsigned>(E);
      const int key = ok ? e : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      int32_t prow = 0;
      if (ok) prow = cnt[e] + __popc(peers & ((1u << lane) - 1u));
      __syncwarp();
      if (ok && lane == 31 - __clz(peers)) cnt[e] += __popc(peers);
      __syncwarp();
      if (ok) {
        m.slot2prow[s] = prow;
        m.prow2slot[prow] = static_cast<int32_t>(s);
        if (slot2row) {
          const int32_t shift = FUSED ? s_poff[e] - s_off[e] : m.poff[e] - m.offsets[e];
          const int32_t row = prow - shift;
          slot2row[s] = row;
          row2slot[row] = static_cast<int32_t>(s);
        }
      } else if (in) {
        m.slot2prow[s] = -1;
        if (slot2row) slot2row[s] = -1;
      }
    }
  }
}

static bool route_fused(const Plan& p) {
  return p.nchunks > 0 && p.nchunks * p.E <= ROUTE_FUSE_MAX && p.E <= ROUTE_FUSE_MAX_E;
}

int route_launches(const Plan& p) { return p.nchunks == 0 ? 1 : (route_fused(p) ? 2 : 3); }

cudaError_t launch_route(const Plan& p, const int32_t* ids, MetaPtrs m, CtrlPtrs c,
                         int32_t* slot2row, int32_t* row2slot, unsigned* status,
                         cudaStream_t st, bool pdl) {
  const int E = static_cast<int>(p.E), Ex = static_cast<int>(p.Ex);
  const int32_t T = static_cast<int32_t>(p.T);
  const unsigned blocks = static_cast<unsigned>(p.nchunks);  // one block per chunk
  cudaError_t err = cudaSuccess;
  if (p.nchunks > 0) {
    err = launch_kernel(route_count_kernel, blocks, RWARPS * 32, sizeof(int32_t) * E, st, pdl, 1,
                        ids, p.TK, E, p.nchunks, c.chunk_base, status);
    if (err != cudaSuccess) return err;
  }
  if (route_fused(p)) {
    const size_t smem = sizeof(int32_t) * (RWARPS * E + 4 * (Ex + 1));
    return launch_kernel(route_rank_kernel<true>, blocks, RWARPS * 32, smem, st, pdl, 1, ids,
                         p.TK, E, Ex, T, p.nchunks, m, c, p.ctrl_zero_count, slot2row, row2slot);
  }
  err = launch_kernel(route_scan_kernel, 1, 1024, 0, st, pdl, 1, E, Ex, T, p.nchunks, m, c,
                      p.ctrl_zero_count);
  if (err != cudaSuccess) return err;
  if (p.nchunks > 0) {
    const size_t smem = sizeof(int32_t) * RWARPS * E;
    err = launch_kernel(route_rank_kernel<false>, blocks, RWARPS * 32, smem, st, pdl, 1, ids,
                        p.TK, E, Ex, T, p.nchunks, m, c, p.ctrl_zero_count, slot2row, row2slot);
  }
  return err;
}

}  // namespace hmm
