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
// Three launches: per-chunk histograms -> one-block scan -> per-chunk stable
// ranks.  A chunk (1024 slots) belongs to one block of 8 warps, 128 slots per
// warp: warp match_any groups equal ids inside each 32-slot step, so the order
// inside a warp follows s, and the warps' per-expert counts are prefix-summed
// in shared memory, so the order across warps follows s too.  Each warp loads
// its ids into registers before the first step, so the steps do not wait on
// global loads one after another.
#include "hmm_internal.h"

namespace hmm {

constexpr int WSLOTS = RCHUNK / RWARPS;  // slots per warp of a chunk
constexpr int RSTEPS = WSLOTS / 32;      // 32-slot steps per warp

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

// Block-wide exclusive scan of one value per thread (blockDim.x == 1024).
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_tot, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t inc = v;
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int32_t wv = warp_tot[lane];
    int32_t winc = wv;
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, winc, d);
      if (lane >= d) winc += n;
    }
    warp_tot[lane] = winc - wv;
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

__global__ void __launch_bounds__(RWARPS * 32) route_rank_kernel(
    const int32_t* __restrict__ ids, int64_t TK, int E, int64_t nchunks, MetaPtrs m,
    const int32_t* __restrict__ chunk_base, int32_t* slot2row, int32_t* row2slot) {
  extern __shared__ int32_t sh[];  // [RWARPS][E]: per-warp counts, then cursors
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* cnt = sh + warp * E;
  const int64_t chunk = blockIdx.x;
  const int64_t c0 = chunk * RCHUNK;
  const int64_t c1 = (c0 + RCHUNK < TK ? c0 + RCHUNK : TK);
  const int64_t s0 = c0 + static_cast<int64_t>(warp) * WSLOTS;
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
  __syncthreads();
  // 2. cursor of warp w for expert e: the padded row of its first slot of e
  //    = the chunk's first row of e + the slots of e in warps 0 .. w-1
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = chunk_base[chunk * E + e] + (m.poff[e] - m.offsets[e]);
#pragma unroll
    for (int w = 0; w < RWARPS; ++w) {
      const int32_t c = sh[w * E + e];
      sh[w * E + e] = run;
      run += c;
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
          const int32_t row = prow - (m.poff[e] - m.offsets[e]);
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

cudaError_t launch_route(const Plan& p, const int32_t* ids, MetaPtrs m, CtrlPtrs c,
                         int32_t* slot2row, int32_t* row2slot, unsigned* status,
                         cudaStream_t st) {
  const int E = static_cast<int>(p.E);
  const int blocks = static_cast<int>(p.nchunks);  // one block per chunk
  const size_t smem = sizeof(int32_t) * RWARPS * E;
  if (p.nchunks > 0) {
    route_count_kernel<<<blocks, RWARPS * 32, sizeof(int32_t) * E, st>>>(ids, p.TK, E, p.nchunks,
                                                                       c.chunk_base, status);
  }
  route_scan_kernel<<<1, 1024, 0, st>>>(E, static_cast<int>(p.Ex), static_cast<int32_t>(p.T),
                                        p.nchunks, m, c, p.ctrl_zero_count);
  if (p.nchunks > 0) {
    route_rank_kernel<<<blocks, RWARPS * 32, smem, st>>>(ids, p.TK, E, p.nchunks, m,
                                                         c.chunk_base, slot2row, row2slot);
  }
  return cudaGetLastError();
}

}  // namespace hmm
