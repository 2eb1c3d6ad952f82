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
// Three launches: per-warp-chunk histograms -> one-block scan -> per-chunk
// stable ranks (warp match_any groups equal ids inside each 32-slot step, so
// the order inside a chunk follows s).
#include "hmm_internal.h"

namespace hmm {

__global__ void __launch_bounds__(RWARPS * 32) route_count_kernel(const int32_t* __restrict__ ids,
                                                                  int64_t TK, int E,
                                                                  int64_t nchunks,
                                                                  int32_t* __restrict__ chunk_cnt,
                                                                  unsigned* status) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* cnt = sh + warp * E;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * RWARPS + warp;
  if (chunk >= nchunks) return;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int64_t s0 = chunk * RCHUNK;
  const int64_t s1 = (s0 + RCHUNK < TK ? s0 + RCHUNK : TK);
  bool bad = false;
  for (int64_t s = s0 + lane; s < s1; s += 32) {
    const int e = ids[s];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&cnt[e], 1);
    else
      bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, HMM_STATUS_EXPERT_ID);
  __syncwarp();
  for (int e = lane; e < E; e += 32) chunk_cnt[chunk * E + e] = cnt[e];
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

__global__ void __launch_bounds__(1024) route_scan_kernel(int E, int64_t nchunks, MetaPtrs m,
                                                          CtrlPtrs c, int64_t zero_count) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t tot_cnt, tot_pad;
  const int e = threadIdx.x;
  int32_t cnt = 0;
  if (e < E) {
    for (int64_t ch = 0; ch < nchunks; ++ch) {
      const int32_t v = c.chunk_base[ch * E + e];
      c.chunk_base[ch * E + e] = cnt;
      cnt += v;
    }
  }
  const int32_t padded = (cnt + BM - 1) / BM * BM;
  const int32_t off = block_exclusive_scan(cnt, warp_tot, &tot_cnt);
  const int32_t poff = block_exclusive_scan(padded, warp_tot, &tot_pad);
  if (e < E) {
    m.counts[e] = cnt;
    m.offsets[e] = off;
    m.poff[e] = poff;
    for (int64_t ch = 0; ch < nchunks; ++ch) c.chunk_base[ch * E + e] += off;
    for (int32_t r = poff + cnt; r < poff + padded; ++r) m.prow2slot[r] = -1;
  }
  if (e == 0) {
    m.offsets[E] = tot_cnt;
    m.poff[E] = tot_pad;
  }
  // tickets, per-M-tile and per-expert ready counters of this call
  for (int64_t i = e; i < zero_count; i += blockDim.x) c.tickets[i] = 0;
}

__global__ void __launch_bounds__(RWARPS * 32) route_rank_kernel(
    const int32_t* __restrict__ ids, int64_t TK, int E, int64_t nchunks, MetaPtrs m,
    const int32_t* __restrict__ chunk_base, int32_t* slot2row, int32_t* row2slot) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* cnt = sh + warp * E;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * RWARPS + warp;
  if (chunk >= nchunks) return;
  for (int e = lane; e < E; e += 32) cnt[e] = chunk_base[chunk * E + e];
  __syncwarp();
  const int64_t s0 = chunk * RCHUNK;
  const int64_t s1 = (s0 + RCHUNK < TK ? s0 + RCHUNK : TK);
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t s = base + lane;
    const bool in = s < s1;
    const int e = in ? ids[s] : -1;
    const bool ok = in && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const int key = ok ? e : -1 - lane;  // invalid lanes never group
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    int32_t row = 0;
    if (ok) row = cnt[e] + __popc(peers & ((1u << lane) - 1u));
    __syncwarp();
    if (ok && lane == 31 - __clz(peers)) cnt[e] += __popc(peers);
    __syncwarp();
    if (ok) {
      const int32_t prow = m.poff[e] + (row - m.offsets[e]);
      m.slot2prow[s] = prow;
      m.prow2slot[prow] = static_cast<int32_t>(s);
      if (slot2row) {
        slot2row[s] = row;
        row2slot[row] = static_cast<int32_t>(s);
      }
    } else if (in) {
      m.slot2prow[s] = -1;
      if (slot2row) slot2row[s] = -1;
    }
  }
}

cudaError_t launch_route(const Plan& p, const int32_t* ids, MetaPtrs m, CtrlPtrs c,
                         int32_t* slot2row, int32_t* row2slot, unsigned* status,
                         cudaStream_t st) {
  const int E = static_cast<int>(p.E);
  const int blocks = static_cast<int>((p.nchunks + RWARPS - 1) / RWARPS);
  const size_t smem = sizeof(int32_t) * RWARPS * E;
  if (p.nchunks > 0) {
    route_count_kernel<<<blocks, RWARPS * 32, smem, st>>>(ids, p.TK, E, p.nchunks, c.chunk_base,
                                                          status);
  }
  route_scan_kernel<<<1, 1024, 0, st>>>(E, p.nchunks, m, c, p.ctrl_zero_count);
  if (p.nchunks > 0) {
    route_rank_kernel<<<blocks, RWARPS * 32, smem, st>>>(ids, p.TK, E, p.nchunks, m,
                                                         c.chunk_base, slot2row, row2slot);
  }
  return cudaGetLastError();
}

}  // namespace hmm
