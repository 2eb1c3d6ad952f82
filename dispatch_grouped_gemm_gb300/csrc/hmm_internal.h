// hmm_internal.h -- declarations shared by the library's translation units
// (not part of the public ABI; the public header is include/hmm.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "hmm.h"

namespace hmm {

// Every expert's rows start on a multiple of BM in the permuted ("padded")
// layout, so no GEMM tile or K block spans two experts; padding rows are
// zero (x_perm, dy_perm) or computed from zeros (a, h, dH, w*a).
constexpr int BM = 128;
constexpr int BK = 64;    // K per pipeline stage (one 128-byte swizzle row of bf16)
// Token blocks of the row-mode GEMMs end at the first multiple of TROWS at or
// past an expert's last row, and so do the weight gradients' K blocks: the
// padding rows up to there are the only ones any kernel reads.
constexpr int TROWS = 64;
constexpr int RCHUNK = 1024;  // slots per routing warp-chunk
constexpr int RWARPS = 8;     // warps per routing block
constexpr int MAX_E = 1024;   // experts supported (routing keeps per-expert counters in smem)
constexpr int NUM_TICKETS = 8;

// Device-side metadata of one call (lives in `saved` when training, else in
// the forward workspace).  All int32.
struct MetaPtrs {
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1]  unpadded exclusive prefix of counts
  int32_t* poff;       // [E+1]  padded prefix: expert e owns rows [poff[e], poff[e+1])
  int32_t* slot2prow;  // [TK]   padded row of slot s (-1 for an invalid id)
  int32_t* prow2slot;  // [R]    slot of a padded row (-1 for padding)
};

// Scratch counters of one call.
struct CtrlPtrs {
  int32_t* chunk_base;  // [nchunks * E]
  int32_t* tickets;     // [NUM_TICKETS]      } contiguous: zeroed together
  int32_t* ready;       // [R / 64]           } at the start of every call
};

struct Plan {
  int64_t T, H, I, E, K, TK;
  int64_t shared;       // 1: the optional shared expert is expert E of the padded rows
  int64_t Ex;           // E + shared: experts of the padded row space
  int64_t R;            // capacity of the padded row space
  int64_t max_mtiles;   // R / BM
  int64_t nchunks;      // routing warp-chunks
  int64_t dwp_ld;       // per-row d_w partials (one per 32 columns of I)
  // row strides (bytes) of the fp8 arrays of the weight-gradient low halves,
  // padded to 16 bytes for TMA: H columns (x_perm8, dy_perm8), 2I (dH_lo8), I (wa_lo8)
  int64_t ld8_h, ld8_2i, ld8_i;
  bool training;
  // byte offsets inside the buffers
  size_t meta_bytes;
  size_t off_counts, off_offsets, off_poff, off_slot2prow, off_prow2slot;  // inside meta
  size_t ctrl_bytes;
  size_t off_chunk_base, off_tickets, off_ready;                           // inside ctrl
  int64_t ctrl_zero_count;  // int32 counters from off_tickets that each call zeroes
  // forward: saved = [meta | x_perm | x_perm8 | h]   (training)
  //          workspace = [ctrl | cmb | a | o]       (training)
  //          workspace = [ctrl | cmb | meta | x_perm | a | o]   (inference)
  // cmb: the fused combine's counters, one per (token, 32-column segment of
  // H): cmb_count int32, zeroed by the dispatch of x when used
  size_t saved_bytes, fwd_ws_bytes;
  size_t sv_meta, sv_xperm, sv_x8, sv_h;
  size_t fw_ctrl, fw_cmb, fw_meta, fw_xperm, fw_a, fw_o;
  int64_t cmb_nseg, cmb_count;
  // backward workspace =
  //   [ctrl | dy_perm | dy_perm8 | wperm | dH | dH_lo8 | wa | wa_lo8 | dX_perm | dwp]
  size_t bwd_ws_bytes;
  size_t bw_ctrl, bw_dyperm, bw_dy8, bw_wperm, bw_dh, bw_dhlo, bw_wa, bw_walo, bw_dxperm, bw_dwp;
};

// HMM_OK, or the error code for a shape outside the supported range (sizes,
// dtype, the shared flag, H / I not multiples of 8, a padded row space past
// 2^31 rows).  Every entry point calls it before any device work.
int check_shape(const hmm_shape* s);
int make_plan(const hmm_shape* s, bool training, Plan* p);
MetaPtrs meta_at(const Plan& p, void* base);
CtrlPtrs ctrl_at(const Plan& p, void* base);

// ------------------------------------------- programmatic dependent launches
// Every kernel of the library may be launched with programmatic stream
// serialization (pdl): it is then scheduled while the previous kernel of its
// stream drains, runs its set-up (barriers, TMEM) meanwhile, and calls
// grid_dep_wait() before its first access to global memory; that returns once
// the previous kernel has completed and its writes are visible, and is a
// no-op in a kernel launched without the attribute.  grid_dep_launch() lets
// the stream's next kernel be scheduled once every CTA has called it (or
// exited): the short kernels call it right after their wait, the persistent
// GEMMs when a CTA has issued the loads of its last tile, so that the next
// kernel's CTAs wait beside the GEMM's tail only.  Event records and waits
// between launches keep their full ordering.
#ifdef __CUDACC__
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Launch `kern` on `st` (clusters of cluster_x CTAs when > 1; with pdl, with
// programmatic stream serialization).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------ kernel launchers
// Each returns a cudaError_t of its launch; pdl as for launch_kernel.
cudaError_t launch_route(const Plan& p, const int32_t* ids, MetaPtrs m, CtrlPtrs c,
                         int32_t* slot2row, int32_t* row2slot, unsigned* status,
                         cudaStream_t st, bool pdl);
int route_launches(const Plan& p);  // kernels launch_route launches for p
// x8 (training, else null): also x_perm as e4m3 (ld8_h bytes per row).  Also
// zeroes zero_count int32 at zero_ptr (may be null).
cudaError_t launch_dispatch_x(const Plan& p, const void* x, MetaPtrs m, void* x_perm, void* x8,
                              int32_t* zero_ptr, int64_t zero_count, cudaStream_t st, bool pdl);
cudaError_t launch_combine_y(const Plan& p, const void* o, const void* w, int w_dtype, MetaPtrs m,
                             void* y, cudaStream_t st, bool pdl);
// also dy_perm as e5m2 (dy8, ld8_h bytes per row)
cudaError_t launch_dispatch_dy(const Plan& p, const void* dy, const void* w, int w_dtype,
                               MetaPtrs m, CtrlPtrs c, void* dy_perm, void* dy8, float* wperm,
                               cudaStream_t st, bool pdl);
cudaError_t launch_combine_dx(const Plan& p, const void* dx_perm, const float* dwp, MetaPtrs m,
                              void* dx, void* dw, int w_dtype, cudaStream_t st, bool pdl);

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct GemmEnv {
  EncodeTiledFn encode;
  int num_sms;
  uint64_t* trace;   // tile timeline buffer of the traced launch (null: off)
  int trace_cap;     // records per CTA
  int trace_which;   // which GEMM launch kind is traced
  int pair_rows;     // forward and data-gradient GEMMs on CTA pairs (2-SM MMA)
  int small_rows;    // ... on single CTAs with token blocks of at most 64 rows
  unsigned* status;
  uint64_t budget_ns;
  cudaStream_t stream;
  bool pdl;          // programmatic dependent launches (launch_kernel)
};

// forward GMM1(+SwiGLU) and GMM2 in one persistent launch with per-token-block
// ready counters, for the routed experts and (p.shared) the shared expert
// (Ws1 [H, 2I], Ws2 [I, H]).  h32 may be null (inference).
// fused_y != null: the combine runs in the GMM2 epilogue (counters cmb, the
// routing weights w of dtype w_dtype) and writes y.
int launch_forward_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                         const void* x_perm, const void* W1, const void* W2, const void* Ws1,
                         const void* Ws2, void* a, float* h32, void* o, bool skip_ready_release,
                         int* cmb, const void* w, int w_dtype, void* fused_y);
// backward data gradients in one persistent launch: act_grad (+SwiGLU grad,
// d_w partials; dH and w*a written as a bf16 high part plus an e5m2 low part)
// and input-grad (released per token block), routed and shared experts.
// skip_ready_release: test-only fault injection (the input-grad waits run out).
int launch_data_grad_gemms(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                           const void* dy_perm, const float* wperm, const float* h32,
                           const void* W1, const void* W2, const void* Ws1, const void* Ws2,
                           void* dH, void* dH_lo, void* wa, void* wa_lo, float* dwp,
                           void* dx_perm, bool skip_ready_release);
// weight gradients on CTA pairs (tcgen05 cta_group::2), 256 x 256 tiles:
// dW1 / dW2 of the routed experts and dWs1 / dWs2 of the shared expert (any
// may be null).  The low parts (dH_lo8, wa_lo8: e5m2) meet fp8 copies of the
// other operand (x8: e4m3, dy8: e5m2) in a second, fp8 MMA.
// Tiles go out longest first by a ticket in c.tickets[2..3] (zeroed by the
// backward dispatch; every launch leaves them zero again).
int launch_wgrad_pair(const GemmEnv& env, const Plan& p, MetaPtrs m, CtrlPtrs c,
                      const void* x_perm,
                      const void* x8, const void* dy_perm, const void* dy8, const void* dH,
                      const void* dH_lo8, const void* wa, const void* wa_lo8, void* dW1,
                      void* dW2, void* dWs1, void* dWs2);

}  // namespace hmm
