// hmm_api.cu -- the C ABI of include/hmm.h: host-side validation, buffer
// planning and the launch sequence of the forward and backward.
//
// [HyperMegaMoE §2.3 / §10] the operator offers a workspace query plus an
// execute call for the forward and for the backward; [§3.3] routing offsets,
// counters, tiling and buffers are internal; [§4.2] bad shapes, dtypes,
// layouts and capacities are rejected at the host boundary before any
// device work; [§5.3] buffer capacity and workspace size are computed and
// checked on the host, and per-call event state is reset so that repeated
// iterations never see stale counters (the routing kernel and the backward
// dispatch kernel zero the tickets and ready counters of their call).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <utility>
#include <vector>

#include "hmm_internal.h"

namespace {

struct PhaseInfo {
  const char* name;
  int kernels;
};
constexpr PhaseInfo kPhases[HMM_NUM_PHASES] = {
    // route launches 2 or 3 kernels (route_launches); 3 is the most
    {"route", 3},       {"dispatch_x", 1},    {"gemm_fwd", 1},        {"combine_y", 1},
    {"dispatch_dy", 1}, {"gemm_bwd_data", 1}, {"gemm_bwd_weight", 1}, {"combine_dx", 1}};
enum Phase {
  PH_ROUTE = 0, PH_DISPATCH_X, PH_GEMM_FWD, PH_COMBINE_Y, PH_DISPATCH_DY, PH_GEMM_BWD_DATA,
  PH_GEMM_BWD_WEIGHT, PH_COMBINE_DX
};

struct ProfRec {
  int phase;
  int kernels;  // kernels the phase launched
  cudaEvent_t begin, end;
};

}  // namespace

struct hmm_ctx {
  int device = -1;
  int num_sms = 0;
  unsigned* status = nullptr;  // device status word
  int validate = 0;
  uint64_t budget_ns = 2000000000ull;
  int inject_skip_ready = 0;
  int profile = 0;
  int pair_rows = 2;  // 0 single CTAs, 1 CTA pairs, 2 automatic, 3 single CTAs, small blocks
  int overlap = 1;    // programmatic dependent launches
  int fused_combine = 0;  // combine in the GMM2 epilogue
  uint64_t* trace = nullptr;
  size_t trace_bytes = 0;
  int trace_which = 0;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> pool;
  hmm::EncodeTiledFn encode = nullptr;
  // second stream of the backward: the dx / d_topk_weights combine runs there
  // beside the weight-gradient GEMMs (fork and join events on the caller's
  // stream)
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

namespace {

cudaEvent_t take_event(hmm_ctx* c) {
  if (!c->pool.empty()) {
    cudaEvent_t e = c->pool.back();
    c->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launch phase with events on the launching stream when
// profiling is on.
struct PhaseScope {
  hmm_ctx* c;
  int phase;
  cudaStream_t st;
  int kernels;
  cudaEvent_t begin = nullptr;
  PhaseScope(hmm_ctx* ctx, int ph, cudaStream_t s, int nkern = -1)
      : c(ctx), phase(ph), st(s), kernels(nkern >= 0 ? nkern : kPhases[ph].kernels) {
    if (c->profile && (begin = take_event(c)) != nullptr) cudaEventRecord(begin, st);
  }
  ~PhaseScope() {
    if (!begin) return;
    cudaEvent_t end = take_event(c);
    if (!end) {
      c->pool.push_back(begin);
      return;
    }
    cudaEventRecord(end, st);
    c->recs.push_back({phase, kernels, begin, end});
  }
};

}  // namespace

namespace hmm {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int make_plan(const hmm_shape* s, bool training, Plan* p) {
  std::memset(p, 0, sizeof(*p));
  p->T = s->T;
  p->H = s->H;
  p->I = s->I;
  p->E = s->E;
  p->K = s->K;
  p->TK = s->T * s->K;
  p->shared = s->shared;
  p->Ex = p->E + p->shared;
  p->training = training;
  const int64_t TK = p->TK;
  // padded rows: the routed slots and the shared expert's T rows, each
  // expert's segment rounded up to BM
  const int64_t rows = TK == 0 ? 0 : TK + p->shared * p->T;
  int64_t R = rows == 0 ? 0 : rows + std::min<int64_t>(p->Ex, rows) * (BM - 1);
  R = (R + BM - 1) / BM * BM;
  p->R = R;
  p->max_mtiles = R / BM;
  p->nchunks = (TK + RCHUNK - 1) / RCHUNK;
  p->dwp_ld = (p->I + 31) / 32;  // one d_w partial per row and 32-column block of I
  p->ld8_h = (p->H + 15) / 16 * 16;
  p->ld8_2i = (2 * p->I + 15) / 16 * 16;
  p->ld8_i = (p->I + 15) / 16 * 16;
  const size_t A = 256;
  size_t o = 0;
  p->off_counts = o;    o = align_up(o + 4 * p->Ex, A);
  p->off_offsets = o;   o = align_up(o + 4 * (p->Ex + 1), A);
  p->off_poff = o;      o = align_up(o + 4 * (p->Ex + 1), A);
  p->off_slot2prow = o; o = align_up(o + 4 * TK, A);
  p->off_prow2slot = o; o = align_up(o + 4 * R, A);
  p->meta_bytes = o;
  o = 0;
  p->off_chunk_base = o; o = align_up(o + 4 * p->nchunks * p->E, A);
  p->off_tickets = o;
  p->off_ready = o + 4 * NUM_TICKETS;  // tickets and ready counters contiguous (zeroed together)
  // one ready counter per 64 padded rows (token blocks start on multiples of 64)
  p->ctrl_zero_count = NUM_TICKETS + R / 64;
  o = align_up(p->off_ready + 4 * (R / 64), A);
  p->ctrl_bytes = o;
  const size_t xperm = align_up(static_cast<size_t>(R) * p->H * 2, A);
  // fp32 pre-activations in 32 x 32 blocks (gate and up), columns padded to 32
  const size_t hbytes = align_up(static_cast<size_t>(R) * 2 * ((p->I + 31) / 32 * 32) * 4, A);
  const size_t abytes = align_up(static_cast<size_t>(R) * p->I * 2, A);
  // o: fp32 with the shared expert (its unweighted term in the y combine),
  // else bf16
  const size_t obytes = align_up(static_cast<size_t>(R) * p->H * (p->shared ? 4 : 2), A);
  // the fused combine's counters: one per token and 32-column segment of H
  p->cmb_nseg = (p->H + 31) / 32;
  p->cmb_count = p->T * p->cmb_nseg;
  const size_t cmb_bytes = align_up(static_cast<size_t>(p->cmb_count) * 4, A);
  if (training) {
    p->sv_meta = 0;
    p->sv_xperm = p->meta_bytes;
    p->sv_x8 = p->sv_xperm + xperm;
    p->sv_h = p->sv_x8 + align_up(static_cast<size_t>(R) * p->ld8_h, A);
    p->saved_bytes = p->sv_h + hbytes;
    p->fw_ctrl = 0;
    p->fw_cmb = p->ctrl_bytes;
    p->fw_a = p->fw_cmb + cmb_bytes;
    p->fw_o = p->fw_a + abytes;
    p->fwd_ws_bytes = p->fw_o + obytes;
  } else {
    p->saved_bytes = 0;
    p->fw_ctrl = 0;
    p->fw_cmb = p->ctrl_bytes;
    p->fw_meta = p->fw_cmb + cmb_bytes;
    p->fw_xperm = p->fw_meta + p->meta_bytes;
    p->fw_a = p->fw_xperm + xperm;
    p->fw_o = p->fw_a + abytes;
    p->fwd_ws_bytes = p->fw_o + obytes;
  }
  o = 0;
  p->bw_ctrl = o;    o = align_up(o + p->ctrl_bytes, A);
  p->bw_dyperm = o;  o = align_up(o + static_cast<size_t>(R) * p->H * 2, A);
  p->bw_dy8 = o;     o = align_up(o + static_cast<size_t>(R) * p->ld8_h, A);
  p->bw_wperm = o;   o = align_up(o + static_cast<size_t>(R) * 4, A);
  p->bw_dh = o;      o = align_up(o + static_cast<size_t>(R) * 2 * p->I * 2, A);
  p->bw_dhlo = o;    o = align_up(o + static_cast<size_t>(R) * p->ld8_2i, A);
  p->bw_wa = o;      o = align_up(o + static_cast<size_t>(R) * p->I * 2, A);
  p->bw_walo = o;    o = align_up(o + static_cast<size_t>(R) * p->ld8_i, A);
  // dX_perm: fp32 with the shared expert (see the dX combine), else bf16
  p->bw_dxperm = o;  o = align_up(o + static_cast<size_t>(R) * p->H * (p->shared ? 4 : 2), A);
  p->bw_dwp = o;     o = align_up(o + static_cast<size_t>(R) * p->dwp_ld * 4, A);
  p->bwd_ws_bytes = o;
  return HMM_OK;
}

MetaPtrs meta_at(const Plan& p, void* base) {
  uint8_t* b = static_cast<uint8_t*>(base);
  MetaPtrs m;
  m.counts = reinterpret_cast<int32_t*>(b + p.off_counts);
  m.offsets = reinterpret_cast<int32_t*>(b + p.off_offsets);
  m.poff = reinterpret_cast<int32_t*>(b + p.off_poff);
  m.slot2prow = reinterpret_cast<int32_t*>(b + p.off_slot2prow);
  m.prow2slot = reinterpret_cast<int32_t*>(b + p.off_prow2slot);
  return m;
}

CtrlPtrs ctrl_at(const Plan& p, void* base) {
  uint8_t* b = static_cast<uint8_t*>(base);
  CtrlPtrs c;
  c.chunk_base = reinterpret_cast<int32_t*>(b + p.off_chunk_base);
  c.tickets = reinterpret_cast<int32_t*>(b + p.off_tickets);
  c.ready = reinterpret_cast<int32_t*>(b + p.off_ready);
  return c;
}

// Host-side limits of every entry point [HyperMegaMoE §4.2: shapes, dtypes
// and layouts are rejected at the boundary, before any device work].
int check_shape(const hmm_shape* s) {
  if (!s) return HMM_ERR_ARG;
  if (s->shared != 0 && s->shared != 1) return HMM_ERR_ARG;
  if (s->weights_dtype != HMM_DTYPE_BF16 && s->weights_dtype != HMM_DTYPE_F32)
    return HMM_ERR_DTYPE;
  if (s->T < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->K <= 0) return HMM_ERR_SHAPE;
  // the shared expert is one more expert and, in the dispatch, one more slot
  if (s->E + s->shared > MAX_E || s->K + s->shared > 32) return HMM_ERR_SHAPE;
  if (s->H > (1 << 20) || s->I > (1 << 20) || s->T > (int64_t(1) << 31)) return HMM_ERR_SHAPE;
  if (s->H % 8 != 0 || s->I % 8 != 0) return HMM_ERR_LAYOUT;
  const int64_t TK = s->T * (s->K + s->shared);
  const int64_t R = TK + std::min<int64_t>(s->E + s->shared, TK) * (BM - 1) + BM;
  if (R >= (int64_t(1) << 31) - 1) return HMM_ERR_SHAPE;
  return HMM_OK;
}

}  // namespace hmm

using namespace hmm;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (ok && prev >= 0) cudaSetDevice(prev);
  }
};

GemmEnv env_of(hmm_ctx* ctx, const Plan& p, cudaStream_t st) {
  GemmEnv e;
  e.encode = ctx->encode;
  e.num_sms = ctx->num_sms;
  // pairs (half the tiles, half the token rows staged per SM) pay off when
  // experts average a full 256-row token block; below 64 rows per expert the
  // launches stream weights, best with small token blocks and more stages
  int mode = ctx->pair_rows;
  if (mode == 2) mode = p.TK >= 2 * BM * p.E ? 1 : (p.TK < 64 * p.E ? 3 : 0);
  e.pair_rows = mode == 1 ? 1 : 0;
  e.small_rows = mode == 3 ? 1 : 0;
  e.trace = ctx->trace;
  e.trace_cap = ctx->trace ? static_cast<int>(ctx->trace_bytes / (64 * ctx->num_sms)) : 0;
  e.trace_which = ctx->trace_which;
  e.status = ctx->status;
  e.budget_ns = ctx->budget_ns;
  e.stream = st;
  e.pdl = ctx->overlap != 0;
  return e;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? HMM_OK : HMM_ERR_CUDA; }

int read_route_error(hmm_ctx* ctx, cudaStream_t st) {
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, ctx->status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return HMM_ERR_CUDA;
  if (v & HMM_STATUS_EXPERT_ID) {
    // clear the bit in stream order (the kernels of this call wrote v; the
    // timeout bit, if any, stays for hmm_status)
    const unsigned keep = v & ~HMM_STATUS_EXPERT_ID;
    if (cudaMemcpyAsync(ctx->status, &keep, sizeof keep, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return HMM_ERR_CUDA;
    return HMM_ERR_EXPERT_ID;
  }
  return HMM_OK;
}

}  // namespace

extern "C" {

int hmm_create(hmm_ctx** out, int device) {
  if (!out) return HMM_ERR_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return HMM_ERR_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return HMM_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return HMM_ERR_DEVICE;
  DeviceGuard g(device);
  if (!g.ok) return HMM_ERR_CUDA;
  hmm_ctx* c = new hmm_ctx();
  c->device = device;
  c->num_sms = prop.multiProcessorCount;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete c;
    return HMM_ERR_CUDA;
  }
  c->encode = reinterpret_cast<EncodeTiledFn>(fn);
  if (cudaMalloc(&c->status, sizeof(unsigned)) != cudaSuccess) {
    delete c;
    return HMM_ERR_CUDA;
  }
  if (cudaMemset(c->status, 0, sizeof(unsigned)) != cudaSuccess ||
      cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming) != cudaSuccess) {
    if (c->side) cudaStreamDestroy(c->side);
    if (c->fork) cudaEventDestroy(c->fork);
    cudaFree(c->status);
    delete c;
    return HMM_ERR_CUDA;
  }
  *out = c;
  return HMM_OK;
}

int hmm_destroy(hmm_ctx* ctx) {
  if (!ctx) return HMM_OK;
  {
    DeviceGuard g(ctx->device);
    for (auto& r : ctx->recs) {
      cudaEventSynchronize(r.end);
      cudaEventDestroy(r.begin);
      cudaEventDestroy(r.end);
    }
    for (cudaEvent_t e : ctx->pool) cudaEventDestroy(e);
    if (ctx->side) {
      cudaStreamSynchronize(ctx->side);
      cudaStreamDestroy(ctx->side);
    }
    if (ctx->fork) cudaEventDestroy(ctx->fork);
    if (ctx->join) cudaEventDestroy(ctx->join);
    if (ctx->status) cudaFree(ctx->status);
  }
  delete ctx;
  return HMM_OK;
}

int hmm_set_option(hmm_ctx* ctx, int option, int64_t value) {
  if (!ctx) return HMM_ERR_ARG;
  switch (option) {
    case HMM_OPT_VALIDATE:
      ctx->validate = value != 0;
      return HMM_OK;
    case HMM_OPT_WAIT_BUDGET_NS:
      if (value < 1000000 || value > 60000000000ll) return HMM_ERR_ARG;
      ctx->budget_ns = static_cast<uint64_t>(value);
      return HMM_OK;
    case HMM_OPT_INJECT_SKIP_READY:
      if (value < 0 || value > 2) return HMM_ERR_ARG;
      ctx->inject_skip_ready = static_cast<int>(value);
      return HMM_OK;
    case HMM_OPT_PROFILE:
      ctx->profile = value != 0;
      return HMM_OK;
    case HMM_OPT_PAIR_ROWS:
      if (value < 0 || value > 3) return HMM_ERR_ARG;
      ctx->pair_rows = static_cast<int>(value);
      return HMM_OK;
    case HMM_OPT_OVERLAP_LAUNCHES:
      ctx->overlap = value != 0;
      return HMM_OK;
    case HMM_OPT_FUSED_COMBINE:
      ctx->fused_combine = value != 0;
      return HMM_OK;
    default:
      return HMM_ERR_ARG;
  }
}

int hmm_workspace_size(const hmm_shape* shape, int training, size_t* fwd, size_t* saved,
                       size_t* bwd) {
  const int rc = check_shape(shape);
  if (rc != HMM_OK) return rc;
  Plan p;
  make_plan(shape, training != 0, &p);
  if (fwd) *fwd = p.fwd_ws_bytes;
  if (saved) *saved = p.saved_bytes;
  if (bwd) *bwd = training ? p.bwd_ws_bytes : 0;
  return HMM_OK;
}

int hmm_route(hmm_ctx* ctx, const hmm_shape* shape, const int32_t* topk_ids, int32_t* counts,
              int32_t* offsets, int32_t* slot2row, int32_t* row2slot, void* workspace,
              size_t workspace_bytes, void* stream) {
  if (!ctx) return HMM_ERR_ARG;
  // routing of the routed experts only: a shape with the shared expert is refused
  if (shape && shape->shared != 0) return HMM_ERR_ARG;
  int rc = check_shape(shape);
  if (rc != HMM_OK) return rc;
  Plan p;
  make_plan(shape, false, &p);
  if (!counts || !offsets || (p.TK > 0 && (!topk_ids || !slot2row || !row2slot)) || !workspace)
    return HMM_ERR_ARG;
  if (!aligned16(workspace)) return HMM_ERR_LAYOUT;
  if (workspace_bytes < p.ctrl_bytes + p.meta_bytes) return HMM_ERR_CAPACITY;
  DeviceGuard g(ctx->device);
  if (!g.ok) return HMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CtrlPtrs c = ctrl_at(p, workspace);
  MetaPtrs m = meta_at(p, static_cast<uint8_t*>(workspace) + p.ctrl_bytes);
  rc = cuda_rc(launch_route(p, topk_ids, m, c, slot2row, row2slot, ctx->status, st,
                                  ctx->overlap != 0));
  if (rc != HMM_OK) return rc;
  rc = cuda_rc(cudaMemcpyAsync(counts, m.counts, 4 * p.E, cudaMemcpyDeviceToDevice, st));
  if (rc != HMM_OK) return rc;
  rc = cuda_rc(cudaMemcpyAsync(offsets, m.offsets, 4 * (p.E + 1), cudaMemcpyDeviceToDevice, st));
  if (rc != HMM_OK) return rc;
  if (ctx->validate) return read_route_error(ctx, st);
  return HMM_OK;
}

namespace {

// hmm_forward and hmm_forward_shared (Ws1, Ws2: the shared expert's weights,
// exactly when shape->shared).
int forward_impl(hmm_ctx* ctx, const hmm_shape* shape, const void* x, const int32_t* topk_ids,
                 const void* topk_weights, const void* up_proj_weight,
                 const void* down_proj_weight, const void* Ws1, const void* Ws2, void* y,
                 void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
                 void* stream) {
  if (!ctx) return HMM_ERR_ARG;
  int rc = check_shape(shape);
  if (rc != HMM_OK) return rc;
  const bool training = saved != nullptr;
  Plan p;
  make_plan(shape, training, &p);
  if (p.TK > 0 && (!x || !topk_ids || !topk_weights || !up_proj_weight || !down_proj_weight ||
                   !y || !workspace || (p.shared && (!Ws1 || !Ws2))))
    return HMM_ERR_ARG;
  if (p.TK == 0) return HMM_OK;
  for (const void* ptr : {x, static_cast<const void*>(topk_ids), topk_weights, up_proj_weight,
                          down_proj_weight, static_cast<const void*>(y),
                          static_cast<const void*>(workspace), Ws1, Ws2})
    if (ptr && !aligned16(ptr)) return HMM_ERR_LAYOUT;
  if (training && !aligned16(saved)) return HMM_ERR_LAYOUT;
  if (workspace_bytes < p.fwd_ws_bytes) return HMM_ERR_CAPACITY;
  if (training && saved_bytes < p.saved_bytes) return HMM_ERR_CAPACITY;
  DeviceGuard g(ctx->device);
  if (!g.ok) return HMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* sv = static_cast<uint8_t*>(saved);
  CtrlPtrs c = ctrl_at(p, ws + p.fw_ctrl);
  MetaPtrs m = meta_at(p, training ? sv + p.sv_meta : ws + p.fw_meta);
  void* x_perm = training ? sv + p.sv_xperm : ws + p.fw_xperm;
  void* x8 = training ? sv + p.sv_x8 : nullptr;
  float* h32 = training ? reinterpret_cast<float*>(sv + p.sv_h) : nullptr;
  void* a = ws + p.fw_a;
  void* o = ws + p.fw_o;

  const bool fused = ctx->fused_combine != 0;
  int32_t* cmb = fused ? reinterpret_cast<int32_t*>(ws + p.fw_cmb) : nullptr;
  {
    PhaseScope ps(ctx, PH_ROUTE, st, route_launches(p));
    rc = cuda_rc(launch_route(p, topk_ids, m, c, nullptr, nullptr, ctx->status, st,
                              ctx->overlap != 0));
  }
  if (rc != HMM_OK) return rc;
  if (ctx->validate) {
    rc = read_route_error(ctx, st);
    if (rc != HMM_OK) return rc;
  }
  {
    PhaseScope ps(ctx, PH_DISPATCH_X, st);
    // (with the fused combine the dispatch also zeroes its counters)
    rc = cuda_rc(launch_dispatch_x(p, x, m, x_perm, x8, cmb, fused ? p.cmb_count : 0, st,
                                   ctx->overlap != 0));
  }
  if (rc != HMM_OK) return rc;
  const bool inject = ctx->inject_skip_ready == 1;
  if (inject) ctx->inject_skip_ready = 0;
  {
    PhaseScope ps(ctx, PH_GEMM_FWD, st);
    rc = launch_forward_gemms(env_of(ctx, p, st), p, m, c, x_perm, up_proj_weight, down_proj_weight,
                              Ws1, Ws2, a, h32, o, inject,
                              cmb, topk_weights, shape->weights_dtype, fused ? y : nullptr);
  }
  if (rc != HMM_OK || fused) return rc;
  PhaseScope ps(ctx, PH_COMBINE_Y, st);
  return cuda_rc(launch_combine_y(p, o, topk_weights, shape->weights_dtype, m, y, st,
                                ctx->overlap != 0));
}

}  // namespace

int hmm_forward(hmm_ctx* ctx, const hmm_shape* shape, const void* x, const int32_t* topk_ids,
                const void* topk_weights, const void* up_proj_weight,
                const void* down_proj_weight, void* y, void* saved, size_t saved_bytes,
                void* workspace, size_t workspace_bytes, void* stream) {
  if (shape && shape->shared != 0) return HMM_ERR_ARG;  // hmm_forward_shared
  return forward_impl(ctx, shape, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                      nullptr, nullptr, y, saved, saved_bytes, workspace, workspace_bytes, stream);
}

int hmm_forward_shared(hmm_ctx* ctx, const hmm_shape* shape, const void* x,
                       const int32_t* topk_ids, const void* topk_weights,
                       const void* up_proj_weight, const void* down_proj_weight,
                       const void* shared_up_proj_weight, const void* shared_down_proj_weight,
                       void* y, void* saved, size_t saved_bytes, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!shape || shape->shared != 1) return HMM_ERR_ARG;
  return forward_impl(ctx, shape, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                      shared_up_proj_weight, shared_down_proj_weight, y, saved, saved_bytes,
                      workspace, workspace_bytes, stream);
}

namespace {

enum BackwardMode { BWD_FULL = 0, BWD_DX = 1, BWD_DW = 2 };

// hmm_backward, hmm_backward_dx and hmm_backward_dw.  BWD_DX runs everything
// but the weight gradients and leaves their operands (dy_perm and its fp8
// copy, dH and w*a as bf16 high + e5m2 low parts) in the workspace; BWD_DW
// runs only the weight gradients from them and the saved x_perm (and its fp8
// copy).
int backward_impl(hmm_ctx* ctx, const hmm_shape* shape, const void* dy, const void* topk_weights,
                  const void* up_proj_weight, const void* down_proj_weight, const void* Ws1,
                  const void* Ws2, const void* saved, size_t saved_bytes, void* dx,
                  void* d_up_proj_weight, void* d_down_proj_weight, void* dWs1, void* dWs2,
                  void* d_topk_weights, void* workspace, size_t workspace_bytes, void* stream,
                  BackwardMode mode) {
  if (!ctx) return HMM_ERR_ARG;
  int rc = check_shape(shape);
  if (rc != HMM_OK) return rc;
  // the split entry points serve layers without a shared expert
  if (mode != BWD_FULL && shape->shared) return HMM_ERR_ARG;
  if (!shape->shared) dWs1 = dWs2 = nullptr;
  if (mode == BWD_DX) d_up_proj_weight = d_down_proj_weight = nullptr;
  if (mode == BWD_DW) dx = d_topk_weights = nullptr;
  Plan p;
  make_plan(shape, true, &p);
  DeviceGuard g(ctx->device);
  if (!g.ok) return HMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.TK == 0) {
    // no token: every weight gradient is exactly zero
    const size_t up = size_t(2) * p.H * 2 * p.I, down = size_t(2) * p.I * p.H;
    for (auto [ptr, bytes] : {std::pair<void*, size_t>{d_up_proj_weight, p.E * up},
                              std::pair<void*, size_t>{d_down_proj_weight, p.E * down},
                              std::pair<void*, size_t>{dWs1, up},
                              std::pair<void*, size_t>{dWs2, down}}) {
      if (!ptr) continue;
      if (!aligned16(ptr)) return HMM_ERR_LAYOUT;
      rc = cuda_rc(cudaMemsetAsync(ptr, 0, bytes, st));
      if (rc != HMM_OK) return rc;
    }
    return rc;
  }
  if (!saved || !workspace) return HMM_ERR_ARG;
  if (mode != BWD_DW && (!dy || !topk_weights || !up_proj_weight || !down_proj_weight))
    return HMM_ERR_ARG;
  if (p.shared && (!Ws1 || !Ws2)) return HMM_ERR_ARG;
  for (const void* ptr : {dy, topk_weights, up_proj_weight, down_proj_weight, Ws1, Ws2, saved,
                          static_cast<const void*>(workspace), static_cast<const void*>(dx),
                          static_cast<const void*>(d_up_proj_weight),
                          static_cast<const void*>(d_down_proj_weight),
                          static_cast<const void*>(dWs1), static_cast<const void*>(dWs2),
                          static_cast<const void*>(d_topk_weights)})
    if (ptr && !aligned16(ptr)) return HMM_ERR_LAYOUT;
  if (saved_bytes < p.saved_bytes) return HMM_ERR_CAPACITY;
  if (workspace_bytes < p.bwd_ws_bytes) return HMM_ERR_CAPACITY;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* sv = const_cast<uint8_t*>(static_cast<const uint8_t*>(saved));
  MetaPtrs m = meta_at(p, sv + p.sv_meta);
  const void* x_perm = sv + p.sv_xperm;
  const void* x8 = sv + p.sv_x8;
  const float* h32 = reinterpret_cast<const float*>(sv + p.sv_h);
  CtrlPtrs c = ctrl_at(p, ws + p.bw_ctrl);
  void* dy_perm = ws + p.bw_dyperm;
  void* dy8 = ws + p.bw_dy8;
  float* wperm = reinterpret_cast<float*>(ws + p.bw_wperm);
  void* dH = ws + p.bw_dh;
  void* dH_lo = ws + p.bw_dhlo;
  void* wa = ws + p.bw_wa;
  void* wa_lo = ws + p.bw_walo;
  void* dx_perm = ws + p.bw_dxperm;
  float* dwp = reinterpret_cast<float*>(ws + p.bw_dwp);
  const GemmEnv env = env_of(ctx, p, st);
  auto weight_gemms = [&]() {
    return launch_wgrad_pair(env, p, m, c, x_perm, x8, dy_perm, dy8, dH, dH_lo, wa, wa_lo,
                             d_up_proj_weight, d_down_proj_weight, dWs1, dWs2);
  };
  const bool weights = d_up_proj_weight || d_down_proj_weight || dWs1 || dWs2;
  if (mode == BWD_DW) {
    if (!weights) return HMM_OK;
    PhaseScope ps(ctx, PH_GEMM_BWD_WEIGHT, st);
    return weight_gemms();
  }

  {
    PhaseScope ps(ctx, PH_DISPATCH_DY, st);
    rc = cuda_rc(
        launch_dispatch_dy(p, dy, topk_weights, shape->weights_dtype, m, c, dy_perm, dy8, wperm,
                           st, ctx->overlap != 0));
  }
  if (rc != HMM_OK) return rc;
  const bool inject = ctx->inject_skip_ready == 2;
  if (inject) ctx->inject_skip_ready = 0;
  {
    PhaseScope ps(ctx, PH_GEMM_BWD_DATA, st);
    rc = launch_data_grad_gemms(env, p, m, c, dy_perm, wperm, h32, up_proj_weight,
                                down_proj_weight, Ws1, Ws2, dH, dH_lo, wa, wa_lo, dwp, dx_perm,
                                inject);
  }
  if (rc != HMM_OK) return rc;
  // dx and d_topk_weights need only part 1: combine them on the side stream
  // while part 2 (the weight gradients) runs; the caller's stream waits for
  // both before anything queued after this call.
  const bool combine = dx || d_topk_weights;
  if (combine) {
    rc = cuda_rc(cudaEventRecord(ctx->fork, st));
    if (rc == HMM_OK) rc = cuda_rc(cudaStreamWaitEvent(ctx->side, ctx->fork, 0));
    if (rc != HMM_OK) return rc;
    {
      PhaseScope pc(ctx, PH_COMBINE_DX, ctx->side);
      // (behind an event wait: launched in plain stream order)
      rc = cuda_rc(launch_combine_dx(p, dx_perm, dwp, m, dx, d_topk_weights,
                                     shape->weights_dtype, ctx->side, false));
    }
    const int rj = cuda_rc(cudaEventRecord(ctx->join, ctx->side));
    if (rc == HMM_OK) rc = rj;
  }
  int r2 = rc;
  if (rc == HMM_OK && weights) {
    PhaseScope ps(ctx, PH_GEMM_BWD_WEIGHT, st);
    r2 = weight_gemms();
  }
  if (combine) {
    const int rw = cuda_rc(cudaStreamWaitEvent(st, ctx->join, 0));
    if (rc == HMM_OK) rc = rw;
  }
  if (rc == HMM_OK) rc = r2;
  return rc;
}

}  // namespace

int hmm_backward(hmm_ctx* ctx, const hmm_shape* shape, const void* dy, const void* topk_weights,
                 const void* up_proj_weight, const void* down_proj_weight, const void* saved,
                 size_t saved_bytes, void* dx, void* d_up_proj_weight, void* d_down_proj_weight,
                 void* d_topk_weights, void* workspace, size_t workspace_bytes, void* stream) {
  if (shape && shape->shared != 0) return HMM_ERR_ARG;  // hmm_backward_shared
  return backward_impl(ctx, shape, dy, topk_weights, up_proj_weight, down_proj_weight, nullptr,
                       nullptr, saved, saved_bytes, dx, d_up_proj_weight, d_down_proj_weight,
                       nullptr, nullptr, d_topk_weights, workspace, workspace_bytes, stream,
                       BWD_FULL);
}

int hmm_backward_shared(hmm_ctx* ctx, const hmm_shape* shape, const void* dy,
                        const void* topk_weights, const void* up_proj_weight,
                        const void* down_proj_weight, const void* shared_up_proj_weight,
                        const void* shared_down_proj_weight, const void* saved,
                        size_t saved_bytes, void* dx, void* d_up_proj_weight,
                        void* d_down_proj_weight, void* d_shared_up_proj_weight,
                        void* d_shared_down_proj_weight, void* d_topk_weights, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!shape || shape->shared != 1) return HMM_ERR_ARG;
  return backward_impl(ctx, shape, dy, topk_weights, up_proj_weight, down_proj_weight,
                       shared_up_proj_weight, shared_down_proj_weight, saved, saved_bytes, dx,
                       d_up_proj_weight, d_down_proj_weight, d_shared_up_proj_weight,
                       d_shared_down_proj_weight, d_topk_weights, workspace, workspace_bytes,
                       stream, BWD_FULL);
}

int hmm_backward_dx(hmm_ctx* ctx, const hmm_shape* shape, const void* dy,
                    const void* topk_weights, const void* up_proj_weight,
                    const void* down_proj_weight, const void* saved, size_t saved_bytes, void* dx,
                    void* d_topk_weights, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(ctx, shape, dy, topk_weights, up_proj_weight, down_proj_weight, nullptr,
                       nullptr, saved, saved_bytes, dx, nullptr, nullptr, nullptr, nullptr,
                       d_topk_weights, workspace, workspace_bytes, stream, BWD_DX);
}

int hmm_backward_dw(hmm_ctx* ctx, const hmm_shape* shape, const void* saved, size_t saved_bytes,
                    void* d_up_proj_weight, void* d_down_proj_weight, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return backward_impl(ctx, shape, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, saved,
                       saved_bytes, nullptr, d_up_proj_weight, d_down_proj_weight, nullptr,
                       nullptr, nullptr, workspace, workspace_bytes, stream, BWD_DW);
}

int hmm_status(hmm_ctx* ctx, void* stream, int* device_error) {
  if (!ctx) return HMM_ERR_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return HMM_ERR_CUDA;
  // read and clear in the caller's stream order only: no device-wide wait
  // (work of other streams keeps running)
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, ctx->status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(ctx->status, 0, sizeof v, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return HMM_ERR_CUDA;
  if (device_error) *device_error = static_cast<int>(v);
  if (v & HMM_STATUS_TIMEOUT) return HMM_ERR_TIMEOUT;
  if (v & HMM_STATUS_EXPERT_ID) return HMM_ERR_EXPERT_ID;
  return HMM_OK;
}

int hmm_profile_read(hmm_ctx* ctx, int n, double* ms, int64_t* launches) {
  if (!ctx || n < 0) return HMM_ERR_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return HMM_ERR_CUDA;
  double acc[HMM_NUM_PHASES] = {0};
  int64_t cnt[HMM_NUM_PHASES] = {0};
  int rc = HMM_OK;
  for (auto& r : ctx->recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.begin, r.end) != cudaSuccess)
      rc = HMM_ERR_CUDA;
    acc[r.phase] += t;
    cnt[r.phase] += r.kernels;
    ctx->pool.push_back(r.begin);
    ctx->pool.push_back(r.end);
  }
  ctx->recs.clear();
  for (int i = 0; i < n && i < HMM_NUM_PHASES; ++i) {
    if (ms) ms[i] = acc[i];
    if (launches) launches[i] = cnt[i];
  }
  return rc;
}

int hmm_set_trace(hmm_ctx* ctx, void* buffer, size_t bytes, int which) {
  if (!ctx || which < 0 || which > 2) return HMM_ERR_ARG;
  if (buffer && (reinterpret_cast<uintptr_t>(buffer) & 15u)) return HMM_ERR_LAYOUT;
  if (buffer && bytes < static_cast<size_t>(64) * ctx->num_sms) return HMM_ERR_CAPACITY;
  ctx->trace = static_cast<uint64_t*>(buffer);
  ctx->trace_bytes = buffer ? bytes : 0;
  ctx->trace_which = which;
  return HMM_OK;
}

const char* hmm_phase_name(int phase) {
  if (phase < 0 || phase >= HMM_NUM_PHASES) return nullptr;
  return kPhases[phase].name;
}

const char* hmm_error_string(int code) {
  switch (code) {
    case HMM_OK: return "ok";
    case HMM_ERR_ARG: return "invalid argument (null pointer, option or context)";
    case HMM_ERR_SHAPE: return "shape out of the supported range or inconsistent";
    case HMM_ERR_DTYPE: return "unsupported dtype";
    case HMM_ERR_LAYOUT: return "misaligned pointer, or H / I not a multiple of 8";
    case HMM_ERR_CAPACITY: return "workspace or saved buffer too small";
    case HMM_ERR_EXPERT_ID: return "a topk_id is outside [0, E)";
    case HMM_ERR_TIMEOUT: return "a bounded device wait ran out";
    case HMM_ERR_CUDA: return "a CUDA call failed";
    case HMM_ERR_DEVICE: return "no such device, or the device is not sm_103";
    default: return "unknown error code";
  }
}

}  // extern "C"
