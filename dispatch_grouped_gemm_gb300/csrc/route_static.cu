// route_static.cu -- hmm_route_static: the routing step with no allocation.
//
// Some callers cannot call cudaMalloc: a serving engine that hands all device
// memory to its own pool at start-up and forbids any later allocation, or a
// plug-in whose host process gives it no allocator and no workspace.  For
// them this entry point runs the same routing kernels as hmm_route, but keeps
// their scratch (per-chunk histograms, the padded layout, counters) in one
// file-scope device array of fixed size instead of a caller workspace.  It
// needs no context either (hmm_create allocates a status word).
//
// The array is part of the library's module: every GPU that loads libhmm.so
// holds kScratchBytes of device memory for it until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "hmm_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

// [0, 256): device status word of these calls; [256, end): ctrl + meta of one call
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
unsigned char* g_addr[kMaxDevices] = {};  // device address of g_scratch, per device
bool g_checked[kMaxDevices] = {};

// Once per device, with that device current: check it is an sm_103 part and
// look up the device address of g_scratch.  (In host code `g_scratch` names a
// host-side shadow, not device memory, so it is never passed to a kernel.)
int setup_device(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_checked[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return HMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return HMM_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return HMM_ERR_CUDA;
    g_addr[dev] = static_cast<unsigned char*>(p);
    g_checked[dev] = true;
  }
  *out = g_addr[dev];
  return HMM_OK;
}

}  // namespace

extern "C" int hmm_route_static(const hmm_shape* shape, const int32_t* topk_ids, int32_t* counts,
                                int32_t* offsets, int32_t* slot2row, int32_t* row2slot,
                                void* stream) {
  using namespace hmm;
  // routing of the routed experts only: a shape with the shared expert is refused
  if (!shape || shape->shared != 0) return HMM_ERR_ARG;
  // the same limits as every other entry point (hmm_route included)
  const int src = check_shape(shape);
  if (src != HMM_OK) return src;
  Plan p;
  make_plan(shape, false, &p);
  if (!counts || !offsets || (p.TK > 0 && (!topk_ids || !slot2row || !row2slot)))
    return HMM_ERR_ARG;
  // scratch of this call: status word, then ctrl, then meta (all 256-aligned)
  const size_t need = 256 + p.ctrl_bytes + p.meta_bytes;
  if (need > kScratchBytes) return HMM_ERR_CAPACITY;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HMM_ERR_DEVICE;
  unsigned char* base = nullptr;
  const int rc = setup_device(dev, &base);
  if (rc != HMM_OK) return rc;
  unsigned* status = reinterpret_cast<unsigned*>(base);
  CtrlPtrs c = ctrl_at(p, base + 256);
  MetaPtrs m = meta_at(p, base + 256 + p.ctrl_bytes);
  // counts and offsets go straight to the caller's arrays
  m.counts = counts;
  m.offsets = offsets;
  // Nothing here must start at zero: the count kernel writes every histogram
  // entry it covers, the scan (its own kernel, or inside the rank kernel)
  // writes the counters and the padded offsets, the rank kernel writes every
  // slot.  Stale contents of a previous call are overwritten before they are
  // read.
  return launch_route(p, topk_ids, m, c, slot2row, row2slot, status,
                      static_cast<cudaStream_t>(stream), true) == cudaSuccess
             ? HMM_OK
             : HMM_ERR_CUDA;
}
