/*
 * hmm.h -- C ABI of the GB300 (sm_103a) fused MoE-FFN library (libhmm.so).
 *
 * The operation is the single-GPU form of the fused MoE-FFN of the
 * HyperMegaMoE issue (hyper-parallel #312):
 *
 *   forward  [HyperMegaMoE §2.1, §3.1, §4.1]
 *     Dispatch -> GMM1/up_proj -> SwiGLU -> GMM2/down_proj -> Combine
 *     y[t] = sum_k topk_weights[t,k] * FFN_{topk_ids[t,k]}(x[t])
 *     FFN_e(v) = (silu(v . W1[e][:, :I]) * (v . W1[e][:, I:])) . W2[e]
 *   backward [HyperMegaMoE §2.2]
 *     dx, d_up_proj_weight, d_down_proj_weight, d_topk_weights
 *     (topk_ids has no gradient).
 *
 * On one GPU "Dispatch" and "Combine" are a device-side permute (token rows
 * gathered into expert-contiguous order) and unpermute (the K expert rows of
 * a token gathered back and merged with its routing weights).  There is no
 * all-to-all and no inter-GPU traffic.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, row-major (C order), on the device of the context,
 *   with 16-byte-aligned base addresses.  Shapes (T, H, I, E, K as in
 *   HyperMegaMoE §3.1):
 *     x, y, dy, dx              bf16   [T, H]
 *     topk_ids                  int32  [T, K]   global expert ids in [0, E)
 *     topk_weights, d_topk_w    bf16 or fp32 [T, K] (hmm_shape.weights_dtype)
 *     up_proj_weight, d_up      bf16   [E, H, 2I]  columns 0..I-1 = gate,
 *                                                  I..2I-1 = up
 *     down_proj_weight, d_down  bf16   [E, I, H]
 *   H and I must be multiples of 8 (16-byte rows).
 * - The caller owns every buffer: inputs, outputs, the per-call workspace and
 *   the "saved" buffer that carries routing metadata and activations from a
 *   forward to its backward.  Sizes come from hmm_workspace_size().  The
 *   library never allocates per call; hmm_create() allocates one small
 *   device status word.
 * - Every call is asynchronous on `stream` (a cudaStream_t, passed as
 *   void*).  Inputs must stay valid and unmodified until the stream reaches
 *   the end of the call.
 * - Returns HMM_OK (0) or a negative HMM_ERR_* code.  Shape, dtype, layout
 *   and capacity are checked on the host before anything is launched
 *   [HyperMegaMoE §4.2: bad input is rejected at the host boundary, not in a
 *   device kernel].  Conditions only the device can see (an expert id out of
 *   range, a bounded wait that ran out) set bits of the context's device
 *   status word, which hmm_status() reads; with HMM_OPT_VALIDATE set,
 *   hmm_forward() and hmm_route() synchronise after the routing step and
 *   return HMM_ERR_EXPERT_ID before any GEMM runs.  Outputs are unspecified
 *   after an error.
 * - Gradients are written, not accumulated (d_up / d_down of an expert that
 *   receives no token are written as exact zeros).
 * - A context may be used from one host thread at a time.  Concurrent calls
 *   on different streams need distinct workspace and saved buffers.
 * - hmm_route, hmm_forward*, hmm_backward* can be captured into a CUDA graph
 *   on `stream` and replayed (the pointers and shape are fixed in the graph;
 *   the inputs may change in place between replays): they allocate nothing,
 *   reset their own counters in every call, and the backward's second stream
 *   joins the capture through its fork and join events.  HMM_OPT_VALIDATE
 *   (a host synchronisation) and HMM_OPT_PROFILE must be off while capturing.
 */
#ifndef HMM_H_
#define HMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define HMM_OK 0
#define HMM_ERR_ARG (-1)       /* null pointer / bad option / bad context */
#define HMM_ERR_SHAPE (-2)     /* dimension out of range or inconsistent */
#define HMM_ERR_DTYPE (-3)     /* unsupported dtype code */
#define HMM_ERR_LAYOUT (-4)    /* misaligned pointer or H, I not multiples of 8 */
#define HMM_ERR_CAPACITY (-5)  /* workspace or saved buffer smaller than required */
#define HMM_ERR_EXPERT_ID (-6) /* a topk_id outside [0, E) (device-detected) */
#define HMM_ERR_TIMEOUT (-7)   /* a bounded device wait ran out (device-detected) */
#define HMM_ERR_CUDA (-8)      /* a CUDA runtime/driver call failed */
#define HMM_ERR_DEVICE (-9)    /* device is not sm_103 / no such device */

/* bits of the device status word (hmm_status) */
#define HMM_STATUS_EXPERT_ID 1u
#define HMM_STATUS_TIMEOUT 2u

/* dtype codes */
#define HMM_DTYPE_BF16 0
#define HMM_DTYPE_F32 1

typedef struct hmm_ctx hmm_ctx;

typedef struct hmm_shape {
  int64_t T;             /* tokens (may be 0) */
  int64_t H;             /* hidden size, multiple of 8 */
  int64_t I;             /* expert intermediate size, multiple of 8 */
  int64_t E;             /* experts, >= 1 */
  int64_t K;             /* experts per token, >= 1 */
  int32_t weights_dtype; /* HMM_DTYPE_BF16 or HMM_DTYPE_F32 for topk_weights */
  int32_t shared;        /* 1: one shared expert [HyperMegaMoE §6.1], used through
                            hmm_forward_shared / hmm_backward_shared (the sizes of
                            hmm_workspace_size include it); 0: none.  With 1,
                            E + 1 <= 1024 and K <= 31. */
} hmm_shape;

/* Create a context bound to CUDA device `device` (must be sm_103).  Allocates
 * the device status word.  *out is NULL on failure. */
int hmm_create(hmm_ctx** out, int device);

/* Destroy a context (frees the status word).  NULL is accepted. */
int hmm_destroy(hmm_ctx* ctx);

/* Context options.
 *   HMM_OPT_VALIDATE      0/1: hmm_forward/hmm_route synchronise after routing
 *                         and return HMM_ERR_EXPERT_ID for a bad id (default 0).
 *   HMM_OPT_WAIT_BUDGET_NS  budget of every bounded device wait, in ns
 *                         (default 2e9; range 1e6 .. 6e10).
 *   HMM_OPT_INJECT_SKIP_READY  test-only fault injection on the host side: when
 *                         1, the next hmm_forward launches its GMM1 tiles
 *                         without releasing the GMM2 ready counters, so every
 *                         GMM2 tile's bounded wait runs out and the call
 *                         reports HMM_STATUS_TIMEOUT; when 2, the next
 *                         hmm_backward (or hmm_backward_dx) does the same to
 *                         its act_grad and input-grad tiles.  Cleared by the
 *                         call it affects.  No device fault is involved: the
 *                         waits end by their budget and every CTA leaves. */
#define HMM_OPT_VALIDATE 1
#define HMM_OPT_WAIT_BUDGET_NS 2
#define HMM_OPT_INJECT_SKIP_READY 3
/*   HMM_OPT_PROFILE       0/1: bracket every launch phase with CUDA events
 *                         recorded on the call's stream (read them with
 *                         hmm_profile_read).  Default 0. */
#define HMM_OPT_PROFILE 4
/*   (option ids 5 and 6 are not used) */
/*   HMM_OPT_PAIR_ROWS     tiling of the forward and data-gradient GEMMs:
 *                         1: CTA pairs with 2-SM MMAs (256 weight columns per
 *                         tile, 128 per CTA, token blocks of up to 256 rows);
 *                         0: single CTAs (128 weight columns, blocks of up to
 *                         256 rows); 3: single CTAs with blocks of up to 64
 *                         rows and deeper pipelines (weight streaming);
 *                         2 (default): automatic, 1 when the routed rows
 *                         average at least 256 per expert (T * K >= 256 * E),
 *                         3 below 64 per expert, else 0.  Results do not
 *                         depend on it. */
#define HMM_OPT_PAIR_ROWS 7
/*   HMM_OPT_OVERLAP_LAUNCHES  0/1: launch every kernel with programmatic
 *                         stream serialization, so that it is scheduled and
 *                         sets itself up while the previous kernel of the
 *                         stream drains; it still reads nothing before that
 *                         kernel has completed.  Default 1.  Results do not
 *                         depend on it. */
#define HMM_OPT_OVERLAP_LAUNCHES 8
/*   HMM_OPT_FUSED_COMBINE  0/1: fold the forward's Combine into the GMM2
 *                         epilogue [HyperMegaMoE §6.2: the unpermute and the
 *                         top-k weighted merge inside the fused operator;
 *                         MoE overlap explainer §6: a per-token completion
 *                         count publishes a token once all of its branches
 *                         are in].  Each GMM2 tile counts its token rows per
 *                         32-column segment; the epilogue warp that completes
 *                         a token's K expert rows (K + 1 with the shared
 *                         expert) of a segment sums them in k order and writes
 *                         y, so no combine launch runs.  y is bit-identical to
 *                         the separate combine (same fp32 operations in the
 *                         same order, one bf16 rounding).  Default 0.  Out-of-
 *                         range expert ids leave the rows of their tokens
 *                         unwritten (outputs are undefined on that error). */
#define HMM_OPT_FUSED_COMBINE 9
int hmm_set_option(hmm_ctx* ctx, int option, int64_t value);

/* Launch phases timed under HMM_OPT_PROFILE (index = phase id):
 *   0 route (2 or 3 kernels)  1 dispatch_x  2 gemm_fwd (GMM1+SwiGLU, GMM2)
 *   3 combine_y (no launch with HMM_OPT_FUSED_COMBINE)   4 dispatch_dy
 *   5 gemm_bwd_data (act_grad + SwiGLU grad, input-grad)
 *   6 gemm_bwd_weight (W2Grad, W1Grad)
 *   7 combine_dx (+ d_topk_weights; on a second stream, beside phase 6)  */
#define HMM_NUM_PHASES 8

/* Tracing: waits for every event recorded since the previous read, then
 * writes, for each phase id < n, the summed GPU time in ms (ms[i]) and the
 * number of kernel launches (launches[i]) recorded since that read, and
 * resets the counters.  Either array may be NULL. */
int hmm_profile_read(hmm_ctx* ctx, int n, double* ms, int64_t* launches);

/* Name of a phase id ("route", "gemm_fwd", ...), or NULL if out of range. */
const char* hmm_phase_name(int phase);

/* Per-tile timeline of one GEMM launch (tracing).  buffer (device memory
 * owned by the caller, 16-byte aligned) receives, for the next launch of GEMM
 * kind `which` (0: forward GEMMs, 1: backward data-gradient GEMMs, 2:
 * backward weight-gradient GEMMs), one record of 8 uint64 per tile and CTA:
 *   [0] (sm id << 48) | (problem << 40) | (expert << 20) | K blocks
 *   [1] scheduler published the tile   [2] first TMA load issued
 *   [3] last TMA load issued           [4] first MMA issued
 *   [5] last MMA committed             [6] epilogue saw the accumulator
 *   [7] epilogue done (one warp)       (globaltimer ns; 0 = not reached)
 * laid out as records[cta * cap + i] with cap = bytes / (64 * grid), where
 * grid is the number of SMs.  Slots a launch does not reach stay as they were.
 * NULL disables tracing. */
int hmm_set_trace(hmm_ctx* ctx, void* buffer, size_t bytes, int which);

/* Buffer sizes in bytes for a shape.  training != 0: the forward keeps its
 * activations in `saved` for the backward; training == 0: they live in the
 * forward workspace and *saved_bytes is 0.  Any output pointer may be NULL. */
int hmm_workspace_size(const hmm_shape* shape, int training,
                       size_t* fwd_workspace_bytes, size_t* saved_bytes,
                       size_t* bwd_workspace_bytes);

/* Routing metadata alone [HyperMegaMoE §3.3 offset/size/group list, §4.1
 * expansion of each token into K slots s = t*K + k; MoE overlap explainer §5:
 * counts, prefix sums, offsets and the token permutation on the device]:
 *   counts[e]   number of slots routed to expert e                  int32 [E]
 *   offsets[e]  exclusive prefix sum of counts, offsets[E] = T*K    int32 [E+1]
 *   slot2row[s] position of slot s in expert-sorted order, stable
 *               (ties by ascending s)                               int32 [T*K]
 *   row2slot[r] inverse permutation                                 int32 [T*K]
 * workspace: at least the forward workspace size of the same shape.
 * No host round trip unless HMM_OPT_VALIDATE is set. */
int hmm_route(hmm_ctx* ctx, const hmm_shape* shape, const int32_t* topk_ids,
              int32_t* counts, int32_t* offsets, int32_t* slot2row,
              int32_t* row2slot, void* workspace, size_t workspace_bytes,
              void* stream);

/* Routing with no allocation and no context.  The paper has no counterpart
 * of this entry point; it exists for callers that cannot allocate device
 * memory (an engine whose memory pool owns the whole device, a plug-in whose
 * host gives it no allocator or workspace).
 *
 * Computes exactly what hmm_route computes (same kernels, same outputs, same
 * argument meaning and layout), on the current CUDA device, asynchronously
 * on `stream`.  Its scratch is one 8 MiB device array inside the library
 * (held by every GPU that loads the library until the process exits); it
 * calls no cudaMalloc, cudaFree or other allocating routine.
 * - The first call on each device looks up the array's device address (and
 *   checks that the device is sm_103); make that first call before any stream
 *   capture on that device.
 * - Every call shares the one array: calls whose GPU work overlaps (on two
 *   streams, or from two host threads) race and give undefined results.
 *   Serialise them on one stream.
 * - The scratch of a shape is 256 bytes plus the routing part of the forward
 *   workspace: with S = T*K slots, C = ceil(S / 1024) and the padded rows
 *   R = S + 127*min(E, S) rounded up to a multiple of 128, about
 *   4*S + 4*R + R/16 + 4*E*C + 12*E + 32 bytes, each array rounded up to
 *   256 bytes (about 8 bytes per slot plus 512 bytes per expert plus 4*E
 *   bytes per 1024 slots).  A shape whose scratch exceeds the array returns
 *   HMM_ERR_CAPACITY before any device work.  Shape limits are those of
 *   hmm_route. 
 * - Ids outside [0, E) are left out: their slot2row is -1 and
 *   offsets[E] < T*K (there is no status word to read). */
int hmm_route_static(const hmm_shape* shape, const int32_t* topk_ids,
                     int32_t* counts, int32_t* offsets, int32_t* slot2row,
                     int32_t* row2slot, void* stream);

/* Fused forward [HyperMegaMoE §2.1]: y = Combine(GMM2(SwiGLU(GMM1(Dispatch(x))))).
 * saved == NULL: inference (the [., 2I] pre-activation is never written to
 * memory).  Otherwise saved (saved_bytes from hmm_workspace_size with
 * training=1) receives what hmm_backward needs: routing metadata, permuted x,
 * gate/up pre-activations, SwiGLU outputs and expert outputs. */
int hmm_forward(hmm_ctx* ctx, const hmm_shape* shape, const void* x,
                const int32_t* topk_ids, const void* topk_weights,
                const void* up_proj_weight, const void* down_proj_weight,
                void* y, void* saved, size_t saved_bytes, void* workspace,
                size_t workspace_bytes, void* stream);

/* Fused backward [HyperMegaMoE §2.2]: from dy and the `saved` buffer of the
 * matching hmm_forward (same shape, same topk_ids, weights unchanged) writes
 *   dx               bf16 [T, H]
 *   d_up_proj_weight bf16 [E, H, 2I]
 *   d_down_proj_weight bf16 [E, I, H]
 *   d_topk_weights   [T, K] in shape->weights_dtype
 * Any of the four outputs may be NULL to skip it. */
int hmm_backward(hmm_ctx* ctx, const hmm_shape* shape, const void* dy,
                 const void* topk_weights, const void* up_proj_weight,
                 const void* down_proj_weight, const void* saved,
                 size_t saved_bytes, void* dx, void* d_up_proj_weight,
                 void* d_down_proj_weight, void* d_topk_weights,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Optional shared expert [HyperMegaMoE §6.1: shared-expert weights whose GMM1,
 * SwiGLU and GMM2 are scheduled with the routed experts' pipeline and whose
 * output is merged at Combine; the interface gains the shared weights only
 * when the feature is used].  shape->shared must be 1 (hmm_forward and
 * hmm_backward refuse such a shape, these refuse shared == 0).
 *   y[t] = sum_k topk_weights[t,k] FFN_{topk_ids[t,k]}(x[t]) + FFN_s(x[t])
 * (reading: every token, unit weight, no gate), FFN_s the expert FFN on
 *   shared_up_proj_weight   bf16 [H, 2I]  (gate | up, like one routed expert)
 *   shared_down_proj_weight bf16 [I, H]
 * The shared expert runs as one more expert of the same launches (its rows
 * are the T tokens in order).  The backward adds its part of dx and writes
 * d_shared_up_proj_weight [H, 2I] and d_shared_down_proj_weight [I, H]
 * (either may be NULL); d_topk_weights is unchanged by it.  Arguments,
 * layouts and errors otherwise as for hmm_forward / hmm_backward; sizes come
 * from hmm_workspace_size with the same shape.  The split entry points
 * hmm_backward_dx / hmm_backward_dw refuse shared == 1. */
int hmm_forward_shared(hmm_ctx* ctx, const hmm_shape* shape, const void* x,
                       const int32_t* topk_ids, const void* topk_weights,
                       const void* up_proj_weight, const void* down_proj_weight,
                       const void* shared_up_proj_weight,
                       const void* shared_down_proj_weight, void* y, void* saved,
                       size_t saved_bytes, void* workspace,
                       size_t workspace_bytes, void* stream);
int hmm_backward_shared(hmm_ctx* ctx, const hmm_shape* shape, const void* dy,
                        const void* topk_weights, const void* up_proj_weight,
                        const void* down_proj_weight,
                        const void* shared_up_proj_weight,
                        const void* shared_down_proj_weight, const void* saved,
                        size_t saved_bytes, void* dx, void* d_up_proj_weight,
                        void* d_down_proj_weight, void* d_shared_up_proj_weight,
                        void* d_shared_down_proj_weight, void* d_topk_weights,
                        void* workspace, size_t workspace_bytes, void* stream);

/* The backward split into its data and weight halves, for schedulers that
 * defer the weight gradients [EP overlap issue §2.3 (W/D split, deferred W
 * queue), §4.5: separate D-only and W-only backward entry points].
 *
 * hmm_backward_dx: what hmm_backward does without the weight gradients
 *   (dispatch dY, act_grad + SwiGLU grad, input-grad, combine dX and
 *   d_topk_weights; dx or d_topk_weights may be NULL).  It leaves in
 *   `workspace` the operands of the weight gradients: dY permuted (bf16 and
 *   an fp8 copy), dH and w*a (bf16 high parts and fp8 low parts).
 * hmm_backward_dw: d_up_proj_weight and d_down_proj_weight (either may be
 *   NULL) from those operands and `saved`.  Call it on the same stream, after
 *   the hmm_backward_dx of the same shape, `saved` and `workspace`; nothing
 *   else may write that workspace or `saved` in between.  The workspace is
 *   held until then: that is the memory cost of deferring W.
 *
 * Together the two write exactly what one hmm_backward call writes (the
 * same kernels on the same inputs: bit-identical results).  Errors as for
 * hmm_backward; hmm_backward_dw checks only shape, saved and workspace. */
int hmm_backward_dx(hmm_ctx* ctx, const hmm_shape* shape, const void* dy,
                    const void* topk_weights, const void* up_proj_weight,
                    const void* down_proj_weight, const void* saved,
                    size_t saved_bytes, void* dx, void* d_topk_weights,
                    void* workspace, size_t workspace_bytes, void* stream);
int hmm_backward_dw(hmm_ctx* ctx, const hmm_shape* shape, const void* saved,
                    size_t saved_bytes, void* d_up_proj_weight,
                    void* d_down_proj_weight, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Read and clear the device status word in `stream` order, then wait for
 * `stream` (only that stream: other streams of the device keep running).
 * Work queued on `stream` before the call has set its bits by then.
 * *device_error receives the HMM_STATUS_* bits.  Returns HMM_OK, or
 * HMM_ERR_EXPERT_ID / HMM_ERR_TIMEOUT if the corresponding bit was set. */
int hmm_status(hmm_ctx* ctx, void* stream, int* device_error);

/* Static description of a return code. */
const char* hmm_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* HMM_H_ */
