/*
 * hmm_oracle.c -- plain, slow fp64 CPU oracle for the fused MoE-FFN
 * (Dispatch -> GMM1/up_proj -> SwiGLU -> GMM2/down_proj -> top-k weighted
 * Combine) and its backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (sources, cited by page title and section):
 *   [HyperMegaMoE §2.1]  forward chain Dispatch -> GMM1 -> SwiGLU -> GMM2 ->
 *                        Combine; output y has the shape of x.
 *   [HyperMegaMoE §3.1]  public arguments x[T,H], topk_ids[T,K] (global expert
 *                        ids, no gradient), topk_weights[T,K],
 *                        up_proj_weight[E,H,2I], down_proj_weight[E,I,H].
 *   [HyperMegaMoE §4.1]  every token expands into K expert slots; each slot
 *                        runs its expert's GMM1 -> SwiGLU -> GMM2; Combine
 *                        merges the K outputs weighted by topk_weights.
 *   [HyperMegaMoE §2.2]  backward: dispatch of dY, act_grad = dY . W2^T,
 *                        SwiGLU grad, input-grad GMM, W2Grad, W1Grad,
 *                        Combine(dX); returns dx, d_up_proj_weight,
 *                        d_down_proj_weight, d_topk_weights.
 *   [MoE overlap explainer §6]  combine: acc[token] += gate * value over the
 *                        token's top-k branches.
 *   [HyperMegaMoE §3.3, §4.1, MoE overlap explainer §5]  routing metadata:
 *                        per-expert counts, exclusive prefix offsets and the
 *                        expert-sorted permutation with its inverse.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of the repository):
 *   - the first I columns of up_proj's 2I outputs are the gate, the second I
 *     the up projection, SwiGLU(g, u) = silu(g) * u, silu(z) = z * sigma(z);
 *   - weights are applied as x . W (no transpose), shapes as in §3.1;
 *   - topk_weights multiply the expert outputs at Combine and are not
 *     renormalised;
 *   - the permutation is the stable sort of slots s = t*K + k by expert id
 *     (ties by ascending s);
 *   - a slot whose expert repeats inside a token is an independent slot;
 *   - ids outside [0, E) are an error, never clamped.
 *
 * Arithmetic: every input value is decoded exactly to double (bf16 is the
 * top half of an IEEE binary32) and all arithmetic is fp64, summed in plain
 * index order.  No blocking, fusion or reordering beyond the definitions.
 *
 * Parity pins for every function here live in the oracle's own CPU tests
 * (brute force, closed forms, a library special case, invariances, finite
 * differences); none of them reads anything produced by the CUDA path.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes for the floating inputs */
#define ORACLE_BF16 0 /* raw bf16 bit patterns, uint16_t */
#define ORACLE_F64 1  /* double */

static inline double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Element i of a floating input of dtype dt, decoded exactly to double. */
static inline double ld(const void* p, int64_t i, int dt) {
  if (dt == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t*)p)[i]);
  return ((const double*)p)[i];
}

static inline double sigma(double z) { return 1.0 / (1.0 + exp(-z)); }

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Routing metadata [HyperMegaMoE §3.3 "offset, size and group list", §4.1
 * "each token expands into K expert slots"; MoE overlap explainer §5 counts,
 * prefix sums, offsets and the token permutation].
 *   counts[e]   = #{ s : ids[s] == e }
 *   offsets[0]  = 0,  offsets[e+1] = offsets[e] + counts[e]
 *   slot2row[s] = offsets[ids[s]] + #{ s' < s : ids[s'] == ids[s] }
 *   row2slot[slot2row[s]] = s
 * Returns the number of out-of-range ids (0 on success); with any such id the
 * arrays are left unspecified.
 */
int64_t oracle_route(int64_t T, int64_t K, int64_t E, const int32_t* ids,
                     int32_t* counts, int32_t* offsets, int32_t* slot2row,
                     int32_t* row2slot) {
  int64_t TK = T * K, bad = 0;
  for (int64_t s = 0; s < TK; ++s)
    if (ids[s] < 0 || ids[s] >= E) ++bad;
  if (bad) return bad;
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < TK; ++s) counts[ids[s]] += 1;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* seen = (int32_t*)calloc((size_t)(E > 0 ? E : 1), sizeof(int32_t));
  for (int64_t s = 0; s < TK; ++s) {
    int32_t e = ids[s];
    slot2row[s] = offsets[e] + seen[e];
    seen[e] += 1;
    row2slot[slot2row[s]] = (int32_t)s;
  }
  free(seen);
  return 0;
}

/*
 * One expert applied to one token row [HyperMegaMoE §2.1 GMM1 -> SwiGLU ->
 * GMM2]:
 *   h = x_row . W1_e            (length 2I, W1_e is [H, 2I])
 *   a = silu(h[0:I]) * h[I:2I]  (length I)
 *   o = a . W2_e                (length H, W2_e is [I, H])
 * x_row, W1_e, W2_e are element offsets into x, W1, W2 of dtype dt.
 */
void oracle_expert_ffn(int64_t H, int64_t I, int dt, const void* x,
                       int64_t x_off, const void* W1, int64_t w1_off,
                       const void* W2, int64_t w2_off, double* h, double* a,
                       double* o) {
  for (int64_t j = 0; j < 2 * I; ++j) h[j] = 0.0;
  for (int64_t i = 0; i < H; ++i) {
    double xi = ld(x, x_off + i, dt);
    int64_t row = w1_off + i * 2 * I;
    for (int64_t j = 0; j < 2 * I; ++j) h[j] += xi * ld(W1, row + j, dt);
  }
  for (int64_t j = 0; j < I; ++j) {
    double g = h[j], u = h[I + j];
    a[j] = g * sigma(g) * u;
  }
  for (int64_t c = 0; c < H; ++c) o[c] = 0.0;
  for (int64_t j = 0; j < I; ++j) {
    double aj = a[j];
    int64_t row = w2_off + j * H;
    for (int64_t c = 0; c < H; ++c) o[c] += aj * ld(W2, row + c, dt);
  }
}

/*
 * Forward [HyperMegaMoE §2.1, §4.1; MoE overlap explainer §6]:
 *   y[t] = sum_{k=0..K-1} topk_weights[t,k] * FFN_{ids[t,k]}(x[t])
 * summed in k order.  y is double [T, H].  Returns the number of invalid ids
 * (y untouched when nonzero).
 */
int64_t oracle_forward(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K,
                       int dt, const void* x, const int32_t* ids,
                       const void* w, const void* W1, const void* W2,
                       double* y) {
  int64_t bad = 0;
  for (int64_t s = 0; s < T * K; ++s)
    if (ids[s] < 0 || ids[s] >= E) ++bad;
  if (bad) return bad;
#pragma omp parallel
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      double* yt = y + t * H;
      for (int64_t c = 0; c < H; ++c) yt[c] = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        int64_t e = ids[t * K + k];
        oracle_expert_ffn(H, I, dt, x, t * H, W1, e * H * 2 * I, W2, e * I * H,
                          h, a, o);
        double wk = ld(w, t * K + k, dt);
        for (int64_t c = 0; c < H; ++c) yt[c] += wk * o[c];
      }
    }
    free(h);
    free(a);
    free(o);
  }
  return 0;
}

/*
 * Backward of one slot, the chain rule through the forward above
 * [HyperMegaMoE §2.2: Dispatch(dY) -> act_grad = dY . W2^T -> SwiGLUGrad ->
 * input-grad GMM; W2Grad; W1Grad; Combine(dX); d_topk_weights]:
 *   dO = w * dy_t                        (gradient reaching the expert output)
 *   dA = dO . W2_e^T                     (act_grad, length I)
 *   dg = dA * u * sigma(g) * (1 + g * (1 - sigma(g)))
 *   du = dA * g * sigma(g)               (SwiGLU grad; dH = [dg, du])
 * Writes dO (length H), dA (I) and dH (2I); h and a come from the forward.
 */
static void slot_backward(int64_t H, int64_t I, int dt, const void* W2,
                          int64_t w2_off, const double* h, double wk,
                          const void* dy, int64_t dy_off, double* dO,
                          double* dA, double* dH) {
  for (int64_t c = 0; c < H; ++c) dO[c] = wk * ld(dy, dy_off + c, dt);
  for (int64_t j = 0; j < I; ++j) {
    double acc = 0.0;
    int64_t row = w2_off + j * H;
    for (int64_t c = 0; c < H; ++c) acc += dO[c] * ld(W2, row + c, dt);
    dA[j] = acc;
  }
  for (int64_t j = 0; j < I; ++j) {
    double g = h[j], u = h[I + j], sg = sigma(g);
    dH[j] = dA[j] * u * sg * (1.0 + g * (1.0 - sg));
    dH[I + j] = dA[j] * g * sg;
  }
}

/*
 * Token-side gradients [HyperMegaMoE §2.2]:
 *   d_topk_weights[t,k] = < dy_t , FFN_{ids[t,k]}(x_t) >
 *   dx[t] = sum_k dH_{t,k} . W1_e^T      (Combine(dX): unweighted, because
 *                                         the weight is already inside dO)
 * dx is double [T,H], dw is double [T,K].  Returns the number of invalid ids.
 */
int64_t oracle_backward_tokens(int64_t T, int64_t H, int64_t I, int64_t E,
                               int64_t K, int dt, const void* x,
                               const int32_t* ids, const void* w,
                               const void* W1, const void* W2, const void* dy,
                               double* dx, double* dw) {
  int64_t bad = 0;
  for (int64_t s = 0; s < T * K; ++s)
    if (ids[s] < 0 || ids[s] >= E) ++bad;
  if (bad) return bad;
#pragma omp parallel
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    double* dO = (double*)malloc(sizeof(double) * (size_t)H);
    double* dA = (double*)malloc(sizeof(double) * (size_t)I);
    double* dH = (double*)malloc(sizeof(double) * (size_t)(2 * I));
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      double* dxt = dx + t * H;
      for (int64_t i = 0; i < H; ++i) dxt[i] = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        int64_t e = ids[t * K + k];
        oracle_expert_ffn(H, I, dt, x, t * H, W1, e * H * 2 * I, W2, e * I * H,
                          h, a, o);
        double d = 0.0;
        for (int64_t c = 0; c < H; ++c) d += ld(dy, t * H + c, dt) * o[c];
        dw[t * K + k] = d;
        slot_backward(H, I, dt, W2, e * I * H, h, ld(w, t * K + k, dt), dy,
                      t * H, dO, dA, dH);
        for (int64_t i = 0; i < H; ++i) {
          double acc = 0.0;
          int64_t row = e * H * 2 * I + i * 2 * I;
          for (int64_t j = 0; j < 2 * I; ++j) acc += dH[j] * ld(W1, row + j, dt);
          dxt[i] += acc;
        }
      }
    }
    free(h);
    free(a);
    free(o);
    free(dO);
    free(dA);
    free(dH);
  }
  return 0;
}

/*
 * Weight gradients of one expert e [HyperMegaMoE §2.2 W2Grad, W1Grad]:
 *   dW2[e] = sum_{slots s routed to e} a_s^T (outer) dO_s      [I, H]
 *   dW1[e] = sum_{slots s routed to e} x_t^T (outer) dH_s      [H, 2I]
 * summed over slots in ascending s.  An expert with no slot gets exact zeros.
 * dW1_e is double [H, 2I], dW2_e is double [I, H].  Returns the number of
 * invalid ids.
 */
int64_t oracle_weight_grad(int64_t T, int64_t H, int64_t I, int64_t E,
                           int64_t K, int dt, int64_t e, const void* x,
                           const int32_t* ids, const void* w, const void* W1,
                           const void* W2, const void* dy, double* dW1_e,
                           double* dW2_e) {
  int64_t bad = 0, n = 0;
  for (int64_t s = 0; s < T * K; ++s) {
    if (ids[s] < 0 || ids[s] >= E) ++bad;
    else if (ids[s] == e) ++n;
  }
  if (bad) return bad;
  for (int64_t i = 0; i < H * 2 * I; ++i) dW1_e[i] = 0.0;
  for (int64_t i = 0; i < I * H; ++i) dW2_e[i] = 0.0;
  if (n == 0) return 0;
  /* the slots routed to e, in ascending s */
  int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
  n = 0;
  for (int64_t s = 0; s < T * K; ++s)
    if (ids[s] == e) slots[n++] = s;
  double* A = (double*)malloc(sizeof(double) * (size_t)(n * I));
  double* DO = (double*)malloc(sizeof(double) * (size_t)(n * H));
  double* DH = (double*)malloc(sizeof(double) * (size_t)(n * 2 * I));
  /* per-slot forward and backward vectors (independent per slot) */
#pragma omp parallel
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    double* dA = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; ++r) {
      int64_t s = slots[r], t = s / K;
      oracle_expert_ffn(H, I, dt, x, t * H, W1, e * H * 2 * I, W2, e * I * H,
                        h, A + r * I, o);
      slot_backward(H, I, dt, W2, e * I * H, h, ld(w, s, dt), dy, t * H,
                    DO + r * H, dA, DH + r * 2 * I);
    }
    free(h);
    free(o);
    free(dA);
  }
  /* outer-product sums; each output row is owned by one thread and summed
     over slots in ascending s */
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < I; ++j)
    for (int64_t r = 0; r < n; ++r) {
      double aj = A[r * I + j];
      for (int64_t c = 0; c < H; ++c) dW2_e[j * H + c] += aj * DO[r * H + c];
    }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < H; ++i)
    for (int64_t r = 0; r < n; ++r) {
      double xi = ld(x, (slots[r] / K) * H + i, dt);
      for (int64_t j = 0; j < 2 * I; ++j)
        dW1_e[i * 2 * I + j] += xi * DH[r * 2 * I + j];
    }
  free(slots);
  free(A);
  free(DO);
  free(DH);
  return 0;
}

/*
 * Optional shared expert [HyperMegaMoE §6.1: shared-expert weights whose
 * GMM1 -> SwiGLU -> GMM2 run beside the routed experts and whose output is
 * merged at Combine].  Reading where the page is silent: every token goes
 * through the shared expert with unit weight (no gate), so
 *   y[t] += FFN_s(x[t])
 * with FFN_s the expert FFN above on Ws1 [H, 2I], Ws2 [I, H].  ys is double
 * [T, H] (the shared term alone).
 */
void oracle_shared_forward(int64_t T, int64_t H, int64_t I, int dt,
                           const void* x, const void* Ws1, const void* Ws2,
                           double* ys) {
#pragma omp parallel
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
      oracle_expert_ffn(H, I, dt, x, t * H, Ws1, 0, Ws2, 0, h, a, ys + t * H);
    free(h);
    free(a);
  }
}

/*
 * Backward of the shared term (the chain rule through y[t] += FFN_s(x[t]),
 * unit weight):
 *   dA_t = dy_t . Ws2^T,  dH_t = SwiGLU grad,  dxs[t] = dH_t . Ws1^T
 *   dWs2 = sum_t a_t^T (outer) dy_t          [I, H]
 *   dWs1 = sum_t x_t^T (outer) dH_t          [H, 2I]
 * summed over tokens in ascending t.  dxs is double [T, H] (the shared
 * term's part of dx alone).
 */
void oracle_shared_backward(int64_t T, int64_t H, int64_t I, int dt,
                            const void* x, const void* Ws1, const void* Ws2,
                            const void* dy, double* dxs, double* dWs1,
                            double* dWs2) {
  double* A = (double*)malloc(sizeof(double) * (size_t)(T * I));
  double* DH = (double*)malloc(sizeof(double) * (size_t)(T * 2 * I));
#pragma omp parallel
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    double* dO = (double*)malloc(sizeof(double) * (size_t)H);
    double* dA = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      oracle_expert_ffn(H, I, dt, x, t * H, Ws1, 0, Ws2, 0, h, A + t * I, o);
      slot_backward(H, I, dt, Ws2, 0, h, 1.0, dy, t * H, dO, dA,
                    DH + t * 2 * I);
      double* dxt = dxs + t * H;
      for (int64_t i = 0; i < H; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < 2 * I; ++j)
          acc += DH[t * 2 * I + j] * ld(Ws1, i * 2 * I + j, dt);
        dxt[i] = acc;
      }
    }
    free(h);
    free(o);
    free(dO);
    free(dA);
  }
  for (int64_t i = 0; i < H * 2 * I; ++i) dWs1[i] = 0.0;
  for (int64_t i = 0; i < I * H; ++i) dWs2[i] = 0.0;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < I; ++j)
    for (int64_t t = 0; t < T; ++t) {
      double aj = A[t * I + j];
      for (int64_t c = 0; c < H; ++c)
        dWs2[j * H + c] += aj * ld(dy, t * H + c, dt);
    }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < H; ++i)
    for (int64_t t = 0; t < T; ++t) {
      double xi = ld(x, t * H + i, dt);
      for (int64_t j = 0; j < 2 * I; ++j)
        dWs1[i * 2 * I + j] += xi * DH[t * 2 * I + j];
    }
  free(A);
  free(DH);
}
