/*
 * moe_oracle.c -- plain, slow, CPU reference of the sparse Mixture-of-Experts
 * feed-forward block.  TEST INFRASTRUCTURE ONLY: nothing on the product path
 * links, loads or calls this file.  It shares no code, header, table or helper
 * with the CUDA library; only the seeded input generators serve both.
 *
 * Source: "Optimizing on-device inference for Apple Silicon" (Perplexity blog,
 * 2026-09-01).  The block it describes, and which this file evaluates:
 *   - section "Qwen creates three distinct workload shapes": a router scores
 *     256 expert sub-networks and picks eight for every token; one shared
 *     expert processes every token as well.
 *   - section "Reduce intermediate traffic and dispatch traffic": an expert is
 *     two input projections followed by a gated activation and one output
 *     projection; the output projection is weighted by the routing score and
 *     summed with the shared expert's result.
 *   - section "Keep expert routing on the GPU": after top-8 selection a
 *     histogram counts the assignments per expert.
 * Where the page leaves a step open the plain reading is taken:
 *   - the routing weight of a chosen expert is its softmax probability over all
 *     E logits, renormalised over the k chosen ones;
 *   - the gated activation is SiLU (SwiGLU): h = silu(W_gate x) * (W_up x),
 *     silu(z) = z / (1 + exp(-z));
 *   - the shared expert has the same shape as a routed one and weight 1;
 *   - no biases inside the expert projections; an optional per-expert bias
 *     enters the router logits;
 *   - ties in the top-k selection go to the lower expert index.
 *
 * Arithmetic: every input element is widened exactly to double and every sum
 * and product runs in double.  One value is narrowed on purpose: the router
 * logit is rounded to float before the top-k decision, because the selection
 * is an integer decision and is taken in the precision the pages give their
 * matrix products (32-bit float accumulation, section "Dequantise weights
 * within matrix multiplication").  The softmax, the weights and the experts
 * then run in double on those logits.
 *
 * Layouts (row-major):  x[T][d]; Wr[E][d]; Wg_e, Wu_e [F][d]; Wd_e [d][F];
 * Sg, Su [F][d]; Sd [d][F].  Element type of x and the router: dtype 0 =
 * bfloat16 bit patterns (uint16), dtype 1 = float32.  Expert weights (routed
 * and shared) have the same type, or, with wdtype 2, the 4-bit group-affine
 * format of section "Dequantise weights within matrix multiplication": each
 * matrix is an oracle_q4 record (below) whose element (r, c) is
 *     w = scale[r][c / 64] * q + bias[r][c / 64],   q = the 4-bit code,
 * codes packed two per byte along the row, the even column in the low nibble,
 * scale and bias bfloat16.  The oracle widens scale, bias and q exactly to
 * double and forms w in double.  Expert weights are passed as an array of E
 * pointers so a caller may hand over only the experts it needs; a selected
 * expert whose pointer is NULL is an error.
 *
 * Parity pins live in tests/test_oracle_pins.py (brute force, library
 * cross-checks, closed forms, invariants) and tests/test_oracle_mutations.py,
 * which rebuilds this file with ORACLE_MUTATION=n and checks that each planted
 * mistake fails at least one pin.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

typedef struct {
  int d;        /* model width */
  int F;        /* expert intermediate width */
  int E;        /* routed experts */
  int k;        /* experts chosen per token */
  int n_shared; /* 0 or 1 */
  int dtype;    /* x and router: 0 = bf16 bits, 1 = f32 */
  int wdtype;   /* expert weights: 0 = bf16 bits, 1 = f32, 2 = 4-bit group-affine */
} oracle_dims;

/* One matrix in the 4-bit group-affine format (wdtype 2). */
typedef struct {
  const uint8_t *codes;   /* [rows][cols / 2] */
  const uint16_t *scales; /* [rows][cols / 64] bfloat16 bits */
  const uint16_t *biases; /* [rows][cols / 64] bfloat16 bits */
} oracle_q4;

#define ORACLE_Q4_GROUP 64

/* Exact widening of one stored element to double. */
static double elem(const void *base, int dtype, size_t i) {
  if (dtype == 1) return (double)((const float *)base)[i];
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double bf16_bits(uint16_t b) {
  uint32_t bits = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Element (r, c) of an R x C expert matrix of type wdtype, in double. */
static double welem(const void *M, int wdtype, size_t r, size_t c, size_t C) {
  if (wdtype != 2) return elem(M, wdtype, r * C + c);
  const oracle_q4 *q = (const oracle_q4 *)M;
  const size_t i = r * C + c;
  const uint8_t byte = q->codes[i / 2];
#if ORACLE_MUTATION == 9
  const unsigned code = (i & 1) ? (byte & 15u) : (byte >> 4); /* planted: nibbles swapped */
#else
  const unsigned code = (i & 1) ? (byte >> 4) : (byte & 15u);
#endif
  const size_t g = r * (C / ORACLE_Q4_GROUP) + c / ORACLE_Q4_GROUP;
  return bf16_bits(q->scales[g]) * (double)code + bf16_bits(q->biases[g]);
}

/* y[r] = sum_c M[r][c] * v[c] for an R x C row-major matrix, double accumulate. */
static void matvec(const void *M, int dtype, int R, int C, const double *v, double *y) {
  for (int r = 0; r < R; ++r) {
    double acc = 0.0;
    for (int c = 0; c < C; ++c) acc += welem(M, dtype, (size_t)r, (size_t)c, (size_t)C) * v[c];
    y[r] = acc;
  }
}

static double silu(double z) {
#if ORACLE_MUTATION == 2
  return z / (1.0 + exp(z)); /* planted: wrong sign */
#else
  return z / (1.0 + exp(-z));
#endif
}

/*
 * Router of one token: logits (rounded to float), top-k selection, routing
 * weights.  Section "Qwen creates three distinct workload shapes" (scores over
 * 256 experts, eight chosen); weights = softmax over all E, renormalised over
 * the chosen k.  sel[] is ordered by descending logit, ties to lower index.
 */
static void route_token(const oracle_dims *D, const double *xv, const void *wr,
                        const float *bias, float *logit, int32_t *sel, double *w) {
  const int E = D->E, d = D->d, k = D->k;
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
#if ORACLE_MUTATION == 6
    for (int i = 0; i < d; ++i) acc += xv[i] * elem(wr, D->dtype, (size_t)i * E + e); /* planted: transposed */
#else
    for (int i = 0; i < d; ++i) acc += xv[i] * elem(wr, D->dtype, (size_t)e * d + i);
#endif
    if (bias) acc += (double)bias[e];
    logit[e] = (float)acc;
  }
  /* selection: k passes, each takes the largest logit not yet taken */
  char *taken = (char *)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
#if ORACLE_MUTATION == 5
      if (best < 0 || logit[e] < logit[best]) best = e; /* planted: smallest instead of largest */
#else
      if (best < 0 || logit[e] > logit[best]) best = e;
#endif
    }
    taken[best] = 1;
    sel[j] = best;
  }
  free(taken);
  /* softmax over all E logits with the maximum subtracted */
  double mx = (double)logit[0];
  for (int e = 1; e < E; ++e)
    if ((double)logit[e] > mx) mx = (double)logit[e];
  double z = 0.0;
  for (int e = 0; e < E; ++e) z += exp((double)logit[e] - mx);
  double psel = 0.0;
  for (int j = 0; j < k; ++j) {
    w[j] = exp((double)logit[sel[j]] - mx) / z;
    psel += w[j];
  }
#if ORACLE_MUTATION != 4 /* mutation 4 plants: no renormalisation */
  for (int j = 0; j < k; ++j) w[j] /= psel;
#endif
}

/*
 * One SwiGLU expert applied to one token, accumulated into out with a scale:
 * out += scale * Wd (silu(Wg x) * (Wu x)).
 * Section "Reduce intermediate traffic and dispatch traffic" (two input
 * projections with their gated activation; output projection with its routing
 * score).
 */
static void expert_token(const oracle_dims *D, const double *xv, const void *wg, const void *wu,
                         const void *wd, double scale, double *out, double *g, double *u,
                         double *y) {
  const int d = D->d, F = D->F;
  matvec(wg, D->wdtype, F, d, xv, g);
  matvec(wu, D->wdtype, F, d, xv, u);
  for (int f = 0; f < F; ++f) {
#if ORACLE_MUTATION == 7
    g[f] = u[f]; /* planted: activation dropped */
#else
    g[f] = silu(g[f]) * u[f];
#endif
  }
#if ORACLE_MUTATION == 3
  for (int i = 0; i < d; ++i) { /* planted: output projection read transposed */
    double acc = 0.0;
    for (int f = 0; f < F; ++f) acc += welem(wd, D->wdtype, (size_t)f, (size_t)i, (size_t)d) * g[f];
    y[i] = acc;
  }
#else
  matvec(wd, D->wdtype, d, F, g, y);
#endif
  for (int i = 0; i < d; ++i) out[i] += scale * y[i];
}

/* counts[e] = #{(t, j) : idx[t][j] == e} -- section "Keep expert routing on the
 * GPU" (a histogram counts the assignments that went to each expert). */
static void histogram(const int32_t *idx, int T, int k, int E, int32_t *counts) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int t = 0; t < T; ++t)
#if ORACLE_MUTATION == 8
    counts[idx[(size_t)t * k]]++; /* planted: only the first choice counted */
#else
    for (int j = 0; j < k; ++j) counts[idx[(size_t)t * k + j]]++;
#endif
}

static int check_dims(const oracle_dims *D) {
  if (!D || D->d <= 0 || D->F <= 0 || D->E <= 0 || D->k <= 0 || D->k > D->E) return -1;
  if (D->n_shared != 0 && D->n_shared != 1) return -1;
  if (D->dtype != 0 && D->dtype != 1) return -1;
  if (D->wdtype != 0 && D->wdtype != 1 && D->wdtype != 2) return -1;
  if (D->wdtype == 2 && (D->d % ORACLE_Q4_GROUP || D->F % ORACLE_Q4_GROUP)) return -1;
  return 0;
}

/*
 * Routing only.  idx[T][k], w[T][k] (double), logits[T][E] (float, may be
 * NULL), counts[E] (may be NULL).  counts[e] = number of tokens that chose e
 * (section "Keep expert routing on the GPU": the histogram step).
 * Returns 0, or -1 on bad arguments.
 */
int oracle_route(const oracle_dims *D, const void *x, int T, const void *wr, const float *bias,
                 int32_t *idx, double *w, float *logits, int32_t *counts, int nthreads) {
  if (check_dims(D) || T < 0 || (T > 0 && (!x || !wr || !idx || !w))) return -1;
  const int E = D->E, d = D->d, k = D->k;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 4)
  for (int t = 0; t < T; ++t) {
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    float *lg = logits ? logits + (size_t)t * E : (float *)malloc(sizeof(float) * (size_t)E);
    for (int i = 0; i < d; ++i) xv[i] = elem(x, D->dtype, (size_t)t * d + i);
    route_token(D, xv, wr, bias, lg, idx + (size_t)t * k, w + (size_t)t * k);
    if (!logits) free(lg);
    free(xv);
  }
  if (counts) histogram(idx, T, k, E, counts);
  return 0;
}

/*
 * The whole block for T tokens:
 *   out[t] = sum_{j<k} w[t][j] * E_{idx[t][j]}(x_t)  +  S(x_t)   (S only if n_shared)
 * out is double [T][d].  wg/wu/wd are arrays of E pointers (entries may be NULL
 * for experts no token selects).  idx, w, counts as in oracle_route (idx and w
 * are required here, counts may be NULL).  Returns 0, -1 on bad arguments, -2
 * when a selected expert has no weights.
 */
int oracle_forward(const oracle_dims *D, const void *x, int T, const void *wr, const float *bias,
                   const void *const *wg, const void *const *wu, const void *const *wd,
                   const void *sg, const void *su, const void *sd, double *out, int32_t *idx,
                   double *w, int32_t *counts, int nthreads) {
  if (check_dims(D) || T < 0) return -1;
  if (T == 0) {
    if (counts)
      for (int e = 0; e < D->E; ++e) counts[e] = 0;
    return 0;
  }
  if (!x || !wr || !wg || !wu || !wd || !out || !idx || !w) return -1;
  if (D->n_shared && (!sg || !su || !sd)) return -1;
  const int E = D->E, d = D->d, F = D->F, k = D->k;
  if (nthreads < 1) nthreads = 1;
  int missing = 0;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : missing)
  for (int t = 0; t < T; ++t) {
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *g = (double *)malloc(sizeof(double) * (size_t)F);
    double *u = (double *)malloc(sizeof(double) * (size_t)F);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    float *lg = (float *)malloc(sizeof(float) * (size_t)E);
    double *o = out + (size_t)t * d;
    for (int i = 0; i < d; ++i) xv[i] = elem(x, D->dtype, (size_t)t * d + i);
    route_token(D, xv, wr, bias, lg, idx + (size_t)t * k, w + (size_t)t * k);
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      if (!wg[e] || !wu[e] || !wd[e]) {
        missing = 1;
        continue;
      }
      expert_token(D, xv, wg[e], wu[e], wd[e], w[(size_t)t * k + j], o, g, u, y);
    }
#if ORACLE_MUTATION != 1 /* mutation 1 plants: shared expert dropped */
    if (D->n_shared) expert_token(D, xv, sg, su, sd, 1.0, o, g, u, y);
#endif
    free(lg);
    free(y);
    free(u);
    free(g);
    free(xv);
  }
  if (counts) histogram(idx, T, k, E, counts);
  return missing ? -2 : 0;
}

/* Version tag so a loader can check it has the file it expects. */
int oracle_version(void) { return 1; }
