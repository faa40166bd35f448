/*
 * Plain CPU oracle for the page-table-aware fused MoE layer of Rimuru
 * ("Rimuru: Unified Memory Management for Modern LLM Serving via Elastic
 * Expert Offloading", arXiv 2610.40305; abstract, and the explainer page
 * "Rimuru unifies serving memory", paragraph on the page-table-aware kernel).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * it is linked by the tests, by the smoke check and by the CPU-baseline leg of
 * the benchmark, and by nothing else.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * What the layer computes (the pages give the mechanism, not the formulas, so
 * the arithmetic below is the standard top-k MoE FFN; every reading is listed
 * in the design notes):
 *   1. each expert projection is read from one page of the expert memory
 *      view: bytes [page_id * page_bytes, page_id * page_bytes + rows*cols*2)
 *      of the shared pool, bf16, row-major [rows][cols]
 *      (memory views: abstract; Figure 6);
 *      w1, w3 are [H][I] and w2 is [I][H] (Table 1, taken literally);
 *   2. routing: the k largest router logits, larger value first, lower expert
 *      index first among equal values; weights are softmax probabilities of the
 *      chosen experts, renormalised over the k chosen ones (or divided by the
 *      full softmax sum when renorm == 0);
 *   3. grouping: assignment f = t*k + j goes to expert ids[f]; assignments are
 *      listed expert by expert, ascending f inside one expert (stable);
 *   4. per assignment: g = x_t W1, u = x_t W3, h = silu(g) * u with
 *      silu(g) = g / (1 + exp(-g)), y = h W2;
 *   5. combine: out_t = sum over j = 0..k-1 of w[t*k+j] * y[t*k+j].
 *
 * Precision: every floating-point value is carried in double (bf16 inputs are
 * widened exactly); nothing is rounded in between.  Routing decisions compare
 * the fp32 logits as given, so they are exact.  Weights are returned rounded
 * to fp32; h, y and out are returned in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes. */
#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_PAGE -2
#define ORACLE_ERR_NONFINITE -3
#define ORACLE_ERR_NOMEM -4

/* bf16 bit pattern -> double, decoded field by field (1 sign bit, 8 exponent
 * bits with bias 127, 7 fraction bits). */
double oracle_bf16_to_f64(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 7) & 0xFF;
  int frac = bits & 0x7F;
  double v;
  if (expo == 0xFF) {
    v = frac ? NAN : INFINITY;
  } else if (expo == 0) {
    v = ldexp((double)frac, -126 - 7); /* subnormal: 0.frac * 2^-126 */
  } else {
    v = ldexp(1.0 + (double)frac / 128.0, expo - 127);
  }
  return sign ? -v : v;
}

/* Step 1: copy one page of the expert view out into a contiguous double
 * matrix [rows][cols].  Fails if the page does not lie inside the pool. */
int oracle_page_to_matrix(const uint8_t* pool, uint64_t pool_bytes, uint64_t page_bytes,
                          int64_t page_id, int rows, int cols, double* out) {
  uint64_t need = (uint64_t)rows * (uint64_t)cols * 2u;
  if (page_id < 0 || need > page_bytes) return ORACLE_ERR_PAGE;
  uint64_t start = (uint64_t)page_id * page_bytes;
  if (start + page_bytes > pool_bytes) return ORACLE_ERR_PAGE;
  const uint8_t* src = pool + start;
  for (int r = 0; r < rows; ++r) {
    for (int c = 0; c < cols; ++c) {
      uint64_t at = ((uint64_t)r * (uint64_t)cols + (uint64_t)c) * 2u;
      uint16_t bits = (uint16_t)(src[at] | ((uint16_t)src[at + 1] << 8)); /* little endian */
      out[(size_t)r * cols + c] = oracle_bf16_to_f64(bits);
    }
  }
  return ORACLE_OK;
}

/* "a ranks before b": larger logit first, lower index first on equal logits. */
static int ranks_before(const float* l, int a, int b) {
  if (l[a] > l[b]) return 1;
  if (l[a] < l[b]) return 0;
  return a < b;
}

/* Step 2: routing for T tokens over E experts, k chosen per token.
 * ids[t*k + j] is the expert in slot j of token t; w the matching weight
 * rounded to fp32; wd (may be NULL) the same weight in double. */
static int route_impl(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                      float* w, double* wd) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return ORACLE_ERR_ARG;
  int* order = (int*)malloc(sizeof(int) * (size_t)E);
  if (!order) return ORACLE_ERR_NOMEM;
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      if (!isfinite(l[e])) { free(order); return ORACLE_ERR_NONFINITE; }
    }
    /* sort 0..E-1 by the key (-logit, index): insertion sort */
    for (int e = 0; e < E; ++e) order[e] = e;
    for (int i = 1; i < E; ++i) {
      int cur = order[i];
      int p = i - 1;
      while (p >= 0 && ranks_before(l, cur, order[p])) {
        order[p + 1] = order[p];
        --p;
      }
      order[p + 1] = cur;
    }
    /* softmax probabilities, shifted by the largest logit */
    double m = (double)l[order[0]];
    double sum_topk = 0.0, sum_all = 0.0;
    for (int j = 0; j < k; ++j) sum_topk += exp((double)l[order[j]] - m);
    for (int e = 0; e < E; ++e) sum_all += exp((double)l[e] - m);
    double denom = renorm ? sum_topk : sum_all;
    for (int j = 0; j < k; ++j) {
      double p = exp((double)l[order[j]] - m) / denom;
      ids[(size_t)t * k + j] = order[j];
      w[(size_t)t * k + j] = (float)p;
      if (wd) wd[(size_t)t * k + j] = p;
    }
  }
  free(order);
  return ORACLE_OK;
}

int oracle_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids, float* w) {
  return route_impl(logits, T, E, k, renorm, ids, w, NULL);
}

/* Step 3: stable counting sort of the A = T*k assignments by expert.
 * offsets[e] .. offsets[e+1]-1 are the positions of expert e in sorted[]. */
int oracle_align(const int32_t* ids, int A, int E, int32_t* sorted, int32_t* offsets) {
  if (A < 0 || E <= 0) return ORACLE_ERR_ARG;
  int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!cursor) return ORACLE_ERR_NOMEM;
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int f = 0; f < A; ++f) {
    if (ids[f] < 0 || ids[f] >= E) { free(cursor); return ORACLE_ERR_ARG; }
    offsets[ids[f] + 1] += 1;
  }
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int f = 0; f < A; ++f) {
    int e = ids[f];
    sorted[cursor[e]] = f;
    cursor[e] += 1;
  }
  free(cursor);
  return ORACLE_OK;
}

/* Step 4 for one assignment: g = x W1, u = x W3, h = silu(g) * u, y = h W2. */
static void expert_ffn(const double* x, const double* w1, const double* w3, const double* w2,
                       int H, int I, double* g, double* u, double* h, double* y) {
  for (int i = 0; i < I; ++i) { g[i] = 0.0; u[i] = 0.0; }
  for (int r = 0; r < H; ++r) {
    for (int i = 0; i < I; ++i) {
      g[i] += x[r] * w1[(size_t)r * I + i];
      u[i] += x[r] * w3[(size_t)r * I + i];
    }
  }
  for (int i = 0; i < I; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
  for (int c = 0; c < H; ++c) y[c] = 0.0;
  for (int i = 0; i < I; ++i) {
    for (int c = 0; c < H; ++c) y[c] += h[i] * w2[(size_t)i * H + c];
  }
}

/*
 * The whole layer.
 *   x        bf16 bits [T][H];   logits fp32 [T][E]
 *   pool     host copy of the shared pool, pool_bytes long
 *   pt       page table of this layer in expert-view page ids, [E][3]
 *            (column 0 = w1, 1 = w3, 2 = w2)
 *   tokens   if n_tokens >= 0, only these tokens get outputs (routing and
 *            grouping still cover all T tokens); NULL/-1 means every token
 * Outputs (any of h, y may be NULL):
 *   ids int32 [T*k], w fp32 [T*k], sorted int32 [T*k], offsets int32 [E+1],
 *   h double [T*k][I], y double [T*k][H] (rows of assignments that were
 *   computed), out double [T][H] (rows of computed tokens; others untouched).
 *   nthreads > 0 sets the OpenMP thread count used across experts.
 */
int oracle_moe_forward(const uint16_t* x, const float* logits, int T, int H, int I, int E,
                       int k, int renorm, const uint8_t* pool, uint64_t pool_bytes,
                       uint64_t page_bytes, const int32_t* pt, const int32_t* tokens,
                       int n_tokens, int nthreads, int32_t* ids, float* w, int32_t* sorted,
                       int32_t* offsets, double* h, double* y, double* out) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E || page_bytes == 0)
    return ORACLE_ERR_ARG;
  const int A = T * k;
  double* wd = (double*)malloc(sizeof(double) * (size_t)(A > 0 ? A : 1));
  if (!wd) return ORACLE_ERR_NOMEM;
  int st = route_impl(logits, T, E, k, renorm, ids, w, wd);
  if (st == ORACLE_OK) st = oracle_align(ids, A, E, sorted, offsets);
  if (st != ORACLE_OK) { free(wd); return st; }

  /* which tokens need outputs */
  uint8_t* want = (uint8_t*)calloc((size_t)(T > 0 ? T : 1), 1);
  double* yall = (double*)malloc(sizeof(double) * (size_t)(A > 0 ? A : 1) * (size_t)H);
  if (!want || !yall) { free(want); free(yall); free(wd); return ORACLE_ERR_NOMEM; }
  if (tokens == NULL || n_tokens < 0) {
    for (int t = 0; t < T; ++t) want[t] = 1;
  } else {
    for (int s = 0; s < n_tokens; ++s) {
      if (tokens[s] < 0 || tokens[s] >= T) { free(want); free(yall); free(wd); return ORACLE_ERR_ARG; }
      want[tokens[s]] = 1;
    }
  }

  int failed = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int e = 0; e < E; ++e) {
    /* does any wanted assignment go to expert e? */
    int used = 0;
    for (int s = offsets[e]; s < offsets[e + 1]; ++s) used |= want[sorted[s] / k];
    if (!used) continue;
    /* the matrices are read only through this expert's own pages */
    double* w1 = (double*)malloc(sizeof(double) * (size_t)H * I);
    double* w3 = (double*)malloc(sizeof(double) * (size_t)H * I);
    double* w2 = (double*)malloc(sizeof(double) * (size_t)I * H);
    double* xt = (double*)malloc(sizeof(double) * (size_t)H);
    double* g = (double*)malloc(sizeof(double) * (size_t)I);
    double* u = (double*)malloc(sizeof(double) * (size_t)I);
    double* hh = (double*)malloc(sizeof(double) * (size_t)I);
    int bad = (!w1 || !w3 || !w2 || !xt || !g || !u || !hh) ? ORACLE_ERR_NOMEM : ORACLE_OK;
    if (bad == ORACLE_OK)
      bad = oracle_page_to_matrix(pool, pool_bytes, page_bytes, pt[e * 3 + 0], H, I, w1);
    if (bad == ORACLE_OK)
      bad = oracle_page_to_matrix(pool, pool_bytes, page_bytes, pt[e * 3 + 1], H, I, w3);
    if (bad == ORACLE_OK)
      bad = oracle_page_to_matrix(pool, pool_bytes, page_bytes, pt[e * 3 + 2], I, H, w2);
    if (bad == ORACLE_OK) {
      for (int s = offsets[e]; s < offsets[e + 1]; ++s) {
        int f = sorted[s];
        int t = f / k;
        if (!want[t]) continue;
        for (int r = 0; r < H; ++r) xt[r] = oracle_bf16_to_f64(x[(size_t)t * H + r]);
        expert_ffn(xt, w1, w3, w2, H, I, g, u, hh, yall + (size_t)f * H);
        if (h) memcpy(h + (size_t)f * I, hh, sizeof(double) * (size_t)I);
      }
    }
    free(w1); free(w3); free(w2); free(xt); free(g); free(u); free(hh);
    if (bad != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
      failed = bad;
    }
  }
  if (failed != ORACLE_OK) { free(want); free(yall); free(wd); return failed; }

  /* Step 5: weighted combine, slots in order j = 0..k-1 */
  for (int t = 0; t < T; ++t) {
    if (!want[t]) continue;
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        int f = t * k + j;
        acc += wd[f] * yall[(size_t)f * H + c];
      }
      out[(size_t)t * H + c] = acc;
    }
    if (y) {
      for (int j = 0; j < k; ++j) {
        int f = t * k + j;
        memcpy(y + (size_t)f * H, yall + (size_t)f * H, sizeof(double) * (size_t)H);
      }
    }
  }
  free(want);
  free(yall);
  free(wd);
  return ORACLE_OK;
}

/* Threads the oracle will use (1 when built without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
