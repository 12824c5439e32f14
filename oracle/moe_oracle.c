/*
 * moe_oracle.c -- plain, slow CPU oracle for the sparse Mixture-of-Experts forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes follows "Distributed Training Part 4: Tensor Parallelism, Hybrid
 * Parallelism, MoE + Expert Parallelism" (jesamkim ai-tech-blog, 2026-04-16):
 *   - §3 "Mixture of Experts", Structure: a router that is a linear layer followed by a
 *     softmax over the experts; each expert an independent FFN; the output
 *     y = sum over i in TopK of G(x)_i * E_i(x), with only the k best experts used.
 *   - §3, Load-Balancing Loss: an auxiliary scalar (Switch Transformer style) that is
 *     smallest when tokens are spread evenly over the experts.
 *   - §4 "Expert Parallelism", Dispatch and Combine: every token is sent to the experts
 *     the router chose and the expert outputs are sent back to the token.
 * Readings where the page is silent (each one also listed in the design notes):
 *   - expert FFN is SwiGLU: E_i(x) = W2_i (SiLU(W1_i x) * (W3_i x)), no biases;
 *   - logits z = (x . W_r[e] + b_e) / tau, gates are the chosen softmax entries, not
 *     renormalised over the k chosen;
 *   - top-k order: descending logit, equal logits -> lower expert index first; the
 *     decision is taken on the logit rounded to fp32, the precision the GPU decides in;
 *   - dispatch order: a counting sort by expert that is stable in token order;
 *   - aux = E * sum_i f_i * P_i, f_i = count_i / (T k), P_i = mean over tokens of p_i.
 *
 * Arithmetic is fp64 throughout, on inputs that are exact fp32 values or bf16 bit
 * patterns widened exactly; every sum runs sequentially in index order.  Tokens are
 * independent, so loops over tokens run under OpenMP without changing any result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NO_MEM 2

typedef struct {
  int64_t T;     /* tokens */
  int32_t d;     /* d_model */
  int32_t E;     /* number of experts */
  int32_t k;     /* experts chosen per token */
  int32_t F;     /* d_expert: hidden width of one expert */
  int32_t dtype; /* storage of x and weights: 0 = fp32, 1 = bf16 bit patterns */
  double tau;    /* router temperature, > 0 */
  int32_t renorm; /* 0: gates are the chosen softmax entries; 1: renormalised over the k chosen */
} orc_cfg;

/* Element i of a fp32 or bf16 array, widened exactly to double. */
static double orc_load(const void* base, int32_t dtype, int64_t i) {
  if (dtype == 1) {
    uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

static int orc_check(const orc_cfg* c) {
  if (!c || c->T < 0 || c->d <= 0 || c->E <= 0 || c->k <= 0 || c->k > c->E || c->F <= 0 ||
      !(c->tau > 0.0) || (c->dtype != 0 && c->dtype != 1) || (c->renorm != 0 && c->renorm != 1))
    return ORC_BAD_ARG;
  return ORC_OK;
}

/*
 * Router (§3 Structure: linear layer + softmax) and top-k selection (§3, the TopK of the
 * output formula).  Per token t:
 *   z[t,e]   = (sum_c x[t,c] W_r[e,c] + b_e) / tau
 *   p[t,e]   = exp(z[t,e] - max_e z) / sum_e' exp(z[t,e'] - max z)
 *   idx[t,:] = the k experts with the largest fp32-rounded z, descending, ties to the
 *              lower index
 *   gate[t,j]= p[t, idx[t,j]]
 * or, with renorm (a variant the page's TopK leaves open), the same entries divided by
 * their sum over the k chosen (summed in j order), i.e. a softmax over the chosen logits.
 * bias may be NULL (no bias).  Any of z, p may be NULL when not wanted.
 */
int orc_router(const orc_cfg* c, const void* x, const void* wr, const float* bias, double* z,
               double* p, int32_t* idx, double* gate) {
  if (orc_check(c) || !x || !wr || !idx || !gate) return ORC_BAD_ARG;
  const int64_t T = c->T;
  const int32_t d = c->d, E = c->E, k = c->k;
  int failed = 0;
#pragma omp parallel
  {
    double* zt = (double*)malloc(sizeof(double) * (size_t)E);
    double* pt = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    if (!zt || !pt || !taken) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) {
          double acc = 0.0;
          for (int32_t col = 0; col < d; ++col)
            acc += orc_load(x, c->dtype, t * d + col) * orc_load(wr, c->dtype, (int64_t)e * d + col);
          if (bias) acc += (double)bias[e];
          zt[e] = acc / c->tau;
        }
        double m = zt[0];
        for (int32_t e = 1; e < E; ++e)
          if (zt[e] > m) m = zt[e];
        double s = 0.0;
        for (int32_t e = 0; e < E; ++e) {
          pt[e] = exp(zt[e] - m);
          s += pt[e];
        }
        for (int32_t e = 0; e < E; ++e) pt[e] /= s;
        /* selection: repeatedly take the best remaining expert; strict '>' keeps the
           lower index on equal fp32 logits */
        memset(taken, 0, (size_t)E);
        for (int32_t j = 0; j < k; ++j) {
          int32_t best = -1;
          float bestv = 0.0f;
          for (int32_t e = 0; e < E; ++e) {
            if (taken[e]) continue;
            float v = (float)zt[e];
            if (best < 0 || v > bestv) {
              best = e;
              bestv = v;
            }
          }
          taken[best] = 1;
          idx[t * k + j] = best;
          gate[t * k + j] = pt[best];
        }
        if (c->renorm) {
          double chosen = 0.0;
          for (int32_t j = 0; j < k; ++j) chosen += gate[t * k + j];
          for (int32_t j = 0; j < k; ++j) gate[t * k + j] /= chosen;
        }
        if (z)
          for (int32_t e = 0; e < E; ++e) z[t * E + e] = zt[e];
        if (p)
          for (int32_t e = 0; e < E; ++e) p[t * E + e] = pt[e];
      }
    }
    free(zt);
    free(pt);
    free(taken);
  }
  return failed ? ORC_NO_MEM : ORC_OK;
}

/*
 * Dispatch (§4 Dispatch: each token goes to the experts its router chose), on one device:
 *   counts[e]        = number of (t, j) with idx[t,j] = e
 *   offsets[e]       = counts[0] + ... + counts[e-1], offsets[E] = T k
 *   perm_src[p]      = token of the p-th row of the expert-contiguous order
 *   perm_slot[p]     = its slot t*k + j
 * Rows of one expert appear in ascending (t, j) order, i.e. a counting sort stable in
 * token order.  perm_src / perm_slot may be NULL.
 */
int orc_dispatch(const orc_cfg* c, const int32_t* idx, int32_t* counts, int32_t* offsets,
                 int32_t* perm_src, int32_t* perm_slot) {
  if (orc_check(c) || !idx || !counts || !offsets) return ORC_BAD_ARG;
  const int64_t T = c->T;
  const int32_t E = c->E, k = c->k;
  for (int32_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < T * k; ++s) {
    if (idx[s] < 0 || idx[s] >= E) return ORC_BAD_ARG;
    counts[idx[s]] += 1;
  }
  offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!cursor) return ORC_NO_MEM;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t j = 0; j < k; ++j) {
      int32_t e = idx[t * k + j];
      int32_t pos = offsets[e] + cursor[e]++;
      if (perm_src) perm_src[pos] = (int32_t)t;
      if (perm_slot) perm_slot[pos] = (int32_t)(t * k + j);
    }
  free(cursor);
  return ORC_OK;
}

/* One expert on one token (§3 Structure: the expert is an FFN; SwiGLU form):
 *   a = W1_e xr,  g = W3_e xr           (W1_e, W3_e are [F, d], rows = hidden units)
 *   h = a * sigmoid(a) * g              (sigmoid(a) = 1 / (1 + exp(-a)))
 *   out = W2_e h                        (W2_e is [d, F])
 * xr has d entries; h (F entries) may be NULL. */
static void orc_expert_row(const orc_cfg* c, const void* w1, const void* w3, const void* w2,
                           int32_t e, const double* xr, double* h, double* out) {
  const int32_t d = c->d, F = c->F;
  const int64_t wbase = (int64_t)e * F * d;
  for (int32_t f = 0; f < F; ++f) {
    double a = 0.0, g = 0.0;
    for (int32_t col = 0; col < d; ++col) {
      a += orc_load(w1, c->dtype, wbase + (int64_t)f * d + col) * xr[col];
      g += orc_load(w3, c->dtype, wbase + (int64_t)f * d + col) * xr[col];
    }
    h[f] = a / (1.0 + exp(-a)) * g;
  }
  for (int32_t r = 0; r < d; ++r) {
    double acc = 0.0;
    for (int32_t f = 0; f < F; ++f) acc += orc_load(w2, c->dtype, wbase + (int64_t)r * F + f) * h[f];
    out[r] = acc;
  }
}

/* Public single (token, expert) evaluation, for checking one routed row at a time:
 * h_out [F] and out [d] receive the SwiGLU hidden vector and the expert output. */
int orc_expert(const orc_cfg* c, const void* x, const void* w1, const void* w3, const void* w2,
               int64_t t, int32_t e, double* h_out, double* out) {
  if (orc_check(c) || !x || !w1 || !w3 || !w2 || !out || t < 0 || t >= c->T || e < 0 || e >= c->E)
    return ORC_BAD_ARG;
  double* xr = (double*)malloc(sizeof(double) * (size_t)c->d);
  double* h = (double*)malloc(sizeof(double) * (size_t)c->F);
  if (!xr || !h) {
    free(xr);
    free(h);
    return ORC_NO_MEM;
  }
  for (int32_t col = 0; col < c->d; ++col) xr[col] = orc_load(x, c->dtype, t * c->d + col);
  orc_expert_row(c, w1, w3, w2, e, xr, h, out);
  if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)c->F);
  free(xr);
  free(h);
  return ORC_OK;
}

/* Many (token, expert) evaluations at once, for checking many routed rows: row i is expert
 * e[i] applied to token t[i], exactly as orc_expert computes it (the same per-row
 * arithmetic, rows independent, so the OpenMP loop over rows changes no result).
 * h_out [n, F] may be NULL; out [n, d] receives the expert outputs. */
int orc_expert_rows(const orc_cfg* c, const void* x, const void* w1, const void* w3, const void* w2, int64_t n,
                    const int64_t* t, const int32_t* e, double* h_out, double* out) {
  if (orc_check(c) || !x || !w1 || !w3 || !w2 || !t || !e || !out || n < 0) return ORC_BAD_ARG;
  for (int64_t i = 0; i < n; ++i)
    if (t[i] < 0 || t[i] >= c->T || e[i] < 0 || e[i] >= c->E) return ORC_BAD_ARG;
  const int32_t d = c->d, F = c->F;
  int failed = 0;
#pragma omp parallel
  {
    double* xr = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)F);
    if (!xr || !h) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < n; ++i) {
        for (int32_t col = 0; col < d; ++col) xr[col] = orc_load(x, c->dtype, t[i] * d + col);
        orc_expert_row(c, w1, w3, w2, e[i], xr, h, out + i * d);
        if (h_out) memcpy(h_out + i * F, h, sizeof(double) * (size_t)F);
      }
    }
    free(xr);
    free(h);
  }
  return failed ? ORC_NO_MEM : ORC_OK;
}

/*
 * Combine (§3 output formula; §4 Combine: expert outputs return to their token):
 *   y[i] = sum_{j=0..k-1} gate[t,j] * E_{idx[t,j]}(x[t]),   t = tokens[i]
 * summed in j order.  tokens == NULL means all tokens 0..T-1 (ntok must equal T).
 * idx / gate are the routing to use (the oracle's own, or any other).
 */
int orc_combine(const orc_cfg* c, const void* x, const void* w1, const void* w3, const void* w2,
                const int32_t* idx, const double* gate, const int64_t* tokens, int64_t ntok,
                double* y) {
  if (orc_check(c) || !x || !w1 || !w3 || !w2 || !idx || !gate || !y || ntok < 0) return ORC_BAD_ARG;
  if (!tokens && ntok != c->T) return ORC_BAD_ARG;
  const int32_t d = c->d, k = c->k;
  int failed = 0;
#pragma omp parallel
  {
    double* xr = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)c->F);
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    if (!xr || !h || !o) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < ntok; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        double* yr = y + i * d;
        if (t < 0 || t >= c->T) {
#pragma omp atomic write
          failed = 2;
          continue;
        }
        for (int32_t col = 0; col < d; ++col) {
          xr[col] = orc_load(x, c->dtype, t * d + col);
          yr[col] = 0.0;
        }
        for (int32_t j = 0; j < k; ++j) {
          int32_t e = idx[t * k + j];
          if (e < 0 || e >= c->E) {
#pragma omp atomic write
            failed = 2;
            break;
          }
          orc_expert_row(c, w1, w3, w2, e, xr, h, o);
          for (int32_t col = 0; col < d; ++col) yr[col] += gate[t * k + j] * o[col];
        }
      }
    }
    free(xr);
    free(h);
    free(o);
  }
  if (failed == 2) return ORC_BAD_ARG;
  return failed ? ORC_NO_MEM : ORC_OK;
}

/*
 * Load-balancing scalar (§3 Load-Balancing Loss; Switch Transformer form):
 *   f_i = counts[i] / (T k),  P_i = (1/T) sum_t p[t,i],  aux = E sum_i f_i P_i.
 * p is the full [T, E] softmax, summed over t in index order.
 */
int orc_aux(const orc_cfg* c, const double* p, const int32_t* counts, double* aux) {
  if (orc_check(c) || !p || !counts || !aux || c->T == 0) return ORC_BAD_ARG;
  const int64_t T = c->T;
  const int32_t E = c->E;
  double total = 0.0;
  for (int32_t i = 0; i < E; ++i) {
    double P = 0.0;
    for (int64_t t = 0; t < T; ++t) P += p[t * E + i];
    P /= (double)T;
    double f = (double)counts[i] / ((double)T * (double)c->k);
    total += f * P;
  }
  *aux = (double)E * total;
  return ORC_OK;
}

/*
 * The whole forward, in the order the page describes it: router, top-k, dispatch,
 * experts, combine, plus the balancing scalar.  Outputs (all host memory):
 *   y [T, d], idx [T, k], gate [T, k], counts [E], offsets [E+1], perm_src [T k],
 *   perm_slot [T k], aux (scalar).  z / p [T, E] may be NULL (then p is kept internally).
 */
int orc_forward(const orc_cfg* c, const void* x, const void* wr, const float* bias, const void* w1,
                const void* w3, const void* w2, double* y, int32_t* idx, double* gate, int32_t* counts,
                int32_t* offsets, int32_t* perm_src, int32_t* perm_slot, double* z, double* p,
                double* aux) {
  if (orc_check(c) || !y || !idx || !gate || !counts || !offsets || !aux) return ORC_BAD_ARG;
  double* pp = p ? p : (double*)malloc(sizeof(double) * (size_t)(c->T * c->E));
  if (!pp) return ORC_NO_MEM;
  int rc = orc_router(c, x, wr, bias, z, pp, idx, gate);
  if (!rc) rc = orc_dispatch(c, idx, counts, offsets, perm_src, perm_slot);
  if (!rc) rc = orc_combine(c, x, w1, w3, w2, idx, gate, NULL, c->T, y);
  if (!rc && c->T > 0) rc = orc_aux(c, pp, counts, aux);
  if (!p) free(pp);
  return rc;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int orc_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      extern int omp_get_num_threads(void);
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}

/*
 * Backward of the layer for the scalar  L = sum_t dy[t] . y[t] + alpha * aux
 * (the page's training setting: the balancing loss is added to the task loss; alpha is its
 * weight).  Routing (top-k choice, counts f_i) is piecewise constant and carries no
 * gradient; the gradient reaches the router through the gate values and through P_i.
 *   per slot (t, j), e = idx, g = gate:
 *     a = W1_e x, b = W3_e x, h = silu(a) b, o = W2_e h
 *     dg  = dy . o                      do = g dy
 *     dW2_e += do h^T                   dh = W2_e^T do
 *     da = dh * b * silu'(a)            db = dh * silu(a),  silu'(a) = s (1 + a (1 - s)), s = sigmoid(a)
 *     dW1_e += da x^T,  dW3_e += db x^T,  dx += W1_e^T da + W3_e^T db
 *   router, per token: dp_e = sum_j [idx_j = e] dg_j  (renormalised gates: dp at the chosen
 *     = (dg_j - sum_j' g_j' dg_j') / S, S = sum of the chosen p)  + alpha E f_e / T
 *     dz = p * (dp - sum_e p_e dp_e),  dl = dz / tau
 *     dW_r[e] += dl_e x,  dbias_e += dl_e,  dx += sum_e dl_e W_r[e]
 * Outputs (host, fp64): dx [T,d], dwr [E,d], dbias [E], dw1, dw3 [E,F,d], dw2 [E,d,F].
 * Weight gradients are summed over tokens in token order (OpenMP over output rows).
 */
int orc_backward(const orc_cfg* c, const void* x, const void* wr, const float* bias, const void* w1, const void* w3,
                 const void* w2, const double* dy, double alpha, double* dx, double* dwr, double* dbias,
                 double* dw1, double* dw3, double* dw2) {
  if (orc_check(c) || !x || !wr || !w1 || !w3 || !w2 || !dy || !dx || !dwr || !dbias || !dw1 || !dw3 || !dw2)
    return ORC_BAD_ARG;
  const int64_t T = c->T, N = c->T * c->k;
  const int32_t d = c->d, E = c->E, k = c->k, F = c->F;
  double* p = (double*)malloc(sizeof(double) * (size_t)(T * E));
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  double* gate = (double*)malloc(sizeof(double) * (size_t)N);
  int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
  double* sa = (double*)malloc(sizeof(double) * (size_t)(N * F)); /* per slot: da */
  double* sb = (double*)malloc(sizeof(double) * (size_t)(N * F)); /* db */
  double* sh = (double*)malloc(sizeof(double) * (size_t)(N * F)); /* h */
  double* dg = (double*)malloc(sizeof(double) * (size_t)N);
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)N); /* slot of each dispatched row */
  int rc = ORC_OK;
  if (!p || !idx || !gate || !counts || !offsets || !sa || !sb || !sh || !dg || !perm) rc = ORC_NO_MEM;
  if (!rc) rc = orc_router(c, x, wr, bias, NULL, p, idx, gate);
  if (!rc) rc = orc_dispatch(c, idx, counts, offsets, NULL, perm);
  int failed = 0;
  if (!rc) {
#pragma omp parallel
    {
      double* xr = (double*)malloc(sizeof(double) * (size_t)d);
      double* av = (double*)malloc(sizeof(double) * (size_t)F);
      double* bv = (double*)malloc(sizeof(double) * (size_t)F);
      double* dh = (double*)malloc(sizeof(double) * (size_t)F);
      double* o = (double*)malloc(sizeof(double) * (size_t)d);
      double* dp = (double*)malloc(sizeof(double) * (size_t)E);
      if (!xr || !av || !bv || !dh || !o || !dp) {
#pragma omp atomic write
        failed = 1;
      } else {
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
          double* dxt = dx + t * d;
          for (int32_t col = 0; col < d; ++col) {
            xr[col] = orc_load(x, c->dtype, t * d + col);
            dxt[col] = 0.0;
          }
          const double* dyt = dy + t * d;
          for (int32_t j = 0; j < k; ++j) {
            const int64_t slot = t * k + j;
            const int32_t e = idx[slot];
            const int64_t wb = (int64_t)e * F * d;
            double* h = sh + slot * F;
            for (int32_t f = 0; f < F; ++f) {
              double a = 0.0, b = 0.0;
              for (int32_t col = 0; col < d; ++col) {
                a += orc_load(w1, c->dtype, wb + (int64_t)f * d + col) * xr[col];
                b += orc_load(w3, c->dtype, wb + (int64_t)f * d + col) * xr[col];
              }
              av[f] = a;
              bv[f] = b;
              h[f] = a / (1.0 + exp(-a)) * b;
            }
            double g = gate[slot], dgs = 0.0;
            for (int32_t r = 0; r < d; ++r) {
              double acc = 0.0;
              for (int32_t f = 0; f < F; ++f) acc += orc_load(w2, c->dtype, wb + (int64_t)r * F + f) * h[f];
              o[r] = acc;
              dgs += dyt[r] * acc;
            }
            dg[slot] = dgs;
            /* dh = W2_e^T (g dy): each dh[f] summed over r in ascending order, walking W2 by rows */
            for (int32_t f = 0; f < F; ++f) dh[f] = 0.0;
            for (int32_t r = 0; r < d; ++r)
              for (int32_t f = 0; f < F; ++f) dh[f] += orc_load(w2, c->dtype, wb + (int64_t)r * F + f) * g * dyt[r];
            double* da = sa + slot * F;
            double* db = sb + slot * F;
            for (int32_t f = 0; f < F; ++f) {
              const double s = 1.0 / (1.0 + exp(-av[f]));
              da[f] = dh[f] * bv[f] * s * (1.0 + av[f] * (1.0 - s));
              db[f] = dh[f] * av[f] * s;
            }
            /* W1_e^T da + W3_e^T db: each column summed over f in ascending order, walking the
               weights by rows; then added to dx */
            for (int32_t col = 0; col < d; ++col) o[col] = 0.0;
            for (int32_t f = 0; f < F; ++f)
              for (int32_t col = 0; col < d; ++col)
                o[col] += orc_load(w1, c->dtype, wb + (int64_t)f * d + col) * da[f] +
                          orc_load(w3, c->dtype, wb + (int64_t)f * d + col) * db[f];
            for (int32_t col = 0; col < d; ++col) dxt[col] += o[col];
          }
          /* router */
          const double* pt = p + t * E;
          for (int32_t e = 0; e < E; ++e) dp[e] = alpha * (double)E * (double)counts[e] / ((double)T * (double)k) / (double)T;
          if (c->renorm) {
            double S = 0.0, gdg = 0.0;
            for (int32_t j = 0; j < k; ++j) S += pt[idx[t * k + j]];
            for (int32_t j = 0; j < k; ++j) gdg += gate[t * k + j] * dg[t * k + j];
            for (int32_t j = 0; j < k; ++j) dp[idx[t * k + j]] += (dg[t * k + j] - gdg) / S;
          } else {
            for (int32_t j = 0; j < k; ++j) dp[idx[t * k + j]] += dg[t * k + j];
          }
          double pdp = 0.0;
          for (int32_t e = 0; e < E; ++e) pdp += pt[e] * dp[e];
          for (int32_t e = 0; e < E; ++e) {
            const double dl = pt[e] * (dp[e] - pdp) / c->tau;
            dp[e] = dl; /* reuse: dlogit */
            for (int32_t col = 0; col < d; ++col) dxt[col] += dl * orc_load(wr, c->dtype, (int64_t)e * d + col);
          }
          for (int32_t e = 0; e < E; ++e) p[t * E + e] = dp[e]; /* keep dlogit for the router weights */
        }
      }
      free(xr);
      free(av);
      free(bv);
      free(dh);
      free(o);
      free(dp);
    }
    if (failed) rc = ORC_NO_MEM;
  }
  if (!rc) {
    /* weight gradients (p now holds dlogit [T,E]); every element sums over the tokens of
       its expert in token order, whichever row of the output a thread takes.
       Router rows and bias: one expert each. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t e = 0; e < E; ++e) {
      double* gr = dwr + (int64_t)e * d;
      memset(gr, 0, sizeof(double) * (size_t)d);
      dbias[e] = 0.0;
      for (int64_t t = 0; t < T; ++t) {
        const double dl = p[t * E + e];
        for (int32_t col = 0; col < d; ++col) gr[col] += dl * orc_load(x, c->dtype, t * d + col);
        dbias[e] += dl;
      }
    }
    /* expert weights: dW1 / dW3 row (e, f) and dW2 row (e, r) over the slots routed to e,
       taken from the dispatch order (ascending token, i.e. the same order as a walk over t) */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t q = 0; q < (int64_t)E * F; ++q) {
      const int32_t e = (int32_t)(q / F), f = (int32_t)(q % F);
      double* g1 = dw1 + q * d;
      double* g3 = dw3 + q * d;
      memset(g1, 0, sizeof(double) * (size_t)d);
      memset(g3, 0, sizeof(double) * (size_t)d);
      for (int32_t i = offsets[e]; i < offsets[e + 1]; ++i) {
        const int64_t slot = perm[i], t = slot / k;
        const double da = sa[slot * F + f], db = sb[slot * F + f];
        for (int32_t col = 0; col < d; ++col) {
          const double xv = orc_load(x, c->dtype, t * d + col);
          g1[col] += da * xv;
          g3[col] += db * xv;
        }
      }
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t q = 0; q < (int64_t)E * d; ++q) {
      const int32_t e = (int32_t)(q / d), r = (int32_t)(q % d);
      double* g2 = dw2 + q * F;
      memset(g2, 0, sizeof(double) * (size_t)F);
      for (int32_t i = offsets[e]; i < offsets[e + 1]; ++i) {
        const int64_t slot = perm[i], t = slot / k;
        const double* h = sh + slot * F;
        const double gdy = gate[slot] * dy[t * d + r];
        for (int32_t f = 0; f < F; ++f) g2[f] += gdy * h[f];
      }
    }
  }
  free(p);
  free(idx);
  free(gate);
  free(counts);
  free(offsets);
  free(sa);
  free(sb);
  free(sh);
  free(dg);
  free(perm);
  return rc;
}
