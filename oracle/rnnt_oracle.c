/*
 * rnnt_oracle.c -- plain fp64 CPU oracle for the RNN-T joint network, output
 * layer and transducer loss, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only at the seeded synthetic inputs.
 *
 * What it computes is the plain definition of the method, in fp64, cell by
 * cell, in the order the sample-wise transducer paper states the five
 * components ("Neural transducer training: reduced memory consumption with
 * sample-wise computation", arXiv 2211.16270):
 *
 *   joint network   (§2, Eq. 3-4):  a = W^A hA[b,t] + W^L hL[b,u] + b^Z,
 *                                   z = tanh(a)       (tanh: the method's name)
 *   output layer    (§2, Eq. 5-6):  h = W^O z + b^O
 *   f^W_1           (§2, Eq. 7):    ln P_D = ln sum_v exp(h_v)   (denominator only)
 *   f^W_2           (§2, Eq. 8):    forward/backward variables alpha, beta
 *   f^W_3           (§2, Eq. 9):    L = -sum_b ln P(y_b | x_b)
 *   f^W_4           (§2, Eq. 10):   dh = dL/dh
 *   backward through the output layer and joint network (§4, Algorithm 1:
 *   gradients dtheta^J, dtheta^O and the encodings' gradients, accumulated
 *   over samples, "identical to batched computation").
 *
 * The extraction of the paper lost the bodies of Eq. 3-10; where it is silent
 * this file takes the standard transducer lattice (the paper defers to
 * Graves' transducer and to warp-transducer for the formal definition, §2):
 *   - labels[b,0] is the prepended blank and is never read; the transition
 *     from label position u to u+1 emits labels[b,u+1]; hL row u is the label
 *     context after u labels (§2: "prepended with the blank token").
 *   - lattice of sample b: t in [0,T_b), u in [0,U_b]; start (0,0); the path
 *     ends with a blank emitted at (T_b-1, U_b).
 *   - lpb(t,u) = h_blank - ln P_D, lpl(t,u) = h_{labels[b,u+1]} - ln P_D for
 *     u < U_b, and -inf on row u = U_b.
 *   - alpha(0,0) = 0; alpha(t,u) = logaddexp(alpha(t-1,u) + lpb(t-1,u),
 *                                            alpha(t,u-1) + lpl(t,u-1)).
 *   - beta(T_b-1,U_b) = lpb(T_b-1,U_b); beta(t,u) = logaddexp(
 *         beta(t+1,u) + lpb(t,u), beta(t,u+1) + lpl(t,u)).
 *   - ln P = alpha(T_b-1,U_b) + lpb(T_b-1,U_b); loss_b = -ln P; the batch
 *     loss is the sum over b (Eq. 9), each term weighted by grad_loss[b].
 *   - posteriors: pb = exp(alpha + lpb + beta(t+1,u) - ln P) with
 *     beta(T_b,U_b) := 0 and beta(T_b,u<U_b) := -inf; pl = exp(alpha + lpl +
 *     beta(t,u+1) - ln P) for u < U_b, else 0.
 *   - dh_v = g_b * ((pb + pl) softmax_v - pb [v = blank] - pl [v = label]).
 *   - cells outside the valid region: saved values -inf, gradients exactly 0.
 *
 * Parallelism: OpenMP over cells in the forward, over (b,t) rows in the
 * backward with per-thread gradient buffers summed in thread order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "rnnt_oracle.h"

static double logaddexp(double a, double b) {
  if (a == -INFINITY && b == -INFINITY) return -INFINITY;
  double m = a > b ? a : b;
  double d = a > b ? b - a : a - b; /* -|a-b| */
  return m + log1p(exp(d));
}

static int max_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* One cell's joint network and output layer (Eq. 3-6), computed directly from
 * the encodings: a = W^A hA + W^L hL + b^Z, z = tanh(a), h = W^O z + b^O. */
static void cell_forward(const oracle_dims* d, const double* hA_bt, const double* hL_bu,
                         const double* WA, const double* WL, const double* bZ,
                         const double* WO, const double* bO, double* z, double* h) {
  const int H = d->H, HA = d->HA, HL = d->HL, V = d->V;
  for (int k = 0; k < H; ++k) {
    double a = bZ ? bZ[k] : 0.0;
    const double* wa = WA + (size_t)k * HA;
    const double* wl = WL + (size_t)k * HL;
    for (int j = 0; j < HA; ++j) a += wa[j] * hA_bt[j];
    for (int j = 0; j < HL; ++j) a += wl[j] * hL_bu[j];
    z[k] = tanh(a);
  }
  for (int v = 0; v < V; ++v) {
    double s = bO ? bO[v] : 0.0;
    const double* wo = WO + (size_t)v * H;
    for (int k = 0; k < H; ++k) s += wo[k] * z[k];
    h[v] = s;
  }
}

/* ln sum_v exp(h_v) with the maximum taken out (Eq. 7, the denominator). */
static double log_denominator(const double* h, int V) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) m = h[v] > m ? h[v] : m;
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp(h[v] - m);
  return m + log(s);
}

int oracle_check_inputs(const oracle_dims* d, const int32_t* labels, const int32_t* T_len,
                        const int32_t* U_len) {
  if (d->B < 0 || d->T < 1 || d->U1 < 1 || d->H < 1 || d->V < 1 || d->HA < 1 || d->HL < 1)
    return ORACLE_ERR_DIMS;
  if (d->blank < 0 || d->blank >= d->V) return ORACLE_ERR_DIMS;
  for (int b = 0; b < d->B; ++b) {
    if (T_len[b] < 1 || T_len[b] > d->T) return ORACLE_ERR_LENGTH;
    if (U_len[b] < 0 || U_len[b] > d->U1 - 1) return ORACLE_ERR_LENGTH;
    for (int u = 0; u < U_len[b]; ++u) {
      int y = labels[(size_t)b * d->U1 + u + 1];
      if (y < 0 || y >= d->V) return ORACLE_ERR_LABEL;
    }
  }
  return ORACLE_OK;
}

int oracle_rnnt(const oracle_dims* d, const double* hA, const double* hL, const double* WA,
                const double* WL, const double* bZ, const double* WO, const double* bO,
                const int32_t* labels, const int32_t* T_len, const int32_t* U_len,
                const double* grad_loss, double* loss, double* lpb_out, double* lpl_out,
                double* lnPD_out, double* alpha_out, double* beta_out, double* lnP_beta,
                double* dh_out, double* dhA, double* dhL, double* dWA, double* dWL, double* dbZ,
                double* dWO, double* dbO, int nthreads) {
  int st = oracle_check_inputs(d, labels, T_len, U_len);
  if (st != ORACLE_OK) return st;
  const int B = d->B, T = d->T, U1 = d->U1, HA = d->HA, HL = d->HL, H = d->H, V = d->V;
  const int blank = d->blank;
  const size_t ncell = (size_t)B * T * U1;
  const int nth = max_threads(nthreads);

  /* Saved per-cell state: the loss needs only these (Eq. 7-9). */
  double* lpb = (double*)malloc(sizeof(double) * ncell);
  double* lpl = (double*)malloc(sizeof(double) * ncell);
  double* lnPD = (double*)malloc(sizeof(double) * ncell);
  double* alpha = (double*)malloc(sizeof(double) * ncell);
  double* beta = (double*)malloc(sizeof(double) * ncell);
  double* lnP = (double*)malloc(sizeof(double) * (B > 0 ? B : 1));
  if (!lpb || !lpl || !lnPD || !alpha || !beta || !lnP) {
    free(lpb); free(lpl); free(lnPD); free(alpha); free(beta); free(lnP);
    return ORACLE_ERR_ALLOC;
  }
  for (size_t i = 0; i < ncell; ++i) {
    lpb[i] = lpl[i] = lnPD[i] = alpha[i] = beta[i] = -INFINITY;
  }

  /* f^J, f^O, f^W_1 per valid cell: ln P_D and the two log-probabilities. */
  const long long nrow = (long long)B * T;
#pragma omp parallel num_threads(nth)
  {
    double* z = (double*)malloc(sizeof(double) * H);
    double* h = (double*)malloc(sizeof(double) * V);
#pragma omp for schedule(dynamic, 1)
    for (long long r = 0; r < nrow; ++r) {
      const int b = (int)(r / T), t = (int)(r % T);
      if (t >= T_len[b]) continue;
      for (int u = 0; u <= U_len[b]; ++u) {
        cell_forward(d, hA + ((size_t)b * T + t) * HA, hL + ((size_t)b * U1 + u) * HL, WA, WL,
                     bZ, WO, bO, z, h);
        const size_t c = ((size_t)b * T + t) * U1 + u;
        const double ld = log_denominator(h, V);
        lnPD[c] = ld;
        lpb[c] = h[blank] - ld;
        lpl[c] = (u < U_len[b]) ? h[labels[(size_t)b * U1 + u + 1]] - ld : -INFINITY;
      }
    }
    free(z);
    free(h);
  }

  /* f^W_2, f^W_3: alpha and beta over each sample's lattice, and the loss. */
#pragma omp parallel for num_threads(nth) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    const int Tb = T_len[b], Ub = U_len[b];
    double* al = alpha + (size_t)b * T * U1;
    double* be = beta + (size_t)b * T * U1;
    const double* pb = lpb + (size_t)b * T * U1;
    const double* pl = lpl + (size_t)b * T * U1;
    for (int t = 0; t < Tb; ++t)
      for (int u = 0; u <= Ub; ++u) {
        if (t == 0 && u == 0) { al[0] = 0.0; continue; }
        double from_t = t > 0 ? al[(t - 1) * U1 + u] + pb[(t - 1) * U1 + u] : -INFINITY;
        double from_u = u > 0 ? al[t * U1 + u - 1] + pl[t * U1 + u - 1] : -INFINITY;
        al[t * U1 + u] = logaddexp(from_t, from_u);
      }
    for (int t = Tb - 1; t >= 0; --t)
      for (int u = Ub; u >= 0; --u) {
        if (t == Tb - 1 && u == Ub) { be[t * U1 + u] = pb[t * U1 + u]; continue; }
        double via_blank = t + 1 < Tb ? be[(t + 1) * U1 + u] + pb[t * U1 + u] : -INFINITY;
        double via_label = u < Ub ? be[t * U1 + u + 1] + pl[t * U1 + u] : -INFINITY;
        be[t * U1 + u] = logaddexp(via_blank, via_label);
      }
    lnP[b] = al[(Tb - 1) * U1 + Ub] + pb[(Tb - 1) * U1 + Ub];
    if (loss) loss[b] = -lnP[b];
    if (lnP_beta) lnP_beta[b] = be[0];
  }

  if (lpb_out) memcpy(lpb_out, lpb, sizeof(double) * ncell);
  if (lpl_out) memcpy(lpl_out, lpl, sizeof(double) * ncell);
  if (lnPD_out) memcpy(lnPD_out, lnPD, sizeof(double) * ncell);
  if (alpha_out) memcpy(alpha_out, alpha, sizeof(double) * ncell);
  if (beta_out) memcpy(beta_out, beta, sizeof(double) * ncell);

  const int want_grad = dhA || dhL || dWA || dWL || dbZ || dWO || dbO || dh_out;
  if (want_grad) {
    if (dh_out) memset(dh_out, 0, sizeof(double) * ncell * V);
    /* Per-thread accumulators for everything that several rows touch. */
    const size_t nWA = (size_t)H * HA, nWL = (size_t)H * HL, nWO = (size_t)V * H;
    const size_t nhL = (size_t)B * U1 * HL;
    const size_t per = nWA + nWL + H + nWO + V + nhL;
    double* acc = (double*)calloc((size_t)nth * per, sizeof(double));
    if (!acc) {
      free(lpb); free(lpl); free(lnPD); free(alpha); free(beta); free(lnP);
      return ORACLE_ERR_ALLOC;
    }
    if (dhA) memset(dhA, 0, sizeof(double) * (size_t)B * T * HA);
#pragma omp parallel num_threads(nth)
    {
#ifdef _OPENMP
      const int me = omp_get_thread_num();
#else
      const int me = 0;
#endif
      double* aWA = acc + (size_t)me * per;
      double* aWL = aWA + nWA;
      double* abZ = aWL + nWL;
      double* aWO = abZ + H;
      double* abO = aWO + nWO;
      double* ahL = abO + V;
      double* z = (double*)malloc(sizeof(double) * H);
      double* h = (double*)malloc(sizeof(double) * V);
      double* dh = (double*)malloc(sizeof(double) * V);
      double* da = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
      for (long long r = 0; r < nrow; ++r) {
        const int b = (int)(r / T), t = (int)(r % T);
        const int Tb = T_len[b], Ub = U_len[b];
        if (t >= Tb) continue;
        const double g = grad_loss ? grad_loss[b] : 1.0;
        const double* hA_bt = hA + ((size_t)b * T + t) * HA;
        for (int u = 0; u <= Ub; ++u) {
          const size_t c = ((size_t)b * T + t) * U1 + u;
          const double* hL_bu = hL + ((size_t)b * U1 + u) * HL;
          /* Recompute the cell (activation checkpointing). */
          cell_forward(d, hA_bt, hL_bu, WA, WL, bZ, WO, bO, z, h);
          /* Posteriors of the blank and label transitions out of (t,u). */
          double beta_next_t;
          if (t + 1 < Tb) beta_next_t = beta[c + U1];
          else beta_next_t = (u == Ub) ? 0.0 : -INFINITY;
          const double pb = exp(alpha[c] + lpb[c] + beta_next_t - lnP[b]);
          const double pl = (u < Ub) ? exp(alpha[c] + lpl[c] + beta[c + 1] - lnP[b]) : 0.0;
          const int y = (u < Ub) ? labels[(size_t)b * U1 + u + 1] : -1;
          /* f^W_4: dh = d(-ln P)/dh, scaled by the incoming gradient. */
          for (int v = 0; v < V; ++v) {
            double sm = exp(h[v] - lnPD[c]);
            double gv = (pb + pl) * sm;
            if (v == blank) gv -= pb;
            if (v == y) gv -= pl;
            dh[v] = g * gv;
          }
          if (dh_out) memcpy(dh_out + c * V, dh, sizeof(double) * V);
          /* Output layer backward: dz = W^O^T dh, dW^O += dh z^T, db^O += dh. */
          for (int k = 0; k < H; ++k) da[k] = 0.0;
          for (int v = 0; v < V; ++v) {
            const double* wo = WO + (size_t)v * H;
            double* awo = aWO + (size_t)v * H;
            const double dv = dh[v];
            abO[v] += dv;
            for (int k = 0; k < H; ++k) {
              da[k] += wo[k] * dv;
              awo[k] += dv * z[k];
            }
          }
          /* tanh backward: da = dz * (1 - z^2). */
          for (int k = 0; k < H; ++k) da[k] *= (1.0 - z[k] * z[k]);
          /* Joint network backward. */
          double* dhA_bt = dhA ? dhA + ((size_t)b * T + t) * HA : NULL;
          double* ahL_bu = ahL + ((size_t)b * U1 + u) * HL;
          for (int k = 0; k < H; ++k) {
            const double dk = da[k];
            abZ[k] += dk;
            const double* wa = WA + (size_t)k * HA;
            const double* wl = WL + (size_t)k * HL;
            double* awa = aWA + (size_t)k * HA;
            double* awl = aWL + (size_t)k * HL;
            for (int j = 0; j < HA; ++j) {
              awa[j] += dk * hA_bt[j];
              if (dhA_bt) dhA_bt[j] += wa[j] * dk;
            }
            for (int j = 0; j < HL; ++j) {
              awl[j] += dk * hL_bu[j];
              ahL_bu[j] += wl[j] * dk;
            }
          }
        }
      }
      free(z); free(h); free(dh); free(da);
    }
    /* Sum the per-thread buffers in thread order (deterministic for a fixed
     * thread count). */
    double* outs[6] = {dWA, dWL, dbZ, dWO, dbO, dhL};
    size_t offs[6] = {0, nWA, nWA + nWL, nWA + nWL + H, nWA + nWL + H + nWO,
                      nWA + nWL + H + nWO + V};
    size_t lens[6] = {nWA, nWL, (size_t)H, nWO, (size_t)V, nhL};
    for (int o = 0; o < 6; ++o) {
      if (!outs[o]) continue;
      memset(outs[o], 0, sizeof(double) * lens[o]);
      for (int th = 0; th < nth; ++th) {
        const double* src = acc + (size_t)th * per + offs[o];
        for (size_t i = 0; i < lens[o]; ++i) outs[o][i] += src[i];
      }
    }
    free(acc);
  }
  free(lpb); free(lpl); free(lnPD); free(alpha); free(beta); free(lnP);
  return ORACLE_OK;
}

int oracle_num_threads(int nthreads) { return max_threads(nthreads); }
