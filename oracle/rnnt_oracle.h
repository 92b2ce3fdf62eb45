/*
 * rnnt_oracle.h -- C interface of the fp64 CPU oracle (test infrastructure
 * only; see rnnt_oracle.c).  Everything is host memory, row-major, fp64 for
 * values and int32 for labels and lengths:
 *   hA [B,T,HA], hL [B,U1,HL], W^A [H,HA], W^L [H,HL], b^Z [H] (or NULL = 0),
 *   W^O [V,H], b^O [V] (or NULL = 0), labels [B,U1] (index 0 = the prepended
 *   blank, never read), T_len [B], U_len [B].
 * Outputs (each may be NULL to skip it):
 *   loss [B] = -ln P(y_b|x_b); lpb, lpl, lnPD, alpha, beta [B,T,U1] with -inf
 *   outside the valid lattice; lnP_beta [B] = beta(0,0); dh [B,T,U1,V] (small
 *   cases only); gradients dhA [B,T,HA], dhL [B,U1,HL], dWA [H,HA], dWL [H,HL],
 *   dbZ [H], dWO [V,H], dbO [V] of sum_b grad_loss[b] * loss[b]
 *   (grad_loss NULL = all ones).  Gradients are overwritten.
 */
#ifndef RNNT_ORACLE_H
#define RNNT_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int B, T, U1, HA, HL, H, V, blank;
} oracle_dims;

enum { ORACLE_OK = 0, ORACLE_ERR_DIMS = 1, ORACLE_ERR_LENGTH = 2, ORACLE_ERR_LABEL = 3,
       ORACLE_ERR_ALLOC = 4 };

int oracle_check_inputs(const oracle_dims* d, const int32_t* labels, const int32_t* T_len,
                        const int32_t* U_len);

int oracle_rnnt(const oracle_dims* d, const double* hA, const double* hL, const double* WA,
                const double* WL, const double* bZ, const double* WO, const double* bO,
                const int32_t* labels, const int32_t* T_len, const int32_t* U_len,
                const double* grad_loss, double* loss, double* lpb, double* lpl, double* lnPD,
                double* alpha, double* beta, double* lnP_beta, double* dh, double* dhA,
                double* dhL, double* dWA, double* dWL, double* dbZ, double* dWO, double* dbO,
                int nthreads);

int oracle_num_threads(int nthreads);

#ifdef __cplusplus
}
#endif
#endif
