/*
 * kda_oracle.h -- declarations of the CPU oracle (test infrastructure only).
 * See kda_oracle.c for what each function computes and the passages it follows.
 * Nothing in the CUDA library includes this header.
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stddef.h>

#define KDAO_D 128                   /* d_k = d_v = head_dim 128                 */
#define KDAO_TMAX 15                 /* rows per verify round, K <= 14           */
#define KDAO_GATE_LOWER_BOUND (-5.0) /* g = -5 * sigmoid(raw)                    */
#define KDAO_L2_EPS 1e-6             /* inside the sqrt of the L2 normalisation  */
#define KDAO_SENTINEL (-1)           /* argmax of a row holding a NaN            */

#define KDAO_TAG_ACCEPT 0xFFFFFFFEu /* counter word 3 of the accept-test uniforms */
#define KDAO_TAG_DRAW 0xFFFFFFFFu   /* counter word 3 of the residual / bonus draw  */

#define KDAO_F32 0
#define KDAO_BF16 1

#define KDAO_OK 0
#define KDAO_EINVAL 1
#define KDAO_ENAN 2
#define KDAO_ENOMEM 5

#ifdef __cplusplus
extern "C" {
#endif

int kdao_prepare(int H, int T, int dtype, const void *xq, const void *xk, const void *xv,
                 const void *xg, const void *xb, const float *conv_w, const float *ring_in,
                 double *q_hat, double *k_hat, double *v_out, double *g_out,
                 double *beta_out, float *ring_out);

int kdao_core(int H, int T, const double *q_hat, const double *k_hat, const double *v,
              const double *g, const double *beta, double *S, double *out);

int kdao_verify(int H, int T, int dtype, const void *xq, const void *xk, const void *xv,
                const void *xg, const void *xb, const float *conv_w, const float *ring_in,
                const float *state_in, float *ring_out, float *state_out, float *out);

int kdao_rollback(int H, int T, int keep, int dtype, const void *xq, const void *xk,
                  const void *xv, const void *xg, const void *xb, const float *conv_w,
                  const float *ring_snap, const float *state_snap, const float *ring_cur,
                  const float *state_cur, float *ring_out, float *state_out);

int kdao_accept(int T, int V, int dtype, const void *logits, const int *drafts, int *vam,
                int *j_out, int *bonus_out);

int kdao_conf_keep(int n, const float *q, float p_min, int pmin0);
int kdao_confidence_vt(int n, const float *raws, float tau, int vt_cap);
int kdao_slot_confidence_vt(int n, const float *raws, float tau, int vt_cap);

int kdao_filtered(int V, int dtype, const void *row, double temperature, int top_k, double top_p,
                  double min_p, double *p);
int kdao_sampled_accept(int T, int V, int dtype, const void *logits, const void *draft_logits,
                        const int *drafts, const double *u_accept, double u_sample, double temperature,
                        int top_k, double top_p, double min_p, int *j_out, int *token_out);

void kdao_philox4x32_10(const unsigned int ctr[4], const unsigned int key[2], unsigned int out[4]);
float kdao_u01(unsigned long long seed, unsigned int counter, unsigned int tag);
int kdao_sampled_accept_session(int T, int V, int dtype, const void *logits, const void *draft_logits,
                                const int *drafts, unsigned long long seed, unsigned int *uctr,
                                unsigned int *sctr, double temperature, int top_k, double top_p,
                                double min_p, int *j_out, int *token_out);

#ifdef __cplusplus
}
#endif

#endif
