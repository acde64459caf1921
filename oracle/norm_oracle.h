/*
 * norm_oracle.h -- declarations of the double-precision CPU oracle.
 * TEST INFRASTRUCTURE ONLY; see norm_oracle.c.  Shares nothing with the CUDA
 * library's headers.
 */
#ifndef NORM_ORACLE_H
#define NORM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_GELU = 2, ORACLE_ACT_SILU = 3, ORACLE_ACT_MISH = 4,
       ORACLE_ACT_LEAKY_RELU = 5, ORACLE_ACT_ELU = 6, ORACLE_ACT_SIGMOID = 7, ORACLE_ACT_CELU = 8,
       ORACLE_ACT_SELU = 9, ORACLE_ACT_RELU6 = 10, ORACLE_ACT_HARDTANH = 11 };

void oracle_layernorm_fwd(int64_t rows, int64_t cols, const double *x,
                          const double *w, const double *b, double eps,
                          double *y, double *mean, double *rstd);
void oracle_layernorm_bwd(int64_t rows, int64_t cols, const double *dy,
                          const double *x, const double *w, double eps,
                          double *dx, double *dw, double *db);
void oracle_layernorm_cf_fwd(int64_t n, int64_t c, int64_t l, const double *x,
                             const double *w, const double *b, double eps,
                             double *y, double *mean, double *rstd);
void oracle_layernorm_cf_bwd(int64_t n, int64_t c, int64_t l, const double *dy,
                             const double *x, const double *w, double eps,
                             double *dx, double *dw, double *db);
void oracle_rmsnorm_fwd(int64_t rows, int64_t cols, const double *x,
                        const double *w, const double *b, double eps, double *y,
                        double *rstd);
void oracle_rmsnorm_bwd(int64_t rows, int64_t cols, const double *dy,
                        const double *x, const double *w, double eps,
                        double *dx, double *dw, double *db);
void oracle_batchnorm_fwd(int64_t n, int64_t c, int64_t l, const double *x,
                          const double *res, const double *w, const double *b,
                          double eps, double momentum, int training, int act,
                          double act_param, double *running_mean, double *running_var,
                          double *y, double *save_mean, double *save_rstd,
                          uint32_t *act_mask, double *z_out);
void oracle_batchnorm_bwd(int64_t n, int64_t c, int64_t l, const double *dy,
                          const double *x, const double *res, const double *w,
                          const double *b, const double *running_mean,
                          const double *running_var, double eps, int training,
                          int act, double act_param, const uint32_t *act_mask, double *dx,
                          double *dres, double *dw, double *db);

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void oracle_dropout_mask(int64_t count, int64_t first, double drop_p, uint32_t seed,
                         uint8_t *keep);
void oracle_act_dropout_fwd(int64_t count, int64_t first, const double *x, int act,
                            double act_param, double drop_p, uint32_t seed, double *y);
void oracle_act_dropout_bwd(int64_t count, int64_t first, const double *dy, const double *x,
                            int act, double act_param, double drop_p, uint32_t seed,
                            double *dx);

#ifdef __cplusplus
}
#endif

#endif /* NORM_ORACLE_H */
