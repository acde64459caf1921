/*
 * c_caller.c -- libnorm called from a plain C program: device memory from the
 * CUDA runtime, the public header include/libnorm.h and nothing else of the
 * library, no Python and no PyTorch.
 *
 * On seeded inputs it runs
 *   - a LayerNorm forward and backward, fp32 [37, 1000] (16-byte vectors, a
 *     ragged last group per row), with weight, bias and both gradients;
 *   - a BatchNorm training forward and backward, fp32 [4, 3, 50], with a
 *     residual and GELU, updating the running statistics;
 * and compares every output element by element with the double-precision CPU
 * oracle (test infrastructure, oracle/norm_oracle.h) within the fp32 parity
 * bound |gpu - oracle| <= 1e-5 + 1e-5*|oracle|.  BatchNorm dw may also differ
 * by 4 ulps of the saved fp32 mean times rstd*|db|: the backward reads the
 * mean the forward saved in fp32, and a mean off by d moves dw by d*rstd*db.
 * Then a call with a bad argument must return NRM_ERR_INVALID_ARG with a
 * message, and nrm_sync_status must report NRM_OK.
 *
 * Prints "ok" and exits 0; names the first mismatch and exits 1; exits 2 when
 * no CUDA device is usable.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "libnorm.h"
#include "norm_oracle.h"

#define FP32_ATOL 1e-5
#define FP32_RTOL 1e-5

static uint64_t g_state = 2024;

/* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the seeded test inputs, nothing else */
static uint64_t next_u64(void)
{
    uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* n values uniform in [lo, hi), stored as float: both sides read these */
static float *fill(size_t n, double lo, double hi)
{
    float *a = (float *)malloc(n * sizeof(float));
    if (!a) exit(3);
    for (size_t i = 0; i < n; ++i)
        a[i] = (float)(lo + (hi - lo) * ((double)(next_u64() >> 11) * 0x1.0p-53));
    return a;
}

static double *widen(const float *a, size_t n)
{
    double *d = (double *)malloc(n * sizeof(double));
    if (!d) exit(3);
    for (size_t i = 0; i < n; ++i) d[i] = a[i];
    return d;
}

static double *zeros(size_t n)
{
    double *d = (double *)calloc(n, sizeof(double));
    if (!d) exit(3);
    return d;
}

static void cuda_ok(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        printf("CUDA error in %s: %s\n", what, cudaGetErrorString(e));
        exit(1);
    }
}

/* a device copy of n floats from host (or uninitialised when h is NULL) */
static float *dev(const float *h, size_t n)
{
    void *d = NULL;
    cuda_ok(cudaMalloc(&d, n * sizeof(float) + 16), "cudaMalloc");
    if (h) cuda_ok(cudaMemcpy(d, h, n * sizeof(float), cudaMemcpyHostToDevice), "upload");
    return (float *)d;
}

static float *back(const float *d, size_t n)
{
    float *h = (float *)malloc(n * sizeof(float));
    if (!h) exit(3);
    cuda_ok(cudaMemcpy(h, d, n * sizeof(float), cudaMemcpyDeviceToHost), "download");
    return h;
}

static int g_failures = 0;

/* element by element: |got - want| <= atol + rtol*|want| (+ slack[i]) */
static void check(const char *what, const float *got, const double *want, size_t n,
                  const double *slack)
{
    for (size_t i = 0; i < n; ++i) {
        double err = fabs((double)got[i] - want[i]);
        double lim = FP32_ATOL + FP32_RTOL * fabs(want[i]) + (slack ? slack[i] : 0.0);
        if (!(err <= lim)) {
            printf("%s: element %zu of %zu: got %.9g, want %.9g (err %.3g > %.3g)\n", what, i, n,
                   (double)got[i], want[i], err, lim);
            ++g_failures;
            return;
        }
    }
}

static void status_ok(nrm_status s, const char *what)
{
    if (s != NRM_OK) {
        printf("%s returned %s: %s\n", what, nrm_status_str(s), nrm_last_error_message());
        exit(1);
    }
}

static void *workspace(size_t bytes)
{
    void *d = NULL;
    if (bytes) cuda_ok(cudaMalloc(&d, bytes), "workspace");
    return d;
}

static void layernorm_case(void)
{
    const int64_t rows = 37, cols = 1000;
    const size_t e = (size_t)(rows * cols);
    const float eps = 1e-5f;
    float *x = fill(e, -1.2, 1.8), *w = fill((size_t)cols, 0.8, 1.2), *b = fill((size_t)cols, -0.2, 0.2);
    float *dy = fill(e, -1.0, 1.0);
    float *d_x = dev(x, e), *d_w = dev(w, (size_t)cols), *d_b = dev(b, (size_t)cols), *d_dy = dev(dy, e);
    float *d_y = dev(NULL, e), *d_mean = dev(NULL, (size_t)rows), *d_rstd = dev(NULL, (size_t)rows);
    float *d_dx = dev(NULL, e), *d_dw = dev(NULL, (size_t)cols), *d_db = dev(NULL, (size_t)cols);

    status_ok(nrm_layernorm_fwd(d_x, d_w, d_b, d_y, d_mean, d_rstd, rows, cols, eps, NRM_F32, NULL),
              "nrm_layernorm_fwd");
    size_t ws_bytes = nrm_workspace_bytes(NRM_OP_LAYERNORM_BWD, rows, cols, NRM_F32);
    if (ws_bytes == 0) {
        printf("nrm_workspace_bytes returned 0\n");
        exit(1);
    }
    void *ws = workspace(ws_bytes);
    status_ok(nrm_layernorm_bwd(d_dy, d_x, d_w, d_mean, d_rstd, d_dx, d_dw, d_db, rows, cols, NRM_F32, ws,
                                ws_bytes, NULL),
              "nrm_layernorm_bwd");
    status_ok(nrm_sync_status(NULL), "nrm_sync_status after LayerNorm");

    double *xd = widen(x, e), *wd = widen(w, (size_t)cols), *bd = widen(b, (size_t)cols), *dyd = widen(dy, e);
    double *y = zeros(e), *mean = zeros((size_t)rows), *rstd = zeros((size_t)rows);
    double *dx = zeros(e), *dw = zeros((size_t)cols), *db = zeros((size_t)cols);
    oracle_layernorm_fwd(rows, cols, xd, wd, bd, (double)eps, y, mean, rstd);
    oracle_layernorm_bwd(rows, cols, dyd, xd, wd, (double)eps, dx, dw, db);

    float *g;
    check("LayerNorm y", g = back(d_y, e), y, e, NULL); free(g);
    check("LayerNorm mean", g = back(d_mean, (size_t)rows), mean, (size_t)rows, NULL); free(g);
    check("LayerNorm rstd", g = back(d_rstd, (size_t)rows), rstd, (size_t)rows, NULL); free(g);
    check("LayerNorm dx", g = back(d_dx, e), dx, e, NULL); free(g);
    check("LayerNorm dw", g = back(d_dw, (size_t)cols), dw, (size_t)cols, NULL); free(g);
    check("LayerNorm db", g = back(d_db, (size_t)cols), db, (size_t)cols, NULL); free(g);

    cudaFree(d_x); cudaFree(d_w); cudaFree(d_b); cudaFree(d_dy); cudaFree(d_y); cudaFree(d_mean);
    cudaFree(d_rstd); cudaFree(d_dx); cudaFree(d_dw); cudaFree(d_db); cudaFree(ws);
    free(x); free(w); free(b); free(dy); free(xd); free(wd); free(bd); free(dyd);
    free(y); free(mean); free(rstd); free(dx); free(dw); free(db);
}

static void batchnorm_case(void)
{
    const int64_t n = 4, c = 3, l = 50;
    const size_t e = (size_t)(n * c * l), cc = (size_t)c;
    const float eps = 1e-5f, momentum = 0.1f;
    float *x = fill(e, -2.0, 3.0), *res = fill(e, -1.0, 1.0), *dy = fill(e, -1.0, 1.0);
    float *w = fill(cc, 0.8, 1.2), *b = fill(cc, -0.2, 0.2);
    float rm0[3] = {0.f, 0.f, 0.f}, rv0[3] = {1.f, 1.f, 1.f};
    float *d_x = dev(x, e), *d_res = dev(res, e), *d_dy = dev(dy, e), *d_w = dev(w, cc), *d_b = dev(b, cc);
    float *d_rm = dev(rm0, cc), *d_rv = dev(rv0, cc);
    float *d_y = dev(NULL, e), *d_sm = dev(NULL, cc), *d_sr = dev(NULL, cc);
    float *d_dx = dev(NULL, e), *d_dres = dev(NULL, e), *d_dw = dev(NULL, cc), *d_db = dev(NULL, cc);
    size_t ws_bytes = nrm_batchnorm_workspace_bytes(n, c, l, NRM_F32);
    void *ws = workspace(ws_bytes);

    status_ok(nrm_batchnorm_fwd(d_x, d_res, d_w, d_b, d_y, d_rm, d_rv, d_sm, d_sr, NULL, n, c, l, eps, momentum,
                                1, NRM_ACT_GELU, 0.f, NRM_F32, ws, ws_bytes, NULL),
              "nrm_batchnorm_fwd");
    status_ok(nrm_batchnorm_bwd(d_dy, d_x, d_res, d_w, d_b, d_sm, d_sr, NULL, d_dx, d_dres, d_dw, d_db, n, c, l,
                                1, NRM_ACT_GELU, 0.f, NRM_F32, ws, ws_bytes, NULL),
              "nrm_batchnorm_bwd");
    status_ok(nrm_sync_status(NULL), "nrm_sync_status after BatchNorm");

    double *xd = widen(x, e), *resd = widen(res, e), *dyd = widen(dy, e), *wd = widen(w, cc), *bd = widen(b, cc);
    double *rm = widen(rm0, cc), *rv = widen(rv0, cc);
    double *y = zeros(e), *sm = zeros(cc), *sr = zeros(cc);
    double *dx = zeros(e), *dres = zeros(e), *dw = zeros(cc), *db = zeros(cc);
    oracle_batchnorm_fwd(n, c, l, xd, resd, wd, bd, (double)eps, (double)momentum, 1, ORACLE_ACT_GELU, 0.0, rm,
                         rv, y, sm, sr, NULL, NULL);
    oracle_batchnorm_bwd(n, c, l, dyd, xd, resd, wd, bd, NULL, NULL, (double)eps, 1, ORACLE_ACT_GELU, 0.0, NULL,
                         dx, dres, dw, db);

    /* 4 ulps of the fp32 mean, times rstd*|db| (see the file comment) */
    double slack[3];
    for (size_t ch = 0; ch < cc; ++ch) {
        float m = fabsf((float)sm[ch]);
        double ulp = (double)nextafterf(m, INFINITY) - (double)m;
        slack[ch] = 4.0 * ulp * sr[ch] * fabs(db[ch]);
    }

    float *g;
    check("BatchNorm y", g = back(d_y, e), y, e, NULL); free(g);
    check("BatchNorm save_mean", g = back(d_sm, cc), sm, cc, NULL); free(g);
    check("BatchNorm save_rstd", g = back(d_sr, cc), sr, cc, NULL); free(g);
    check("BatchNorm running_mean", g = back(d_rm, cc), rm, cc, NULL); free(g);
    check("BatchNorm running_var", g = back(d_rv, cc), rv, cc, NULL); free(g);
    check("BatchNorm dx", g = back(d_dx, e), dx, e, NULL); free(g);
    check("BatchNorm dres", g = back(d_dres, e), dres, e, NULL); free(g);
    check("BatchNorm db", g = back(d_db, cc), db, cc, NULL); free(g);
    check("BatchNorm dw", g = back(d_dw, cc), dw, cc, slack); free(g);

    cudaFree(d_x); cudaFree(d_res); cudaFree(d_dy); cudaFree(d_w); cudaFree(d_b); cudaFree(d_rm);
    cudaFree(d_rv); cudaFree(d_y); cudaFree(d_sm); cudaFree(d_sr); cudaFree(d_dx); cudaFree(d_dres);
    cudaFree(d_dw); cudaFree(d_db); cudaFree(ws);
    free(x); free(res); free(dy); free(w); free(b); free(xd); free(resd); free(dyd); free(wd); free(bd);
    free(rm); free(rv); free(y); free(sm); free(sr); free(dx); free(dres); free(dw); free(db);
}

static void error_case(void)
{
    /* cols = 0 is rejected on the host, before anything is enqueued */
    nrm_status s = nrm_layernorm_fwd(NULL, NULL, NULL, NULL, NULL, NULL, 4, 0, 1e-5f, NRM_F32, NULL);
    if (s != NRM_ERR_INVALID_ARG) {
        printf("a LayerNorm call with cols = 0 returned %s, not NRM_ERR_INVALID_ARG\n", nrm_status_str(s));
        ++g_failures;
    } else if (strlen(nrm_last_error_message()) == 0) {
        printf("no message after NRM_ERR_INVALID_ARG\n");
        ++g_failures;
    }
    status_ok(nrm_sync_status(NULL), "nrm_sync_status after a rejected call");
}

int main(void)
{
    int devices = 0;
    if (cudaGetDeviceCount(&devices) != cudaSuccess || devices == 0) {
        printf("no CUDA device\n");
        return 2;
    }
    layernorm_case();
    batchnorm_case();
    error_case();
    if (g_failures) return 1;
    printf("ok (libnorm %d)\n", nrm_version());
    return 0;
}
