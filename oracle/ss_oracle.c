/*
 * Selective-scan oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, sequential f64 CPU evaluation of the Mamba-1 selective scan,
 * forward and backward.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline leg may load this library; the CUDA path never does,
 * and the two share no code.
 *
 * What it computes (baracuda-kernels `selective_scan.rs`, module doc
 * "Algorithm summary" and "Shape contract"), for every row (b, d):
 *
 *   x_t     = delta[b,t,d] + delta_bias[d]        (bias term only if given)
 *   Delta_t = softplus(x_t)  if softplus, else x_t
 *   h_{-1}  = h0[b,d,:]  if an initial state is given, else 0
 *   a_{t,n} = exp(Delta_t * A[d,n])
 *   h_{t,n} = a_{t,n} * h_{t-1,n} + Delta_t * B[b,t,n] * u[b,t,d]
 *   y0_t    = sum_n h_{t,n} * C[b,t,n]  +  D[d] * u[b,t,d]   (D term if given)
 *   y_t     = y0_t * silu(z[b,t,d])                          (if z given)
 *   last_state[b,d,n] = h_{L-1,n}
 *
 * The backward is the chain rule of that definition for the loss
 * sum_t dy_t * y_t + sum_n dlast_n * last_state_n (dlast optional, else 0),
 * with the structure of mamba-rs `gpu/backward.rs`
 * (B2 gating backward, B3 SSM BPTT with per-row local gradients followed by
 * reductions, B4 softplus backward taking the raw pre-softplus input):
 *
 *   g_t        = dy_t * silu(z_t)                      (dy_t if no z)
 *   dz_t       = dy_t * y0_t * sig(z_t) * (1 + z_t * (1 - sig(z_t)))
 *   lam_{t,n}  = g_t * C[b,t,n] + a_{t+1,n} * lam_{t+1,n},   a_{L,n} lam_{L,n} = dlast_n
 *   du_t       = g_t * D[d] + sum_n lam_{t,n} * Delta_t * B[b,t,n]
 *   dDelta_t   = sum_n lam_{t,n} * (A[d,n] * a_{t,n} * h_{t-1,n} + B[b,t,n] * u_t)
 *   ddelta_t   = dDelta_t * sig(x_t)  if softplus, else dDelta_t
 *   dA[d,n]   += lam_{t,n} * Delta_t * a_{t,n} * h_{t-1,n}   (summed over b, t)
 *   dD[d]     += g_t * u_t                                   (summed over b, t)
 *   dbias[d]  += ddelta_t                                    (summed over b, t)
 *   dB[b,t,n] += lam_{t,n} * Delta_t * u_t                   (summed over d)
 *   dC[b,t,n] += g_t * h_{t,n}                               (summed over d)
 *   dh0[b,d,n] = a_{0,n} * lam_{0,n}   (dlast_n when L = 0)
 *
 * Readings where the pages say nothing: softplus(x) = log(1 + e^x) (stable
 * form), silu(z) = z * sig(z), the initial state is zero unless one is
 * given, the bias is added even when softplus is off, D is added before the
 * gate, and last_state receives no incoming gradient unless dlast is given.
 *
 * Inputs are f64 arrays (values of the I/O precision convert exactly);
 * every operation is carried out in f64.  Rows are independent and are
 * spread over threads; per-row outputs do not depend on the thread count.
 * dB and dC are summed per thread over that thread's contiguous block of
 * rows, then the thread partials are added in thread order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *u, *delta, *A, *B, *C, *D, *z, *bias, *dy;
    int softplus;
    int64_t Bsz, L, Dch, N;
    const double *h0, *dlast; /* [Bsz][Dch][N], nullable */
} problem;

static double softplus_f64(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

static double sigmoid_f64(double x)
{
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

static double silu_f64(double z) { return z * sigmoid_f64(z); }

/* index helpers: [Bsz, L, Dch], [Bsz, L, N], [Dch, N] */
static int64_t at_bld(const problem *p, int64_t b, int64_t t, int64_t d) { return (b * p->L + t) * p->Dch + d; }
static int64_t at_bln(const problem *p, int64_t b, int64_t t, int64_t n) { return (b * p->L + t) * p->N + n; }
static int64_t at_dn(const problem *p, int64_t d, int64_t n) { return d * p->N + n; }
static int64_t at_bdn(const problem *p, int64_t b, int64_t d, int64_t n) { return (b * p->Dch + d) * p->N + n; }

/* h_{-1,n} of row (b, d) */
static double h_init(const problem *p, int64_t b, int64_t d, int64_t n) { return p->h0 ? p->h0[at_bdn(p, b, d, n)] : 0.0; }

static double delta_eff(const problem *p, int64_t b, int64_t t, int64_t d, double *x_out)
{
    double x = p->delta[at_bld(p, b, t, d)];
    if (p->bias) x += p->bias[d];
    if (x_out) *x_out = x;
    return p->softplus ? softplus_f64(x) : x;
}

/* Forward over one row.  h: scratch [N].  y, y0: [L] (nullable).  last: [N] (nullable). */
static void fwd_row(const problem *p, int64_t b, int64_t d, double *h, double *y, double *y0, double *last)
{
    for (int64_t n = 0; n < p->N; n++) h[n] = h_init(p, b, d, n);
    for (int64_t t = 0; t < p->L; t++) {
        double dt = delta_eff(p, b, t, d, NULL);
        double ut = p->u[at_bld(p, b, t, d)];
        double acc = 0.0;
        for (int64_t n = 0; n < p->N; n++) {
            double a = exp(dt * p->A[at_dn(p, d, n)]);
            h[n] = a * h[n] + dt * p->B[at_bln(p, b, t, n)] * ut;
            acc += h[n] * p->C[at_bln(p, b, t, n)];
        }
        if (p->D) acc += p->D[d] * ut;
        if (y0) y0[t] = acc;
        double out = acc;
        if (p->z) out *= silu_f64(p->z[at_bld(p, b, t, d)]);
        if (y) y[t] = out;
    }
    if (last)
        for (int64_t n = 0; n < p->N; n++) last[n] = h[n];
}

typedef struct {
    double *a;   /* [L][N]  a_{t,n}              */
    double *h;   /* [L][N]  h_{t,n}              */
    double *lam; /* [N]     running adjoint      */
} row_scratch;

/* Backward over one row.  Per-row outputs are written (dh0: [N], nullable); dB/dC
 * contributions are added into dB_acc/dC_acc ([Bsz][L][N], nullable). */
static void bwd_row(const problem *p, int64_t b, int64_t d, row_scratch *s, double *du, double *ddelta,
                    double *dz, double *dA, double *dD, double *dbias, double *dh0, double *dB_acc, double *dC_acc)
{
    const int64_t L = p->L, N = p->N;
    /* forward sweep, keeping every a_{t,n} and h_{t,n} */
    for (int64_t t = 0; t < L; t++) {
        double dt = delta_eff(p, b, t, d, NULL);
        double ut = p->u[at_bld(p, b, t, d)];
        for (int64_t n = 0; n < N; n++) {
            double hprev = t > 0 ? s->h[(t - 1) * N + n] : h_init(p, b, d, n);
            double a = exp(dt * p->A[at_dn(p, d, n)]);
            s->a[t * N + n] = a;
            s->h[t * N + n] = a * hprev + dt * p->B[at_bln(p, b, t, n)] * ut;
        }
    }
    /* lam holds lam_{t+1}; a_{L} lam_{L} stands for the incoming gradient of h_{L-1} */
    for (int64_t n = 0; n < N; n++) { s->lam[n] = p->dlast ? p->dlast[at_bdn(p, b, d, n)] : 0.0; dA[n] = 0.0; }
    double dD_sum = 0.0, dbias_sum = 0.0;
    /* reverse sweep */
    for (int64_t t = L - 1; t >= 0; t--) {
        double x;
        double dt = delta_eff(p, b, t, d, &x);
        double ut = p->u[at_bld(p, b, t, d)];
        double dyt = p->dy[at_bld(p, b, t, d)];
        double g = dyt;
        if (p->z) {
            double zt = p->z[at_bld(p, b, t, d)];
            double y0 = 0.0;
            for (int64_t n = 0; n < N; n++) y0 += s->h[t * N + n] * p->C[at_bln(p, b, t, n)];
            if (p->D) y0 += p->D[d] * ut;
            double sg = sigmoid_f64(zt);
            g = dyt * silu_f64(zt);
            if (dz) dz[t] = dyt * y0 * sg * (1.0 + zt * (1.0 - sg));
        }
        double du_t = p->D ? g * p->D[d] : 0.0;
        double dDelta = 0.0;
        for (int64_t n = 0; n < N; n++) {
            double Bn = p->B[at_bln(p, b, t, n)];
            double Cn = p->C[at_bln(p, b, t, n)];
            double a_next = t + 1 < L ? s->a[(t + 1) * N + n] : 1.0;
            double lam = g * Cn + a_next * s->lam[n];
            s->lam[n] = lam;
            double hprev = t > 0 ? s->h[(t - 1) * N + n] : h_init(p, b, d, n);
            double a = s->a[t * N + n];
            du_t += lam * dt * Bn;
            dDelta += lam * (p->A[at_dn(p, d, n)] * a * hprev + Bn * ut);
            dA[n] += lam * dt * a * hprev;
            if (dB_acc) dB_acc[at_bln(p, b, t, n)] += lam * dt * ut;
            if (dC_acc) dC_acc[at_bln(p, b, t, n)] += g * s->h[t * N + n];
        }
        double dx = p->softplus ? dDelta * sigmoid_f64(x) : dDelta;
        du[t] = du_t;
        ddelta[t] = dx;
        dD_sum += g * ut;
        dbias_sum += dx;
    }
    *dD = dD_sum;
    *dbias = dbias_sum;
    /* h_0 = a_0 h_{-1} + ..., so the gradient of h_{-1} is a_0 lam_0 (lam_0 is in s->lam) */
    if (dh0)
        for (int64_t n = 0; n < N; n++) dh0[n] = L > 0 ? s->a[n] * s->lam[n] : s->lam[n];
}

/* ---------------------------------------------------------------- threading */

typedef struct {
    const problem *p;
    const int64_t *rows;
    int64_t lo, hi; /* slice of the row list */
    int mode;       /* 0 fwd, 1 bwd */
    /* fwd */
    double *y_rows, *y0_rows, *last_rows;
    /* bwd */
    double *du_rows, *ddelta_rows, *dz_rows, *dA_rows, *dD_rows, *dbias_rows, *dh0_rows;
    double *dB_part, *dC_part; /* private [Bsz][L][N] accumulators, or NULL */
    int failed;
} job;

static int64_t row_id(const job *j, int64_t i) { return j->rows ? j->rows[i] : i; }

static void *run_job(void *arg)
{
    job *j = (job *)arg;
    const problem *p = j->p;
    const int64_t L = p->L, N = p->N;
    if (j->mode == 0) {
        double *h = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        if (!h) { j->failed = 1; return NULL; }
        for (int64_t i = j->lo; i < j->hi; i++) {
            int64_t r = row_id(j, i), b = r / p->Dch, d = r % p->Dch;
            fwd_row(p, b, d, h, j->y_rows ? j->y_rows + i * L : NULL, j->y0_rows ? j->y0_rows + i * L : NULL,
                    j->last_rows ? j->last_rows + i * N : NULL);
        }
        free(h);
    } else {
        row_scratch s;
        size_t ln = (size_t)(L > 0 ? L : 1) * (size_t)(N > 0 ? N : 1);
        s.a = (double *)malloc(ln * sizeof(double));
        s.h = (double *)malloc(ln * sizeof(double));
        s.lam = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        if (!s.a || !s.h || !s.lam) {
            free(s.a); free(s.h); free(s.lam);
            j->failed = 1;
            return NULL;
        }
        for (int64_t i = j->lo; i < j->hi; i++) {
            int64_t r = row_id(j, i), b = r / p->Dch, d = r % p->Dch;
            bwd_row(p, b, d, &s, j->du_rows + i * L, j->ddelta_rows + i * L, j->dz_rows ? j->dz_rows + i * L : NULL,
                    j->dA_rows + i * N, j->dD_rows + i, j->dbias_rows + i, j->dh0_rows ? j->dh0_rows + i * N : NULL,
                    j->dB_part, j->dC_part);
        }
        free(s.a); free(s.h); free(s.lam);
    }
    return NULL;
}

static int run_threads(job *proto, int64_t n_rows, int nthreads, double *dB, double *dC)
{
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > n_rows) nthreads = (int)(n_rows > 0 ? n_rows : 1);
    const problem *p = proto->p;
    size_t bln = (size_t)(p->Bsz * p->L * p->N);
    job *jobs = (job *)calloc((size_t)nthreads, sizeof(job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 2; }
    int rc = 0;
    for (int k = 0; k < nthreads; k++) {
        jobs[k] = *proto;
        jobs[k].lo = n_rows * k / nthreads;
        jobs[k].hi = n_rows * (k + 1) / nthreads;
        jobs[k].dB_part = NULL;
        jobs[k].dC_part = NULL;
        if (proto->mode == 1 && dB) jobs[k].dB_part = (double *)calloc(bln ? bln : 1, sizeof(double));
        if (proto->mode == 1 && dC) jobs[k].dC_part = (double *)calloc(bln ? bln : 1, sizeof(double));
        if ((dB && proto->mode == 1 && !jobs[k].dB_part) || (dC && proto->mode == 1 && !jobs[k].dC_part)) rc = 2;
    }
    int started = 0;
    if (rc == 0) {
        for (int k = 0; k < nthreads; k++) {
            if (pthread_create(&th[k], NULL, run_job, &jobs[k]) != 0) { rc = 3; break; }
            started++;
        }
        for (int k = 0; k < started; k++) pthread_join(th[k], NULL);
        for (int k = 0; k < started; k++) if (jobs[k].failed) rc = 2;
    }
    if (rc == 0 && proto->mode == 1) {
        /* thread partials summed in thread order */
        for (int k = 0; k < nthreads; k++) {
            if (dB) for (size_t i = 0; i < bln; i++) dB[i] += jobs[k].dB_part[i];
            if (dC) for (size_t i = 0; i < bln; i++) dC[i] += jobs[k].dC_part[i];
        }
    }
    for (int k = 0; k < nthreads; k++) { free(jobs[k].dB_part); free(jobs[k].dC_part); }
    free(jobs);
    free(th);
    return rc;
}

/* ---------------------------------------------------------------- C entry points */

/*
 * Forward.  rows: list of row ids r = b*Dch + d (NULL: every row in order).
 * h0 (nullable) [Bsz][Dch][N]: the state before t = 0.
 * y_rows [n_rows][L], y0_rows (pre-gate, nullable) [n_rows][L], last_rows (nullable) [n_rows][N].
 * Returns 0 on success, 1 on bad arguments, 2 on allocation failure, 3 on thread failure.
 */
int ss_oracle_fwd(const double *u, const double *delta, const double *A, const double *B, const double *C,
                  const double *D, const double *z, const double *delta_bias, int softplus, int64_t Bsz,
                  int64_t L, int64_t Dch, int64_t N, const int64_t *rows, int64_t n_rows, double *y_rows,
                  double *y0_rows, double *last_rows, int nthreads, const double *h0)
{
    if (Bsz < 0 || L < 0 || Dch < 0 || N < 0) return 1;
    problem p = {u, delta, A, B, C, D, z, delta_bias, NULL, softplus, Bsz, L, Dch, N, h0, NULL};
    if (!rows) n_rows = Bsz * Dch;
    if (n_rows == 0) return 0;
    if (!u || !delta || !A || !B || !C) return 1;
    for (int64_t i = 0; rows && i < n_rows; i++)
        if (rows[i] < 0 || rows[i] >= Bsz * Dch) return 1;
    job proto;
    memset(&proto, 0, sizeof proto);
    proto.p = &p;
    proto.rows = rows;
    proto.mode = 0;
    proto.y_rows = y_rows;
    proto.y0_rows = y0_rows;
    proto.last_rows = last_rows;
    return run_threads(&proto, n_rows, nthreads, NULL, NULL);
}

/*
 * Backward.  Per-row outputs: du/ddelta/dz [n_rows][L] (dz nullable), dA_rows [n_rows][N],
 * dD_rows [n_rows], dbias_rows [n_rows] -- the row's own contributions to dA[d], dD[d], dbias[d].
 * dB, dC (nullable) [Bsz][L][N]: the given rows' contributions are ADDED into them.
 * h0, dlast (nullable) [Bsz][Dch][N]: initial state and incoming gradient of last_state;
 * dh0_rows (nullable) [n_rows][N]: gradient of the initial state.
 */
int ss_oracle_bwd(const double *u, const double *delta, const double *A, const double *B, const double *C,
                  const double *D, const double *z, const double *delta_bias, int softplus, const double *dy,
                  int64_t Bsz, int64_t L, int64_t Dch, int64_t N, const int64_t *rows, int64_t n_rows,
                  double *du_rows, double *ddelta_rows, double *dz_rows, double *dA_rows, double *dD_rows,
                  double *dbias_rows, double *dB, double *dC, int nthreads, const double *h0, const double *dlast,
                  double *dh0_rows)
{
    if (Bsz < 0 || L < 0 || Dch < 0 || N < 0) return 1;
    problem p = {u, delta, A, B, C, D, z, delta_bias, dy, softplus, Bsz, L, Dch, N, h0, dlast};
    if (!rows) n_rows = Bsz * Dch;
    if (n_rows == 0) return 0;
    if (!u || !delta || !A || !B || !C || !dy || !du_rows || !ddelta_rows || !dA_rows || !dD_rows || !dbias_rows)
        return 1;
    for (int64_t i = 0; rows && i < n_rows; i++)
        if (rows[i] < 0 || rows[i] >= Bsz * Dch) return 1;
    job proto;
    memset(&proto, 0, sizeof proto);
    proto.p = &p;
    proto.rows = rows;
    proto.mode = 1;
    proto.du_rows = du_rows;
    proto.ddelta_rows = ddelta_rows;
    proto.dz_rows = dz_rows;
    proto.dA_rows = dA_rows;
    proto.dD_rows = dD_rows;
    proto.dbias_rows = dbias_rows;
    proto.dh0_rows = dh0_rows;
    return run_threads(&proto, n_rows, nthreads, dB, dC);
}
