/*
 * Float64 CPU oracle for the selective state-space scans.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * include this file: only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark run it. It shares no code with the CUDA
 * library.
 *
 * What it computes is the plain token-by-token definition of each scan, in
 * float64, with no chunking, blocking or reordering:
 *
 *   Mamba-2 SSD, per batch b and head h (group g = h / (H/G)):
 *     alpha_t   = exp(dt_t * A_h)
 *     h_t[p,n]  = alpha_t * h_{t-1}[p,n] + dt_t * x_t[p] * B_t[n]
 *     y_t[p]    = sum_n C_t[n] * h_t[p,n] + D_h * x_t[p]
 *   This is the generic selective update h_t = A_t h_{t-1} + B_t x_t,
 *   y_t = C_t h_t + D_t x_t of "COREY: Entropy-Guided Runtime Chunk Scheduling
 *   for Selective Scan Kernels" (section 3.1, Preliminaries), with the scalar
 *   per-head decay exp(dt*A) and the Euler input term dt*B of the Mamba-2 SSD
 *   layer ("Compiler-First State Space Duality ...", abstract: diagonal
 *   per-head dynamics). y uses the updated state h_t.
 *
 *   Decode step: the same update for one token, applied in place to a carried
 *   state (the O(1) cached decode of the same page, Figure 1).
 *
 *   Mamba-1 diagonal scan, per batch b and channel d:
 *     h_t[n] = exp(dt_t * A[d,n]) * h_{t-1}[n] + dt_t * x_t * B_t[n]
 *     y_t    = sum_n C_t[n] * h_t[n] + D_d * x_t
 *   (the selective_scan_fn workload of the COREY page, section 5.1).
 *   Its options (the same page's kernel-level timing, section 7, which runs
 *   selective_scan_fn with delta_softplus set): a per-channel delta_bias is
 *   added to dt, then with delta_softplus the step is softplus of that sum,
 *       dt_t = softplus(dt_raw_t + delta_bias_d),  softplus(v) = log(1 + e^v),
 *   and an optional gate z[B,L,Dm] multiplies the output by silu(z):
 *       out_t = y_t * z_t / (1 + exp(-z_t)).
 *
 *   SSD backward (the training step of "Compiler-First State Space Duality
 *   ...", appendix Table 13, forward + backward): reverse-mode differentiation
 *   of the same token loop. With gbar the adjoint of h_t, walking t downwards
 *   from gbar = dL/dh_{L-1} (the final-state cotangent, or 0):
 *     gbar += dy_t C_t^T                      (y_t reads h_t)
 *     dC_t += dy_t^T h_t;  dD += dy_t . x_t
 *     dx_t  = D dy_t + dt_t gbar B_t
 *     dB_t += dt_t gbar^T x_t
 *     dalpha = <gbar, h_{t-1}>;  alpha = exp(dt_t A)
 *     ddt_t = dalpha alpha A + x_t . (gbar B_t);  dA += dalpha alpha dt_t
 *     gbar  = alpha gbar                      (adjoint of h_{t-1})
 *   and the initial-state cotangent is the last gbar. States h_t are
 *   recomputed forward from checkpoints every 64 tokens (the same arithmetic
 *   as the forward loop, so the same values).
 *
 *   Decode-layer neighbours (the fused Mamba-2 decode layer sketched on
 *   "Mamba-2 SSD fused layer via VGpuWarp — design sketch", section "What has
 *   to become a device op", items 1 and 2):
 *     causal conv step, per (b, c), with a rolling window of the last W
 *     inputs, oldest first:  window <- (window[1..W-1], x_t);
 *       out = act(sum_k w[c,k] * window[k] + bias[c]), act = identity or silu;
 *     gated RMS norm, per (b, group of channels):  g = y * silu(z);
 *       out = g / sqrt(mean over the group of g^2 + eps) * w.
 *
 * Layouts (row-major, innermost last):
 *   SSD:    x[B,L,H,P]  dt[B,L,H]  A[H]  Bm,Cm[B,L,G,N]  D[H]  state[B,H,P,N]
 *           y[B,L,H,P]
 *   decode: x[B,H,P]    dt[B,H]    A[H]  Bm,Cm[B,G,N]    D[H]  state[B,H,P,N]
 *           y[B,H,P]
 *   diag:   x,dt[B,L,Dm]  A[Dm,N]  Bm,Cm[B,L,N]  D[Dm]  state[B,Dm,N]  y[B,L,Dm]
 *   conv:   x[B,C]  window state[B,C,W]  w[C,W]  bias[C]  out[B,C]
 *   norm:   y,z[B,D]  w[D]  out[B,D]
 * D and the initial state may be NULL (read as zero); a NULL final state is
 * not written. Independent (b,h) or (b,d) units run on nthreads POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, L, H, P, N, G;
    const double *x, *dt, *A, *Bm, *Cm, *D, *init;
    double *y, *final_state;
    int64_t next_unit, n_units;
    pthread_mutex_t lock;
} ssd_job;

static int64_t take_unit(int64_t *next, int64_t n, pthread_mutex_t *lock) {
    pthread_mutex_lock(lock);
    int64_t u = *next < n ? (*next)++ : -1;
    pthread_mutex_unlock(lock);
    return u;
}

/* One (b,h) unit of the SSD recurrence, token by token. */
static void ssd_unit(const ssd_job *j, int64_t b, int64_t h, double *st) {
    const int64_t L = j->L, H = j->H, P = j->P, N = j->N, G = j->G;
    const int64_t g = h / (H / G);
    const double Ah = j->A[h];
    const double Dh = j->D ? j->D[h] : 0.0;
    if (j->init)
        memcpy(st, j->init + (b * H + h) * P * N, sizeof(double) * P * N);
    else
        memset(st, 0, sizeof(double) * P * N);
    for (int64_t t = 0; t < L; ++t) {
        const double dt = j->dt[(b * L + t) * H + h];
        const double alpha = exp(dt * Ah);
        const double *xt = j->x + ((b * L + t) * H + h) * P;
        const double *Bt = j->Bm + ((b * L + t) * G + g) * N;
        const double *Ct = j->Cm + ((b * L + t) * G + g) * N;
        double *yt = j->y + ((b * L + t) * H + h) * P;
        for (int64_t p = 0; p < P; ++p) {
            double *row = st + p * N;
            const double u = dt * xt[p];
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                row[n] = alpha * row[n] + u * Bt[n];
                acc += Ct[n] * row[n];
            }
            yt[p] = acc + Dh * xt[p];
        }
    }
    if (j->final_state)
        memcpy(j->final_state + (b * H + h) * P * N, st, sizeof(double) * P * N);
}

static void *ssd_worker(void *arg) {
    ssd_job *j = (ssd_job *)arg;
    double *st = (double *)malloc(sizeof(double) * (size_t)(j->P * j->N > 0 ? j->P * j->N : 1));
    for (;;) {
        int64_t u = take_unit(&j->next_unit, j->n_units, &j->lock);
        if (u < 0) break;
        ssd_unit(j, u / j->H, u % j->H, st);
    }
    free(st);
    return NULL;
}

static void run_threads(void *(*fn)(void *), void *job, int nthreads, int64_t n_units) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = (int)(n_units > 0 ? n_units : 1);
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&tid[started], NULL, fn, job) == 0) ++started;
    fn(job);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
}

/* Returns 0 on success, -1 on invalid sizes. */
int oracle_ssd_seq(int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                   const double *x, const double *dt, const double *A, const double *Bm,
                   const double *Cm, const double *D, const double *init_state, double *y,
                   double *final_state, int nthreads) {
    if (B < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G != 0) return -1;
    ssd_job j = {B, L, H, P, N, G, x, dt, A, Bm, Cm, D, init_state, y, final_state, 0, B * H};
    pthread_mutex_init(&j.lock, NULL);
    run_threads(ssd_worker, &j, nthreads, B * H);
    pthread_mutex_destroy(&j.lock);
    return 0;
}

/* One decode token, state updated in place: the L=1 case of the same unit. */
int oracle_ssd_decode(int64_t B, int64_t H, int64_t P, int64_t N, int64_t G, double *state,
                      const double *x, const double *dt, const double *A, const double *Bm,
                      const double *Cm, const double *D, double *y, int nthreads) {
    return oracle_ssd_seq(B, 1, H, P, N, G, x, dt, A, Bm, Cm, D, state, y, state, nthreads);
}

typedef struct {
    int64_t B, L, Dm, N;
    const double *x, *dt, *A, *Bm, *Cm, *D, *init;
    double *y, *final_state;
    const double *delta_bias, *z;
    int delta_softplus;
    int64_t next_unit, n_units;
    pthread_mutex_t lock;
} diag_job;

/* softplus(v) = log(1 + e^v), written so that e^v cannot overflow. */
static double softplus(double v) { return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v)); }

/* One (b,d) unit of the Mamba-1 diagonal recurrence. */
static void diag_unit(const diag_job *j, int64_t b, int64_t d, double *st) {
    const int64_t L = j->L, Dm = j->Dm, N = j->N;
    const double *Ad = j->A + d * N;
    const double Dd = j->D ? j->D[d] : 0.0;
    if (j->init)
        memcpy(st, j->init + (b * Dm + d) * N, sizeof(double) * N);
    else
        memset(st, 0, sizeof(double) * N);
    const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double dt = j->dt[(b * L + t) * Dm + d] + bias;
        if (j->delta_softplus) dt = softplus(dt);
        const double xt = j->x[(b * L + t) * Dm + d];
        const double *Bt = j->Bm + (b * L + t) * N;
        const double *Ct = j->Cm + (b * L + t) * N;
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            st[n] = exp(dt * Ad[n]) * st[n] + dt * xt * Bt[n];
            acc += Ct[n] * st[n];
        }
        double out = acc + Dd * xt;
        if (j->z) {
            const double zt = j->z[(b * L + t) * Dm + d];
            out *= zt / (1.0 + exp(-zt));
        }
        j->y[(b * L + t) * Dm + d] = out;
    }
    if (j->final_state) memcpy(j->final_state + (b * Dm + d) * N, st, sizeof(double) * N);
}

static void *diag_worker(void *arg) {
    diag_job *j = (diag_job *)arg;
    double *st = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    for (;;) {
        int64_t u = take_unit(&j->next_unit, j->n_units, &j->lock);
        if (u < 0) break;
        diag_unit(j, u / j->Dm, u % j->Dm, st);
    }
    free(st);
    return NULL;
}

int oracle_diag_seq_ex(int64_t B, int64_t L, int64_t Dm, int64_t N, const double *x,
                       const double *dt, const double *A, const double *Bm, const double *Cm,
                       const double *D, const double *z, const double *delta_bias, int delta_softplus,
                       const double *init_state, double *y, double *final_state, int nthreads) {
    if (B < 0 || L < 0 || Dm < 1 || N < 1) return -1;
    diag_job j = {B, L, Dm, N, x, dt, A, Bm, Cm, D, init_state, y, final_state,
                  delta_bias, z, delta_softplus != 0, 0, B * Dm};
    pthread_mutex_init(&j.lock, NULL);
    run_threads(diag_worker, &j, nthreads, B * Dm);
    pthread_mutex_destroy(&j.lock);
    return 0;
}

int oracle_diag_seq(int64_t B, int64_t L, int64_t Dm, int64_t N, const double *x,
                    const double *dt, const double *A, const double *Bm, const double *Cm,
                    const double *D, const double *init_state, double *y, double *final_state,
                    int nthreads) {
    return oracle_diag_seq_ex(B, L, Dm, N, x, dt, A, Bm, Cm, D, NULL, NULL, 0, init_state, y,
                              final_state, nthreads);
}

typedef struct {
    int64_t B, L, H, P, N, G;
    const double *x, *dt, *A, *Bm, *Cm, *D, *init, *dy, *dfinal;
    double *dx, *ddt, *dA_part, *dB, *dC, *dD_part, *dinit;
    int64_t next_unit, n_units;
    pthread_mutex_t lock;
} bwd_job;

enum { kCkpt = 64 };

/* Backward of one (b, g) unit: the heads of group g in order, so that the
   shared dB, dC of the group are accumulated by this unit alone. */
static void bwd_unit(const bwd_job *j, int64_t b, int64_t g) {
    const int64_t L = j->L, H = j->H, P = j->P, N = j->N, G = j->G, PN = j->P * j->N;
    const int64_t hpg = H / G, nck = (L + kCkpt - 1) / kCkpt;
    double *ck = (double *)malloc(sizeof(double) * (size_t)(nck > 0 ? nck : 1) * PN);
    double *seg = (double *)malloc(sizeof(double) * (size_t)(kCkpt + 1) * PN);
    double *gbar = (double *)malloc(sizeof(double) * PN);
    for (int64_t t = 0; t < L; ++t)
        for (int64_t n = 0; n < N; ++n) {
            j->dB[((b * L + t) * G + g) * N + n] = 0.0;
            j->dC[((b * L + t) * G + g) * N + n] = 0.0;
        }
    for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
        const double Ah = j->A[h], Dh = j->D ? j->D[h] : 0.0;
        double dA = 0.0, dD = 0.0;
        /* forward: the state entering every kCkpt-token segment */
        double *st = seg;
        if (j->init)
            memcpy(st, j->init + (b * H + h) * PN, sizeof(double) * PN);
        else
            memset(st, 0, sizeof(double) * PN);
        for (int64_t t = 0; t < L; ++t) {
            if (t % kCkpt == 0) memcpy(ck + (t / kCkpt) * PN, st, sizeof(double) * PN);
            const double dt = j->dt[(b * L + t) * H + h], alpha = exp(dt * Ah);
            const double *xt = j->x + ((b * L + t) * H + h) * P, *Bt = j->Bm + ((b * L + t) * G + g) * N;
            for (int64_t p = 0; p < P; ++p)
                for (int64_t n = 0; n < N; ++n) st[p * N + n] = alpha * st[p * N + n] + dt * xt[p] * Bt[n];
        }
        if (j->dfinal)
            memcpy(gbar, j->dfinal + (b * H + h) * PN, sizeof(double) * PN);
        else
            memset(gbar, 0, sizeof(double) * PN);
        for (int64_t c = nck - 1; c >= 0; --c) {
            const int64_t t0 = c * kCkpt, t1 = t0 + kCkpt < L ? t0 + kCkpt : L;
            /* seg[k] = h_{t0 + k - 1}: the entering state, then each token's state */
            memcpy(seg, ck + c * PN, sizeof(double) * PN);
            for (int64_t t = t0; t < t1; ++t) {
                const double dt = j->dt[(b * L + t) * H + h], alpha = exp(dt * Ah);
                const double *xt = j->x + ((b * L + t) * H + h) * P, *Bt = j->Bm + ((b * L + t) * G + g) * N;
                const double *prev = seg + (t - t0) * PN;
                double *cur = seg + (t - t0 + 1) * PN;
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t n = 0; n < N; ++n) cur[p * N + n] = alpha * prev[p * N + n] + dt * xt[p] * Bt[n];
            }
            for (int64_t t = t1 - 1; t >= t0; --t) {
                const double dt = j->dt[(b * L + t) * H + h], alpha = exp(dt * Ah);
                const double *xt = j->x + ((b * L + t) * H + h) * P, *dyt = j->dy + ((b * L + t) * H + h) * P;
                const double *Bt = j->Bm + ((b * L + t) * G + g) * N, *Ct = j->Cm + ((b * L + t) * G + g) * N;
                const double *ht = seg + (t - t0 + 1) * PN, *hprev = seg + (t - t0) * PN;
                double *dxt = j->dx + ((b * L + t) * H + h) * P;
                double *dBt = j->dB + ((b * L + t) * G + g) * N, *dCt = j->dC + ((b * L + t) * G + g) * N;
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t n = 0; n < N; ++n) gbar[p * N + n] += dyt[p] * Ct[n];
                for (int64_t n = 0; n < N; ++n) {
                    double c_ = 0.0, b_ = 0.0;
                    for (int64_t p = 0; p < P; ++p) {
                        c_ += dyt[p] * ht[p * N + n];
                        b_ += gbar[p * N + n] * xt[p];
                    }
                    dCt[n] += c_;
                    dBt[n] += dt * b_;
                }
                double dalpha = 0.0, xgb = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    double gb = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        gb += gbar[p * N + n] * Bt[n];
                        dalpha += gbar[p * N + n] * hprev[p * N + n];
                    }
                    dxt[p] = Dh * dyt[p] + dt * gb;
                    xgb += xt[p] * gb;
                    dD += dyt[p] * xt[p];
                }
                j->ddt[(b * L + t) * H + h] = dalpha * alpha * Ah + xgb;
                dA += dalpha * alpha * dt;
                for (int64_t k = 0; k < PN; ++k) gbar[k] *= alpha;
            }
        }
        if (j->dinit) memcpy(j->dinit + (b * H + h) * PN, gbar, sizeof(double) * PN);
        j->dA_part[b * H + h] = dA;
        j->dD_part[b * H + h] = dD;
    }
    free(ck);
    free(seg);
    free(gbar);
}

static void *bwd_worker(void *arg) {
    bwd_job *j = (bwd_job *)arg;
    for (;;) {
        int64_t u = take_unit(&j->next_unit, j->n_units, &j->lock);
        if (u < 0) break;
        bwd_unit(j, u / j->G, u % j->G);
    }
    return NULL;
}

/* Gradients of the SSD scan: dx[B,L,H,P], ddt[B,L,H], dA[H], dB/dC[B,L,G,N],
   dD[H], dinit[B,H,P,N] (may be NULL) for cotangents dy[B,L,H,P] and dfinal
   [B,H,P,N] (may be NULL: 0). dA and dD sum the per-(b, h) parts in b order. */
int oracle_ssd_seq_bwd(int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G, const double *x,
                       const double *dt, const double *A, const double *Bm, const double *Cm, const double *D,
                       const double *init_state, const double *dy, const double *dfinal, double *dx,
                       double *ddt, double *dA, double *dB, double *dC, double *dD, double *dinit, int nthreads) {
    if (B < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G != 0) return -1;
    double *dA_part = (double *)calloc((size_t)(B * H > 0 ? B * H : 1), sizeof(double));
    double *dD_part = (double *)calloc((size_t)(B * H > 0 ? B * H : 1), sizeof(double));
    bwd_job j = {B, L, H, P, N, G, x, dt, A, Bm, Cm, D, init_state, dy, dfinal,
                 dx, ddt, dA_part, dB, dC, dD_part, dinit, 0, B * G};
    pthread_mutex_init(&j.lock, NULL);
    run_threads(bwd_worker, &j, nthreads, B * G);
    pthread_mutex_destroy(&j.lock);
    for (int64_t h = 0; h < H; ++h) {
        double a = 0.0, d = 0.0;
        for (int64_t b = 0; b < B; ++b) {
            a += dA_part[b * H + h];
            d += dD_part[b * H + h];
        }
        dA[h] = a;
        if (dD) dD[h] = d;
    }
    free(dA_part);
    free(dD_part);
    return 0;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* One causal depthwise convolution step, the window updated in place. */
int oracle_conv1d_step(int64_t B, int64_t C, int64_t W, double *state, const double *x, const double *w,
                       const double *bias, int act, double *out) {
    if (B < 0 || C < 1 || W < 1) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t c = 0; c < C; ++c) {
            double *win = state + (b * C + c) * W;
            for (int64_t k = 0; k + 1 < W; ++k) win[k] = win[k + 1];
            win[W - 1] = x[b * C + c];
            double acc = bias ? bias[c] : 0.0;
            for (int64_t k = 0; k < W; ++k) acc += w[c * W + k] * win[k];
            out[b * C + c] = act ? silu(acc) : acc;
        }
    return 0;
}

/* Gated RMS norm over groups of `group` consecutive channels (D % group == 0). */
int oracle_gated_rmsnorm(int64_t B, int64_t D, int64_t group, const double *y, const double *z, const double *w,
                         double eps, double *out) {
    if (B < 0 || D < 1 || group < 1 || D % group != 0) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g0 = 0; g0 < D; g0 += group) {
            double ss = 0.0;
            for (int64_t i = g0; i < g0 + group; ++i) {
                const double g = y[b * D + i] * (z ? silu(z[b * D + i]) : 1.0);
                ss += g * g;
            }
            const double r = 1.0 / sqrt(ss / (double)group + eps);
            for (int64_t i = g0; i < g0 + group; ++i) {
                const double g = y[b * D + i] * (z ? silu(z[b * D + i]) : 1.0);
                out[b * D + i] = g * r * w[i];
            }
        }
    return 0;
}
