/*
 * linattn_oracle.c -- fp64 CPU oracle for elu(x)+1 kernelized linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Every routine is the plain definition from the pages, written out in
 * double precision with straightforward loops (no blocking, no fusion, no
 * reordering beyond what the definition states).  Citations name the page
 * and the section / equation each step follows:
 *
 *   [P1] "Linear Attention/es" (marovi.ai)
 *        - "Reformulación con núcleos", eq. y_i = phi(q_i)^T S / phi(q_i)^T z
 *          with S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j).
 *        - "Mapas de características", phi(x) = elu(x) + 1.
 *        - "Forma recurrente e inferencia autorregresiva", S_t = S_{t-1} +
 *          phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t), y_t = phi(q_t)^T S_t /
 *          phi(q_t)^T z_t.
 *        - "Entrenamiento: forma paralela", blockwise form: masked
 *          intra-block pairs plus an inter-block linear state update.
 *   [P2] "Linear Transformer (Transformers are RNNs)" (visibilidadia.com)
 *        - "La función ELU + 1": ELU(x) = x for x > 0, e^x - 1 for x <= 0.
 *        - "La formulación recurrente paso a paso": S_t, z_t, o_t.
 *        - The worked PyTorch examples divide by the denominator clamped
 *          from below by eps (clamp_min), which is what max(den, eps) is.
 *
 * Layouts (all row-major, contiguous, fp64):
 *   q, k : [BH][N][d]      v, y : [BH][N][dv]
 *   S    : [BH][d][dv]     z    : [BH][d]
 * BH is batch*heads; heads are independent and are split across threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* [P1] "Mapas de características": phi(x) = elu(x) + 1, with
 * [P2] "La función ELU + 1": ELU(x) = x (x > 0), e^x - 1 (x <= 0).  The same
 * section simplifies the sum to phi(x) = x + 1 (x > 0), e^x (x <= 0); that
 * form is used because it is exact in double precision and keeps phi > 0
 * (the section stresses positivity), whereas (e^x - 1) + 1 rounds e^x away
 * once e^x < 2^-53.                                                         */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* Denominator clamp used by the pages' examples: max(den, eps). */
static double clamp_den(double den, double eps) { return den < eps ? eps : den; }

/* [P1] "Mapas de características" lists the feature maps: kind 0 is the
 * canonical elu(x) + 1 above; kind 1 is the identity map phi(x) = x, which
 * "reduces the layer to a simple bilinear attention".  (The random-feature
 * map changes the feature dimension and is oracle_random_features below.)  */
static double feature(double x, int kind) { return kind == 1 ? x : phi(x); }

void oracle_phi(const double *x, double *out, long n)
{
    for (long i = 0; i < n; ++i) out[i] = phi(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Per-head work items and a tiny pthread pool over heads.                  */
/* ------------------------------------------------------------------------ */
typedef struct {
    int kind;              /* 0 recurrent causal, 1 non-causal, 2 quadratic, 3 chunked */
    const double *q, *k, *v;
    double *y;
    const double *S_in, *z_in; /* nullable: zero state */
    double *S_out, *z_out;     /* nullable */
    int BH, N, d, dv, causal, chunk;
    double eps;
    const double *gamma;       /* nullable: per-head decay (recurrent form only) */
    const double *gate;        /* nullable: per-token gate [BH][N][gate_dim] (recurrent form) */
    int gate_dim;              /* 1 (one gate per token) or d (one per token and feature) */
    int phi_kind;              /* feature map, see feature() */
    int h_begin, h_end;
} job_t;

/* [P1] "Forma recurrente ..." / [P2] "La formulación recurrente paso a paso":
 * for t = 1..N: S += phi(k_t) v_t^T, z += phi(k_t) (update first), then
 * y_t = phi(q_t)^T S / max(phi(q_t)^T z, eps).
 * With a decay ([P1] "Variantes y extensiones", RetNet: S_t = gamma S_{t-1}
 * + phi(k_t) v_t^T, one gamma per head for the multi-scale retention the
 * section mentions) the state is first multiplied by gamma; z is decayed
 * the same way so that y_t stays a normalised average.                    */
/* With a gate ([P1] "Variantes y extensiones": gated linear attention
 * replaces the scalar decay by a data-dependent gate; the pages print no
 * equation, so the reading is the decay's update with the decay taken per
 * token): S_t = diag(g_t) S_{t-1} + phi(k_t) v_t^T and z_t = g_t * z_{t-1} +
 * phi(k_t), g_t in [0, 1] given per token as one value (gate_dim = 1) or one
 * per feature row of S (gate_dim = d, the per-channel gates of the Gated
 * DeltaNet passage).                                                         */
static void head_recurrent(const job_t *J, int h)
{
    const int N = J->N, d = J->d, dv = J->dv, fkind = J->phi_kind;
    const double *q = J->q + (long)h * N * d, *k = J->k + (long)h * N * d;
    const double *v = J->v + (long)h * N * dv;
    double *y = J->y + (long)h * N * dv;
    double *S = calloc((size_t)d * dv, sizeof(double));
    double *z = calloc((size_t)d, sizeof(double));
    double *fk = malloc(sizeof(double) * d), *fq = malloc(sizeof(double) * d);
    if (J->S_in) memcpy(S, J->S_in + (long)h * d * dv, sizeof(double) * d * dv);
    if (J->z_in) memcpy(z, J->z_in + (long)h * d, sizeof(double) * d);
    for (int t = 0; t < N; ++t) {
        for (int a = 0; a < d; ++a) fk[a] = feature(k[(long)t * d + a], fkind);
        if (J->gamma) {
            const double g = J->gamma[h];
            for (int a = 0; a < d; ++a) {
                for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= g;
                z[a] *= g;
            }
        }
        if (J->gate) {
            const double *gt = J->gate + ((long)h * N + t) * J->gate_dim;
            for (int a = 0; a < d; ++a) {
                const double g = gt[J->gate_dim == 1 ? 0 : a];
                for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= g;
                z[a] *= g;
            }
        }
        for (int a = 0; a < d; ++a) {
            for (int b = 0; b < dv; ++b) S[(long)a * dv + b] += fk[a] * v[(long)t * dv + b];
            z[a] += fk[a];
        }
        for (int a = 0; a < d; ++a) fq[a] = feature(q[(long)t * d + a], fkind);
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += fq[a] * z[a];
        den = clamp_den(den, J->eps);
        for (int b = 0; b < dv; ++b) {
            double num = 0.0;
            for (int a = 0; a < d; ++a) num += fq[a] * S[(long)a * dv + b];
            y[(long)t * dv + b] = num / den;
        }
    }
    if (J->S_out) memcpy(J->S_out + (long)h * d * dv, S, sizeof(double) * d * dv);
    if (J->z_out) memcpy(J->z_out + (long)h * d, z, sizeof(double) * d);
    free(S); free(z); free(fk); free(fq);
}

/* [P1] "Reformulación con núcleos": S = sum_j phi(k_j) v_j^T and
 * z = sum_j phi(k_j) over the whole sequence, then for every query
 * y_i = phi(q_i)^T S / max(phi(q_i)^T z, eps).                             */
static void head_noncausal(const job_t *J, int h)
{
    const int N = J->N, d = J->d, dv = J->dv, fkind = J->phi_kind;
    const double *q = J->q + (long)h * N * d, *k = J->k + (long)h * N * d;
    const double *v = J->v + (long)h * N * dv;
    double *y = J->y + (long)h * N * dv;
    double *S = calloc((size_t)d * dv, sizeof(double));
    double *z = calloc((size_t)d, sizeof(double));
    double *f = malloc(sizeof(double) * d);
    for (int j = 0; j < N; ++j) {
        for (int a = 0; a < d; ++a) f[a] = feature(k[(long)j * d + a], fkind);
        for (int a = 0; a < d; ++a) {
            for (int b = 0; b < dv; ++b) S[(long)a * dv + b] += f[a] * v[(long)j * dv + b];
            z[a] += f[a];
        }
    }
    for (int i = 0; i < N; ++i) {
        for (int a = 0; a < d; ++a) f[a] = feature(q[(long)i * d + a], fkind);
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += f[a] * z[a];
        den = clamp_den(den, J->eps);
        for (int b = 0; b < dv; ++b) {
            double num = 0.0;
            for (int a = 0; a < d; ++a) num += f[a] * S[(long)a * dv + b];
            y[(long)i * dv + b] = num / den;
        }
    }
    if (J->S_out) memcpy(J->S_out + (long)h * d * dv, S, sizeof(double) * d * dv);
    if (J->z_out) memcpy(J->z_out + (long)h * d, z, sizeof(double) * d);
    free(S); free(z); free(f);
}

/* [P1] "Reformulación con núcleos", first equality, evaluated pair by pair:
 * y_i = sum_j w_ij v_j / max(sum_j w_ij, eps), w_ij = phi(q_i)^T phi(k_j),
 * over j <= i (causal) or all j.  O(N^2 d): brute force for small cases.   */
static void head_quadratic(const job_t *J, int h)
{
    const int N = J->N, d = J->d, dv = J->dv;
    const double *q = J->q + (long)h * N * d, *k = J->k + (long)h * N * d;
    const double *v = J->v + (long)h * N * dv;
    double *y = J->y + (long)h * N * dv;
    double *num = malloc(sizeof(double) * dv);
    for (int i = 0; i < N; ++i) {
        const int jmax = J->causal ? i : N - 1;
        double den = 0.0;
        for (int b = 0; b < dv; ++b) num[b] = 0.0;
        for (int j = 0; j <= jmax; ++j) {
            double w = 0.0;
            for (int a = 0; a < d; ++a)
                w += feature(q[(long)i * d + a], J->phi_kind) * feature(k[(long)j * d + a], J->phi_kind);
            den += w;
            for (int b = 0; b < dv; ++b) num[b] += w * v[(long)j * dv + b];
        }
        den = clamp_den(den, J->eps);
        for (int b = 0; b < dv; ++b) y[(long)i * dv + b] = num[b] / den;
    }
    free(num);
}

/* [P1] "Entrenamiento: forma paralela": split the sequence into blocks of C
 * tokens.  Inside block c the output combines the masked pairwise term over
 * the block (j <= i, both in c) with the linear term phi(q_i)^T S_prev over
 * all earlier blocks; after the block, S_prev += sum_{j in c} phi(k_j) v_j^T
 * and z_prev += sum_{j in c} phi(k_j).                                      */
static void head_chunked(const job_t *J, int h)
{
    const int N = J->N, d = J->d, dv = J->dv, C = J->chunk;
    const double *q = J->q + (long)h * N * d, *k = J->k + (long)h * N * d;
    const double *v = J->v + (long)h * N * dv;
    double *y = J->y + (long)h * N * dv;
    double *S = calloc((size_t)d * dv, sizeof(double));
    double *z = calloc((size_t)d, sizeof(double));
    double *fq = malloc(sizeof(double) * (size_t)C * d);
    double *fk = malloc(sizeof(double) * (size_t)C * d);
    double *num = malloc(sizeof(double) * dv);
    if (J->S_in) memcpy(S, J->S_in + (long)h * d * dv, sizeof(double) * d * dv);
    if (J->z_in) memcpy(z, J->z_in + (long)h * d, sizeof(double) * d);
    for (int c0 = 0; c0 < N; c0 += C) {
        const int L = (N - c0) < C ? (N - c0) : C;
        for (int i = 0; i < L; ++i)
            for (int a = 0; a < d; ++a) {
                fq[(long)i * d + a] = phi(q[(long)(c0 + i) * d + a]);
                fk[(long)i * d + a] = phi(k[(long)(c0 + i) * d + a]);
            }
        for (int i = 0; i < L; ++i) {
            /* inter-block: phi(q_i)^T S_prev and phi(q_i)^T z_prev */
            double den = 0.0;
            for (int a = 0; a < d; ++a) den += fq[(long)i * d + a] * z[a];
            for (int b = 0; b < dv; ++b) {
                double s = 0.0;
                for (int a = 0; a < d; ++a) s += fq[(long)i * d + a] * S[(long)a * dv + b];
                num[b] = s;
            }
            /* intra-block: masked pairs j <= i inside the block */
            for (int j = 0; j <= i; ++j) {
                double w = 0.0;
                for (int a = 0; a < d; ++a) w += fq[(long)i * d + a] * fk[(long)j * d + a];
                den += w;
                for (int b = 0; b < dv; ++b) num[b] += w * v[(long)(c0 + j) * dv + b];
            }
            den = clamp_den(den, J->eps);
            for (int b = 0; b < dv; ++b) y[(long)(c0 + i) * dv + b] = num[b] / den;
        }
        /* state update after the block */
        for (int j = 0; j < L; ++j)
            for (int a = 0; a < d; ++a) {
                for (int b = 0; b < dv; ++b)
                    S[(long)a * dv + b] += fk[(long)j * d + a] * v[(long)(c0 + j) * dv + b];
                z[a] += fk[(long)j * d + a];
            }
    }
    if (J->S_out) memcpy(J->S_out + (long)h * d * dv, S, sizeof(double) * d * dv);
    if (J->z_out) memcpy(J->z_out + (long)h * d, z, sizeof(double) * d);
    free(S); free(z); free(fq); free(fk); free(num);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    for (int h = J->h_begin; h < J->h_end; ++h) {
        switch (J->kind) {
        case 0: head_recurrent(J, h); break;
        case 1: head_noncausal(J, h); break;
        case 2: head_quadratic(J, h); break;
        default: head_chunked(J, h); break;
        }
    }
    return NULL;
}

static int run_jobs(job_t base, int nthreads)
{
    if (base.BH < 0 || base.N < 0 || base.d <= 0 || base.dv <= 0) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > base.BH) nthreads = base.BH > 0 ? base.BH : 1;
    job_t *jobs = malloc(sizeof(job_t) * nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].h_begin = (int)((long)base.BH * t / nthreads);
        jobs[t].h_end = (int)((long)base.BH * (t + 1) / nthreads);
    }
    char *joined = calloc((size_t)nthreads, 1);
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) == 0) joined[t] = 1;
        else worker(&jobs[t]); /* fall back to running it on this thread */
    worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t]) pthread_join(th[t], NULL);
    free(joined);
    free(jobs); free(th);
    return 0;
}

/* Causal, recurrent (token by token).  S_in/z_in may be NULL (zero state);
 * S_out/z_out may be NULL.  Returns 0 on success.                          */
int oracle_causal_recurrent(const double *q, const double *k, const double *v, double *y,
                            int BH, int N, int d, int dv, double eps,
                            const double *S_in, const double *z_in,
                            double *S_out, double *z_out, int nthreads)
{
    job_t J = {0};
    J.kind = 0; J.q = q; J.k = k; J.v = v; J.y = y; J.S_in = S_in; J.z_in = z_in;
    J.S_out = S_out; J.z_out = z_out; J.BH = BH; J.N = N; J.d = d; J.dv = dv; J.eps = eps;
    return run_jobs(J, nthreads);
}

/* Causal recurrent form with a per-head decay gamma[BH] (0 < gamma <= 1). */
int oracle_causal_recurrent_decay(const double *q, const double *k, const double *v, double *y,
                                  int BH, int N, int d, int dv, double eps, const double *gamma,
                                  const double *S_in, const double *z_in,
                                  double *S_out, double *z_out, int nthreads)
{
    if (!gamma) return 1;
    job_t J = {0};
    J.kind = 0; J.q = q; J.k = k; J.v = v; J.y = y; J.S_in = S_in; J.z_in = z_in;
    J.S_out = S_out; J.z_out = z_out; J.BH = BH; J.N = N; J.d = d; J.dv = dv; J.eps = eps;
    J.gamma = gamma;
    return run_jobs(J, nthreads);
}

/* Non-causal matrix form.  S_out/z_out (the full-sequence sums) may be NULL. */
int oracle_noncausal(const double *q, const double *k, const double *v, double *y,
                     int BH, int N, int d, int dv, double eps,
                     double *S_out, double *z_out, int nthreads)
{
    job_t J = {0};
    J.kind = 1; J.q = q; J.k = k; J.v = v; J.y = y; J.S_out = S_out; J.z_out = z_out;
    J.BH = BH; J.N = N; J.d = d; J.dv = dv; J.eps = eps;
    return run_jobs(J, nthreads);
}

/* Brute-force pairwise form; causal != 0 restricts to j <= i. */
int oracle_quadratic(const double *q, const double *k, const double *v, double *y,
                     int BH, int N, int d, int dv, double eps, int causal, int nthreads)
{
    job_t J = {0};
    J.kind = 2; J.q = q; J.k = k; J.v = v; J.y = y; J.BH = BH; J.N = N; J.d = d; J.dv = dv;
    J.eps = eps; J.causal = causal;
    return run_jobs(J, nthreads);
}

/* Causal recurrent form with a gate per token (gate_dim = 1) or per token
 * and feature (gate_dim = d), gate[BH][N][gate_dim] in [0, 1] (NULL: none),
 * and feature map phi_kind (see feature()).                               */
int oracle_causal_gated(const double *q, const double *k, const double *v, double *y,
                        int BH, int N, int d, int dv, double eps, int phi_kind,
                        const double *gate, int gate_dim, const double *S_in,
                        const double *z_in, double *S_out, double *z_out, int nthreads)
{
    if (gate && gate_dim != 1 && gate_dim != d) return 1;
    if (phi_kind != 0 && phi_kind != 1) return 1;
    job_t J = {0};
    J.kind = 0; J.q = q; J.k = k; J.v = v; J.y = y; J.S_in = S_in; J.z_in = z_in;
    J.S_out = S_out; J.z_out = z_out; J.BH = BH; J.N = N; J.d = d; J.dv = dv; J.eps = eps;
    J.gate = gate; J.gate_dim = gate ? gate_dim : 1; J.phi_kind = phi_kind;
    return run_jobs(J, nthreads);
}

/* Non-causal matrix form with feature map phi_kind. */
int oracle_noncausal_phi(const double *q, const double *k, const double *v, double *y,
                         int BH, int N, int d, int dv, double eps, int phi_kind,
                         double *S_out, double *z_out, int nthreads)
{
    if (phi_kind != 0 && phi_kind != 1) return 1;
    job_t J = {0};
    J.kind = 1; J.q = q; J.k = k; J.v = v; J.y = y; J.S_out = S_out; J.z_out = z_out;
    J.BH = BH; J.N = N; J.d = d; J.dv = dv; J.eps = eps; J.phi_kind = phi_kind;
    return run_jobs(J, nthreads);
}

/* Brute-force pairwise form with feature map phi_kind. */
int oracle_quadratic_phi(const double *q, const double *k, const double *v, double *y,
                         int BH, int N, int d, int dv, double eps, int causal, int phi_kind,
                         int nthreads)
{
    if (phi_kind != 0 && phi_kind != 1) return 1;
    job_t J = {0};
    J.kind = 2; J.q = q; J.k = k; J.v = v; J.y = y; J.BH = BH; J.N = N; J.d = d; J.dv = dv;
    J.eps = eps; J.causal = causal; J.phi_kind = phi_kind;
    return run_jobs(J, nthreads);
}

/* [P1] "Mapas de características", random-feature maps (Performer): positive
 * random features phi(x) proportional to exp(W x - ||x||^2 / 2), W holding
 * the random projections as rows.  The constant of proportionality is read
 * as 1 / sqrt(m) for m rows, so that phi(q) . phi(k) is the average over the
 * m rows w of exp(w.q + w.k - (||q||^2 + ||k||^2) / 2); for Gaussian rows
 * w ~ N(0, I) its expectation is exp(q . k), the softmax kernel the section
 * says the map recovers in expectation.  x: [rows][d], W: [m][d] (given:
 * the random numbers are an input), out: [rows][m].                          */
int oracle_random_features(const double *x, const double *W, double *out, long rows, int d,
                           int m)
{
    if (rows < 0 || d <= 0 || m <= 0) return 1;
    const double scale = 1.0 / sqrt((double)m);
    for (long r = 0; r < rows; ++r) {
        double nrm = 0.0;
        for (int a = 0; a < d; ++a) nrm += x[r * d + a] * x[r * d + a];
        for (int f = 0; f < m; ++f) {
            double wx = 0.0;
            for (int a = 0; a < d; ++a) wx += W[(long)f * d + a] * x[r * d + a];
            out[r * m + f] = scale * exp(wx - 0.5 * nrm);
        }
    }
    return 0;
}

/* Blockwise causal form with block length `chunk` (>= 1). */
int oracle_causal_chunked(const double *q, const double *k, const double *v, double *y,
                          int BH, int N, int d, int dv, double eps, int chunk,
                          const double *S_in, const double *z_in,
                          double *S_out, double *z_out, int nthreads)
{
    if (chunk < 1) return 1;
    job_t J = {0};
    J.kind = 3; J.q = q; J.k = k; J.v = v; J.y = y; J.S_in = S_in; J.z_in = z_in;
    J.S_out = S_out; J.z_out = z_out; J.BH = BH; J.N = N; J.d = d; J.dv = dv; J.eps = eps;
    J.chunk = chunk;
    return run_jobs(J, nthreads);
}

/* One recurrent decode step per head on a stored state (in place):
 * S += phi(k) v^T, z += phi(k), then y = phi(q)^T S / max(phi(q)^T z, eps).
 * q, k: [BH][d]; v, y: [BH][dv]; S: [BH][d][dv]; z: [BH][d].               */
int oracle_decode_step(const double *q, const double *k, const double *v, double *y,
                       double *S, double *z, int BH, int d, int dv, double eps, int nthreads)
{
    /* A decode step is the recurrent form with N = 1 continuing from (S, z). */
    job_t J = {0};
    J.kind = 0; J.q = q; J.k = k; J.v = v; J.y = y; J.S_in = S; J.z_in = z;
    J.S_out = S; J.z_out = z; J.BH = BH; J.N = 1; J.d = d; J.dv = dv; J.eps = eps;
    return run_jobs(J, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Gradients of the causal form.                                            */
/* ------------------------------------------------------------------------ */
/* [P1] "Entrenamiento: forma paralela" names training through the causal
 * recurrence as the reason for the parallel form; training needs the
 * gradients of a scalar loss L with respect to q, k, v.  Given dy_t = dL/dy_t
 * they follow from the recurrence of "Forma recurrente e inferencia
 * autorregresiva" by the chain rule, taken in the recurrence's own order
 * (forward in t, then backward in t):
 *
 *   with D_t = max(den_t, eps), den_t = phi(q_t)^T z_t, y_t = S_t^T phi(q_t) / D_t:
 *     g_t   = dy_t / D_t                         dL/d(num_t)
 *     e_t   = -(dy_t . y_t) / D_t  if den_t >= eps, else 0   dL/d(den_t)
 *     dL/dphi(q_t) = S_t g_t + z_t e_t
 *   the state gradients run backwards from t = N:
 *     Sh_t = sum_{s >= t} phi(q_s) g_s^T,   zh_t = sum_{s >= t} phi(q_s) e_s
 *     dL/dphi(k_t) = Sh_t v_t + zh_t,   dL/dv_t = Sh_t^T phi(k_t)
 *   and dL/dS_in = Sh_1, dL/dz_in = zh_1.
 * phi'(x) = 1 (x > 0), e^x (x <= 0), the derivative of the piecewise form of
 * [P2] "La función ELU + 1"; both branches give 1 at x = 0.
 * The clamp passes the gradient when den_t >= eps (it is inactive there) and
 * blocks it below eps, as clamp_min does in the pages' examples.           */
static double dphi(double x) { return x > 0.0 ? 1.0 : exp(x); }

typedef struct {
    const double *q, *k, *v, *dy;
    double *dq, *dk, *dvv;
    const double *S_in, *z_in;
    double *dS_in, *dz_in;
    int BH, N, d, dv;
    double eps;
    const double *gamma;   /* nullable: per-head decay */
    int h_begin, h_end;
} bjob_t;

static void head_backward(const bjob_t *J, int h)
{
    const int N = J->N, d = J->d, dv = J->dv;
    const double *q = J->q + (long)h * N * d, *k = J->k + (long)h * N * d;
    const double *v = J->v + (long)h * N * dv, *dy = J->dy + (long)h * N * dv;
    double *dq = J->dq + (long)h * N * d, *dk = J->dk + (long)h * N * d;
    double *dvv = J->dvv + (long)h * N * dv;
    double *S = calloc((size_t)d * dv, sizeof(double));
    double *z = calloc((size_t)d, sizeof(double));
    double *fk = malloc(sizeof(double) * d), *fq = malloc(sizeof(double) * d);
    double *y = malloc(sizeof(double) * dv);
    double *g = malloc(sizeof(double) * ((size_t)N * dv + 1));  /* g_t for every t */
    double *e = malloc(sizeof(double) * ((size_t)N + 1));       /* e_t for every t */
    if (J->S_in) memcpy(S, J->S_in + (long)h * d * dv, sizeof(double) * d * dv);
    if (J->z_in) memcpy(z, J->z_in + (long)h * d, sizeof(double) * d);
    const double gam = J->gamma ? J->gamma[h] : 1.0;
    /* forward in t: the state after token t, then dL/dphi(q_t) */
    for (int t = 0; t < N; ++t) {
        for (int a = 0; a < d; ++a) fk[a] = phi(k[(long)t * d + a]);
        if (J->gamma)
            for (int a = 0; a < d; ++a) {
                for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= gam;
                z[a] *= gam;
            }
        for (int a = 0; a < d; ++a) {
            for (int b = 0; b < dv; ++b) S[(long)a * dv + b] += fk[a] * v[(long)t * dv + b];
            z[a] += fk[a];
        }
        for (int a = 0; a < d; ++a) fq[a] = phi(q[(long)t * d + a]);
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += fq[a] * z[a];
        const double D = clamp_den(den, J->eps);
        double dyy = 0.0;
        for (int b = 0; b < dv; ++b) {
            double num = 0.0;
            for (int a = 0; a < d; ++a) num += fq[a] * S[(long)a * dv + b];
            y[b] = num / D;
            dyy += dy[(long)t * dv + b] * y[b];
        }
        for (int b = 0; b < dv; ++b) g[(long)t * dv + b] = dy[(long)t * dv + b] / D;
        e[t] = den >= J->eps ? -dyy / D : 0.0;
        for (int a = 0; a < d; ++a) {
            double s = z[a] * e[t];
            for (int b = 0; b < dv; ++b) s += S[(long)a * dv + b] * g[(long)t * dv + b];
            dq[(long)t * d + a] = s * dphi(q[(long)t * d + a]);
        }
    }
    /* backward in t: Sh, zh include token t itself (y_s reads S_s for s >= t);
     * with a decay, S_s holds phi(k_t) v_t^T times gamma^(s-t), so
     * Sh_t = phi(q_t) g_t^T + gamma Sh_{t+1}                                  */
    memset(S, 0, sizeof(double) * d * dv);
    memset(z, 0, sizeof(double) * d);
    for (int t = N - 1; t >= 0; --t) {
        for (int a = 0; a < d; ++a) fq[a] = phi(q[(long)t * d + a]);
        if (J->gamma)
            for (int a = 0; a < d; ++a) {
                for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= gam;
                z[a] *= gam;
            }
        for (int a = 0; a < d; ++a) {
            for (int b = 0; b < dv; ++b) S[(long)a * dv + b] += fq[a] * g[(long)t * dv + b];
            z[a] += fq[a] * e[t];
        }
        for (int a = 0; a < d; ++a) fk[a] = phi(k[(long)t * d + a]);
        for (int a = 0; a < d; ++a) {
            double s = z[a];
            for (int b = 0; b < dv; ++b) s += S[(long)a * dv + b] * v[(long)t * dv + b];
            dk[(long)t * d + a] = s * dphi(k[(long)t * d + a]);
        }
        for (int b = 0; b < dv; ++b) {
            double s = 0.0;
            for (int a = 0; a < d; ++a) s += S[(long)a * dv + b] * fk[a];
            dvv[(long)t * dv + b] = s;
        }
    }
    /* S_t holds S_in times gamma^(t+1): dL/dS_in = gamma Sh_1 */
    if (J->dS_in)
        for (long i = 0; i < (long)d * dv; ++i) J->dS_in[(long)h * d * dv + i] = gam * S[i];
    if (J->dz_in)
        for (int a = 0; a < d; ++a) J->dz_in[(long)h * d + a] = gam * z[a];
    free(S); free(z); free(fk); free(fq); free(y); free(g); free(e);
}

static void *bworker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    for (int h = J->h_begin; h < J->h_end; ++h) head_backward(J, h);
    return NULL;
}

/* Gradients of sum_t dy_t . y_t for the causal recurrent form.  q, k, dq, dk:
 * [BH][N][d]; v, dy, dvv: [BH][N][dv].  S_in/z_in may be NULL (zero state);
 * dS_in [BH][d][dv] and dz_in [BH][d] may be NULL.  Returns 0 on success.   */
int oracle_causal_backward_decay(const double *q, const double *k, const double *v,
                                 const double *dy, double *dq, double *dk, double *dvv,
                                 int BH, int N, int d, int dv, double eps, const double *gamma,
                                 const double *S_in, const double *z_in,
                                 double *dS_in, double *dz_in, int nthreads);

int oracle_causal_backward(const double *q, const double *k, const double *v,
                           const double *dy, double *dq, double *dk, double *dvv,
                           int BH, int N, int d, int dv, double eps,
                           const double *S_in, const double *z_in,
                           double *dS_in, double *dz_in, int nthreads)
{
    return oracle_causal_backward_decay(q, k, v, dy, dq, dk, dvv, BH, N, d, dv, eps, NULL,
                                        S_in, z_in, dS_in, dz_in, nthreads);
}

/* The same with a per-head decay gamma[BH] (NULL: none), the gradients of
 * the recurrence S_t = gamma S_{t-1} + phi(k_t) v_t^T, z_t likewise.        */
int oracle_causal_backward_decay(const double *q, const double *k, const double *v,
                                 const double *dy, double *dq, double *dk, double *dvv,
                                 int BH, int N, int d, int dv, double eps, const double *gamma,
                                 const double *S_in, const double *z_in,
                                 double *dS_in, double *dz_in, int nthreads)
{
    if (BH < 0 || N < 0 || d <= 0 || dv <= 0) return 1;
    bjob_t base = {0};
    base.q = q; base.k = k; base.v = v; base.dy = dy; base.dq = dq; base.dk = dk;
    base.dvv = dvv; base.S_in = S_in; base.z_in = z_in; base.dS_in = dS_in;
    base.dz_in = dz_in; base.BH = BH; base.N = N; base.d = d; base.dv = dv; base.eps = eps;
    base.gamma = gamma;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = BH > 0 ? BH : 1;
    bjob_t *jobs = malloc(sizeof(bjob_t) * nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].h_begin = (int)((long)BH * t / nthreads);
        jobs[t].h_end = (int)((long)BH * (t + 1) / nthreads);
    }
    char *joined = calloc((size_t)nthreads, 1);
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, bworker, &jobs[t]) == 0) joined[t] = 1;
        else bworker(&jobs[t]); /* fall back to running it on this thread */
    bworker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t]) pthread_join(th[t], NULL);
    free(joined);
    free(jobs); free(th);
    return 0;
}
