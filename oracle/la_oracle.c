/*
 * la_oracle.c -- fp64 CPU oracle for the Lightning Attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library, and it is deliberately plain: no blocking, no fusion, no
 * reordering beyond the definitions it restates.
 *
 * What it computes (MiniMax-01 deep dive, Hugging Face blog, section
 * "Hybrid Modeling", the four-step mechanism of the 7/8 linear-attention
 * layers; MiniMax-M1 article, "Extractos del reporte tecnico", which calls
 * the layer an I/O-aware linear-attention variant):
 *
 *   step 2  q^ = SiLU(q), k^ = SiLU(k), v^ = SiLU(v)      SiLU(x) = x / (1 + e^-x)
 *   step 3  Y  = Q^ (K^T V)  taken as the causal product with the d x d state
 *              S_t = S_{t-1} + k^_t^T v^_t,   y_t = q^_t S_t    (inclusive: s <= t)
 *           (the O(d^2 n) route the same section contrasts with O(n^2 d))
 *   step 4  out = RMSNorm(Y) * sigmoid(G)
 *              r_t = 1 / sqrt(mean over the H*d features of y_t^2 + eps),
 *              out = y * r_t * 1/(1+e^-g)          (unit RMSNorm weight)
 *
 * Readings of points the pages leave open (listed with reasons in the
 * design notes): the inputs q,k,v,g are the projection outputs before the
 * activation; g gets no SiLU; no 1/sqrt(d) scale; no decay; no q.sum(k)
 * denominator; the norm spans all H*d features of a token.
 *
 * Layouts (row-major): q,k,v,g,y,out [B][N][H][d]; state S [B][H][d][d] with
 * S[i][j] = sum_s k^_s[i] * v^_s[j].
 *
 * Build: gcc -O2 -fPIC -shared -pthread la_oracle.c -o liblaoracle.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ */
/* Step 2 of the mechanism: SiLU, the textbook definition.            */
/* ------------------------------------------------------------------ */
static double silu(double x) { return x / (1.0 + exp(-x)); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

void la_oracle_silu(const double* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = silu(x[i]);
}

/* ------------------------------------------------------------------ */
/* Step 3: the causal linear-attention recurrence, one (b,h) at a time */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *qh, *kh, *vh, *S0;
    double *y, *S_final;
    int B, H, d;
    int64_t N;
    int64_t first, last; /* range of (b*H + h) indices this worker owns */
} core_job;

static void core_one_head(const core_job* jb, int64_t bh) {
    const int H = jb->H, d = jb->d;
    const int64_t N = jb->N;
    const int64_t b = bh / H, h = bh % H;
    double* S = (double*)malloc((size_t)d * d * sizeof(double));
    if (jb->S0)
        memcpy(S, jb->S0 + bh * (int64_t)d * d, (size_t)d * d * sizeof(double));
    else
        memset(S, 0, (size_t)d * d * sizeof(double));

    for (int64_t t = 0; t < N; ++t) {
        const int64_t row = ((b * N + t) * H + h) * (int64_t)d; /* [b][t][h][:] */
        const double* kt = jb->kh + row;
        const double* vt = jb->vh + row;
        /* S_t = S_{t-1} + k_t^T v_t : update first, so the sum is over s <= t */
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) S[i * d + j] += kt[i] * vt[j];
        if (jb->y) {
            const double* qt = jb->qh + row;
            double* yt = jb->y + row;
            /* y_t[j] = sum_i q_t[i] S_t[i][j] */
            for (int j = 0; j < d; ++j) yt[j] = 0.0;
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j) yt[j] += qt[i] * S[i * d + j];
        }
    }
    if (jb->S_final)
        memcpy(jb->S_final + bh * (int64_t)d * d, S, (size_t)d * d * sizeof(double));
    free(S);
}

static void* core_worker(void* arg) {
    const core_job* jb = (const core_job*)arg;
    for (int64_t bh = jb->first; bh < jb->last; ++bh) core_one_head(jb, bh);
    return NULL;
}

static int pick_threads(int nthreads, int64_t work) {
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > work) nthreads = (int)(work > 0 ? work : 1);
    if (nthreads > 512) nthreads = 512;
    return nthreads;
}

/*
 * Core recurrence on already-activated inputs q^, k^, v^ (any values; the
 * identity of step 3).  y may be NULL (state-only pass); S0 may be NULL (zero
 * initial state); S_final may be NULL.  The (b,h) recurrences are independent
 * and are split across threads; each is run in token order.
 * Returns the number of threads used.
 */
int la_oracle_core(const double* qh, const double* kh, const double* vh, const double* S0,
                   int B, int H, int64_t N, int d, double* y, double* S_final, int nthreads) {
    const int64_t work = (int64_t)B * H;
    if (work <= 0) return 0;
    nthreads = pick_threads(nthreads, work);
    pthread_t tid[512];
    core_job jobs[512];
    for (int w = 0; w < nthreads; ++w) {
        core_job* jb = &jobs[w];
        jb->qh = qh; jb->kh = kh; jb->vh = vh; jb->S0 = S0;
        jb->y = y; jb->S_final = S_final;
        jb->B = B; jb->H = H; jb->d = d; jb->N = N;
        jb->first = work * w / nthreads;
        jb->last = work * (w + 1) / nthreads;
    }
    for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, core_worker, &jobs[w]);
    core_worker(&jobs[0]);
    for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
    return nthreads;
}

/* ------------------------------------------------------------------ */
/* Step 4: RMSNorm over each token's H*d features, then the gate      */
/* ------------------------------------------------------------------ */
/*
 * y, g, out are [rows][width] (rows = B*N tokens, width = H*d).  out may alias
 * neither input.  r = 1/sqrt(sum(y^2)/width + eps); out = y * r * sigmoid(g).
 * If rstd is not NULL it receives r per row.
 */
void la_oracle_rmsnorm_gate(const double* y, const double* g, int64_t rows, int width,
                            double eps, double* out, double* rstd) {
    for (int64_t r = 0; r < rows; ++r) {
        const double* yr = y + r * width;
        const double* gr = g + r * width;
        double ss = 0.0;
        for (int c = 0; c < width; ++c) ss += yr[c] * yr[c];
        const double inv = 1.0 / sqrt(ss / (double)width + eps);
        if (rstd) rstd[r] = inv;
        for (int c = 0; c < width; ++c) out[r * width + c] = yr[c] * inv * sigmoid(gr[c]);
    }
}

/* ------------------------------------------------------------------ */
/* The whole layer forward (prefill): steps 2, 3 and 4 in order.      */
/* ------------------------------------------------------------------ */
/*
 * q,k,v,g: raw inputs [B][N][H][d] (before the activation).
 * S0: initial state [B][H][d][d] or NULL (zeros).
 * out: [B][N][H][d]; y (pre-norm, optional) [B][N][H][d]; S_final (optional).
 * Returns 0, or -1 if a scratch allocation failed.
 */
int la_oracle_prefill(const double* q, const double* k, const double* v, const double* g,
                      const double* S0, int B, int H, int64_t N, int d, double eps,
                      double* out, double* y, double* S_final, int nthreads) {
    const int64_t n = (int64_t)B * N * H * d;
    double* qh = (double*)malloc((size_t)n * sizeof(double));
    double* kh = (double*)malloc((size_t)n * sizeof(double));
    double* vh = (double*)malloc((size_t)n * sizeof(double));
    double* yy = y ? y : (double*)malloc((size_t)n * sizeof(double));
    if (!qh || !kh || !vh || !yy) {
        free(qh); free(kh); free(vh);
        if (!y) free(yy);
        return -1;
    }
    la_oracle_silu(q, qh, n);
    la_oracle_silu(k, kh, n);
    la_oracle_silu(v, vh, n);
    la_oracle_core(qh, kh, vh, S0, B, H, N, d, yy, S_final, nthreads);
    la_oracle_rmsnorm_gate(yy, g, (int64_t)B * N, H * d, eps, out, NULL);
    free(qh); free(kh); free(vh);
    if (!y) free(yy);
    return 0;
}

/* ------------------------------------------------------------------ */
/* One-token decode against the carried state.                        */
/* ------------------------------------------------------------------ */
/*
 * S: [B][H][d][d], updated in place (S += k^T v, then y = q S: the same
 * inclusive order as the prefill recurrence).  q,k,v,g,out,y: [B][H][d].
 * y may be NULL.  The norm spans the H*d features of each sequence b.
 */
int la_oracle_decode_step(double* S, const double* q, const double* k, const double* v,
                          const double* g, int B, int H, int d, double eps, double* out,
                          double* y) {
    const int64_t n = (int64_t)B * H * d;
    double* qh = (double*)malloc((size_t)n * sizeof(double));
    double* kh = (double*)malloc((size_t)n * sizeof(double));
    double* vh = (double*)malloc((size_t)n * sizeof(double));
    double* yy = y ? y : (double*)malloc((size_t)n * sizeof(double));
    if (!qh || !kh || !vh || !yy) {
        free(qh); free(kh); free(vh);
        if (!y) free(yy);
        return -1;
    }
    la_oracle_silu(q, qh, n);
    la_oracle_silu(k, kh, n);
    la_oracle_silu(v, vh, n);
    /* A decode step is the recurrence over a sequence of length 1 whose
       initial and final state are the same buffer: [B][1][H][d] == [B][H][d]. */
    double* Snew = (double*)malloc((size_t)B * H * d * d * sizeof(double));
    if (!Snew) {
        free(qh); free(kh); free(vh);
        if (!y) free(yy);
        return -1;
    }
    la_oracle_core(qh, kh, vh, S, B, H, 1, d, yy, Snew, 0);
    memcpy(S, Snew, (size_t)B * H * d * d * sizeof(double));
    la_oracle_rmsnorm_gate(yy, g, B, H * d, eps, out, NULL);
    free(Snew); free(qh); free(kh); free(vh);
    if (!y) free(yy);
    return 0;
}
