/*
 * HSTU jagged causal attention -- fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never calls it and shares no code with it.
 *
 * What it computes (ai6s.net "HSTU fused operator" post, section 1, the
 * HSTU formula and its PyTorch definition; section 3.2, the block mask is
 * a lower-triangular mask including the diagonal; section 4.2, jagged
 * values + offsets storage; HSTU paper section 3.1, pointwise aggregated
 * attention without softmax normalisation):
 *
 *   for every sequence b, head h and local row i in [0, n_b), t = off[b] + i:
 *     out[t,h,:] = inv_n * sum_{j=0..i} silu(alpha * <q[t,h,:], k[off[b]+j,h,:]>)
 *                                       * v[off[b]+j,h,:]
 *   silu(x) = x / (1 + exp(-x))
 *
 * Inputs are fp32 arrays that hold bf16-rounded values (exact in fp32 and in
 * fp64); every product and sum is taken in fp64 in plain loops, in the order
 * of the formula.  Masked terms (j > i) are never formed, which equals
 * multiplying them by zero for finite inputs.
 *
 * Layout: q, k, v, out are row-major (total, heads, d); offsets has batch+1
 * non-decreasing entries starting at 0.
 *
 * Candidate (M-FALCON) variant (HSTU paper section 3.4 and Appendix H,
 * Algorithm 1 steps 4-5): the last num_targets[b] tokens of sequence b are
 * ranking candidates.  With hist = n_b - num_targets[b], the causal mask is
 * further restricted at positions i, j >= hist with i != j, so a candidate
 * sees every history token and itself but no other candidate:
 *
 *     term j of row i is kept  iff  j <= i  and  (j < hist or j == i).
 *
 * With no candidates (hist = n_b) this is the causal formula above.
 *
 * hstu_oracle_fwd_rab_f64 adds the relative attention bias rab_{p,t}
 * (see rab_t) to the scores; hstu_oracle_norm_gate_f64 (at the end of the
 * file) applies the HSTU layer's output stage, Norm(A V) (.) U, to rows the
 * functions above made.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* silu(x) = x * sigmoid(x) = x / (1 + e^{-x}).  For x -> -inf, e^{-x}
 * overflows to +inf and the quotient is -0, which is the limit. */
double hstu_oracle_silu(double x) { return x / (1.0 + exp(-x)); }

/*
 * Relative attention bias rab_{p,t} (HSTU paper section 3: a bias that
 * merges relative position p and time t, added inside the attention's
 * nonlinearity; section 3.4: M-FALCON modifies it for candidates; Appendix G
 * fuses its construction into the attention operator).  The construction
 * is lost in extraction; the plain reading taken, in the style of bucketed
 * relative position biases:
 *
 *   bias(i, j) = pos[min(floor(log2(dp + 1)), npos - 1)]
 *              + time[min(floor(log2(dt + 1)), ntime - 1)]
 *   dp = p(i) - p(j),  dt = max(ts[i] - ts[j], 0)
 *
 * with p(i) = i for history tokens and p(i) = hist for every candidate: a
 * candidate sits right after the history, as in its own causal pass
 * (Appendix H), so the identity one pass == separate causal passes holds
 * with the bias too.  The bias is added to the scaled score:
 * silu(alpha * <q_i, k_j> + bias(i, j)).
 */
typedef struct {
    const int64_t* ts;  /* timestamp per token */
    const float* pos;   /* npos entries */
    int npos;
    const float* time;  /* ntime entries */
    int ntime;
} rab_t;

/* floor(log2(x)) for x >= 1, by halving. */
static int floor_log2_u64(uint64_t x) {
    int r = 0;
    while (x > 1) {
        x >>= 1;
        ++r;
    }
    return r;
}

int hstu_oracle_rab_bucket(int64_t delta, int nbuckets) {
    if (delta < 0) delta = 0;
    const int b = floor_log2_u64((uint64_t)delta + 1);
    return b < nbuckets - 1 ? b : nbuckets - 1;
}

/* The position and time buckets of pair (i, j) (sequence-local). */
static void rab_buckets(const rab_t* R, int64_t seq_start, int64_t i, int64_t j, int64_t hist,
                        int* bp, int* bt) {
    const int64_t pi = i < hist ? i : hist, pj = j < hist ? j : hist;
    *bp = hstu_oracle_rab_bucket(pi - pj, R->npos);
    *bt = hstu_oracle_rab_bucket(R->ts[seq_start + i] - R->ts[seq_start + j], R->ntime);
}

static double rab_bias(const rab_t* R, int64_t seq_start, int64_t i, int64_t j, int64_t hist) {
    int bp, bt;
    rab_buckets(R, seq_start, i, j, hist, &bp, &bt);
    return (double)R->pos[bp] + (double)R->time[bt];
}

/* Term j of row i is kept (sequence-local indices): the causal mask, and a
 * candidate (i >= hist) sees no other candidate. */
static int kept(int64_t i, int64_t j, int64_t hist) { return j <= i && (j < hist || j == i); }

/* One output row: out_row[c] for c < d, fp64.  hist: the number of history
 * tokens of the sequence (its length when it has no candidates).  R: the
 * relative attention bias, or NULL. */
static void oracle_row(const float* q, const float* k, const float* v, const rab_t* R,
                       int64_t seq_start, int64_t i, int64_t hist, int heads, int d, int h,
                       double alpha, double inv_n, double* acc /* d doubles, scratch */,
                       double* out_row) {
    const int64_t t = seq_start + i;
    const float* qr = q + (t * heads + h) * (int64_t)d;
    for (int c = 0; c < d; ++c) acc[c] = 0.0;
    for (int64_t j = 0; j <= i; ++j) {
        if (!kept(i, j, hist)) continue;
        const int64_t s = seq_start + j;
        const float* kr = k + (s * heads + h) * (int64_t)d;
        const float* vr = v + (s * heads + h) * (int64_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += (double)qr[c] * (double)kr[c];
        const double bias = R ? rab_bias(R, seq_start, i, j, hist) : 0.0;
        const double p = hstu_oracle_silu(alpha * dot + bias);
        for (int c = 0; c < d; ++c) acc[c] += p * (double)vr[c];
    }
    for (int c = 0; c < d; ++c) out_row[c] = inv_n * acc[c];
}

typedef struct {
    const float *q, *k, *v;
    const int64_t* offsets;
    const int64_t* num_targets; /* candidates per sequence, or NULL: none */
    const rab_t* rab;           /* relative attention bias, or NULL: none */
    int batch, heads, d;
    double alpha, inv_n;
    double* out;
    /* row-sample mode: rows_t/rows_h/nrows set, out is (nrows, d) */
    const int64_t* rows_t;
    const int32_t* rows_h;
    int64_t nrows;
    /* shared work counter */
    pthread_mutex_t* mu;
    int64_t* next;
} job_t;

static int64_t take(job_t* J, int64_t chunk) {
    pthread_mutex_lock(J->mu);
    int64_t w = *J->next;
    *J->next += chunk;
    pthread_mutex_unlock(J->mu);
    return w;
}

/* Locate the sequence that holds token t (linear scan: plain, not fast). */
static int seq_of(const int64_t* offsets, int batch, int64_t t) {
    for (int b = 0; b < batch; ++b)
        if (t >= offsets[b] && t < offsets[b + 1]) return b;
    return -1;
}

static int64_t hist_of(const job_t* J, int b) {
    const int64_t n = J->offsets[b + 1] - J->offsets[b];
    return J->num_targets ? n - J->num_targets[b] : n;
}

static void* worker_full(void* arg) {
    job_t* J = (job_t*)arg;
    double* acc = (double*)malloc(sizeof(double) * (size_t)J->d);
    const int64_t units = (int64_t)J->batch * J->heads;
    for (;;) {
        const int64_t u = take(J, 1);
        if (u >= units) break;
        const int b = (int)(u / J->heads), h = (int)(u % J->heads);
        const int64_t s0 = J->offsets[b], n = J->offsets[b + 1] - J->offsets[b];
        const int64_t hist = hist_of(J, b);
        for (int64_t i = 0; i < n; ++i)
            oracle_row(J->q, J->k, J->v, J->rab, s0, i, hist, J->heads, J->d, h, J->alpha, J->inv_n, acc,
                       J->out + ((s0 + i) * J->heads + h) * (int64_t)J->d);
    }
    free(acc);
    return NULL;
}

static void* worker_rows(void* arg) {
    job_t* J = (job_t*)arg;
    double* acc = (double*)malloc(sizeof(double) * (size_t)J->d);
    for (;;) {
        const int64_t r = take(J, 1);
        if (r >= J->nrows) break;
        const int64_t t = J->rows_t[r];
        const int b = seq_of(J->offsets, J->batch, t);
        double* o = J->out + r * (int64_t)J->d;
        if (b < 0) { /* token outside every sequence: not a row */
            for (int c = 0; c < J->d; ++c) o[c] = NAN;
            continue;
        }
        const int64_t s0 = J->offsets[b];
        oracle_row(J->q, J->k, J->v, J->rab, s0, t - s0, hist_of(J, b), J->heads, J->d, J->rows_h[r],
                   J->alpha, J->inv_n, acc, o);
    }
    free(acc);
    return NULL;
}

static int run(job_t* J, int nthreads, void* (*fn)(void*)) {
    pthread_mutex_t mu = PTHREAD_MUTEX_INITIALIZER;
    int64_t next = 0;
    J->mu = &mu;
    J->next = &next;
    if (nthreads < 1) nthreads = 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, fn, J) == 0) ++started;
    if (started == 0) fn(J); /* could not start threads: run inline */
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return 0;
}

static int check_offsets(const int64_t* offsets, int batch) {
    if (batch < 0 || !offsets) return -1;
    if (offsets[0] != 0) return -1;
    for (int b = 0; b < batch; ++b)
        if (offsets[b + 1] < offsets[b]) return -1;
    return 0;
}

/* 0 <= num_targets[b] <= n_b for every sequence (NULL: no candidates). */
static int check_targets(const int64_t* offsets, const int64_t* num_targets, int batch) {
    if (!num_targets) return 0;
    for (int b = 0; b < batch; ++b)
        if (num_targets[b] < 0 || num_targets[b] > offsets[b + 1] - offsets[b]) return -1;
    return 0;
}

/* Every row of every sequence.  out: (total, heads, d) fp64.  Returns 0 or -1. */
int hstu_oracle_fwd_f64(const float* q, const float* k, const float* v, const int64_t* offsets,
                        int batch, int heads, int d, double alpha, double inv_n, double* out,
                        int nthreads) {
    if (check_offsets(offsets, batch) || heads < 1 || d < 1) return -1;
    job_t J = {q, k, v, offsets, NULL, NULL, batch, heads, d, alpha, inv_n, out, NULL, NULL, 0, NULL,
               NULL};
    return run(&J, nthreads, worker_full);
}

/* Selected rows only: row r is token rows_t[r], head rows_h[r]; out: (nrows, d) fp64.
 * A token that lies in no sequence yields a row of NaN. */
int hstu_oracle_rows_f64(const float* q, const float* k, const float* v, const int64_t* offsets,
                         int batch, int heads, int d, double alpha, double inv_n,
                         const int64_t* rows_t, const int32_t* rows_h, int64_t nrows, double* out,
                         int nthreads) {
    if (check_offsets(offsets, batch) || heads < 1 || d < 1 || nrows < 0) return -1;
    job_t J = {q, k, v, offsets, NULL, NULL, batch, heads, d, alpha, inv_n, out, rows_t, rows_h, nrows,
               NULL, NULL};
    return run(&J, nthreads, worker_rows);
}

/* Candidate variant of hstu_oracle_fwd_f64: the last num_targets[b] tokens of
 * sequence b are candidates (see the header). */
int hstu_oracle_fwd_targets_f64(const float* q, const float* k, const float* v,
                                const int64_t* offsets, const int64_t* num_targets, int batch,
                                int heads, int d, double alpha, double inv_n, double* out,
                                int nthreads) {
    if (check_offsets(offsets, batch) || check_targets(offsets, num_targets, batch) ||
        heads < 1 || d < 1)
        return -1;
    job_t J = {q, k, v, offsets, num_targets, NULL, batch, heads, d, alpha, inv_n, out, NULL, NULL, 0,
               NULL, NULL};
    return run(&J, nthreads, worker_full);
}

/* Candidate variant of hstu_oracle_rows_f64. */
int hstu_oracle_rows_targets_f64(const float* q, const float* k, const float* v,
                                 const int64_t* offsets, const int64_t* num_targets, int batch,
                                 int heads, int d, double alpha, double inv_n,
                                 const int64_t* rows_t, const int32_t* rows_h, int64_t nrows,
                                 double* out, int nthreads) {
    if (check_offsets(offsets, batch) || check_targets(offsets, num_targets, batch) ||
        heads < 1 || d < 1 || nrows < 0)
        return -1;
    job_t J = {q, k, v, offsets, num_targets, NULL, batch, heads, d, alpha, inv_n, out, rows_t, rows_h,
               nrows, NULL, NULL};
    return run(&J, nthreads, worker_rows);
}

/* With the relative attention bias (see rab_t): ts has one timestamp per
 * token, pos npos >= 1 and time ntime >= 1 entries.  num_targets may be
 * NULL (no candidates).  Otherwise as hstu_oracle_fwd_targets_f64. */
int hstu_oracle_fwd_rab_f64(const float* q, const float* k, const float* v, const int64_t* offsets,
                            const int64_t* num_targets, const int64_t* ts, const float* pos,
                            int npos, const float* time, int ntime, int batch, int heads, int d,
                            double alpha, double inv_n, double* out, int nthreads) {
    if (check_offsets(offsets, batch) || (num_targets && check_targets(offsets, num_targets, batch)) ||
        heads < 1 || d < 1 || npos < 1 || ntime < 1)
        return -1;
    const rab_t R = {ts, pos, npos, time, ntime};
    job_t J = {q, k, v, offsets, num_targets, &R, batch, heads, d, alpha, inv_n, out, NULL, NULL, 0,
               NULL, NULL};
    return run(&J, nthreads, worker_full);
}

/* Sampled rows with the relative attention bias. */
int hstu_oracle_rows_rab_f64(const float* q, const float* k, const float* v,
                             const int64_t* offsets, const int64_t* num_targets, const int64_t* ts,
                             const float* pos, int npos, const float* time, int ntime, int batch,
                             int heads, int d, double alpha, double inv_n, const int64_t* rows_t,
                             const int32_t* rows_h, int64_t nrows, double* out, int nthreads) {
    if (check_offsets(offsets, batch) || (num_targets && check_targets(offsets, num_targets, batch)) ||
        heads < 1 || d < 1 || nrows < 0 || npos < 1 || ntime < 1)
        return -1;
    const rab_t R = {ts, pos, npos, time, ntime};
    job_t J = {q, k, v, offsets, num_targets, &R, batch, heads, d, alpha, inv_n, out, rows_t, rows_h,
               nrows, NULL, NULL};
    return run(&J, nthreads, worker_rows);
}

/*
 * Backward pass (HSTU paper Appendix G: the backward recomputes the
 * attention; its gradients are those of the forward definition above).
 * With s_ij = alpha <q_i, k_j> (+ bias), P_ij = inv_n silu(s_ij) on kept
 * pairs and out_i = sum_j P_ij v_j, the chain rule gives, for dO = d out:
 *
 *   dv_j  = sum_i P_ij do_i
 *   dp_ij = <do_i, v_j>
 *   ds_ij = inv_n silu'(s_ij) dp_ij,   silu'(x) = sig(x) (1 + x (1 - sig(x)))
 *   dq_i  = alpha sum_j ds_ij k_j
 *   dk_j  = alpha sum_i ds_ij q_i
 *
 * summed over kept pairs only (the same mask as the forward, candidates
 * included).  All in fp64 from the bf16-valued fp32 inputs.
 */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void* worker_bwd(void* arg);

typedef struct {
    job_t base;          /* q, k, v, offsets, num_targets, rab, batch, heads, d, alpha, inv_n */
    const float* dout;   /* (total, heads, d) */
    double *dq, *dk, *dv;
    double *dpos, *dtime; /* the bias tables' gradients (npos, ntime), or NULL */
} bwd_job_t;

/* The terms of pair (i, j) (sequence-local, kept): P_ij and ds_ij. */
static void bwd_terms(const job_t* J, const float* dout, int64_t s0, int64_t hist, int h,
                      int64_t i, int64_t j, double* p_out, double* ds_out) {
    const int d = J->d, heads = J->heads;
    const float* qi = J->q + ((s0 + i) * heads + h) * (int64_t)d;
    const float* doi = dout + ((s0 + i) * heads + h) * (int64_t)d;
    const float* kj = J->k + ((s0 + j) * heads + h) * (int64_t)d;
    const float* vj = J->v + ((s0 + j) * heads + h) * (int64_t)d;
    double dot = 0.0, dp = 0.0;
    for (int c = 0; c < d; ++c) {
        dot += (double)qi[c] * (double)kj[c];
        dp += (double)doi[c] * (double)vj[c];
    }
    const double bias = J->rab ? rab_bias(J->rab, s0, i, j, hist) : 0.0;
    const double x = J->alpha * dot + bias;
    const double sg = sigmoid(x);
    *p_out = J->inv_n * x * sg;
    *ds_out = J->inv_n * sg * (1.0 + x * (1.0 - sg)) * dp;
}

/* The bias tables' gradients: x_ij = alpha q_i.k_j + pos[bp] + time[bt], so
 * d pos[b] = sum of ds_ij over the kept pairs (all heads) whose position
 * bucket is b, and d time likewise by time bucket.  gp, gt: this worker's
 * partial sums. */
static void bwd_seq_head(const bwd_job_t* B, int b, int h, double* gp, double* gt) {
    const job_t* J = &B->base;
    const int64_t s0 = J->offsets[b], n = J->offsets[b + 1] - s0;
    const int64_t hist = hist_of(J, b);
    const int d = J->d, heads = J->heads;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t ti = s0 + i;
        const float* qi = J->q + (ti * heads + h) * (int64_t)d;
        const float* doi = B->dout + (ti * heads + h) * (int64_t)d;
        double* dqi = B->dq + (ti * heads + h) * (int64_t)d;
        for (int64_t j = 0; j < n; ++j) {
            if (!kept(i, j, hist)) continue;
            const int64_t tj = s0 + j;
            const float* kj = J->k + (tj * heads + h) * (int64_t)d;
            double* dkj = B->dk + (tj * heads + h) * (int64_t)d;
            double* dvj = B->dv + (tj * heads + h) * (int64_t)d;
            double p, ds;
            bwd_terms(J, B->dout, s0, hist, h, i, j, &p, &ds);
            if (gp) {
                int bp, bt;
                rab_buckets(J->rab, s0, i, j, hist, &bp, &bt);
                gp[bp] += ds;
                gt[bt] += ds;
            }
            for (int c = 0; c < d; ++c) {
                dvj[c] += p * (double)doi[c];
                dqi[c] += J->alpha * ds * (double)kj[c];
                dkj[c] += J->alpha * ds * (double)qi[c];
            }
        }
    }
}

/* Sequences are independent and a (sequence, head) pair writes only its own
 * rows, so the workers take whole pairs. */
static void* worker_bwd(void* arg) {
    bwd_job_t* B = (bwd_job_t*)arg;
    job_t* J = &B->base;
    const int64_t units = (int64_t)J->batch * J->heads;
    double *gp = NULL, *gt = NULL;
    if (B->dpos) {
        gp = (double*)calloc((size_t)J->rab->npos, sizeof(double));
        gt = (double*)calloc((size_t)J->rab->ntime, sizeof(double));
    }
    for (;;) {
        const int64_t u = take(J, 1);
        if (u >= units) break;
        bwd_seq_head(B, (int)(u / J->heads), (int)(u % J->heads), gp, gt);
    }
    if (gp) { /* this worker's table sums into the totals */
        pthread_mutex_lock(J->mu);
        for (int e = 0; e < J->rab->npos; ++e) B->dpos[e] += gp[e];
        for (int e = 0; e < J->rab->ntime; ++e) B->dtime[e] += gt[e];
        pthread_mutex_unlock(J->mu);
        free(gp);
        free(gt);
    }
    return NULL;
}

/* Sampled gradient rows: for token t = rows_t[r], head h = rows_h[r],
 *   dq[r] = alpha sum_{j: kept(i, j)} ds_ij k_j        (i = t's position)
 *   dk[r] = alpha sum_{i: kept(i, j)} ds_ij q_i        (j = t's position)
 *   dv[r] = sum_{i: kept(i, j)} P_ij do_i
 * each (nrows, d): the same terms as the full backward, summed one row at a
 * time.  num_targets and the rab arguments as hstu_oracle_fwd_rab_f64
 * (NULL: causal, no bias). */
int hstu_oracle_bwd_rows_f64(const float* q, const float* k, const float* v, const float* dout,
                             const int64_t* offsets, const int64_t* num_targets, const int64_t* ts,
                             const float* pos, int npos, const float* time, int ntime, int batch,
                             int heads, int d, double alpha, double inv_n, const int64_t* rows_t,
                             const int32_t* rows_h, int64_t nrows, double* dq, double* dk,
                             double* dv) {
    if (check_offsets(offsets, batch) || (num_targets && check_targets(offsets, num_targets, batch)) ||
        heads < 1 || d < 1 || nrows < 0 || (ts && (npos < 1 || ntime < 1)))
        return -1;
    const rab_t R = {ts, pos, npos, time, ntime};
    job_t J = {q, k, v, offsets, num_targets, ts ? &R : NULL, batch, heads, d, alpha, inv_n, NULL,
               NULL, NULL, 0, NULL, NULL};
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t t = rows_t[r];
        const int h = rows_h[r];
        const int b = seq_of(offsets, batch, t);
        if (b < 0 || h < 0 || h >= heads) return -1;
        const int64_t s0 = offsets[b], n = offsets[b + 1] - s0, pos = t - s0;
        const int64_t hist = hist_of(&J, b);
        double* dqr = dq + r * (int64_t)d;
        double* dkr = dk + r * (int64_t)d;
        double* dvr = dv + r * (int64_t)d;
        for (int c = 0; c < d; ++c) dqr[c] = dkr[c] = dvr[c] = 0.0;
        for (int64_t j = 0; j < n; ++j) {  /* keys of row pos */
            if (!kept(pos, j, hist)) continue;
            double p, ds;
            bwd_terms(&J, dout, s0, hist, h, pos, j, &p, &ds);
            const float* kj = k + ((s0 + j) * heads + h) * (int64_t)d;
            for (int c = 0; c < d; ++c) dqr[c] += alpha * ds * (double)kj[c];
        }
        for (int64_t i = 0; i < n; ++i) {  /* rows that see key pos */
            if (!kept(i, pos, hist)) continue;
            double p, ds;
            bwd_terms(&J, dout, s0, hist, h, i, pos, &p, &ds);
            const float* qi = q + ((s0 + i) * heads + h) * (int64_t)d;
            const float* doi = dout + ((s0 + i) * heads + h) * (int64_t)d;
            for (int c = 0; c < d; ++c) {
                dkr[c] += alpha * ds * (double)qi[c];
                dvr[c] += p * (double)doi[c];
            }
        }
    }
    return 0;
}

/* dq, dk, dv: fp64 (total, heads, d), written (zeroed here first).
 * num_targets and the rab arguments as hstu_oracle_fwd_rab_f64 (ts NULL:
 * no bias); with the bias, dpos and dtime (npos, ntime; may be NULL)
 * receive the tables' gradients. */
int hstu_oracle_bwd_f64(const float* q, const float* k, const float* v, const float* dout,
                        const int64_t* offsets, const int64_t* num_targets, const int64_t* ts,
                        const float* pos, int npos, const float* time, int ntime, int batch,
                        int heads, int d, double alpha, double inv_n, double* dq, double* dk,
                        double* dv, double* dpos, double* dtime, int nthreads) {
    if (check_offsets(offsets, batch) || (num_targets && check_targets(offsets, num_targets, batch)) ||
        heads < 1 || d < 1 || (ts && (npos < 1 || ntime < 1)))
        return -1;
    const int64_t total = batch ? offsets[batch] : 0;
    for (int64_t e = 0; e < total * heads * (int64_t)d; ++e) dq[e] = dk[e] = dv[e] = 0.0;
    const rab_t R = {ts, pos, npos, time, ntime};
    bwd_job_t B;
    job_t J = {q, k, v, offsets, num_targets, ts ? &R : NULL, batch, heads, d, alpha, inv_n, NULL,
               NULL, NULL, 0, NULL, NULL};
    B.base = J;
    B.dout = dout;
    B.dq = dq;
    B.dk = dk;
    B.dv = dv;
    B.dpos = ts ? dpos : NULL;
    B.dtime = ts ? dtime : NULL;
    if (B.dpos) {
        for (int e = 0; e < npos; ++e) dpos[e] = 0.0;
        for (int e = 0; e < ntime; ++e) dtime[e] = 0.0;
    }
    /* run() hands each worker the job pointer; the job is the first member */
    return run(&B.base, nthreads, worker_bwd);
}

/*
 * The HSTU layer's output stage applied to attention rows: Norm(A V) (.) U
 * (HSTU paper section 3, the layer's spatial aggregation followed by the
 * pointwise transformation; section 3.1 requires a layer norm after the
 * pointwise pooling; the feature-interaction paragraph writes the term as
 * Norm(A(X) V(X)) (.) U(X)).  The paper's equations are lost in
 * extraction; the plainest reading is taken:
 *
 *   Norm is a layer norm over one token's attention output with all heads
 *   concatenated (width = heads * d): mean and biased variance over the
 *   width, then (x - mean) / sqrt(var + eps) * gamma + beta, gamma and beta
 *   of that width;
 *   (.) U multiplies elementwise by U, which already went through the
 *   SiLU of the paper's first sub-layer (phi_1 acts on U).
 *
 * x: fp64 (rows, width), the attention output; u: fp32 (rows, width)
 * holding bf16 values; gamma, beta: fp32 (width); y: fp64 (rows, width).
 * Mean and variance are two plain passes over the row in fp64.
 */
int hstu_oracle_norm_gate_f64(const double* x, const float* u, const float* gamma,
                              const float* beta, double eps, int64_t rows, int64_t width,
                              double* y) {
    if (rows < 0 || width < 1 || !(eps >= 0.0)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * width;
        double mean = 0.0;
        for (int64_t c = 0; c < width; ++c) mean += xr[c];
        mean /= (double)width;
        double var = 0.0;
        for (int64_t c = 0; c < width; ++c) var += (xr[c] - mean) * (xr[c] - mean);
        var /= (double)width;
        const double rstd = 1.0 / sqrt(var + eps);
        for (int64_t c = 0; c < width; ++c) {
            const double normed = (xr[c] - mean) * rstd * (double)gamma[c] + (double)beta[c];
            y[r * width + c] = normed * (double)u[r * width + c];
        }
    }
    return 0;
}
