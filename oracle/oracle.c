/*
 * oracle.c -- plain, slow, fp64 CPU statement of packed RoPE attention (forward).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes follows hanzo-kernel 0.2.42 packed.rs:
 *   - module doc: qkv [T, 3*H*D] with q | k | v blocks, heads contiguous in each block;
 *     cu [S+1] the first token of each sequence; cos, sin [P, D/2] by position within a
 *     sequence; "window + 1 (0: every key)".
 *   - fn attend_ref ("the composite in f64: rotation, scaled scores, the window, a softmax
 *     over each sequence's keys, the product with the values"): half-split rotation
 *     r[t] = x[t] c - x[t+32] s, r[t+32] = x[t] s + x[t+32] c at the in-sequence position;
 *     score = scale * (q . k) for keys with |i - j| <= w (every key when the window is
 *     off), otherwise -inf; lse = m + ln(sum exp(s - m)); out = sum_j exp(s_j - m)/Z v_j.
 * The score row of each query is materialised in full (the per-sequence score matrix one
 * row at a time), as the reference composite does.
 *
 * The tile schedule (oracle_schedule) states, as a plain sequential walk over the
 * sequences, the tile records the library's device scheduler must reproduce bit for bit.
 * Its first part is packed.rs fn layout (each sequence cut into BR-row tiles at rows
 * 0, BR, 2BR, ...) with the key range clipped to the window (fn attend, key-range
 * clipping); its second part packs short sequences greedily into tiles of at most BR
 * rows.
 *
 * Inputs may be given in fp64, fp32, bf16 (bit patterns) or fp16 (bit patterns); every
 * value is widened to fp64 exactly before use.
 *
 * ORACLE_MUTANT (compile-time, tests only): plants one known mistake so the pin tests can
 * show that they catch it. 0 (default) is the oracle proper.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define HD 64      /* head dimension D */
#define HALF 32    /* D / 2 */

enum { DT_F64 = 0, DT_F32 = 1, DT_BF16 = 2, DT_F16 = 3 };

/* ---------------------------------------------------------------------------------------
 * exact widening of the storage types */

static double half_bits_to_double(uint16_t h) {
    /* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;                /* bfloat16 is the top half of binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double ld(const void *base, int dt, int64_t i) {
    switch (dt) {
    case DT_F64: return ((const double *)base)[i];
    case DT_F32: return (double)((const float *)base)[i];
    case DT_BF16: return bf16_bits_to_double(((const uint16_t *)base)[i]);
    default: return half_bits_to_double(((const uint16_t *)base)[i]);
    }
}

/* ---------------------------------------------------------------------------------------
 * the rotation (packed.rs fn attend_ref, closure `rot`; fn attend, "the query tile,
 * rotated and scaled"): pairs (t, t + 32), angle taken from the tables at `pos`. */

static void rope_row(const void *x, int dt, int64_t at, int64_t pos, const void *cosb,
                     const void *sinb, int tdt, double *y) {
    for (int t = 0; t < HALF; t++) {
        double c = ld(cosb, tdt, pos * HALF + t);
        double s = ld(sinb, tdt, pos * HALF + t);
#if ORACLE_MUTANT == 2
        double x1 = ld(x, dt, at + 2 * t);         /* planted: interleaved pairs (2t, 2t+1) */
        double x2 = ld(x, dt, at + 2 * t + 1);
#else
        double x1 = ld(x, dt, at + t);
        double x2 = ld(x, dt, at + t + HALF);
#endif
#if ORACLE_MUTANT == 1
        y[t] = x1 * c + x2 * s;                    /* planted: rotation by -angle */
        y[t + HALF] = -x1 * s + x2 * c;
#else
        y[t] = x1 * c - x2 * s;
        y[t + HALF] = x1 * s + x2 * c;
#endif
    }
}

void oracle_rope(const void *x, int dt, int64_t pos, const void *cosb, const void *sinb, int tdt,
                 double *y) {
    rope_row(x, dt, 0, pos, cosb, sinb, tdt, y);
}

/* ---------------------------------------------------------------------------------------
 * one query row of one head of one sequence */

typedef struct {
    const void *qkv;
    int dt;
    const void *cosb, *sinb;
    int tdt;
    const uint32_t *cu;
    int S;
    int64_t T;
    int H;
    int window;
    double scale;
} problem;

/* kr: the sequence's rotated keys [L][64]; sc: scratch [L] */
static void one_row(const problem *p, int64_t start, int64_t L, int h, int64_t i, const double *kr,
                    double *sc, double *out_row, double *lse_out) {
    const int64_t ldq = 3 * (int64_t)p->H * HD;
    const int64_t hd = (int64_t)p->H * HD;
    double q[HD];
#if ORACLE_MUTANT == 3
    rope_row(p->qkv, p->dt, (start + i) * ldq + h * HD, start + i, p->cosb, p->sinb, p->tdt, q);
    /* planted: global token index as the position */
#else
    rope_row(p->qkv, p->dt, (start + i) * ldq + h * HD, i, p->cosb, p->sinb, p->tdt, q);
#endif
    double m = -INFINITY;
    for (int64_t j = 0; j < L; j++) {
        int64_t gap = i > j ? i - j : j - i;
#if ORACLE_MUTANT == 4
        int reach = p->window == 0 || gap < p->window;   /* planted: exclusive window */
#else
        int reach = p->window == 0 || gap <= p->window;
#endif
        if (reach) {
            double dot = 0.0;
            for (int d = 0; d < HD; d++) dot += q[d] * kr[j * HD + d];
#if ORACLE_MUTANT == 5
            sc[j] = dot;                                  /* planted: scale dropped */
#else
            sc[j] = p->scale * dot;
#endif
        } else {
            sc[j] = -INFINITY;
        }
        if (sc[j] > m) m = sc[j];
    }
    /* weights exp(s_j - m) (masked keys weigh exp(-inf) = 0), their sum and the lse */
    double z = 0.0;
    for (int64_t j = 0; j < L; j++) {
        sc[j] = exp(sc[j] - m);
        z += sc[j];
    }
#if ORACLE_MUTANT == 6
    *lse_out = m + log2(z);                               /* planted: wrong log base */
#elif ORACLE_MUTANT == 24
    *lse_out = log(z);                                    /* planted: the max left out */
#else
    *lse_out = m + log(z);
#endif
#if ORACLE_MUTANT == 23
    /* planted: the values rotated like the keys */
    double *vr = malloc(sizeof(double) * L * HD);
    if (vr) {
        for (int64_t j = 0; j < L; j++)
            rope_row(p->qkv, p->dt, (start + j) * ldq + 2 * hd + h * HD, j, p->cosb, p->sinb, p->tdt, vr + j * HD);
        for (int d = 0; d < HD; d++) {
            double acc = 0.0;
            for (int64_t j = 0; j < L; j++) acc += sc[j] / z * vr[j * HD + d];
            out_row[d] = acc;
        }
        free(vr);
        return;
    }
#endif
    for (int d = 0; d < HD; d++) {
        double acc = 0.0;
        for (int64_t j = 0; j < L; j++) {
#if ORACLE_MUTANT == 7
            double v = ld(p->qkv, p->dt, (start + j) * ldq + hd + h * HD + d);  /* planted: k for v */
#else
            double v = ld(p->qkv, p->dt, (start + j) * ldq + 2 * hd + h * HD + d);
#endif
            acc += sc[j] / z * v;
        }
        out_row[d] = acc;
    }
}

/* rotated keys of sequence [start, start+L) for head h */
static void rotate_keys(const problem *p, int64_t start, int64_t L, int h, double *kr) {
    const int64_t ldq = 3 * (int64_t)p->H * HD;
    const int64_t hd = (int64_t)p->H * HD;
    for (int64_t j = 0; j < L; j++) {
#if ORACLE_MUTANT == 3
        rope_row(p->qkv, p->dt, (start + j) * ldq + hd + h * HD, start + j, p->cosb, p->sinb,
                 p->tdt, kr + j * HD);
#else
        rope_row(p->qkv, p->dt, (start + j) * ldq + hd + h * HD, j, p->cosb, p->sinb, p->tdt,
                 kr + j * HD);
#endif
    }
}

/* ---------------------------------------------------------------------------------------
 * whole forward: units are (sequence, head) pairs, spread over worker threads */

typedef struct {
    const problem *p;
    double *out, *lse;
    atomic_long next;
    int64_t units;
    int64_t maxlen;
    int failed;
} fwd_job;

static void *fwd_worker(void *arg) {
    fwd_job *job = (fwd_job *)arg;
    const problem *p = job->p;
    double *kr = malloc(sizeof(double) * (size_t)(job->maxlen > 0 ? job->maxlen : 1) * HD);
    double *sc = malloc(sizeof(double) * (size_t)(job->maxlen > 0 ? job->maxlen : 1));
    if (!kr || !sc) {
        job->failed = 1;
        free(kr);
        free(sc);
        return NULL;
    }
    const int64_t hd = (int64_t)p->H * HD;
    for (;;) {
        int64_t u = atomic_fetch_add(&job->next, 1);
        if (u >= job->units) break;
        int s = (int)(u / p->H);
        int h = (int)(u % p->H);
        int64_t start = p->cu[s];
        int64_t L = (int64_t)p->cu[s + 1] - start;
        if (L <= 0) continue;
        rotate_keys(p, start, L, h, kr);
        for (int64_t i = 0; i < L; i++) {
            double l;
            one_row(p, start, L, h, i, kr, sc, job->out + (start + i) * hd + h * HD, &l);
            job->lse[h * p->T + start + i] = l;
        }
    }
    free(kr);
    free(sc);
    return NULL;
}

int oracle_threads(void) {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof set, &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    return 1;
}

static int check_cu(const uint32_t *cu, int S, int64_t T) {
    if (S < 0 || T < 0) return -1;
    if (cu[0] != 0) return -1;
    for (int s = 0; s < S; s++)
        if (cu[s + 1] < cu[s]) return -1;
    if ((int64_t)cu[S] != T) return -1;
    return 0;
}

/*
 * out [T, H*64] and lse [H, T] in fp64. Returns 0, or -1 on malformed arguments (cu not a
 * non-decreasing offset list from 0 to T, H < 1, window < 0), -2 on allocation failure.
 * The caller guarantees cos/sin hold at least max(L) rows.
 */
int oracle_attend(const void *qkv, int dt, const void *cosb, const void *sinb, int tdt,
                  const uint32_t *cu, int S, int64_t T, int H, int window, double scale,
                  double *out, double *lse, int nthreads) {
    if (H < 1 || window < 0 || check_cu(cu, S, T)) return -1;
    problem p = {qkv, dt, cosb, sinb, tdt, cu, S, T, H, window, scale};
    int64_t maxlen = 0;
    for (int s = 0; s < S; s++) {
        int64_t L = (int64_t)cu[s + 1] - cu[s];
        if (L > maxlen) maxlen = L;
    }
    fwd_job job;
    job.p = &p;
    job.out = out;
    job.lse = lse;
    atomic_init(&job.next, 0);
    job.units = (int64_t)S * H;
    job.maxlen = maxlen;
    job.failed = 0;
    if (nthreads <= 0) nthreads = oracle_threads();
    if (nthreads > 1024) nthreads = 1024;
    pthread_t tid[1024];
    int started = 0;
    for (int k = 1; k < nthreads; k++) {
        if (pthread_create(&tid[started], NULL, fwd_worker, &job) == 0) started++;
    }
    fwd_worker(&job);
    for (int k = 0; k < started; k++) pthread_join(tid[k], NULL);
    return job.failed ? -2 : 0;
}

/*
 * Selected rows only: for each n, token rows_tok[n] and head rows_head[n]; writes
 * out_rows [n, 64] and lse_rows [n]. Each row is computed on its own (its sequence's keys
 * rotated afresh), so any row of a workload of any size can be checked one by one.
 */
typedef struct {
    const problem *p;
    const int64_t *tok;
    const int32_t *head;
    int64_t n;
    double *out_rows, *lse_rows;
    atomic_long next;
    int failed;
} rows_job;

static int64_t seq_of(const uint32_t *cu, int S, int64_t a) {
    /* the sequence holding token a: largest s with cu[s] <= a and a < cu[s+1] */
    int64_t lo = 0, hi = S; /* answer in [lo, hi) */
    while (hi - lo > 1) {
        int64_t mid = (lo + hi) / 2;
#if ORACLE_MUTANT == 27
        if ((int64_t)cu[mid] < a) lo = mid; else hi = mid;  /* planted: a sequence's first token given to the one before */
#else
        if ((int64_t)cu[mid] <= a) lo = mid; else hi = mid;
#endif
    }
#if ORACLE_MUTANT != 27
    while (lo < S && (int64_t)cu[lo + 1] <= a) lo++;   /* step over empty sequences */
#endif
    return lo;
}

static void *rows_worker(void *arg) {
    rows_job *job = (rows_job *)arg;
    const problem *p = job->p;
    for (;;) {
        int64_t n = atomic_fetch_add(&job->next, 1);
        if (n >= job->n) break;
        int64_t a = job->tok[n];
#if ORACLE_MUTANT == 28
        int h = 0;                                       /* planted: the row's head ignored */
#else
        int h = job->head[n];
#endif
        int64_t s = seq_of(p->cu, p->S, a);
        int64_t start = p->cu[s];
        int64_t L = (int64_t)p->cu[s + 1] - start;
        double *kr = malloc(sizeof(double) * (size_t)L * HD);
        double *sc = malloc(sizeof(double) * (size_t)L);
        if (!kr || !sc) {
            job->failed = 1;
            free(kr);
            free(sc);
            continue;
        }
        rotate_keys(p, start, L, h, kr);
        one_row(p, start, L, h, a - start, kr, sc, job->out_rows + n * HD, job->lse_rows + n);
        free(kr);
        free(sc);
    }
    return NULL;
}

int oracle_attend_rows(const void *qkv, int dt, const void *cosb, const void *sinb, int tdt,
                       const uint32_t *cu, int S, int64_t T, int H, int window, double scale,
                       const int64_t *rows_tok, const int32_t *rows_head, int64_t n,
                       double *out_rows, double *lse_rows, int nthreads) {
    if (H < 1 || window < 0 || check_cu(cu, S, T)) return -1;
    for (int64_t k = 0; k < n; k++)
        if (rows_tok[k] < 0 || rows_tok[k] >= T || rows_head[k] < 0 || rows_head[k] >= H) return -1;
    problem p = {qkv, dt, cosb, sinb, tdt, cu, S, T, H, window, scale};
    rows_job job;
    job.p = &p;
    job.tok = rows_tok;
    job.head = rows_head;
    job.n = n;
    job.out_rows = out_rows;
    job.lse_rows = lse_rows;
    atomic_init(&job.next, 0);
    job.failed = 0;
    if (nthreads <= 0) nthreads = oracle_threads();
    if (nthreads > 1024) nthreads = 1024;
    pthread_t tid[1024];
    int started = 0;
    for (int k = 1; k < nthreads; k++)
        if (pthread_create(&tid[started], NULL, rows_worker, &job) == 0) started++;
    rows_worker(&job);
    for (int k = 0; k < started; k++) pthread_join(tid[k], NULL);
    return job.failed ? -2 : 0;
}

/* ---------------------------------------------------------------------------------------
 * the standalone rotation (the pages' rope op: the first `dims` features of a head vector
 * rotated in pairs -- the two halves, or interleaved pairs ("traditional") -- forwards, or
 * inversely for the gradient; kime's rope step applies it to the q and k of a packed qkv)
 *
 * For a head vector x (64 features) at in-sequence position p, with h = dims / 2 and table
 * entries c_j = cos[p h + j], s_j = sin[p h + j] (tables of width h):
 *   pair j < h: (a, b) = (j, j + h) for the halves, (2j, 2j + 1) for interleaved pairs
 *   forward:  y_a = x_a c_j - x_b s_j,   y_b = x_a s_j + x_b c_j
 *   inverse:  y_a = x_a c_j + x_b s_j,   y_b = x_b c_j - x_a s_j   (the transposed rotation)
 *   features dims .. 63 are copied.
 */
static void rope_vector(const void *x, int dt, int64_t at, int64_t pos, const void *cosb, const void *sinb,
                        int tdt, int dims, int traditional, int inverse, double *y) {
    const int h = dims / 2;
    for (int f = dims; f < HD; f++) y[f] = ld(x, dt, at + f);
#if ORACLE_MUTANT == 14
    for (int f = dims; f < HD; f++) y[f] = 0.0;                    /* planted: tail not copied */
#endif
    for (int j = 0; j < h; j++) {
#if ORACLE_MUTANT == 13
        int a = j, b = j + h;                                      /* planted: layout ignored */
#elif ORACLE_MUTANT == 21
        int a = traditional ? 2 * j : j;
        int b = traditional ? 2 * j + 1 : j + HD / 2;              /* planted: pairs across the head */
#else
        int a = traditional ? 2 * j : j;
        int b = traditional ? 2 * j + 1 : j + h;
#endif
#if ORACLE_MUTANT == 22
        double c = ld(sinb, tdt, pos * h + j), sn = ld(cosb, tdt, pos * h + j);  /* planted: swapped */
#else
        double c = ld(cosb, tdt, pos * h + j), sn = ld(sinb, tdt, pos * h + j);
#endif
        double xa = ld(x, dt, at + a), xb = ld(x, dt, at + b);
#if ORACLE_MUTANT == 12
        int fwd = 1;                                               /* planted: direction ignored */
#else
        int fwd = !inverse;
#endif
        if (fwd) {
            y[a] = xa * c - xb * sn;
            y[b] = xa * sn + xb * c;
        } else {
            y[a] = xa * c + xb * sn;
            y[b] = xb * c - xa * sn;
        }
    }
}

/*
 * Every q and k head vector of qkv [T, 3 H 64] rotated at its token's in-sequence position
 * (the token minus the start of its sequence in cu); v copied. y [T, 3 H 64] in f64.
 * Returns 0, or -1 on bad arguments (dims odd or outside [2, 64], H < 1, malformed cu, a
 * position at or past P table rows).
 */
int oracle_rope_qkv(const void *qkv, int dt, const void *cosb, const void *sinb, int tdt, int64_t P,
                    const uint32_t *cu, int S, int64_t T, int H, int dims, int traditional, int inverse,
                    double *y) {
    if (H < 1 || dims < 2 || dims > HD || (dims & 1) || check_cu(cu, S, T)) return -1;
    const int64_t W = 3LL * H * HD;
    for (int sq = 0; sq < S; sq++) {
        for (int64_t t = cu[sq]; t < (int64_t)cu[sq + 1]; t++) {
            const int64_t pos = t - cu[sq];
            if (pos >= P) return -1;
            for (int part = 0; part < 3; part++)
                for (int hh = 0; hh < H; hh++) {
                    const int64_t at = t * W + (int64_t)part * H * HD + (int64_t)hh * HD;
                    if (part == 2) {
                        for (int f = 0; f < HD; f++) y[at + f] = ld(qkv, dt, at + f);
                    } else {
                        rope_vector(qkv, dt, at, pos, cosb, sinb, tdt, dims, traditional, inverse, y + at);
                    }
                }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * the backward pass (the pages' attend_back and its f64 reference): the gradient of
 * L = sum(dout * out) with respect to qkv, through the rotation. Per sequence and head, with
 * q'_i = rot(q_i, i), k'_j = rot(k_j, j), s_ij = scale q'_i . k'_j on visible pairs,
 * P = softmax_j(s), O_i = sum_j P_ij v_j:
 *   D_i = dout_i . O_i,   dP_ij = dout_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
 *   dv_j = sum_i P_ij dout_i,   dq'_i = scale sum_j dS_ij k'_j,   dk'_j = scale sum_i dS_ij q'_i
 *   dq_i = rot^T(dq'_i, i),   dk_j = rot^T(dk'_j, j)   (the transposed rotation)
 * Everything from the inputs in f64 (the forward is recomputed here, not read).
 */
int oracle_attend_backward(const void *qkv, int dt, const void *cosb, const void *sinb, int tdt,
                           const uint32_t *cu, int S, int64_t T, int H, int window, double scale,
                           const void *dout, int ddt, double *dqkv) {
    if (H < 1 || window < 0 || check_cu(cu, S, T)) return -1;
    const int64_t ldq = 3LL * H * HD, hd = (int64_t)H * HD;
    int64_t maxlen = 1;
    for (int sq = 0; sq < S; sq++)
        if ((int64_t)cu[sq + 1] - cu[sq] > maxlen) maxlen = (int64_t)cu[sq + 1] - cu[sq];
    double *qr = malloc(sizeof(double) * maxlen * HD), *kr = malloc(sizeof(double) * maxlen * HD);
    double *dk = malloc(sizeof(double) * maxlen * HD), *dv = malloc(sizeof(double) * maxlen * HD);
    double *pr = malloc(sizeof(double) * maxlen), *dsr = malloc(sizeof(double) * maxlen);
    if (!qr || !kr || !dk || !dv || !pr || !dsr) {
        free(qr); free(kr); free(dk); free(dv); free(pr); free(dsr);
        return -2;
    }
    for (int64_t e = 0; e < T * ldq; e++) dqkv[e] = 0.0;
    for (int sq = 0; sq < S; sq++) {
        const int64_t start = cu[sq], L = (int64_t)cu[sq + 1] - cu[sq];
        if (L <= 0) continue;
        for (int h = 0; h < H; h++) {
            for (int64_t j = 0; j < L; j++) {
                rope_row(qkv, dt, (start + j) * ldq + h * HD, j, cosb, sinb, tdt, qr + j * HD);
                rope_row(qkv, dt, (start + j) * ldq + hd + h * HD, j, cosb, sinb, tdt, kr + j * HD);
            }
            for (int64_t e = 0; e < L * HD; e++) dk[e] = dv[e] = 0.0;
            for (int64_t i = 0; i < L; i++) {
                /* this row's probabilities */
                double m = -INFINITY;
                for (int64_t j = 0; j < L; j++) {
                    int64_t gap = i > j ? i - j : j - i;
                    if (window == 0 || gap <= window) {
                        double dot = 0.0;
                        for (int d = 0; d < HD; d++) dot += qr[i * HD + d] * kr[j * HD + d];
                        pr[j] = scale * dot;
                    } else {
                        pr[j] = -INFINITY;
                    }
                    if (pr[j] > m) m = pr[j];
                }
                double z = 0.0;
                for (int64_t j = 0; j < L; j++) {
                    pr[j] = exp(pr[j] - m);
                    z += pr[j];
                }
#if ORACLE_MUTANT != 20
                for (int64_t j = 0; j < L; j++) pr[j] /= z;
#endif                                                    /* planted (20): not normalised */
                /* D_i = dout_i . O_i */
                double di = 0.0;
                for (int d = 0; d < HD; d++) {
                    double o = 0.0;
                    for (int64_t j = 0; j < L; j++)
                        o += pr[j] * ld(qkv, dt, (start + j) * ldq + 2 * hd + h * HD + d);
                    di += ld(dout, ddt, (start + i) * hd + h * HD + d) * o;
                }
                /* dS_ij, dv, dk' */
                for (int64_t j = 0; j < L; j++) {
                    double dp = 0.0;
                    for (int d = 0; d < HD; d++)
                        dp += ld(dout, ddt, (start + i) * hd + h * HD + d) *
                              ld(qkv, dt, (start + j) * ldq + 2 * hd + h * HD + d);
#if ORACLE_MUTANT == 15
                    dsr[j] = pr[j] * dp;                                  /* planted: D dropped */
#else
                    dsr[j] = pr[j] * (dp - di);
#endif
                    for (int d = 0; d < HD; d++) {
#if ORACLE_MUTANT == 19
                        dv[j * HD + d] += dsr[j] * ld(dout, ddt, (start + i) * hd + h * HD + d);  /* planted */
#else
                        dv[j * HD + d] += pr[j] * ld(dout, ddt, (start + i) * hd + h * HD + d);
#endif
                        dk[j * HD + d] += scale * dsr[j] * qr[i * HD + d];
                    }
                }
                /* dq'_i, rotated back */
                double dq[HD], y[HD];
                for (int d = 0; d < HD; d++) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < L; j++) acc += dsr[j] * kr[j * HD + d];
#if ORACLE_MUTANT == 17
                    dq[d] = acc;                                          /* planted: scale missing */
#else
                    dq[d] = scale * acc;
#endif
                }
#if ORACLE_MUTANT == 18
                rope_vector(dq, DT_F64, 0, i, cosb, sinb, tdt, HD, 0, 0, y);  /* planted: forwards */
#else
                rope_vector(dq, DT_F64, 0, i, cosb, sinb, tdt, HD, 0, 1, y);
#endif
                for (int d = 0; d < HD; d++) dqkv[(start + i) * ldq + h * HD + d] = y[d];
            }
            for (int64_t j = 0; j < L; j++) {
                double y[HD];
#if ORACLE_MUTANT == 16
                rope_vector(dk + j * HD, DT_F64, 0, j, cosb, sinb, tdt, HD, 0, 0, y);  /* planted: forwards */
#else
                rope_vector(dk + j * HD, DT_F64, 0, j, cosb, sinb, tdt, HD, 0, 1, y);
#endif
                for (int d = 0; d < HD; d++) {
                    dqkv[(start + j) * ldq + hd + h * HD + d] = y[d];
                    dqkv[(start + j) * ldq + 2 * hd + h * HD + d] = dv[j * HD + d];
                }
            }
        }
    }
    free(qr); free(kr); free(dk); free(dv); free(pr); free(dsr);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * the tile schedule
 *
 * Records of 8 uint32: {q0, rows, k0, nk, seq, nseq, kind, ktiles}
 *   q0, rows  query tokens [q0, q0 + rows)
 *   k0, nk    key tokens [k0, k0 + nk): every key some row of the tile can see
 *   seq, nseq the sequences [seq, seq + nseq) whose rows the tile holds
 *   kind      0: a BR-row piece of one sequence; 1: a group of whole short sequences
 *   ktiles    ceil(nk / BC)
 * Constants: BR = BC = 128 rows per tile; a sequence is short when its length is at most
 * SHORT = 64. Short (and empty) sequences are grouped within WIN = 1024-token windows
 * [1024 w, 1024 w + 1024), a sequence belonging to the window of its first token: taken in
 * order, they are packed greedily -- a group takes the next sequence while that sequence is
 * short, belongs to the group's window and keeps the group within BR rows; anything else
 * closes it (a group of empty sequences only has no rows and gives no record).
 * Records are listed by increasing q0.
 */
#define SCH_BR 128
#define SCH_BC 128
#define SCH_SHORT 64
#define SCH_WIN 1024
/* capacity unit: at most 3 records per 64 tokens (plus one) */
#define SCH_CAP_UNIT 64

static int64_t emit(uint32_t *tiles, int64_t cap, int64_t nt, int64_t q0, int64_t rows, int64_t k0,
                    int64_t k1, int64_t seq, int64_t nseq, int kind) {
    if (nt < cap) {
        uint32_t *r = tiles + 8 * nt;
        r[0] = (uint32_t)q0;
        r[1] = (uint32_t)rows;
        r[2] = (uint32_t)k0;
        r[3] = (uint32_t)(k1 - k0);
        r[4] = (uint32_t)seq;
        r[5] = (uint32_t)nseq;
        r[6] = (uint32_t)kind;
        r[7] = (uint32_t)((k1 - k0 + SCH_BC - 1) / SCH_BC);
    }
    return nt + 1;
}

/*
 * Writes up to `cap` records to tiles [cap][8] and their total count to *nt. Returns 0, or
 * -1 when cu is malformed (then *nt = 0).
 */
int oracle_schedule(const uint32_t *cu, int S, int64_t T, int window, uint32_t *tiles, int64_t cap,
                    int64_t *nt_out) {
    *nt_out = 0;
    if (window < 0 || check_cu(cu, S, T)) return -1;
    int64_t nt = 0;
    /* the open group of short sequences: window, first member, last member */
    int64_t g_w = -1, g_first = -1, g_last = -1;
    for (int s = 0; s <= S; s++) {
        int64_t start = s < S ? cu[s] : T;
        int64_t L = s < S ? (int64_t)cu[s + 1] - cu[s] : 0;
        int is_short = s < S && L <= SCH_SHORT;
        int64_t w = start / SCH_WIN;
        /* close the open group when this sequence does not join it */
#if ORACLE_MUTANT == 10
        int joins = g_w >= 0 && is_short && w == g_w && start + L - cu[g_first] <= SCH_BR + 1; /* planted */
#elif ORACLE_MUTANT == 11
        int joins = g_w >= 0 && is_short && start + L - cu[g_first] <= SCH_BR;  /* planted: no window */
#else
        int joins = g_w >= 0 && is_short && w == g_w && start + L - cu[g_first] <= SCH_BR;
#endif
        if (g_w >= 0 && !joins) {
            int64_t q0 = cu[g_first];
            int64_t rows = (int64_t)cu[g_last + 1] - q0;
            if (rows > 0)
                nt = emit(tiles, cap, nt, q0, rows, q0, q0 + rows, g_first, g_last - g_first + 1, 1);
            g_w = -1;
        }
        if (s == S) break;
        if (is_short) {
            if (g_w < 0) {
                g_w = w;
                g_first = s;
            }
            g_last = s;
            continue;
        }
        /* a long sequence: packed.rs fn layout's tiles at rows 0, BR, 2BR, ... with the key
         * range of each clipped to the window */
        for (int64_t i0 = 0; i0 < L; i0 += SCH_BR) {
#if ORACLE_MUTANT == 26
            int64_t rows = SCH_BR;                                  /* planted: last piece overruns */
#else
            int64_t rows = L - i0 < SCH_BR ? L - i0 : SCH_BR;
#endif
            int64_t q0 = start + i0;
            int64_t k0 = start, k1 = start + L;
            if (window > 0) {
#if ORACLE_MUTANT == 8
                if (q0 + rows + window - 1 < k1) k1 = q0 + rows + window - 1;  /* planted: short */
                if (q0 - window > k0) k0 = q0 - window;
#elif ORACLE_MUTANT == 9
                if (q0 - window - 1 > k0) k0 = q0 - window - 1;              /* planted: loose */
                if (q0 + rows + window < k1) k1 = q0 + rows + window;
#elif ORACLE_MUTANT == 25
                if (q0 - window > k0) k0 = q0 - window;
                k1 = q0 + rows + window;                     /* planted: not clipped at the end */
#else
                if (q0 - window > k0) k0 = q0 - window;
                if (q0 + rows + window < k1) k1 = q0 + rows + window;
#endif
            }
            nt = emit(tiles, cap, nt, q0, rows, k0, k1, s, 1, 0);
        }
    }
    *nt_out = nt;
    return 0;
}

/* an upper bound on the number of records for T tokens (what a caller should allocate) */
int64_t oracle_schedule_cap(int64_t T) { return 3 * ((T + SCH_CAP_UNIT - 1) / SCH_CAP_UNIT) + 1; }
