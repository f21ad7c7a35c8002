/*
 * gdn_oracle.c -- plain sequential CPU oracle for ReplaySSM-style handling of
 * Gated DeltaNet (GDN) recurrent state under speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header
 * or table with the CUDA library it checks.
 *
 * What it computes (sources: "The inference stack behind OCRia" (LlamaIndex
 * engineering blog), section "Making speculative verification cheaper": per
 * sequence a checkpoint of the GDN state and a short buffer of the inputs
 * committed since; draft outputs come from replaying buffer and draft over the
 * checkpoint, the checkpoint is rewritten only when the buffer is flushed, and
 * a rejection only shortens the buffer; "Inference Engineering", chapter 5,
 * speculative decoding: drafts are accepted up to the first rejected token).
 *
 * The pages do not print the GDN recurrence; it is the gated delta rule of
 * Yang, Kautz & Hatamizadeh, "Gated Delta Networks" (ICLR 2025):
 *     S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t (scale * q_t),  alpha_t = exp(g_t),  scale = 1/sqrt(d_k)
 * with S of shape [d_v, d_k].  Expanding the product gives the rank-one form
 * used below, S_t = alpha S + w k^T with w = beta (v - alpha S k); the test
 * suite checks that expansion against the explicit matrix product.
 *
 * Precision: every quantity is a double.  With fp32_mode set, each single
 * operation is rounded to binary32 right after it is performed in double,
 * which for +, -, * equals the binary32 operation itself; that mode exists
 * only for the bit-exact schedule invariants.  At a flush the state is
 * rounded to binary32 because the checkpoint is stored as fp32.
 *
 * Parity pins (brute force, closed forms, invariants) live in the tests.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, H, dk, dv, T, cap, threshold, n_slot;
    double scale;
    int fp32_mode;
    int n_threads;
} orc_dims;

/* status bits, OR-ed into *status */
#define ORC_BAD_ACCEPT 1   /* accepted count outside [0, T] */
#define ORC_NO_ROOM    2   /* len + T > cap at verify */
#define ORC_BAD_LEN    4   /* len outside [0, cap] (or len + p > cap at accept) */

static double rnd(const orc_dims *d, double x) {
    return d->fp32_mode ? (double)(float)x : x;
}

/* One token of the gated delta rule on one [dv, dk] state, in place.
 * When q is given, o[i] = sum_j S_t[i,j] * (scale * q[j]) with the updated state. */
static void delta_rule_token(const orc_dims *d, double *S,
                             const double *k, const double *v, double g, double beta,
                             const double *q, double *o)
{
    const int dk = d->dk, dv = d->dv;
    const double alpha = rnd(d, exp(g));
    for (int i = 0; i < dv; ++i) {
        double *row = S + (size_t)i * dk;
        double sk = 0.0;                               /* (S_{t-1} k_t)_i */
        for (int j = 0; j < dk; ++j) sk = rnd(d, sk + rnd(d, row[j] * k[j]));
        const double w = rnd(d, beta * rnd(d, v[i] - rnd(d, alpha * sk)));
        for (int j = 0; j < dk; ++j) row[j] = rnd(d, rnd(d, alpha * row[j]) + rnd(d, w * k[j]));
        if (q) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc = rnd(d, acc + rnd(d, row[j] * rnd(d, d->scale * q[j])));
            o[i] = acc;
        }
    }
}

/* Straight sequential run: apply n tokens to S (in place).  Token t reads
 * k + t*k_stride, v + t*v_stride, g[t*gb_stride], beta[t*gb_stride]; when q is
 * non-NULL, the output of token t goes to o + t*o_stride. */
int orc_recur(const orc_dims *d, double *S, int n,
              const double *k, long k_stride, const double *v, long v_stride,
              const double *g, const double *beta, long gb_stride,
              const double *q, long q_stride, double *o, long o_stride)
{
    for (int t = 0; t < n; ++t)
        delta_rule_token(d, S, k + t * k_stride, v + t * v_stride,
                         g[t * gb_stride], beta[t * gb_stride],
                         q ? q + t * q_stride : NULL, q ? o + t * o_stride : NULL);
    return 0;
}

/* ---------------------------------------------------------------- layouts */
/* state    [n_slot, H, dv, dk]      buf_k [n_slot, H, cap, dk]
 * buf_v    [n_slot, H, cap, dv]     buf_g, buf_beta [n_slot, H, cap]
 * q, k     [B, T, H, dk]            v, out [B, T, H, dv]
 * g, beta  [B, T, H]                buf_len [n_slot], state_idx [B] (NULL: identity) */

static size_t st_off(const orc_dims *d, int slot, int h) { return ((size_t)slot * d->H + h) * d->dv * d->dk; }
static size_t bk_off(const orc_dims *d, int slot, int h, int t) { return (((size_t)slot * d->H + h) * d->cap + t) * d->dk; }
static size_t bv_off(const orc_dims *d, int slot, int h, int t) { return (((size_t)slot * d->H + h) * d->cap + t) * d->dv; }
static size_t bg_off(const orc_dims *d, int slot, int h, int t) { return ((size_t)slot * d->H + h) * d->cap + t; }
static size_t dk_off(const orc_dims *d, int b, int t, int h) { return (((size_t)b * d->T + t) * d->H + h) * d->dk; }
static size_t dv_off(const orc_dims *d, int b, int t, int h) { return (((size_t)b * d->T + t) * d->H + h) * d->dv; }
static size_t dg_off(const orc_dims *d, int b, int t, int h) { return ((size_t)b * d->T + t) * d->H + h; }

static int slot_of(const int32_t *state_idx, int b) { return state_idx ? state_idx[b] : b; }

/* ------------------------------------------------------ parallel (b,h) loop */
typedef void (*unit_fn)(void *ctx, int b, int h);
typedef struct { unit_fn fn; void *ctx; int B, H, tid, nthr; } worker_arg;

static void *worker(void *p) {
    worker_arg *a = (worker_arg *)p;
    for (int u = a->tid; u < a->B * a->H; u += a->nthr) a->fn(a->ctx, u / a->H, u % a->H);
    return NULL;
}

static void for_each_unit(const orc_dims *d, unit_fn fn, void *ctx) {
    int nthr = d->n_threads > 0 ? d->n_threads : 1;
    if (nthr > d->B * d->H) nthr = d->B * d->H;
    if (nthr <= 1) {
        for (int b = 0; b < d->B; ++b)
            for (int h = 0; h < d->H; ++h) fn(ctx, b, h);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthr);
    worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * nthr);
    for (int i = 0; i < nthr; ++i) {
        args[i] = (worker_arg){fn, ctx, d->B, d->H, i, nthr};
        pthread_create(&th[i], NULL, worker, &args[i]);
    }
    for (int i = 0; i < nthr; ++i) pthread_join(th[i], NULL);
    free(th);
    free(args);
}

/* ------------------------------------------------------------------ verify */
typedef struct {
    const orc_dims *d;
    const double *state; const int32_t *state_idx;
    double *buf_k, *buf_v, *buf_g, *buf_beta; const int32_t *buf_len;
    const double *q, *k, *v, *g, *beta;
    double *out; const unsigned char *skip;
} verify_ctx;

static void verify_unit(void *p, int b, int h) {
    verify_ctx *c = (verify_ctx *)p;
    const orc_dims *d = c->d;
    if (c->skip[b]) return;
    const int slot = slot_of(c->state_idx, b);
    const int len = c->buf_len[slot];
    const size_t n = (size_t)d->dv * d->dk;
    double *S = (double *)malloc(n * sizeof(double));
    memcpy(S, c->state + st_off(d, slot, h), n * sizeof(double));   /* the checkpoint is only read */
    /* committed tokens from the buffer, outputs discarded */
    orc_recur(d, S, len,
              c->buf_k + bk_off(d, slot, h, 0), d->dk, c->buf_v + bv_off(d, slot, h, 0), d->dv,
              c->buf_g + bg_off(d, slot, h, 0), c->buf_beta + bg_off(d, slot, h, 0), 1,
              NULL, 0, NULL, 0);
    /* the draft block, emitting o_t */
    const long tk = (long)d->H * d->dk, tv = (long)d->H * d->dv, tg = d->H;
    orc_recur(d, S, d->T,
              c->k + dk_off(d, b, 0, h), tk, c->v + dv_off(d, b, 0, h), tv,
              c->g + dg_off(d, b, 0, h), c->beta + dg_off(d, b, 0, h), tg,
              c->q + dk_off(d, b, 0, h), tk, c->out + dv_off(d, b, 0, h), tv);
    free(S);
    /* stage the draft block behind the committed tokens so that accepting p
     * tokens later is only a length update */
    for (int t = 0; t < d->T; ++t) {
        memcpy(c->buf_k + bk_off(d, slot, h, len + t), c->k + dk_off(d, b, t, h), d->dk * sizeof(double));
        memcpy(c->buf_v + bv_off(d, slot, h, len + t), c->v + dv_off(d, b, t, h), d->dv * sizeof(double));
        c->buf_g[bg_off(d, slot, h, len + t)] = c->g[dg_off(d, b, t, h)];
        c->buf_beta[bg_off(d, slot, h, len + t)] = c->beta[dg_off(d, b, t, h)];
    }
}

int orc_verify(const orc_dims *d, const double *state, const int32_t *state_idx,
               double *buf_k, double *buf_v, double *buf_g, double *buf_beta, const int32_t *buf_len,
               const double *q, const double *k, const double *v, const double *g, const double *beta,
               double *out, int32_t *status)
{
    unsigned char *skip = (unsigned char *)calloc(d->B > 0 ? d->B : 1, 1);
    for (int b = 0; b < d->B; ++b) {
        const int len = buf_len[slot_of(state_idx, b)];
        if (len < 0 || len + d->T > d->cap) { *status |= ORC_NO_ROOM; skip[b] = 1; }
    }
    verify_ctx c = {d, state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len,
                    q, k, v, g, beta, out, skip};
    for_each_unit(d, verify_unit, &c);
    free(skip);
    return 0;
}

/* ------------------------------------------------------------------ accept */
int orc_accept(const orc_dims *d, int32_t *buf_len, const int32_t *state_idx,
               const int32_t *accepted, int32_t *status)
{
    for (int b = 0; b < d->B; ++b) {
        const int slot = slot_of(state_idx, b);
        const int p = accepted[b], len = buf_len[slot];
        if (p < 0 || p > d->T) { *status |= ORC_BAD_ACCEPT; continue; }
        if (len < 0 || len + p > d->cap) { *status |= ORC_BAD_LEN; continue; }
        buf_len[slot] = len + p;     /* rejection of the rest is implicit */
    }
    return 0;
}

/* ------------------------------------------------------------------- flush */
typedef struct {
    const orc_dims *d;
    double *state; const int32_t *state_idx;
    const double *buf_k, *buf_v, *buf_g, *buf_beta; const int32_t *lens;
} flush_ctx;

static void flush_unit(void *p, int b, int h) {
    flush_ctx *c = (flush_ctx *)p;
    const orc_dims *d = c->d;
    const int len = c->lens[b];
    if (len <= 0) return;
    const int slot = slot_of(c->state_idx, b);
    double *S = c->state + st_off(d, slot, h);
    orc_recur(d, S, len,
              c->buf_k + bk_off(d, slot, h, 0), d->dk, c->buf_v + bv_off(d, slot, h, 0), d->dv,
              c->buf_g + bg_off(d, slot, h, 0), c->buf_beta + bg_off(d, slot, h, 0), 1,
              NULL, 0, NULL, 0);
    for (size_t e = 0; e < (size_t)d->dv * d->dk; ++e) S[e] = (double)(float)S[e];  /* fp32 checkpoint */
}

int orc_flush(const orc_dims *d, double *state, const int32_t *state_idx,
              const double *buf_k, const double *buf_v, const double *buf_g, const double *buf_beta,
              int32_t *buf_len, int force, int32_t *status)
{
    int32_t *lens = (int32_t *)calloc(d->B > 0 ? d->B : 1, sizeof(int32_t));  /* tokens to fold per b, 0 = none */
    for (int b = 0; b < d->B; ++b) {
        const int len = buf_len[slot_of(state_idx, b)];
        if (len < 0 || len > d->cap) { *status |= ORC_BAD_LEN; continue; }
        if (len >= d->threshold || (force && len > 0)) lens[b] = len;
    }
    flush_ctx c = {d, state, state_idx, buf_k, buf_v, buf_g, buf_beta, lens};
    for_each_unit(d, flush_unit, &c);
    for (int b = 0; b < d->B; ++b)
        if (lens[b] > 0) buf_len[slot_of(state_idx, b)] = 0;
    free(lens);
    return 0;
}

/* ------------------------------------------------- non-replay baseline
 * The data movement ReplaySSM avoids ("The inference stack behind OCRia",
 * section "Making speculative verification cheaper": restoring a recurrent
 * state after a rejection moves a lot of data).  Without a buffer the state is
 * always current; so that a rejection can go back to the state after the
 * accepted prefix, the verify stores the state after every draft token, and
 * the accept copies the snapshot of the accepted prefix over the state.
 *
 * layouts: state [n_slot, H, dv, dk]; snap [B, H, T, dv, dk] (per batch row,
 * stored as binary32 like the checkpoint); draft inputs and out as above.
 * Status: a slot outside [0, n_slot) sets ORC_BAD_SLOT and skips the row; an
 * accepted count outside [0, T] sets ORC_BAD_ACCEPT and skips the row. */
#define ORC_BAD_SLOT 8

typedef struct {
    const orc_dims *d;
    const double *state; const int32_t *state_idx;
    const double *q, *k, *v, *g, *beta;
    double *out, *snap; const unsigned char *skip;
} nr_verify_ctx;

static void nr_verify_unit(void *p, int b, int h) {
    nr_verify_ctx *c = (nr_verify_ctx *)p;
    const orc_dims *d = c->d;
    if (c->skip[b]) return;
    const int slot = slot_of(c->state_idx, b);
    const size_t n = (size_t)d->dv * d->dk;
    double *S = (double *)malloc(n * sizeof(double));
    memcpy(S, c->state + st_off(d, slot, h), n * sizeof(double));   /* the state is only read */
    const long tk = (long)d->H * d->dk, tv = (long)d->H * d->dv, tg = d->H;
    for (int t = 0; t < d->T; ++t) {
        orc_recur(d, S, 1,
                  c->k + dk_off(d, b, t, h), tk, c->v + dv_off(d, b, t, h), tv,
                  c->g + dg_off(d, b, t, h), c->beta + dg_off(d, b, t, h), tg,
                  c->q + dk_off(d, b, t, h), tk, c->out + dv_off(d, b, t, h), tv);
        double *dst = c->snap + (((size_t)b * d->H + h) * d->T + t) * n;
        for (size_t e = 0; e < n; ++e) dst[e] = (double)(float)S[e];   /* stored as binary32 */
    }
    free(S);
}

int orc_nr_verify(const orc_dims *d, const double *state, const int32_t *state_idx,
                  const double *q, const double *k, const double *v, const double *g, const double *beta,
                  double *out, double *snap, int32_t *status)
{
    unsigned char *skip = (unsigned char *)calloc(d->B > 0 ? d->B : 1, 1);
    for (int b = 0; b < d->B; ++b) {
        const int slot = slot_of(state_idx, b);
        if (slot < 0 || slot >= d->n_slot) { *status |= ORC_BAD_SLOT; skip[b] = 1; }
    }
    nr_verify_ctx c = {d, state, state_idx, q, k, v, g, beta, out, snap, skip};
    for_each_unit(d, nr_verify_unit, &c);
    free(skip);
    return 0;
}

int orc_nr_accept(const orc_dims *d, double *state, const int32_t *state_idx, const double *snap,
                  const int32_t *accepted, int32_t *status)
{
    const size_t n = (size_t)d->dv * d->dk;
    for (int b = 0; b < d->B; ++b) {
        const int slot = slot_of(state_idx, b), p = accepted[b];
        if (slot < 0 || slot >= d->n_slot) { *status |= ORC_BAD_SLOT; continue; }
        if (p < 0 || p > d->T) { *status |= ORC_BAD_ACCEPT; continue; }
        if (p == 0) continue;                     /* everything rejected: the state stays */
        for (int h = 0; h < d->H; ++h)
            memcpy(state + st_off(d, slot, h), snap + (((size_t)b * d->H + h) * d->T + (p - 1)) * n,
                   n * sizeof(double));
    }
    return 0;
}
