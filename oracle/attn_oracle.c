/*
 * attn_oracle.c -- fp64 CPU oracle for exact context-parallel attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA library: no headers, no helpers, no tables.
 *
 * Every routine is the plain definition written out, in double precision,
 * with no blocking, fusion or reordering beyond what the cited passage states.
 * Tensors are contiguous row-major [B, L, H, D] (batch, sequence, head, head
 * dim), as in the verify script of the juejin.cn ring-attention debugging
 * article (section 三); lse is [B, L, H], natural log
 * (same page, section 五, local_attn_lse returns lse of shape (B, Sq, H)).
 *
 * Routines:
 *   oracle_attention       naive softmax(QK^T / sqrt(D)) V for chosen query rows
 *                          ("序列并行与 Ring Attention", section 3.1, the SDPA
 *                          equation; causal rule j <= i on global positions,
 *                          section 3.4)
 *   oracle_ring_attention  the blockwise online-softmax recurrence (section
 *                          3.2: m, l, u, alpha, o = u/l) applied in ring order,
 *                          shard r meeting the K/V of shard (r - t) mod P at
 *                          step t (section 3.3), skipping wholly-future shards
 *                          under causal masking (section 3.4)
 *   oracle_merge           log-sum-exp combine of two partial results
 *                          (juejin page, section 四 "combine")
 *   oracle_seq2head /      Ulysses layout transpose [B, L/P, H, D] per rank
 *   oracle_head2seq        <-> [B, L, H/P, D] per rank ("序列并行与 Ring
 *                          Attention", section 3.5)
 *   oracle_attention_bwd   gradients dQ, dK, dV by the chain rule (the backward
 *                          of sections 3.3 and 6.2, summed on one device), and
 *                          the same for chosen query rows (..._dq_rows) or key
 *                          rows (..._dkdv_rows) at long sequence lengths
 *
 * Conventions for sets with no visible key (cannot arise under the causal rule
 * j <= i, but can for a merge input): output 0 and lse = -inf, which is the
 * limit the recurrence reaches when the running denominator stays 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* tiny work-sharing pool: n_items independent items, claimed by an atomic    */
/* counter; each worker owns a scratch buffer of scratch_doubles doubles.     */

typedef void (*item_fn)(void* ctx, long item, double* scratch);

typedef struct {
    item_fn fn;
    void* ctx;
    long n_items;
    long next;            /* atomic */
    long scratch_doubles;
    int failed;           /* atomic */
} pool_t;

static void* pool_worker(void* arg)
{
    pool_t* p = (pool_t*)arg;
    double* scratch = NULL;
    if (p->scratch_doubles > 0) {
        scratch = (double*)malloc(sizeof(double) * (size_t)p->scratch_doubles);
        if (!scratch) { __atomic_store_n(&p->failed, 1, __ATOMIC_SEQ_CST); return NULL; }
    }
    for (;;) {
        long it = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

static int run_pool(item_fn fn, void* ctx, long n_items, long scratch_doubles, int n_threads)
{
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.n_items = n_items; p.next = 0;
    p.scratch_doubles = scratch_doubles; p.failed = 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((long)n_threads > n_items) n_threads = (int)(n_items > 0 ? n_items : 1);
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i) {
        if (pthread_create(&th[started], NULL, pool_worker, &p) != 0) break;
        ++started;
    }
    pool_worker(&p);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    return p.failed ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* naive attention over an explicit key range                                */

typedef struct {
    const double *q, *k, *v;
    double *out, *lse;
    long B, Lq, Lk, H, D;
    long Hk;                 /* key/value heads; query head h reads key/value head h / (H / Hk) */
    int causal;
    long q_pos0, k_pos0;     /* global position of q row 0 / key 0 */
    const long* rows;        /* query rows to evaluate (indices into Lq), or NULL for all */
    long n_rows;
} attn_ctx_t;

/* One query row against every key: the stable softmax of section 3.1, written
 * as max-subtraction, exponentials, their sum, then the weighted mean of V. */
static void attn_item(void* vctx, long item, double* w)
{
    const attn_ctx_t* c = (const attn_ctx_t*)vctx;
    const long D = c->D, H = c->H;
    const long ri = item % c->n_rows;
    const long bh = item / c->n_rows;
    const long h = bh % H, b = bh / H;
    const long i = c->rows ? c->rows[ri] : ri;
    const long hk = h / (H / c->Hk);
    const long q_pos = c->q_pos0 + i;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    const double* qrow = c->q + ((b * c->Lq + i) * H + h) * D;

    double m = -INFINITY;
    for (long j = 0; j < c->Lk; ++j) {
        if (c->causal && c->k_pos0 + j > q_pos) { w[j] = -INFINITY; continue; }
        const double* krow = c->k + ((b * c->Lk + j) * c->Hk + hk) * D;
        double s = 0.0;
        for (long d = 0; d < D; ++d) s += qrow[d] * krow[d];
        s *= inv_sqrt_d;
        w[j] = s;
        if (s > m) m = s;
    }
    double* orow = c->out + ((b * c->n_rows + ri) * H + h) * D;
    double* lrow = c->lse + (b * c->n_rows + ri) * H + h;
    if (m == -INFINITY) {            /* no visible key */
        for (long d = 0; d < D; ++d) orow[d] = 0.0;
        *lrow = -INFINITY;
        return;
    }
    double den = 0.0;
    for (long j = 0; j < c->Lk; ++j) {
        w[j] = (w[j] == -INFINITY) ? 0.0 : exp(w[j] - m);
        den += w[j];
    }
    /* acc[d] = sum_j w_j v[j][d], keys taken in order j = 0, 1, ... for every d */
    double* acc = w + c->Lk;
    for (long d = 0; d < D; ++d) acc[d] = 0.0;
    for (long j = 0; j < c->Lk; ++j) {
        if (w[j] == 0.0) continue;
        const double* vrow = c->v + ((b * c->Lk + j) * c->Hk + hk) * D;
        for (long d = 0; d < D; ++d) acc[d] += w[j] * vrow[d];
    }
    for (long d = 0; d < D; ++d) orow[d] = acc[d] / den;
    *lrow = m + log(den);
}

/*
 * out: [B, n_rows, H, D]; lse: [B, n_rows, H].  q: [B, Lq, H, D]; k, v: [B, Lk, Hk, D].
 * rows == NULL means every query row (n_rows must equal Lq).
 * Query row i sits at global position q_pos0 + i, key j at k_pos0 + j; under
 * causal masking key j is visible to row i iff its position <= the row's.
 * Grouped key/value heads ("序列并行与 Ring Attention", sections 3.5 and 6.4 count
 * them apart from the query heads): H must be a multiple of Hk, and the H / Hk
 * consecutive query heads h = g*(H/Hk) .. (g+1)*(H/Hk) - 1 share key/value head g.
 */
int oracle_attention_gqa(const double* q, const double* k, const double* v,
                         double* out, double* lse,
                         long B, long Lq, long Lk, long H, long Hk, long D, int causal,
                         long q_pos0, long k_pos0,
                         const long* rows, long n_rows, int n_threads)
{
    if (!q || !k || !v || !out || !lse || B < 0 || Lq < 0 || Lk < 0 || H < 0 || D <= 0) return -1;
    if (Hk <= 0 || (H > 0 && H % Hk != 0)) return -2;
    if (!rows) n_rows = Lq;
    if (n_rows < 0) return -1;
    if (rows) for (long i = 0; i < n_rows; ++i) if (rows[i] < 0 || rows[i] >= Lq) return -1;
    attn_ctx_t c = { q, k, v, out, lse, B, Lq, Lk, H, D, Hk, causal, q_pos0, k_pos0, rows, n_rows };
    long n_items = B * H * n_rows;
    if (n_items == 0) return 0;
    return run_pool(attn_item, &c, n_items, (Lk > 0 ? Lk : 1) + D, n_threads);
}

/* The same with as many key/value heads as query heads. */
int oracle_attention(const double* q, const double* k, const double* v,
                     double* out, double* lse,
                     long B, long Lq, long Lk, long H, long D, int causal,
                     long q_pos0, long k_pos0,
                     const long* rows, long n_rows, int n_threads)
{
    return oracle_attention_gqa(q, k, v, out, lse, B, Lq, Lk, H, H > 0 ? H : 1, D, causal,
                                q_pos0, k_pos0, rows, n_rows, n_threads);
}

/* ------------------------------------------------------------------------- */
/* ring-order blockwise recurrence                                           */

typedef struct {
    const double *q, *k, *v;
    double *out, *lse;
    long B, L, H, D, P;
    int causal;
} ring_ctx_t;

static long ring_source(long r, long t, long P) { return ((r - t) % P + P) % P; }

/* One query row of shard r.  Section 3.2's recurrence, one K/V block per ring
 * step: m_{t+1} = max(m_t, max_j s_j), alpha = exp(m_t - m_{t+1}),
 * l_{t+1} = alpha l_t + sum_j exp(s_j - m_{t+1}),
 * u_{t+1} = alpha u_t + sum_j exp(s_j - m_{t+1}) v_j, and finally o = u / l.
 * scratch: Ls score slots followed by D accumulator slots. */
static void ring_item(void* vctx, long item, double* scratch)
{
    const ring_ctx_t* c = (const ring_ctx_t*)vctx;
    const long L = c->L, H = c->H, D = c->D, P = c->P, Ls = L / P;
    const long i = item % L;                 /* global query position */
    const long bh = item / L;
    const long h = bh % H, b = bh / H;
    const long r = i / Ls;                    /* owning shard */
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    const double* qrow = c->q + ((b * L + i) * H + h) * D;
    double* s = scratch;
    double* u = scratch + Ls;

    double m = -INFINITY, l = 0.0;
    for (long d = 0; d < D; ++d) u[d] = 0.0;

    for (long t = 0; t < P; ++t) {
        const long src = ring_source(r, t, P);
        if (c->causal && src > r) continue;   /* wholly in the future */
        const long j0 = src * Ls;
        double mb = -INFINITY;
        for (long jj = 0; jj < Ls; ++jj) {
            const long j = j0 + jj;
            if (c->causal && j > i) { s[jj] = -INFINITY; continue; }
            const double* krow = c->k + ((b * L + j) * H + h) * D;
            double acc = 0.0;
            for (long d = 0; d < D; ++d) acc += qrow[d] * krow[d];
            s[jj] = acc * inv_sqrt_d;
            if (s[jj] > mb) mb = s[jj];
        }
        const double m_new = (mb > m) ? mb : m;
        if (m_new == -INFINITY) continue;     /* nothing visible yet */
        const double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        double block_sum = 0.0;
        for (long d = 0; d < D; ++d) u[d] *= alpha;
        for (long jj = 0; jj < Ls; ++jj) {
            if (s[jj] == -INFINITY) continue;
            const double e = exp(s[jj] - m_new);
            block_sum += e;
            const double* vrow = c->v + ((b * L + j0 + jj) * H + h) * D;
            for (long d = 0; d < D; ++d) u[d] += e * vrow[d];
        }
        l = alpha * l + block_sum;
        m = m_new;
    }
    double* orow = c->out + ((b * L + i) * H + h) * D;
    if (l == 0.0) {
        for (long d = 0; d < D; ++d) orow[d] = 0.0;
        c->lse[(b * L + i) * H + h] = -INFINITY;
        return;
    }
    for (long d = 0; d < D; ++d) orow[d] = u[d] / l;
    c->lse[(b * L + i) * H + h] = m + log(l);
}

/*
 * Ring-order reference.  out [B, L, H, D], lse [B, L, H].  trace, if not NULL,
 * receives a P x P int table: trace[r * P + t] = source shard visited by shard
 * r at step t, or -1 where that step is skipped as wholly future.
 * Requires L % P == 0 (equal shards, section 3.3).
 */
int oracle_ring_attention(const double* q, const double* k, const double* v,
                          double* out, double* lse,
                          long B, long L, long H, long D, long P, int causal,
                          int* trace, int n_threads)
{
    if (!q || !k || !v || !out || !lse || B < 0 || L < 0 || H < 0 || D <= 0 || P <= 0) return -1;
    if (L % P != 0) return -2;
    if (trace) {
        for (long r = 0; r < P; ++r)
            for (long t = 0; t < P; ++t) {
                const long src = ring_source(r, t, P);
                trace[r * P + t] = (causal && src > r) ? -1 : (int)src;
            }
    }
    ring_ctx_t c = { q, k, v, out, lse, B, L, H, D, P, causal };
    long n_items = B * H * L;
    if (n_items == 0) return 0;
    return run_pool(ring_item, &c, n_items, L / P + D, n_threads);
}

/* ------------------------------------------------------------------------- */
/* LSE merge of two partial results                                          */

/*
 * o = o_a * exp(lse_a - lse) + o_b * exp(lse_b - lse), lse = log(e^lse_a + e^lse_b).
 * A partial whose lse is -inf covers no key and gets weight 0; if both are
 * -inf the merged output is 0 and lse is -inf.  o_*: [rows, D]; lse_*: [rows].
 */
int oracle_merge(const double* o_a, const double* lse_a,
                 const double* o_b, const double* lse_b,
                 double* o, double* lse, long rows, long D)
{
    if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse || rows < 0 || D <= 0) return -1;
    for (long i = 0; i < rows; ++i) {
        const double a = lse_a[i], b = lse_b[i];
        if (a == -INFINITY && b == -INFINITY) {
            lse[i] = -INFINITY;
            for (long d = 0; d < D; ++d) o[i * D + d] = 0.0;
            continue;
        }
        const double hi = a > b ? a : b;
        const double lo = a > b ? b : a;
        const double l = hi + log1p(exp(lo - hi));   /* logaddexp */
        const double wa = exp(a - l), wb = exp(b - l);
        for (long d = 0; d < D; ++d) o[i * D + d] = o_a[i * D + d] * wa + o_b[i * D + d] * wb;
        lse[i] = l;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Ulysses layout transposes                                                 */

/*
 * Sequence-sharded buffer: P rank slices, rank r holding [B, L/P, H, D] for
 * tokens [r L/P, (r+1) L/P).  Head-sharded buffer: P rank slices, rank g
 * holding [B, L, H/P, D] for heads [g H/P, (g+1) H/P).  Element by element:
 *   head[g][b][r*Ls + l][hh][d] = seq[r][b][l][g*Hg + hh][d].
 * Elements are opaque byte strings of elem_bytes.
 */
int oracle_seq2head(const void* in, void* out, long B, long L, long H, long D,
                    long P, long elem_bytes)
{
    if (!in || !out || B < 0 || L < 0 || H < 0 || D <= 0 || P <= 0 || elem_bytes <= 0) return -1;
    if (L % P != 0 || H % P != 0) return -2;
    const long Ls = L / P, Hg = H / P;
    const unsigned char* src = (const unsigned char*)in;
    unsigned char* dst = (unsigned char*)out;
    for (long g = 0; g < P; ++g)
        for (long b = 0; b < B; ++b)
            for (long lg = 0; lg < L; ++lg)
                for (long hh = 0; hh < Hg; ++hh)
                    for (long d = 0; d < D; ++d) {
                        const long r = lg / Ls, l = lg % Ls, hgl = g * Hg + hh;
                        const long di = (((g * B + b) * L + lg) * Hg + hh) * D + d;
                        const long si = (((r * B + b) * Ls + l) * H + hgl) * D + d;
                        memcpy(dst + di * elem_bytes, src + si * elem_bytes, (size_t)elem_bytes);
                    }
    return 0;
}

/* The inverse transpose: seq[r][b][l][g*Hg + hh][d] = head[g][b][r*Ls + l][hh][d]. */
int oracle_head2seq(const void* in, void* out, long B, long L, long H, long D,
                    long P, long elem_bytes)
{
    if (!in || !out || B < 0 || L < 0 || H < 0 || D <= 0 || P <= 0 || elem_bytes <= 0) return -1;
    if (L % P != 0 || H % P != 0) return -2;
    const long Ls = L / P, Hg = H / P;
    const unsigned char* src = (const unsigned char*)in;
    unsigned char* dst = (unsigned char*)out;
    for (long r = 0; r < P; ++r)
        for (long b = 0; b < B; ++b)
            for (long l = 0; l < Ls; ++l)
                for (long hgl = 0; hgl < H; ++hgl)
                    for (long d = 0; d < D; ++d) {
                        const long g = hgl / Hg, hh = hgl % Hg, lg = r * Ls + l;
                        const long di = (((r * B + b) * Ls + l) * H + hgl) * D + d;
                        const long si = (((g * B + b) * L + lg) * Hg + hh) * D + d;
                        memcpy(dst + di * elem_bytes, src + si * elem_bytes, (size_t)elem_bytes);
                    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* backward: gradients of the attention output                               */

typedef struct {
    const double *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    long B, L, H, D;
    int causal;
} bwd_ctx_t;

/*
 * One (batch, head): the chain rule through O = softmax(S) V with
 * S = Q K^T / sqrt(D) (masked entries excluded):
 *   dV = P^T dO,  dP = dO V^T,  dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik),
 *   dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D).
 * The backward that "序列并行与 Ring Attention" (sections 3.3 and 6.2) describes
 * recomputes the probabilities from the saved row statistics and returns dK, dV
 * to the shard that owns K, V; on one device that is this same sum.
 * scratch: P (L*L) then dP (L*L).
 */
static void bwd_item(void* vctx, long item, double* scratch)
{
    const bwd_ctx_t* c = (const bwd_ctx_t*)vctx;
    const long L = c->L, H = c->H, D = c->D;
    const long h = item % H, b = item / H;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    double* P = scratch;
    double* dP = scratch + L * L;
#define AT(t, i) ((t) + ((b * L + (i)) * H + h) * D)
    for (long i = 0; i < L; ++i) {
        double m = -INFINITY;
        for (long j = 0; j < L; ++j) {
            if (c->causal && j > i) { P[i * L + j] = -INFINITY; continue; }
            double s = 0.0;
            for (long d = 0; d < D; ++d) s += AT(c->q, i)[d] * AT(c->k, j)[d];
            s *= inv_sqrt_d;
            P[i * L + j] = s;
            if (s > m) m = s;
        }
        double den = 0.0;
        for (long j = 0; j < L; ++j) {
            P[i * L + j] = (P[i * L + j] == -INFINITY) ? 0.0 : exp(P[i * L + j] - m);
            den += P[i * L + j];
        }
        for (long j = 0; j < L; ++j) P[i * L + j] /= den;
    }
    for (long i = 0; i < L; ++i)
        for (long j = 0; j < L; ++j) {
            double s = 0.0;
            for (long d = 0; d < D; ++d) s += AT(c->dout, i)[d] * AT(c->v, j)[d];
            dP[i * L + j] = s;
        }
    /* dS overwrites dP */
    for (long i = 0; i < L; ++i) {
        double rowdot = 0.0;
        for (long j = 0; j < L; ++j) rowdot += P[i * L + j] * dP[i * L + j];
        for (long j = 0; j < L; ++j) dP[i * L + j] = P[i * L + j] * (dP[i * L + j] - rowdot);
    }
    for (long i = 0; i < L; ++i)
        for (long d = 0; d < D; ++d) {
            double s = 0.0;
            for (long j = 0; j < L; ++j) s += dP[i * L + j] * AT(c->k, j)[d];
            AT(c->dq, i)[d] = s * inv_sqrt_d;
        }
    for (long j = 0; j < L; ++j)
        for (long d = 0; d < D; ++d) {
            double sk = 0.0, sv = 0.0;
            for (long i = 0; i < L; ++i) {
                sk += dP[i * L + j] * AT(c->q, i)[d];
                sv += P[i * L + j] * AT(c->dout, i)[d];
            }
            AT(c->dk, j)[d] = sk * inv_sqrt_d;
            AT(c->dv, j)[d] = sv;
        }
#undef AT
}

/* Gradients of O = attention(Q, K, V) against an upstream gradient dO.
 * All tensors [B, L, H, D]; meant for small L (keeps two L x L matrices per thread). */
int oracle_attention_bwd(const double* q, const double* k, const double* v, const double* dout,
                         double* dq, double* dk, double* dv,
                         long B, long L, long H, long D, int causal, int n_threads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 0 || L < 0 || H < 0 || D <= 0) return -1;
    bwd_ctx_t c = { q, k, v, dout, dq, dk, dv, B, L, H, D, causal };
    long n_items = B * H;
    if (n_items == 0 || L == 0) return 0;
    return run_pool(bwd_item, &c, n_items, 2 * L * L, n_threads);
}

/* ------------------------------------------------------------------------- */
/* backward for chosen query rows: dq of row i needs only row i's scores     */

typedef struct {
    const double *q, *k, *v, *dout;
    double* dq;
    long B, L, H, D;
    int causal;
    const long* rows;
    long n_rows;
} bwd_rows_ctx_t;

/* dq_i = sum_j P_ij (dP_ij - sum_k P_ik dP_ik) k_j / sqrt(D) with P_i. = softmax of
 * row i's scores and dP_ij = dO_i . v_j: the same chain rule as bwd_item, one row.
 * scratch: P (L) then dP (L). */
static void bwd_rows_item(void* vctx, long item, double* scratch)
{
    const bwd_rows_ctx_t* c = (const bwd_rows_ctx_t*)vctx;
    const long L = c->L, H = c->H, D = c->D;
    const long ri = item % c->n_rows;
    const long bh = item / c->n_rows;
    const long h = bh % H, b = bh / H;
    const long i = c->rows[ri];
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    const long n = c->causal ? i + 1 : L;     /* visible keys 0..n-1 */
    double* P = scratch;
    double* dP = scratch + L;
#define AT(t, r) ((t) + ((b * L + (r)) * H + h) * D)
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        double s = 0.0;
        for (long d = 0; d < D; ++d) s += AT(c->q, i)[d] * AT(c->k, j)[d];
        P[j] = s * inv_sqrt_d;
        if (P[j] > m) m = P[j];
    }
    double den = 0.0;
    for (long j = 0; j < n; ++j) { P[j] = exp(P[j] - m); den += P[j]; }
    double rowdot = 0.0;
    for (long j = 0; j < n; ++j) {
        P[j] /= den;
        double s = 0.0;
        for (long d = 0; d < D; ++d) s += AT(c->dout, i)[d] * AT(c->v, j)[d];
        dP[j] = s;
        rowdot += P[j] * s;
    }
    double* out = c->dq + ((b * c->n_rows + ri) * H + h) * D;
    for (long d = 0; d < D; ++d) out[d] = 0.0;
    for (long j = 0; j < n; ++j) {
        const double ds = P[j] * (dP[j] - rowdot);
        for (long d = 0; d < D; ++d) out[d] += ds * AT(c->k, j)[d];
    }
    for (long d = 0; d < D; ++d) out[d] *= inv_sqrt_d;
#undef AT
}

/* dq of the listed query rows only: dq_rows [B, n_rows, H, D]. */
int oracle_attention_bwd_dq_rows(const double* q, const double* k, const double* v,
                                 const double* dout, double* dq_rows,
                                 long B, long L, long H, long D, int causal,
                                 const long* rows, long n_rows, int n_threads)
{
    if (!q || !k || !v || !dout || !dq_rows || !rows || B < 0 || L <= 0 || H < 0 || D <= 0) return -1;
    for (long r = 0; r < n_rows; ++r) if (rows[r] < 0 || rows[r] >= L) return -1;
    bwd_rows_ctx_t c = { q, k, v, dout, dq_rows, B, L, H, D, causal, rows, n_rows };
    long n_items = B * H * n_rows;
    if (n_items == 0) return 0;
    return run_pool(bwd_rows_item, &c, n_items, 2 * L, n_threads);
}

/* ------------------------------------------------------------------------- */
/* backward for chosen key rows: dk_j and dv_j sum over every query that      */
/* sees key j, so they need each such query's softmax normaliser and row dot; */
/* the naive forward gives both for every query row first, then the key rows  */
/* are the chain rule's column sums.                                          */

typedef struct {
    const double *q, *k, *v, *dout;
    double *lse, *rowdot;       /* [B, L, H]: per query row */
    double* o;                  /* [B, L, H, D]: the attention output of every query row */
    double *dk, *dv;            /* [B, n_rows, H, D] */
    long B, L, H, D;
    int causal;
    const long* rows;
    long n_rows;
} bwd_key_rows_ctx_t;

/* Query row i of (b, h), the stable softmax of section 3.1: lse_i = ln sum_j e^{s_ij}
 * over the keys it sees (s_ij = q_i . k_j / sqrt(D); causal: j <= i), its output
 * O_i = sum_j e^{s_ij - lse_i} v_j, and rowdot_i = dO_i . O_i, which equals
 * sum_j P_ij dP_ij (dP_ij = dO_i . v_j): the term the chain rule subtracts in
 * dS_ij = P_ij (dP_ij - rowdot_i).  scratch: the row's scores (L). */
static void query_stats_item(void* vctx, long item, double* scratch)
{
    const bwd_key_rows_ctx_t* c = (const bwd_key_rows_ctx_t*)vctx;
    const long L = c->L, H = c->H, D = c->D;
    const long i = item % L;
    const long bh = item / L;
    const long h = bh % H, b = bh / H;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    const long n = c->causal ? i + 1 : L;     /* visible keys 0..n-1 */
#define AT(t, r) ((t) + ((b * L + (r)) * H + h) * D)
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        double s = 0.0;
        for (long d = 0; d < D; ++d) s += AT(c->q, i)[d] * AT(c->k, j)[d];
        scratch[j] = s * inv_sqrt_d;
        if (scratch[j] > m) m = scratch[j];
    }
    double den = 0.0;
    for (long j = 0; j < n; ++j) den += exp(scratch[j] - m);
    const double lse = m + log(den);
    double* o = AT(c->o, i);
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    for (long j = 0; j < n; ++j) {
        const double p = exp(scratch[j] - lse);
        for (long d = 0; d < D; ++d) o[d] += p * AT(c->v, j)[d];
    }
    double rowdot = 0.0;
    for (long d = 0; d < D; ++d) rowdot += AT(c->dout, i)[d] * o[d];
    c->lse[(b * L + i) * H + h] = lse;
    c->rowdot[(b * L + i) * H + h] = rowdot;
#undef AT
}

/* Key row j of (b, h):
 *   dv_j = sum_i P_ij dO_i,   dk_j = sum_i dS_ij q_i / sqrt(D),
 * over the queries i that see key j (causal: i >= j), with P_ij = e^{s_ij - lse_i}
 * and dS_ij = P_ij (dO_i . v_j - rowdot_i): the columns of the chain rule that
 * bwd_item evaluates as whole matrices. */
static void key_rows_item(void* vctx, long item, double* scratch)
{
    (void)scratch;
    const bwd_key_rows_ctx_t* c = (const bwd_key_rows_ctx_t*)vctx;
    const long L = c->L, H = c->H, D = c->D;
    const long rj = item % c->n_rows;
    const long bh = item / c->n_rows;
    const long h = bh % H, b = bh / H;
    const long j = c->rows[rj];
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#define AT(t, r) ((t) + ((b * L + (r)) * H + h) * D)
    double* dk = c->dk + ((b * c->n_rows + rj) * H + h) * D;
    double* dv = c->dv + ((b * c->n_rows + rj) * H + h) * D;
    for (long d = 0; d < D; ++d) { dk[d] = 0.0; dv[d] = 0.0; }
    for (long i = c->causal ? j : 0; i < L; ++i) {
        double s = 0.0, dp = 0.0;
        for (long d = 0; d < D; ++d) {
            s += AT(c->q, i)[d] * AT(c->k, j)[d];
            dp += AT(c->dout, i)[d] * AT(c->v, j)[d];
        }
        const long si = (b * L + i) * H + h;
        const double p = exp(s * inv_sqrt_d - c->lse[si]);
        const double ds = p * (dp - c->rowdot[si]);
        for (long d = 0; d < D; ++d) {
            dv[d] += p * AT(c->dout, i)[d];
            dk[d] += ds * AT(c->q, i)[d];
        }
    }
    for (long d = 0; d < D; ++d) dk[d] *= inv_sqrt_d;
#undef AT
}

/* dk and dv of the listed key rows only: dk_rows, dv_rows [B, n_rows, H, D].  The
 * per-query pass costs one sweep over all (query, key) pairs; the key rows then cost
 * O(L D) each, so this works at long sequence lengths.  lse_out [B, L, H] and
 * o_out [B, L, H, D] (either may be NULL) receive the per-query lse and output the
 * routine computed on the way. */
int oracle_attention_bwd_dkdv_rows(const double* q, const double* k, const double* v,
                                   const double* dout, double* dk_rows, double* dv_rows,
                                   long B, long L, long H, long D, int causal,
                                   const long* rows, long n_rows, double* lse_out,
                                   double* o_out, int n_threads)
{
    if (!q || !k || !v || !dout || !dk_rows || !dv_rows || !rows || B < 0 || L <= 0 || H < 0 ||
        D <= 0 || n_rows < 0)
        return -1;
    for (long r = 0; r < n_rows; ++r) if (rows[r] < 0 || rows[r] >= L) return -1;
    if (B * H * n_rows == 0) return 0;
    double* stats = (double*)malloc((size_t)(2 * B * L * H) * sizeof(double));
    double* o = o_out ? o_out : (double*)malloc((size_t)(B * L * H * D) * sizeof(double));
    if (!stats || !o) {
        free(stats);
        if (!o_out) free(o);
        return -2;
    }
    bwd_key_rows_ctx_t c = { q, k, v, dout, stats, stats + B * L * H, o, dk_rows, dv_rows,
                             B, L, H, D, causal, rows, n_rows };
    int rc = run_pool(query_stats_item, &c, B * H * L, L, n_threads);
    if (rc == 0) rc = run_pool(key_rows_item, &c, B * H * n_rows, 0, n_threads);
    if (rc == 0 && lse_out) memcpy(lse_out, stats, (size_t)(B * L * H) * sizeof(double));
    free(stats);
    if (!o_out) free(o);
    return rc;
}
