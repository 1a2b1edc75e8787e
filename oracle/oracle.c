/*
 * oracle.c -- CPU oracle for blockwise ring attention.  TEST INFRASTRUCTURE
 * ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg call
 * it; the product library never does.  It shares no code with the CUDA path.
 *
 * Everything is plain fp64 with scalar loops.  Threads only split independent
 * work (query rows, keys, heads); they never change the order of a sum.
 *
 * Sources (web pages on sequence parallelism and ring attention):
 *   [ZZ]  "Context parallelism and zig-zag ring attention" (Chinese translation
 *         of Khang Pham's article), section "Zig Zag Ring Attention".
 *   [SP]  "Sequenzparallelitaet und Ringaufmerksamkeit" (aiunderstanding.org),
 *         sections "Tiefer Einblick" and the FAQ.
 *   [TH]  "Sequence Parallelism and Ring Attention", Thai edition of [SP],
 *         section "technical insight".
 *
 * Tensor layouts (row-major, natural token order unless stated):
 *   q, out, dout, dq : [B][S][H][D]      k, v, dk, dv : [B][S][Hkv][D]
 *   lse              : [B][H][S]
 * Query head h reads key/value head h / (H / Hkv)  (grouped heads).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OL_CONTIGUOUS 0
#define OL_STRIPED 1
#define OL_ZIGZAG 2

/* ------------------------------------------------------------------------ */
/* Layout maps.                                                              */
/* ------------------------------------------------------------------------ */

/*
 * oracle_layout_positions: for every shard r and local slot j, the global
 * token position held there, written pos[r * n + j], n = S / P.  Built by
 * dealing tokens out one by one, never by a closed-form formula:
 *   contiguous ([SP] "Tiefer Einblick": each GPU owns a contiguous run of
 *     tokens): shard r receives tokens r*n ... r*n + n - 1 in turn;
 *   striped ([ZZ]: GPU 0 gets tokens 0, 4, 8, ..., GPU 1 gets 1, 5, 9, ...;
 *     that page calls this interleaving "zig-zag"): token i is dealt to shard
 *     i mod P, round-robin like cards;
 *   zig-zag ([SP] "Die Zukunft ..." names striped and zig-zag variants; the
 *     pages do not spell it out, the reading used is: cut the sequence into
 *     2P equal chunks, shard r holds chunk r followed by chunk 2P-1-r).
 * Within a shard the positions come out increasing.  Returns 0 on success,
 * -1 on bad arguments (P < 1, S not divisible by P, or by 2P for zig-zag).
 */
int oracle_layout_positions(int64_t S, int P, int layout, int64_t *pos)
{
    if (P < 1 || S < 0 || S % P != 0) return -1;
    int64_t n = S / P;
    if (layout == OL_CONTIGUOUS) {
        int64_t next = 0;
        for (int r = 0; r < P; ++r)
            for (int64_t j = 0; j < n; ++j) pos[r * n + j] = next++;
        return 0;
    }
    if (layout == OL_STRIPED) {
        int64_t *fill = calloc((size_t)P, sizeof(int64_t));
        if (!fill) return -1;
        for (int64_t i = 0; i < S; ++i) {
            int r = (int)(i % P);           /* the dealer's next hand */
            pos[r * n + fill[r]] = i;
            fill[r] += 1;
        }
        free(fill);
        return 0;
    }
    if (layout == OL_ZIGZAG) {
        if (S % (2 * (int64_t)P) != 0) return -1;
        int64_t C = S / (2 * (int64_t)P);
        for (int r = 0; r < P; ++r) {
            int64_t j = 0;
            int chunks[2] = {r, 2 * P - 1 - r};
            for (int c = 0; c < 2; ++c)
                for (int64_t t = 0; t < C; ++t) pos[r * n + j++] = (int64_t)chunks[c] * C + t;
        }
        return 0;
    }
    return -1;
}

/* ------------------------------------------------------------------------ */
/* Thread pool helper: run fn(ctx, item) for item in [0, count).             */
/* ------------------------------------------------------------------------ */

typedef void (*item_fn)(void *ctx, int64_t item);
typedef struct {
    item_fn fn;
    void *ctx;
    int64_t count;
    int64_t next;
    pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int64_t it = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (it >= p->count) break;
        p->fn(p->ctx, it);
    }
    return NULL;
}

static void run_items(item_fn fn, void *ctx, int64_t count, int nthreads)
{
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.count = count; p.next = 0;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > count) nthreads = (int)(count > 0 ? count : 1);
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, pool_worker, &p) == 0) ++started;
    pool_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------------ */
/* Full attention, the plain definition.                                     */
/* ------------------------------------------------------------------------ */

/*
 * For query (b, h) at global position i, with g = h / (H/Hkv) and visible
 * keys V_i = {j <= i} if causal else all j ([ZZ]: in an autoregressive model
 * a token only sees earlier tokens):
 *   s_j   = scale * sum_d q[b,i,h,d] k[b,j,g,d]
 *   m     = max_j s_j,   l = sum_j exp(s_j - m)
 *   out   = sum_j exp(s_j - m) v[b,j,g,:] / l,    lse = m + ln l.
 * qrows holds only the queries asked for: qrows[b][t][h][d] is the query at
 * position rows[t].  Results go to out[b][t][h][d] and lse[b][h][t].
 */
typedef struct {
    const double *qrows, *k, *v;
    const int64_t *rows;
    int64_t nrows, S;
    int B, H, Hkv, D, causal;
    double scale;
    double *out, *lse;
} fwd_ctx;

static void fwd_item(void *vctx, int64_t item)
{
    fwd_ctx *c = (fwd_ctx *)vctx;
    const int B = c->B, H = c->H, Hkv = c->Hkv, D = c->D;
    const int64_t S = c->S, nr = c->nrows;
    int64_t t = item % nr;
    int h = (int)((item / nr) % H);
    int b = (int)(item / (nr * H));
    (void)B;
    int g = h / (H / Hkv);
    int64_t i = c->rows[t];
    int64_t last = c->causal ? i : S - 1;
    const double *qi = c->qrows + (((int64_t)b * nr + t) * H + h) * D;
    double *sc = malloc(sizeof(double) * (size_t)(last + 1));
    double m = -INFINITY;
    for (int64_t j = 0; j <= last; ++j) {
        const double *kj = c->k + (((int64_t)b * S + j) * Hkv + g) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
        sc[j] = c->scale * dot;
        if (sc[j] > m) m = sc[j];
    }
    double l = 0.0;
    double *o = c->out + (((int64_t)b * nr + t) * H + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        double p = exp(sc[j] - m);
        l += p;
        const double *vj = c->v + (((int64_t)b * S + j) * Hkv + g) * D;
        for (int d = 0; d < D; ++d) o[d] += p * vj[d];
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    c->lse[((int64_t)b * H + h) * nr + t] = m + log(l);
    free(sc);
}

int oracle_attn_fwd_rows(const double *qrows, const double *k, const double *v, int B, int H,
                         int Hkv, int64_t S, int D, int causal, double scale,
                         const int64_t *rows, int64_t nrows, double *out, double *lse,
                         int nthreads)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || S < 1 || nrows < 0) return -1;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= S) return -1;
    fwd_ctx c = {qrows, k, v, rows, nrows, S, B, H, Hkv, D, causal, scale, out, lse};
    run_items(fwd_item, &c, (int64_t)B * H * nrows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Blockwise ring order with online softmax.                                 */
/* ------------------------------------------------------------------------ */

/*
 * The ring algorithm as the pages tell it ([SP] "Tiefer Einblick", [TH]
 * "technical insight"): shard r keeps its queries; at ring step t it holds
 * the key/value block of shard s = (r - t) mod P (each rank receives from the
 * previous one).  For each arriving block it computes partial attention and
 * folds it into a running maximum m and running normaliser l, rescaling the
 * earlier partial sums when a larger score appears.  After P steps every
 * query has met every key.  Natural-order output, same layout as the full
 * definition above (all S rows).
 */
typedef struct {
    const double *q, *k, *v;
    const int64_t *pos; /* [P][n] */
    int64_t S, n;
    int P, B, H, Hkv, D, causal;
    double scale;
    double *out, *lse;
} ring_ctx;

static void ring_item(void *vctx, int64_t item)
{
    ring_ctx *c = (ring_ctx *)vctx;
    const int H = c->H, Hkv = c->Hkv, D = c->D, P = c->P;
    const int64_t S = c->S, n = c->n;
    int64_t j = item % n;
    int r = (int)((item / n) % P);
    int h = (int)((item / (n * P)) % H);
    int b = (int)(item / (n * P * H));
    int g = h / (H / Hkv);
    int64_t i = c->pos[(int64_t)r * n + j];
    const double *qi = c->q + (((int64_t)b * S + i) * H + h) * D;
    double m = -INFINITY, l = 0.0;
    double *acc = calloc((size_t)D, sizeof(double));
    double *sc = malloc(sizeof(double) * (size_t)n);
    for (int t = 0; t < P; ++t) {
        int s = ((r - t) % P + P) % P;
        /* partial scores against the arriving block */
        double mb = -INFINITY;
        for (int64_t u = 0; u < n; ++u) {
            int64_t jj = c->pos[(int64_t)s * n + u];
            if (c->causal && jj > i) { sc[u] = -INFINITY; continue; }
            const double *kj = c->k + (((int64_t)b * S + jj) * Hkv + g) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
            sc[u] = c->scale * dot;
            if (sc[u] > mb) mb = sc[u];
        }
        if (mb == -INFINITY) continue; /* nothing visible in this block */
        double mnew = m > mb ? m : mb;
        double corr = exp(m - mnew); /* exp(-inf) = 0 on the first block */
        l *= corr;
        for (int d = 0; d < D; ++d) acc[d] *= corr;
        for (int64_t u = 0; u < n; ++u) {
            if (sc[u] == -INFINITY) continue;
            int64_t jj = c->pos[(int64_t)s * n + u];
            double p = exp(sc[u] - mnew);
            l += p;
            const double *vj = c->v + (((int64_t)b * S + jj) * Hkv + g) * D;
            for (int d = 0; d < D; ++d) acc[d] += p * vj[d];
        }
        m = mnew;
    }
    double *o = c->out + (((int64_t)b * S + i) * H + h) * D;
    for (int d = 0; d < D; ++d) o[d] = acc[d] / l;
    c->lse[((int64_t)b * H + h) * S + i] = m + log(l);
    free(acc);
    free(sc);
}

int oracle_ring_fwd(const double *q, const double *k, const double *v, int B, int H, int Hkv,
                    int64_t S, int D, int P, int layout, int causal, double scale, double *out,
                    double *lse, int nthreads)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || S < 1 || P < 1) return -1;
    int64_t *pos = malloc(sizeof(int64_t) * (size_t)S);
    if (!pos) return -1;
    if (oracle_layout_positions(S, P, layout, pos) != 0) { free(pos); return -1; }
    ring_ctx c = {q, k, v, pos, S, S / P, P, B, H, Hkv, D, causal, scale, out, lse};
    run_items(ring_item, &c, (int64_t)B * H * S, nthreads);
    free(pos);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One ring hop: partial attention of shard r against block s.               */
/* ------------------------------------------------------------------------ */

/*
 * The unit one ring hop produces ([SP] "Tiefer Einblick": on each arriving
 * block the GPU computes a partial attention): the queries of shard r against
 * the keys of shard s only, causal on GLOBAL positions, normalised within the
 * block.  Inputs are in shard-local order: q_shard[b][j][h][d] is the query at
 * position pos_r(j), k_shard/v_shard[b][u][g][d] the key/value at pos_s(u).
 * Outputs: out_part[b][j][h][d] (normalised partial) and lse_part[b][h][j].
 * A query that sees no key of the block gets out 0 and lse -infinity.
 */
typedef struct {
    const double *q, *k, *v;
    const int64_t *pos;
    int64_t n;
    int P, r, s, B, H, Hkv, D, causal;
    double scale;
    double *out, *lse;
} step_ctx;

static void step_item(void *vctx, int64_t item)
{
    step_ctx *c = (step_ctx *)vctx;
    const int H = c->H, Hkv = c->Hkv, D = c->D;
    const int64_t n = c->n;
    int64_t j = item % n;
    int h = (int)((item / n) % H);
    int b = (int)(item / (n * H));
    int g = h / (H / Hkv);
    int64_t i = c->pos[(int64_t)c->r * n + j];
    const double *qi = c->q + (((int64_t)b * n + j) * H + h) * D;
    double *sc = malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int64_t u = 0; u < n; ++u) {
        int64_t pu = c->pos[(int64_t)c->s * n + u];
        if (c->causal && pu > i) { sc[u] = -INFINITY; continue; }
        const double *ku = c->k + (((int64_t)b * n + u) * Hkv + g) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qi[d] * ku[d];
        sc[u] = c->scale * dot;
        if (sc[u] > m) m = sc[u];
    }
    double *o = c->out + (((int64_t)b * n + j) * H + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    double *lse = c->lse + ((int64_t)b * H + h) * n + j;
    if (m == -INFINITY) { *lse = -INFINITY; free(sc); return; }
    double l = 0.0;
    for (int64_t u = 0; u < n; ++u) {
        if (sc[u] == -INFINITY) continue;
        double p = exp(sc[u] - m);
        l += p;
        const double *vu = c->v + (((int64_t)b * n + u) * Hkv + g) * D;
        for (int d = 0; d < D; ++d) o[d] += p * vu[d];
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
    free(sc);
}

int oracle_step(const double *q_shard, const double *k_shard, const double *v_shard, int B,
                int H, int Hkv, int64_t S, int D, int P, int layout, int r, int s, int causal,
                double scale, double *out_part, double *lse_part, int nthreads)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || S < 1 || P < 1) return -1;
    if (r < 0 || r >= P || s < 0 || s >= P) return -1;
    int64_t *pos = malloc(sizeof(int64_t) * (size_t)S);
    if (!pos) return -1;
    if (oracle_layout_positions(S, P, layout, pos) != 0) { free(pos); return -1; }
    step_ctx c = {q_shard, k_shard, v_shard, pos, S / P, P, r, s, B, H, Hkv, D, causal, scale,
                  out_part, lse_part};
    run_items(step_item, &c, (int64_t)B * H * (S / P), nthreads);
    free(pos);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Merge of two partial results.                                             */
/* ------------------------------------------------------------------------ */

/*
 * Folding one hop's partial into the running result ([SP] "Tiefer Einblick":
 * results are accumulated with online softmax).  With each partial normalised
 * by its own sum, the running state (m, l) of the pages is carried as
 * lse = m + ln l, and the fold is
 *   lse = ln(exp(lse1) + exp(lse2)),  out = exp(lse1-lse) out1 + exp(lse2-lse) out2.
 * out_*: [B][n][H][D], lse_*: [B][H][n].  (out_acc, lse_acc) is updated in
 * place.  Both -infinity: the row stays (0, -infinity).
 */
void oracle_merge(double *out_acc, double *lse_acc, const double *out_part,
                  const double *lse_part, int B, int H, int64_t n, int D)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t j = 0; j < n; ++j) {
                double *la = lse_acc + ((int64_t)b * H + h) * n + j;
                double lp = lse_part[((int64_t)b * H + h) * n + j];
                double *oa = out_acc + (((int64_t)b * n + j) * H + h) * D;
                const double *op = out_part + (((int64_t)b * n + j) * H + h) * D;
                double l1 = *la, l2 = lp;
                if (l1 == -INFINITY && l2 == -INFINITY) {
                    for (int d = 0; d < D; ++d) oa[d] = 0.0;
                    continue;
                }
                double mx = l1 > l2 ? l1 : l2;
                double lse = mx + log(exp(l1 - mx) + exp(l2 - mx));
                double w1 = exp(l1 - lse), w2 = exp(l2 - lse);
                for (int d = 0; d < D; ++d) oa[d] = w1 * oa[d] + w2 * op[d];
                *la = lse;
            }
}

/* ------------------------------------------------------------------------ */
/* Backward of full attention (the pages are silent; textbook gradient).     */
/* ------------------------------------------------------------------------ */

/*
 * Gradients of out = softmax(scale q k^T + mask) v with respect to q, k, v,
 * given dout:  P_ij = exp(s_ij - lse_i),  delta_i = sum_d dout_id out_id,
 *   dv_j = sum_i P_ij dout_i,   dP_ij = dout_i . v_j,
 *   dS_ij = P_ij (dP_ij - delta_i),
 *   dq_i = scale sum_j dS_ij k_j,   dk_j = scale sum_i dS_ij q_i.
 * out and lse are recomputed here in fp64 from q, k, v.  Computed for a list
 * of (b, g) pairs (g a key/value head; all H/Hkv query heads of the group):
 *   dq_sel[t][G][S][D], dk_sel[t][S][D], dv_sel[t][S][D]   for t < npairs,
 * where G = H / Hkv and query head h = g*G + e is stored at index e.
 */
typedef struct {
    const double *q, *k, *v, *dout;
    const int *bg;
    int64_t S;
    int B, H, Hkv, D, causal, G;
    double scale;
    double *lse, *delta;            /* [npairs][G][S] scratch */
    double *dq, *dk, *dv;
} bwd_ctx;

#define QIDX(c, b, i, h) ((((int64_t)(b) * (c)->S + (i)) * (c)->H + (h)) * (c)->D)
#define KIDX(c, b, j, g) ((((int64_t)(b) * (c)->S + (j)) * (c)->Hkv + (g)) * (c)->D)

/* pass 1, one item per (pair, e, query row): lse, delta and dq */
static void bwd_rows_item(void *vctx, int64_t item)
{
    bwd_ctx *c = (bwd_ctx *)vctx;
    const int64_t S = c->S;
    const int D = c->D, G = c->G;
    int64_t i = item % S;
    int e = (int)((item / S) % G);
    int t = (int)(item / (S * G));
    int b = c->bg[2 * t], g = c->bg[2 * t + 1];
    int h = g * G + e;
    int64_t last = c->causal ? i : S - 1;
    const double *qi = c->q + QIDX(c, b, i, h);
    const double *doi = c->dout + QIDX(c, b, i, h);
    double *sc = malloc(sizeof(double) * (size_t)(last + 1));
    double m = -INFINITY;
    for (int64_t j = 0; j <= last; ++j) {
        const double *kj = c->k + KIDX(c, b, j, g);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
        sc[j] = c->scale * dot;
        if (sc[j] > m) m = sc[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j <= last; ++j) l += exp(sc[j] - m);
    double lse = m + log(l);
    /* out_i, then delta_i = dout_i . out_i */
    double *o = calloc((size_t)D, sizeof(double));
    for (int64_t j = 0; j <= last; ++j) {
        double p = exp(sc[j] - lse);
        const double *vj = c->v + KIDX(c, b, j, g);
        for (int d = 0; d < D; ++d) o[d] += p * vj[d];
    }
    double delta = 0.0;
    for (int d = 0; d < D; ++d) delta += doi[d] * o[d];
    int64_t si = ((int64_t)t * G + e) * S + i;
    c->lse[si] = lse;
    c->delta[si] = delta;
    double *dq = c->dq + si * D;
    for (int d = 0; d < D; ++d) dq[d] = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        double p = exp(sc[j] - lse);
        const double *vj = c->v + KIDX(c, b, j, g);
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += doi[d] * vj[d];
        double ds = p * (dp - delta);
        const double *kj = c->k + KIDX(c, b, j, g);
        for (int d = 0; d < D; ++d) dq[d] += ds * kj[d];
    }
    for (int d = 0; d < D; ++d) dq[d] *= c->scale;
    free(o);
    free(sc);
}

/* pass 2, one item per (pair, key row): dk and dv summed over the group */
static void bwd_keys_item(void *vctx, int64_t item)
{
    bwd_ctx *c = (bwd_ctx *)vctx;
    const int64_t S = c->S;
    const int D = c->D, G = c->G;
    int64_t j = item % S;
    int t = (int)(item / S);
    int b = c->bg[2 * t], g = c->bg[2 * t + 1];
    const double *kj = c->k + KIDX(c, b, j, g);
    const double *vj = c->v + KIDX(c, b, j, g);
    double *dk = c->dk + ((int64_t)t * S + j) * D;
    double *dv = c->dv + ((int64_t)t * S + j) * D;
    for (int d = 0; d < D; ++d) { dk[d] = 0.0; dv[d] = 0.0; }
    for (int e = 0; e < G; ++e) {
        int h = g * G + e;
        int64_t first = c->causal ? j : 0;
        for (int64_t i = first; i < S; ++i) {
            const double *qi = c->q + QIDX(c, b, i, h);
            const double *doi = c->dout + QIDX(c, b, i, h);
            int64_t si = ((int64_t)t * G + e) * S + i;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
            double p = exp(c->scale * dot - c->lse[si]);
            double dp = 0.0;
            for (int d = 0; d < D; ++d) dp += doi[d] * vj[d];
            double ds = p * (dp - c->delta[si]);
            for (int d = 0; d < D; ++d) {
                dv[d] += p * doi[d];
                dk[d] += ds * qi[d];
            }
        }
    }
    for (int d = 0; d < D; ++d) dk[d] *= c->scale;
}

int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int B, int H, int Hkv, int64_t S, int D, int causal, double scale,
                    const int *bg_pairs, int npairs, double *dq_sel, double *dk_sel,
                    double *dv_sel, int nthreads)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || S < 1 || npairs < 1) return -1;
    for (int t = 0; t < npairs; ++t)
        if (bg_pairs[2 * t] < 0 || bg_pairs[2 * t] >= B || bg_pairs[2 * t + 1] < 0 ||
            bg_pairs[2 * t + 1] >= Hkv)
            return -1;
    int G = H / Hkv;
    double *lse = malloc(sizeof(double) * (size_t)npairs * G * S);
    double *delta = malloc(sizeof(double) * (size_t)npairs * G * S);
    if (!lse || !delta) { free(lse); free(delta); return -1; }
    bwd_ctx c = {q, k, v, dout, bg_pairs, S, B, H, Hkv, D, causal, G, scale,
                 lse, delta, dq_sel, dk_sel, dv_sel};
    run_items(bwd_rows_item, &c, (int64_t)npairs * G * S, nthreads);
    run_items(bwd_keys_item, &c, (int64_t)npairs * S, nthreads);
    free(lse);
    free(delta);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Per-shard work census (causal load balance, [ZZ]).                        */
/* ------------------------------------------------------------------------ */

/*
 * [ZZ] explains that under a causal mask a plain contiguous split leaves the
 * later ranks with more work and the earlier ones idle, and that interleaving
 * evens it out.  This counts, by brute force over every (query, key) pair:
 *   pairs[r]  = number of visible (query, key) pairs whose query lives on
 *               shard r (all key blocks of the ring);
 *   tiles[r]  = number of (query tile, key tile) blocks with at least one
 *               visible pair.
 * A tile is `tile` consecutive local slots of one shard.  With run > 0 the
 * local slots are first cut into runs of `run` slots and no tile straddles two
 * runs (the last tile of a run may be shorter): run = C gives tiles that stay
 * inside one zig-zag chunk, which is how a kernel that loads each tile as one
 * run of consecutive positions must cut them.  run = 0 cuts only at the end
 * of the shard.  Threads split the shards r; each shard's counts are summed
 * in one thread.  O(S^2) work.
 */
typedef struct {
    const int64_t *pos;
    int64_t n, run, tiles_per_run, nt;
    int P, causal, tile;
    int64_t *pairs, *tiles;
    unsigned char *seen;   /* nt * nt flags per thread slot, indexed by shard r */
} census_ctx;

static int64_t census_tile_of(const census_ctx *c, int64_t j)
{
    return (j / c->run) * c->tiles_per_run + (j % c->run) / c->tile;
}

static void census_item(void *vctx, int64_t r)
{
    census_ctx *c = (census_ctx *)vctx;
    unsigned char *seen = c->seen + r * c->nt * c->nt;
    int64_t npairs = 0, ntiles = 0;
    for (int s = 0; s < c->P; ++s) {
        memset(seen, 0, (size_t)(c->nt * c->nt));
        for (int64_t j = 0; j < c->n; ++j) {
            int64_t qp = c->pos[r * c->n + j];
            int64_t tq = census_tile_of(c, j);
            for (int64_t u = 0; u < c->n; ++u) {
                if (c->causal && c->pos[(int64_t)s * c->n + u] > qp) continue;
                npairs += 1;
                seen[tq * c->nt + census_tile_of(c, u)] = 1;
            }
        }
        for (int64_t t = 0; t < c->nt * c->nt; ++t) ntiles += seen[t];
    }
    c->pairs[r] = npairs;
    c->tiles[r] = ntiles;
}

int oracle_work_census(int64_t S, int P, int layout, int causal, int tile, int64_t run,
                       int64_t *pairs, int64_t *tiles, int nthreads)
{
    if (tile < 1 || run < 0) return -1;
    int64_t *pos = malloc(sizeof(int64_t) * (size_t)(S > 0 ? S : 1));
    if (!pos) return -1;
    if (oracle_layout_positions(S, P, layout, pos) != 0) { free(pos); return -1; }
    census_ctx c;
    c.pos = pos;
    c.n = S / P;
    c.run = run > 0 && run < c.n ? run : c.n;
    if (c.run < 1) c.run = 1;
    c.tiles_per_run = (c.run + tile - 1) / tile;
    c.nt = ((c.n + c.run - 1) / c.run) * c.tiles_per_run;
    c.P = P; c.causal = causal; c.tile = tile;
    c.pairs = pairs; c.tiles = tiles;
    c.seen = malloc((size_t)(P * c.nt * c.nt > 0 ? P * c.nt * c.nt : 1));
    if (!c.seen) { free(pos); return -1; }
    run_items(census_item, &c, P, nthreads);
    free(c.seen);
    free(pos);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Row permutation by the layout map (byte copy).                            */
/* ------------------------------------------------------------------------ */

/*
 * Gathers token rows into shard-major order: dst[o][r*n + j] = src[o][pos_r(j)]
 * for each of `outer` independent slabs of S rows of row_bytes bytes.  With
 * inverse != 0 it scatters them back: dst[o][pos_r(j)] = src[o][r*n + j].
 */
int oracle_permute(const unsigned char *src, unsigned char *dst, int64_t outer, int64_t S,
                   int64_t row_bytes, int P, int layout, int inverse)
{
    int64_t *pos = malloc(sizeof(int64_t) * (size_t)S);
    if (!pos) return -1;
    if (oracle_layout_positions(S, P, layout, pos) != 0) { free(pos); return -1; }
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t slot = 0; slot < S; ++slot) {
            int64_t g = pos[slot];
            const unsigned char *from = src + (o * S + (inverse ? slot : g)) * row_bytes;
            unsigned char *to = dst + (o * S + (inverse ? g : slot)) * row_bytes;
            memcpy(to, from, (size_t)row_bytes);
        }
    free(pos);
    return 0;
}
