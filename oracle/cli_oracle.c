/*
 * Float64 CPU oracle of the in-batch contrastive scoring path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing of the product path links, loads or calls
 * this file: only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline
 * leg (and its `--impl reference` arm) use it.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Every function is the plain definition of what the method computes, written
 * from the UForm 4 documentation pages:
 *   - "UForm" (uform.md), section "Matryoshka-Like Multi-Scale Embedders": the
 *     SigLIP loss, one independent sigmoid cross-entropy per cell of the score
 *     matrix, with inverse temperature t and bias b.
 *   - "Training" (uform/c/training.md), `uform_pair_loss_form_t`
 *     (`sigmoid`: every repel weighed like an attract), `uform_contrastive_t`
 *     (t, b, negatives, ambient_repulsion_weight), `uform_negatives_t`,
 *     `uform_edges_view_t` and `uform_relations_view_t` (resolution order:
 *     ignore, then attract, then repel, then the run's negatives).
 *   - "UForm", section "ColBERT-Style Late-Interaction Rerankers": the hard
 *     MaxSim score, each query token keeping its single best document token,
 *     with the gradient routed through that best match alone.
 *   - "Arenas" (uform/c/arenas.md), "Rows and Tapes": ragged tapes are data
 *     end to end plus count + 1 offsets.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   - loss normalisation: L = (1/N) * sum over anchors i of the anchor's row
 *     sum (SigLIP's per-anchor loss averaged over the batch's anchors);
 *   - the pooled diagonal (i, i) is never scored;
 *   - dt is dL/dt for the inverse temperature itself;
 *   - hard MaxSim defaults to the sum over query tokens; `mean` divides by |q|;
 *   - ties of the max go to the lowest document-local index.
 *
 * No blocking, fusion or reordering beyond the definitions: dot products are
 * summed in index order, the per-anchor row work of the pooled loss is split
 * over threads by anchor, and per-anchor partial sums are added in anchor
 * order, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* scalar helpers                                                            */
/* ------------------------------------------------------------------------ */

/* sigma(x) = 1 / (1 + exp(-x)), evaluated on the side that cannot overflow. */
double oracle_sigmoid(double x) {
    if (x >= 0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* softplus(x) = log(1 + exp(x)) = max(x, 0) + log1p(exp(-|x|)). */
double oracle_softplus(double x) { return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x))); }

static double dot(const double *a, const double *b, int64_t width) {
    double s = 0.0;
    for (int64_t k = 0; k < width; ++k) s += a[k] * b[k];
    return s;
}

/* ------------------------------------------------------------------------ */
/* relations                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint64_t *offsets; /* count + 1, or NULL for "no edges" */
    const uint32_t *ids;
    const double *weights;   /* NULL: every edge weighs one */
} edges_t;

/* Is (i -> j) in the edge set?  Linear scan of row i; *w gets its weight. */
static int edge_lookup(const edges_t *set, int64_t i, int64_t j, double *w) {
    if (!set->offsets) return 0;
    for (uint64_t k = set->offsets[i]; k < set->offsets[i + 1]; ++k) {
        if ((int64_t)set->ids[k] == j) {
            if (w) *w = set->weights ? set->weights[k] : 1.0;
            return 1;
        }
    }
    return 0;
}

/*
 * Resolution of one ordered pair (training.md, `uform_relations_view_t`):
 * ignore first, then attract, then repel, then the run's negatives.
 * Returns 0 when the pair is skipped; otherwise *y = +1 (attract) or -1
 * (repel) and *w = its weight.
 */
static int resolve(const edges_t *att, const edges_t *rep, const edges_t *ign, int named,
                   double ambient, int64_t i, int64_t j, double *y, double *w) {
    if (edge_lookup(ign, i, j, NULL)) return 0;
    if (edge_lookup(att, i, j, w)) { *y = +1.0; return 1; }
    if (edge_lookup(rep, i, j, w)) { *y = -1.0; return 1; }
    if (named) return 0;
    *y = -1.0;
    *w = ambient;
    return 1;
}

/* One cell: loss w * (-log sigma(y z)) and its derivative with respect to z. */
static void cell(double y, double w, double z, double *loss, double *dloss_dz) {
    *loss = w * oracle_softplus(-y * z);      /* -log sigma(yz) = softplus(-yz) */
    *dloss_dz = -w * y * oracle_sigmoid(-y * z);
}

/* ------------------------------------------------------------------------ */
/* tiny thread pool over an index range                                       */
/* ------------------------------------------------------------------------ */

typedef void (*range_fn)(void *ctx, int64_t begin, int64_t end, int slot);
typedef struct { range_fn fn; void *ctx; int64_t begin, end; int slot; } job_t;

static void *job_main(void *p) {
    job_t *j = (job_t *)p;
    j->fn(j->ctx, j->begin, j->end, j->slot);
    return NULL;
}

/* Splits [0, n) into `threads` contiguous slices; slice s runs with slot s. */
static void parallel_for(int64_t n, int threads, range_fn fn, void *ctx) {
    if (threads < 1) threads = 1;
    if (threads > n) threads = (int)(n > 0 ? n : 1);
    pthread_t tid[256];
    job_t jobs[256];
    if (threads > 256) threads = 256;
    for (int s = 0; s < threads; ++s) {
        jobs[s].fn = fn;
        jobs[s].ctx = ctx;
        jobs[s].begin = n * s / threads;
        jobs[s].end = n * (s + 1) / threads;
        jobs[s].slot = s;
    }
    for (int s = 1; s < threads; ++s) pthread_create(&tid[s], NULL, job_main, &jobs[s]);
    job_main(&jobs[0]);
    for (int s = 1; s < threads; ++s) pthread_join(tid[s], NULL);
}

/* ------------------------------------------------------------------------ */
/* pooled sigmoid pair loss                                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t n, width;
    const double *e;
    double t, b;
    edges_t att, rep, ign;
    int named;
    double ambient;
    const int64_t *rows; /* anchors to evaluate; NULL = all, in order */
    double *row_loss;    /* per evaluated anchor: (1/N) sum_j l_ij */
    double *de;          /* per evaluated anchor: dL/de_i (width values) */
    double *part;        /* per evaluated anchor: its loss, dt and db shares */
} pooled_ctx;

/*
 * Anchor i's share of the loss, and the full gradient with respect to e_i.
 * L = (1/N) sum_i sum_{j != i} l_ij with l_ij = w_ij softplus(-y_ij z_ij),
 * z_ij = t <e_i, e_j> + b.  e_i enters z_ij and z_ji, so
 * dL/de_i = (t/N) sum_j (dl_ij/dz + dl_ji/dz) e_j, while dL/dt and dL/db
 * collect every ordered pair once; here each anchor adds its own pairs (i, j).
 */
static void pooled_rows(void *p, int64_t begin, int64_t end, int slot) {
    (void)slot;
    pooled_ctx *c = (pooled_ctx *)p;
    const double inv_n = 1.0 / (double)c->n;
    for (int64_t r = begin; r < end; ++r) {
        double dt = 0, db = 0;
        int64_t i = c->rows ? c->rows[r] : r;
        const double *ei = c->e + i * c->width;
        double *gi = c->de ? c->de + r * c->width : NULL;
        if (gi) memset(gi, 0, sizeof(double) * (size_t)c->width);
        double row_loss = 0;
        for (int64_t j = 0; j < c->n; ++j) {
            if (j == i) continue; /* the diagonal is never scored */
            const double *ej = c->e + j * c->width;
            double s = dot(ei, ej, c->width);
            double z = c->t * s + c->b;
            double y, w, l, g_ij = 0, g_ji = 0;
            if (resolve(&c->att, &c->rep, &c->ign, c->named, c->ambient, i, j, &y, &w)) {
                cell(y, w, z, &l, &g_ij);
                row_loss += l;
                dt += g_ij * inv_n * s;
                db += g_ij * inv_n;
            }
            if (resolve(&c->att, &c->rep, &c->ign, c->named, c->ambient, j, i, &y, &w)) {
                cell(y, w, z, &l, &g_ji); /* z_ji = z_ij */
            }
            if (gi) {
                double coef = c->t * (g_ij + g_ji) * inv_n;
                for (int64_t k = 0; k < c->width; ++k) gi[k] += coef * ej[k];
            }
        }
        if (c->row_loss) c->row_loss[r] = row_loss * inv_n;
        c->part[3 * r + 0] = row_loss * inv_n;
        c->part[3 * r + 1] = dt;
        c->part[3 * r + 2] = db;
    }
}

/*
 * Pooled sigmoid pair loss over all anchors, or over the `nrows` anchors
 * listed in `rows` (then `loss`, `dt`, `db` are those anchors' shares and
 * `de`/`row_loss` hold one entry per listed anchor).
 * Edge sets: offsets[n+1] (NULL = none), ids, optional weights.
 */
int oracle_pair_loss_sigmoid(int64_t n, int64_t width, const double *e, double t, double b,
                             const uint64_t *att_off, const uint32_t *att_ids, const double *att_w,
                             const uint64_t *rep_off, const uint32_t *rep_ids, const double *rep_w,
                             const uint64_t *ign_off, const uint32_t *ign_ids,
                             int negatives_named, double ambient_weight,
                             int64_t nrows, const int64_t *rows,
                             double *loss, double *de, double *row_loss, double *dt, double *db,
                             int threads) {
    if (n <= 0 || width <= 0 || !e) return 1;
    pooled_ctx c = {n, width, e, t, b, {att_off, att_ids, att_w}, {rep_off, rep_ids, rep_w},
                    {ign_off, ign_ids, NULL}, negatives_named, ambient_weight, rows, row_loss, de, NULL};
    int64_t m = rows ? nrows : n;
    double *part = (double *)calloc((size_t)(3 * (m > 0 ? m : 1)), sizeof(double));
    if (!part) return 2;
    c.part = part;
    parallel_for(m, threads, pooled_rows, &c);
    /* anchors' shares added in anchor order: independent of the thread count */
    double L = 0, T = 0, B = 0;
    for (int64_t r = 0; r < m; ++r) { L += part[3 * r]; T += part[3 * r + 1]; B += part[3 * r + 2]; }
    free(part);
    if (loss) *loss = L;
    if (dt) *dt = T;
    if (db) *db = B;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* the same loss over a given rectangular score matrix                        */
/* ------------------------------------------------------------------------ */

/*
 * L = (1/R) sum_{i<R} sum_{j<C} w_ij softplus(-y_ij (t S_ij + b)); no implicit
 * diagonal rule (rows and columns are different roles).  With `sides`
 * (R == C), a row whose item is not query-capable (sides & 1 == 0) or a
 * column whose item is not document-capable (sides & 2 == 0) is ignored.
 * dS_ij = t * dl_ij/dz / R; dt = sum g S; db = sum g (g = dl/dz / R).
 */
int oracle_pair_loss_sigmoid_scores(int64_t r_count, int64_t c_count, const double *scores, double t,
                                    double b, const uint64_t *att_off, const uint32_t *att_ids,
                                    const double *att_w, const uint64_t *rep_off, const uint32_t *rep_ids,
                                    const double *rep_w, const uint64_t *ign_off, const uint32_t *ign_ids,
                                    const uint8_t *sides, int negatives_named, double ambient_weight,
                                    double *loss, double *dscores, double *dt, double *db) {
    if (r_count <= 0 || c_count <= 0 || !scores) return 1;
    edges_t att = {att_off, att_ids, att_w}, rep = {rep_off, rep_ids, rep_w}, ign = {ign_off, ign_ids, NULL};
    double inv_r = 1.0 / (double)r_count, L = 0, T = 0, B = 0;
    for (int64_t i = 0; i < r_count; ++i) {
        for (int64_t j = 0; j < c_count; ++j) {
            double s = scores[i * c_count + j], g = 0, y, w, l;
            int scored = !(sides && (!(sides[i] & 1) || !(sides[j] & 2)));
            if (scored && resolve(&att, &rep, &ign, negatives_named, ambient_weight, i, j, &y, &w)) {
                cell(y, w, t * s + b, &l, &g);
                L += l * inv_r;
                T += g * inv_r * s;
                B += g * inv_r;
            }
            if (dscores) dscores[i * c_count + j] = t * g * inv_r;
        }
    }
    *loss = L;
    if (dt) *dt = T;
    if (db) *db = B;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* hard MaxSim                                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t nq, nd, width;
    const uint64_t *q_off, *d_off;
    const double *q, *d;
    int mean;
    int64_t rows_q;
    /* forward over a list of (query, doc) pairs */
    int64_t npairs;
    const int64_t *pq, *pd;
    double *score;      /* per pair */
    int32_t *argmax;    /* per pair, |q| entries at arg_off[pair] */
    double *gap;        /* same indexing, or NULL */
    const int64_t *arg_off;
} maxsim_ctx;

/*
 * One query token t against document d: the best document row (lowest local
 * index on ties: strict ">" while scanning in ascending order), its value,
 * and the gap to the best value among the other rows (+inf if |d| = 1).
 */
static void best_match(const maxsim_ctx *c, int64_t t, int64_t d, double *best, int32_t *arg,
                       double *gap) {
    double b1 = -INFINITY, b2 = -INFINITY;
    int32_t a = -1;
    for (uint64_t s = c->d_off[d]; s < c->d_off[d + 1]; ++s) {
        double v = dot(c->q + t * c->width, c->d + (int64_t)s * c->width, c->width);
        if (v > b1) { b2 = b1; b1 = v; a = (int32_t)(s - c->d_off[d]); }
        else if (v > b2) { b2 = v; }
    }
    *best = b1;
    *arg = a;
    if (gap) *gap = b1 - b2;
}

/* S(q, d) = sum_{t in q} max_{s in d} <q_t, d_s>  (divided by |q| when mean). */
static void pair_rows(void *p, int64_t begin, int64_t end, int slot) {
    (void)slot;
    maxsim_ctx *c = (maxsim_ctx *)p;
    for (int64_t k = begin; k < end; ++k) {
        int64_t q = c->pq[k], d = c->pd[k];
        double S = 0;
        int64_t o = c->arg_off[k];
        for (uint64_t t = c->q_off[q]; t < c->q_off[q + 1]; ++t) {
            double best, gap;
            int32_t a;
            best_match(c, (int64_t)t, d, &best, &a, &gap);
            S += best;
            int64_t local = (int64_t)(t - c->q_off[q]);
            if (c->argmax) c->argmax[o + local] = a;
            if (c->gap) c->gap[o + local] = gap;
        }
        if (c->mean) S /= (double)(c->q_off[q + 1] - c->q_off[q]);
        c->score[k] = S;
    }
}

/*
 * MaxSim forward over listed (query, document) pairs.  For pair k the
 * |q| argmax entries (document-local indices) and top-2 gaps are written at
 * arg_off[k] (a caller-computed prefix sum of the listed queries' lengths).
 */
int oracle_maxsim_pairs(int64_t nq, const uint64_t *q_off, const double *q, int64_t nd,
                        const uint64_t *d_off, const double *d, int64_t width, int mean,
                        int64_t npairs, const int64_t *pq, const int64_t *pd, const int64_t *arg_off,
                        double *score, int32_t *argmax, double *gap, int threads) {
    if (nq <= 0 || nd <= 0 || width <= 0) return 1;
    maxsim_ctx c = {nq, nd, width, q_off, d_off, q, d, mean, (int64_t)q_off[nq],
                    npairs, pq, pd, score, argmax, gap, arg_off};
    parallel_for(npairs, threads, pair_rows, &c);
    return 0;
}

/*
 * MaxSim forward over all pairs.  scores: [nq][nd]; argmax, gap: document
 * major, [nd][rows_q] (entry [d][t] for query token t of the query tape).
 */
typedef struct { maxsim_ctx *c; double *scores; int32_t *argmax; double *gap; } all_ctx;

static void all_rows(void *p, int64_t begin, int64_t end, int slot) {
    (void)slot;
    all_ctx *a = (all_ctx *)p;
    const maxsim_ctx *c = a->c;
    for (int64_t q = begin; q < end; ++q) {
        for (int64_t d = 0; d < c->nd; ++d) {
            double S = 0;
            for (uint64_t t = c->q_off[q]; t < c->q_off[q + 1]; ++t) {
                double best, gap;
                int32_t arg;
                best_match(c, (int64_t)t, d, &best, &arg, &gap);
                S += best;
                if (a->argmax) a->argmax[d * c->rows_q + (int64_t)t] = arg;
                if (a->gap) a->gap[d * c->rows_q + (int64_t)t] = gap;
            }
            if (c->mean) S /= (double)(c->q_off[q + 1] - c->q_off[q]);
            a->scores[q * c->nd + d] = S;
        }
    }
}

int oracle_maxsim_forward(int64_t nq, const uint64_t *q_off, const double *q, int64_t nd,
                          const uint64_t *d_off, const double *d, int64_t width, int mean,
                          double *scores, int32_t *argmax, double *gap, int threads) {
    if (nq <= 0 || nd <= 0 || width <= 0) return 1;
    maxsim_ctx c = {nq, nd, width, q_off, d_off, q, d, mean, (int64_t)q_off[nq],
                    0, NULL, NULL, NULL, NULL, NULL, NULL};
    all_ctx a = {&c, scores, argmax, gap};
    parallel_for(nq, threads, all_rows, &a);
    return 0;
}

/*
 * MaxSim backward through the argmax: with c = dS[q][d] (divided by |q| when
 * mean), every query token t of q and its match a = argmax[d][t] give
 * dQ[t] += c * D[a] and dD[a] += c * Q[t].  The query side is split over
 * threads by query and the document side by document, so every output row
 * has one writer.
 */
typedef struct {
    const maxsim_ctx *c;
    const int32_t *argmax;
    const double *ds;
    double *dq, *dd;
} bwd_ctx;

static void bwd_queries(void *p, int64_t begin, int64_t end, int slot) {
    (void)slot;
    bwd_ctx *b = (bwd_ctx *)p;
    const maxsim_ctx *c = b->c;
    for (int64_t q = begin; q < end; ++q) {
        double len = (double)(c->q_off[q + 1] - c->q_off[q]);
        for (uint64_t t = c->q_off[q]; t < c->q_off[q + 1]; ++t) {
            double *g = b->dq + (int64_t)t * c->width;
            memset(g, 0, sizeof(double) * (size_t)c->width);
            for (int64_t d = 0; d < c->nd; ++d) {
                double coef = b->ds[q * c->nd + d] / (c->mean ? len : 1.0);
                int64_t row = (int64_t)c->d_off[d] + b->argmax[d * c->rows_q + (int64_t)t];
                for (int64_t k = 0; k < c->width; ++k) g[k] += coef * c->d[row * c->width + k];
            }
        }
    }
}

static void bwd_docs(void *p, int64_t begin, int64_t end, int slot) {
    (void)slot;
    bwd_ctx *b = (bwd_ctx *)p;
    const maxsim_ctx *c = b->c;
    for (int64_t d = begin; d < end; ++d) {
        memset(b->dd + (int64_t)c->d_off[d] * c->width, 0,
               sizeof(double) * (size_t)((c->d_off[d + 1] - c->d_off[d]) * (uint64_t)c->width));
        for (int64_t q = 0; q < c->nq; ++q) {
            double len = (double)(c->q_off[q + 1] - c->q_off[q]);
            double coef = b->ds[q * c->nd + d] / (c->mean ? len : 1.0);
            for (uint64_t t = c->q_off[q]; t < c->q_off[q + 1]; ++t) {
                int64_t row = (int64_t)c->d_off[d] + b->argmax[d * c->rows_q + (int64_t)t];
                for (int64_t k = 0; k < c->width; ++k)
                    b->dd[row * c->width + k] += coef * c->q[(int64_t)t * c->width + k];
            }
        }
    }
}

int oracle_maxsim_backward(int64_t nq, const uint64_t *q_off, const double *q, int64_t nd,
                           const uint64_t *d_off, const double *d, int64_t width, int mean,
                           const int32_t *argmax, const double *dscores, double *dq, double *dd,
                           int threads) {
    if (nq <= 0 || nd <= 0 || width <= 0) return 1;
    maxsim_ctx c = {nq, nd, width, q_off, d_off, q, d, mean, (int64_t)q_off[nq],
                    0, NULL, NULL, NULL, NULL, NULL, NULL};
    bwd_ctx b = {&c, argmax, dscores, dq, dd};
    if (dq) parallel_for(nq, threads, bwd_queries, &b);
    if (dd) parallel_for(nd, threads, bwd_docs, &b);
    return 0;
}

/*
 * Gradient rows of one query (dQ for its |q| tokens, given the dS row
 * dscores_row[nd]) or of one document (dD for its |d| rows, given the dS
 * column dscores_col[nq]), each computing the argmax it needs itself.  These
 * let a caller check sampled outputs of a workload too large for the full
 * oracle.
 */
int oracle_maxsim_grad_query(int64_t nq, const uint64_t *q_off, const double *q, int64_t nd,
                             const uint64_t *d_off, const double *d, int64_t width, int mean,
                             int64_t qi, const double *dscores_row, double *dq_rows) {
    maxsim_ctx c = {nq, nd, width, q_off, d_off, q, d, mean, (int64_t)q_off[nq],
                    0, NULL, NULL, NULL, NULL, NULL, NULL};
    double len = (double)(q_off[qi + 1] - q_off[qi]);
    for (uint64_t t = q_off[qi]; t < q_off[qi + 1]; ++t) {
        double *g = dq_rows + (int64_t)(t - q_off[qi]) * width;
        memset(g, 0, sizeof(double) * (size_t)width);
        for (int64_t dd = 0; dd < nd; ++dd) {
            double best;
            int32_t a;
            best_match(&c, (int64_t)t, dd, &best, &a, NULL);
            double coef = dscores_row[dd] / (mean ? len : 1.0);
            int64_t row = (int64_t)d_off[dd] + a;
            for (int64_t k = 0; k < width; ++k) g[k] += coef * d[row * width + k];
        }
    }
    return 0;
}

int oracle_maxsim_grad_doc(int64_t nq, const uint64_t *q_off, const double *q, int64_t nd,
                           const uint64_t *d_off, const double *d, int64_t width, int mean,
                           int64_t di, const double *dscores_col, double *dd_rows) {
    maxsim_ctx c = {nq, nd, width, q_off, d_off, q, d, mean, (int64_t)q_off[nq],
                    0, NULL, NULL, NULL, NULL, NULL, NULL};
    memset(dd_rows, 0, sizeof(double) * (size_t)((d_off[di + 1] - d_off[di]) * (uint64_t)width));
    for (int64_t qq = 0; qq < nq; ++qq) {
        double len = (double)(q_off[qq + 1] - q_off[qq]);
        double coef = dscores_col[qq] / (mean ? len : 1.0);
        for (uint64_t t = q_off[qq]; t < q_off[qq + 1]; ++t) {
            double best;
            int32_t a;
            best_match(&c, (int64_t)t, di, &best, &a, NULL);
            for (int64_t k = 0; k < width; ++k) dd_rows[(int64_t)a * width + k] += coef * q[(int64_t)t * width + k];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* the `balanced` and `ranked` pair-loss forms over a score matrix            */
/* ------------------------------------------------------------------------ */

/*
 * "Training", `uform_pair_loss_form_t`:
 *   balanced -- the sigmoid cross-entropy of every cell, its attract and repel
 *               halves normalized apart;
 *   ranked   -- the sigmoid cross-entropy of every positive's score over every
 *               negative's, where the bias cancels.
 * Readings (the pages give words only):
 *   balanced: per row p, l_p = sum_{attract} w l / sum_{attract} w
 *                            + sum_{repel} w l / sum_{repel} w,
 *             each half present only when the row has such cells, with the
 *             sigmoid cell loss l = softplus(-y (t S + b));
 *   ranked:   per row p, l_p = sum_{i in P, j in N} w_i w_j softplus(-t (S_pi - S_pj))
 *                            / sum_{i in P, j in N} w_i w_j,
 *             P the row's attract cells, N its repel cells (explicit or ambient),
 *             0 when either is empty;
 *   both:     L = (1/R) sum_p l_p; relations and sides resolve cells exactly
 *             as in oracle_pair_loss_sigmoid_scores.
 * form: 1 = balanced, 2 = ranked (the pages' enumerator values).
 */
int oracle_pair_loss_scores_form(int form, int64_t r_count, int64_t c_count, const double *scores, double t,
                                 double b, const uint64_t *att_off, const uint32_t *att_ids, const double *att_w,
                                 const uint64_t *rep_off, const uint32_t *rep_ids, const double *rep_w,
                                 const uint64_t *ign_off, const uint32_t *ign_ids, const uint8_t *sides,
                                 int negatives_named, double ambient_weight, double *loss, double *dscores,
                                 double *dt, double *db) {
    if (r_count <= 0 || c_count <= 0 || !scores || (form != 1 && form != 2)) return 1;
    edges_t att = {att_off, att_ids, att_w}, rep = {rep_off, rep_ids, rep_w}, ign = {ign_off, ign_ids, NULL};
    double *y = (double *)malloc(sizeof(double) * (size_t)c_count);
    double *w = (double *)malloc(sizeof(double) * (size_t)c_count);
    if (!y || !w) { free(y); free(w); return 2; }
    const double inv_r = 1.0 / (double)r_count;
    double L = 0, T = 0, B = 0;
    if (dscores) memset(dscores, 0, sizeof(double) * (size_t)(r_count * c_count));
    for (int64_t i = 0; i < r_count; ++i) {
        const double *s = scores + i * c_count;
        double *ds = dscores ? dscores + i * c_count : NULL;
        double wa = 0, wr = 0;
        for (int64_t j = 0; j < c_count; ++j) {
            y[j] = 0;
            w[j] = 0;
            int scored = !(sides && (!(sides[i] & 1) || !(sides[j] & 2)));
            if (scored && resolve(&att, &rep, &ign, negatives_named, ambient_weight, i, j, &y[j], &w[j])) {
                if (y[j] > 0) wa += w[j]; else wr += w[j];
            } else {
                y[j] = 0;
                w[j] = 0;
            }
        }
        if (form == 1) {
            for (int64_t j = 0; j < c_count; ++j) {
                if (y[j] == 0) continue;
                const double norm = y[j] > 0 ? wa : wr;
                double l, g;
                cell(y[j], w[j], t * s[j] + b, &l, &g);   /* g = dl/dz */
                L += l / norm * inv_r;
                T += g / norm * inv_r * s[j];
                B += g / norm * inv_r;
                if (ds) ds[j] = t * g / norm * inv_r;
            }
        } else {
            double z = 0;
            for (int64_t a = 0; a < c_count; ++a)
                if (y[a] > 0)
                    for (int64_t n = 0; n < c_count; ++n)
                        if (y[n] < 0) z += w[a] * w[n];
            if (z <= 0) continue;
            for (int64_t a = 0; a < c_count; ++a) {
                if (y[a] <= 0) continue;
                for (int64_t n = 0; n < c_count; ++n) {
                    if (y[n] >= 0) continue;
                    const double pw = w[a] * w[n] / z * inv_r;
                    const double m = t * (s[a] - s[n]);
                    /* softplus(-m) = -log sigma(m); d/dm = -sigma(-m) */
                    L += pw * oracle_softplus(-m);
                    const double dm = -pw * oracle_sigmoid(-m);
                    T += dm * (s[a] - s[n]);
                    if (ds) {
                        ds[a] += dm * t;
                        ds[n] -= dm * t;
                    }
                }
            }
        }
    }
    free(y);
    free(w);
    *loss = L;
    if (dt) *dt = T;
    if (db) *db = B;
    return 0;
}
