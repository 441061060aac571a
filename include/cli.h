/*
 * cli.h -- in-batch contrastive scoring on one GB300 (sm_103a): a stateless C ABI.
 *
 * Two operations of a multi-modal byte-encoder trainer's contrastive step, as
 * the UForm 4 documentation pages describe them:
 *
 *   1. the pooled pair loss in SigLIP's `sigmoid` form over N pooled
 *      embeddings, with a learnable inverse temperature t and bias b and
 *      attract / repel / ignore relations given as CSR edge sets
 *      ("UForm", section "Matryoshka-Like Multi-Scale Embedders", the SigLIP
 *      loss; "Training", `uform_pair_loss_form_t`, `uform_contrastive_t`,
 *      `uform_negatives_t`, `uform_edges_view_t`, `uform_relations_view_t`);
 *   2. ColBERT-style hard MaxSim between query and document token vectors held
 *      in Arrow-style ragged tapes, with a backward pass routed through the
 *      argmax ("UForm", section "ColBERT-Style Late-Interaction Rerankers";
 *      "Arenas", section "Rows and Tapes").
 *
 * Conventions, after the pages' C API ("Arenas"; "Training"):
 *   - Callers lend memory and never a way to allocate it: every input, output
 *     and workspace is a caller-owned device buffer, and the library allocates
 *     nothing.  It enqueues work on the caller's stream and returns; it keeps
 *     no pointer past return and holds no global state (one entry point,
 *     maxsim_backward_no_alloc, keeps a fixed scratch array instead of a
 *     lent workspace; see there).
 *   - Each verb takes one argument struct.
 *   - Outputs are overwritten, never accumulated into.
 *   - A fault the host can see (a NULL pointer, a bad size, an output
 *     overlapping an input, a workspace that is too small, a misaligned
 *     pointer) returns a status synchronously and enqueues nothing.
 *   - A fault only the device can see (offsets that decrease or run past the
 *     data, ids out of range or not strictly ascending, an empty query or
 *     document, an argmax entry outside its document where the backward reads
 *     it, i.e. for a pair with c != 0) is written to the
 *     caller-lent `device_status` word (0 = success) by a validation kernel
 *     that runs first on the stream; the compute kernels then do nothing and
 *     the outputs are unspecified.  Nothing ever traps.  A device wait that
 *     runs out of its bound reports CLI_INTERNAL there too.
 *   - Status names are static strings (nothing allocates on failure).
 *
 * Element types: bf16 data are passed as `const void *` holding IEEE bfloat16
 * values; every other element type is spelled out.  All pointers named
 * "device" must be device memory of the current CUDA device; `stream` is a
 * cudaStream_t (NULL = the legacy default stream).
 */
#ifndef CLI_H
#define CLI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Statuses; the names follow the pages' status enumeration ("Python", section
 * "Errors": shape-mismatch, unsupported, invalid-argument, device, malformed,
 * internal). */
typedef enum {
    CLI_OK = 0,
    CLI_INVALID_ARGUMENT = 1,
    CLI_SHAPE_MISMATCH = 2,
    CLI_UNSUPPORTED = 3,
    CLI_DEVICE = 4,
    CLI_MALFORMED = 5,
    CLI_INTERNAL = 6
} cli_status_t;

/* Static name of a status ("ok", "invalid-argument", ...); "unknown" otherwise. */
const char *cli_status_name(int status);

/* One edge set over `count` items as compressed sparse rows ("Training",
 * `uform_edges_view_t`): item i links to ids[offsets[i]] .. ids[offsets[i+1]-1],
 * strictly ascending.  All three arrays are device memory; `offsets` NULL names
 * no edges; `weights` NULL weighs every edge one.  `edges` must equal
 * offsets[count] (checked on the device). */
typedef struct {
    const uint64_t *offsets; /* device, count + 1 */
    const uint32_t *ids;     /* device, edges */
    const float *weights;    /* device, edges, or NULL */
    size_t edges;            /* host-side total, = offsets[count] */
} cli_edges_t;

/* Contrastive targets, resolved per ordered pair in this order ("Training",
 * `uform_relations_view_t`): a pair `ignore` names is skipped, one `attract`
 * names pulls (y = +1, its weight), one `repel` names pushes (y = -1, its
 * weight), and every other pair follows the negatives: ambient
 * (`negatives_named` = 0) repels at `ambient_weight`, named (1) skips it
 * (`uform_negatives_t`).  Ignore weights are not read. */
typedef struct {
    cli_edges_t attract, repel, ignore;
    int negatives_named;
    float ambient_weight;
} cli_relations_t;

/*
 * pair_loss_sigmoid_fwd_bwd -- the pooled sigmoid pair loss and its gradients.
 *
 * For every ordered pair (i, j), i != j, with resolved (y_ij, w_ij):
 *     z_ij = t <e_i, e_j> + b,   l_ij = w_ij * (-log sigma(y_ij z_ij)),
 *     L = (1/N) sum_{i != j} l_ij                        ("world mean"),
 * and dL/dE (fp32), dL/dt, dL/db.  The N x N score matrix never reaches
 * device memory: scores, sigmoids, log-sigmoids, relation masking and both
 * gradient contractions are fused into one kernel over tiles.
 *
 *   count, width    N (> 1) and D (a multiple of 8, at most 4096)
 *   embeddings      device bf16 [count x ld], row stride ld >= width (a
 *                   multiple of 8), 16-byte aligned; the caller normalises
 *   inverse_temperature, bias   device fp32 scalars t and b
 *   relations       see cli_relations_t; a step naming no attract edge is
 *                   refused with CLI_INVALID_ARGUMENT ("Training",
 *                   `uform_trainer_step`, `relations`)
 *   loss, d_inverse_temperature, d_bias   device fp32 scalars (written)
 *   d_embeddings    device fp32 [count x ld_d_embeddings] (written), row
 *                   stride a multiple of 4 and >= width, 16-byte aligned
 *   workspace       device, >= pair_loss_sigmoid_workspace_bytes(...),
 *                   256-byte aligned; contents on entry are ignored
 *   device_status   device int32 (written: 0 or a cli_status_t)
 *   stream          cudaStream_t
 *   row_begin, row_count   the anchor band: only ordered pairs (i, j) with
 *                   row_begin <= i < row_begin + row_count are scored, and
 *                   L, dL/dt, dL/db and dE (over all N rows) are that band's
 *                   shares, still divided by N, so the results of bands that
 *                   partition 0 .. N-1 add up to the whole call's.  This is
 *                   one device's part when the loss is sharded across
 *                   devices ("UForm", section "Matryoshka-Like Multi-Scale
 *                   Embedders": the per-rank embeddings all-gathered into
 *                   one similarity band, the gradients reduce-scattered
 *                   back), read as each rank scoring its own items' rows
 *                   against every gathered column.  (0, 0):
 *                   every row.  A band past the batch, or row_count = 0 with
 *                   row_begin > 0, is CLI_SHAPE_MISMATCH.
 *
 * dE sums tile contributions with reductions in whatever order the GPU runs
 * them, so it is reproducible to rounding, not bit for bit; L, dt and db are
 * reduced in a fixed order and are bit-reproducible.
 */
typedef struct {
    size_t count, width, ld;
    const void *embeddings;
    const float *inverse_temperature;
    const float *bias;
    cli_relations_t relations;
    float *loss;
    float *d_embeddings;
    size_t ld_d_embeddings;
    float *d_inverse_temperature;
    float *d_bias;
    void *workspace;
    size_t workspace_bytes;
    int32_t *device_status;
    void *stream;
    size_t row_begin, row_count;
} cli_pair_loss_sigmoid_t;

cli_status_t pair_loss_sigmoid_fwd_bwd(const cli_pair_loss_sigmoid_t *args);

/* Workspace bytes for pair_loss_sigmoid_fwd_bwd; `edges` = the sum of the
 * three edge sets' sizes. */
size_t pair_loss_sigmoid_workspace_bytes(size_t count, size_t width, size_t edges);

/*
 * pair_loss_sigmoid_groups_fwd_bwd -- the pooled sigmoid pair loss with
 * temperature groups ("Training", `uform_contrastive_t`, `temperature_groups`:
 * learnable (inverse temperature, bias) pairs, one per group a step's items
 * select).  Item i selects group g(i), and a cell takes its anchor's pair:
 *     z_ij = t[g(i)] <e_i, e_j> + b[g(i)],  l_ij = w_ij softplus(-y_ij z_ij),
 *     L = (1/N) sum_{i != j} l_ij,  dE, and dt[g], db[g] per group.
 *
 *   base            every field as in cli_pair_loss_sigmoid_t, except that
 *                   inverse_temperature, bias are device fp32 [group_count]
 *                   and d_inverse_temperature, d_bias device fp32
 *                   [group_count] (written); the workspace is sized by
 *                   pair_loss_sigmoid_workspace_bytes
 *   groups          device int32 [count], item i's group; a value outside
 *                   [0, group_count) sets CLI_MALFORMED in the device status
 *   group_count     at least 1
 *
 * With one group the call is pair_loss_sigmoid_fwd_bwd.  With more, z is not
 * symmetric, so every ordered pair of tiles is visited (twice the tensor work)
 * and the per-group dt, db are summed with atomic adds: they reproduce to
 * rounding, not bit for bit.
 */
typedef struct {
    cli_pair_loss_sigmoid_t base;
    const int32_t *groups;
    size_t group_count;
} cli_pair_loss_groups_t;

cli_status_t pair_loss_sigmoid_groups_fwd_bwd(const cli_pair_loss_groups_t *args);

/*
 * pair_loss_sigmoid_matryoshka_fwd_bwd -- the pooled sigmoid pair loss over
 * nested prefixes of the embeddings ("Training", `uform_contrastive_t`,
 * `matryoshka_dimensions`: prefix widths strictly ascending, each a multiple
 * of 8, at most 8, every one scored; "UForm", section "Matryoshka-Like
 * Multi-Scale Embedders": each prefix is trained under the SigLIP loss on
 * cosine similarities):
 *     u_p,i = e_i[:p] / |e_i[:p]|,   L = sum_p L_sigmoid(u_p),
 * with one (t, b) for every prefix; dE, dt and db are the gradients of that
 * sum.  The library normalises each prefix (the caller's rows need not be unit
 * vectors), scores a bf16 copy of it (nearest-even rounding) and passes the
 * gradient through the normalisation; a prefix of zero norm scores the zero
 * vector and passes no gradient.  The full width is scored only if listed.
 *
 *   base            every field as in cli_pair_loss_sigmoid_t; `base.workspace`
 *                   must hold pair_loss_sigmoid_matryoshka_workspace_bytes
 *   prefix_widths   host array of prefix_count widths, read before the call
 *                   returns; 1 <= prefix_count <= CLI_MATRYOSHKA_MAX_PREFIXES,
 *                   strictly ascending, multiples of 8, at most base.width
 *                   (CLI_SHAPE_MISMATCH otherwise)
 *   prefix_loss     device fp32 [prefix_count] (written), each prefix's loss;
 *                   may be NULL
 */
#define CLI_MATRYOSHKA_MAX_PREFIXES 8
typedef struct {
    cli_pair_loss_sigmoid_t base;
    const size_t *prefix_widths;
    size_t prefix_count;
    float *prefix_loss;
} cli_pair_loss_matryoshka_t;

cli_status_t pair_loss_sigmoid_matryoshka_fwd_bwd(const cli_pair_loss_matryoshka_t *args);

/* Workspace bytes for pair_loss_sigmoid_matryoshka_fwd_bwd (any prefix list). */
size_t pair_loss_sigmoid_matryoshka_workspace_bytes(size_t count, size_t width, size_t edges);

/*
 * pair_loss_sigmoid_scores_fwd_bwd -- the same sigmoid pair loss over a given
 * rows x cols score matrix S (e.g. hard MaxSim scores of queries against
 * documents, "UForm", section "ColBERT-Style Late-Interaction Rerankers":
 * the MaxSim scores fill the same band the embedder builds, and the SigLIP
 * form stays selectable):
 *     l_ij = w_ij * (-log sigma(y_ij (t S_ij + b))),  L = (1/rows) sum l_ij,
 *     dS_ij = dL/dS_ij, dt, db.
 * There is no implicit diagonal rule: rows and columns are different roles,
 * and relations index rows -> columns.  With `sides` (rows == cols; one byte
 * per item: bit 0 = can be a query, bit 1 = can be a document, after
 * "Training", `uform_late_interaction_side_t`), every cell whose row item is
 * not a query or whose column item is not a document is ignored.
 *
 *   scores          device fp32 [rows x ld]
 *   d_scores        device fp32 [rows x ld_d_scores] (written)
 *   other fields as in cli_pair_loss_sigmoid_t.
 */
typedef struct {
    size_t rows, cols, ld;
    const float *scores;
    const float *inverse_temperature;
    const float *bias;
    cli_relations_t relations;
    const uint8_t *sides; /* device, rows bytes, or NULL */
    float *loss;
    float *d_scores;
    size_t ld_d_scores;
    float *d_inverse_temperature;
    float *d_bias;
    void *workspace;
    size_t workspace_bytes;
    int32_t *device_status;
    void *stream;
} cli_pair_loss_sigmoid_scores_t;

cli_status_t pair_loss_sigmoid_scores_fwd_bwd(const cli_pair_loss_sigmoid_scores_t *args);
size_t pair_loss_sigmoid_scores_workspace_bytes(size_t rows, size_t cols);

/* Pair-loss forms ("Training", `uform_pair_loss_form_t`; the values are the
 * pages' enumerators). */
typedef enum {
    CLI_FORM_BALANCED = 1, /* the sigmoid cross-entropy of every cell, its attract and repel halves normalized apart */
    CLI_FORM_RANKED = 2,   /* the sigmoid cross-entropy of every positive's score over every negative's; b cancels */
    CLI_FORM_SIGMOID = 3   /* SigLIP's sigmoid cross-entropy of every cell, each repel weighed like an attract */
} cli_pair_loss_form_t;

/*
 * pair_loss_scores_fwd_bwd -- a pair loss of the chosen form over a given
 * rows x cols score matrix ("UForm", section "ColBERT-Style Late-Interaction
 * Rerankers": each query's row of hard MaxSim scores is scored by the ranked
 * form by default, and the balanced and SigLIP forms stay selectable).  The
 * pages define balanced and ranked in words only; this library reads them as
 *   balanced: l_p = sum_{attract} w l / sum_{attract} w + sum_{repel} w l / sum_{repel} w
 *             with l the sigmoid form's cell loss, each half present only
 *             when the row has such cells;
 *   ranked:   l_p = sum_{i attract, j repel} w_i w_j softplus(-t (S_pi - S_pj))
 *                   / (sum_i w_i sum_j w_j),  0 when either set is empty;
 *   L = (1/rows) sum_p l_p.
 * Cells are resolved exactly as in pair_loss_sigmoid_scores_fwd_bwd (relations,
 * sides, negatives); form CLI_FORM_SIGMOID computes that verb's result.  db is
 * 0 for the ranked form (the bias cancels).
 */
typedef struct {
    int form;
    cli_pair_loss_sigmoid_scores_t args;   /* every other field, as for the sigmoid form */
} cli_pair_loss_scores_t;

cli_status_t pair_loss_scores_fwd_bwd(const cli_pair_loss_scores_t *args);
size_t pair_loss_scores_workspace_bytes(int form, size_t rows, size_t cols);

/* A ragged tape of `count` items ("Arenas", "Rows and Tapes"): item k owns rows
 * offsets[k] .. offsets[k+1]-1 of `data`, which packs `rows` rows of `width`
 * bf16 values end to end.  `data` and `offsets` are device memory; `rows`
 * must equal offsets[count] (checked on the device); no item may be empty. */
typedef struct {
    const void *data;          /* device bf16 [rows x width], 16-byte aligned */
    const uint64_t *offsets;   /* device, count + 1 */
    size_t count, rows;
} cli_tape_t;

/*
 * maxsim_scores -- hard MaxSim of every query against every document:
 *     S(q, d) = sum_{t in q} max_{s in d} <q_t, d_s>       (mean = 0)
 *     S(q, d) = (1/|q|) sum_{t in q} max_{s in d} <q_t, d_s>  (mean = 1)
 * plus the argmax, the document-local index of the best row, lowest index on
 * ties, for every query token and document ("UForm", section "ColBERT-Style
 * Late-Interaction Rerankers": each query token keeps its single best match).
 * Scores are compared in float32 with the low 5 mantissa bits dropped (under
 * 2^-18 relative), so scores closer than that count as tied; where a token's
 * best score over a document is not a positive normal number (every score of
 * the document <= 0 for that token, or subnormal) the argmax is found again
 * in float64 from the tapes, again the lowest index among equal scores.
 *
 *   width     token width D, a multiple of 8, at most 256 (the pages: a
 *             multiple of 8, 128 by default)
 *   scores    device fp32 [queries.count x ld_scores] (written)
 *   argmax    device int32, document-major: argmax[d * ld_argmax + t] for
 *             query-tape row t (ld_argmax >= queries.rows) (written)
 *   workspace device, >= maxsim_workspace_bytes(...), 256-byte aligned
 */
typedef struct {
    cli_tape_t queries, documents;
    size_t width;
    int mean;
    float *scores;
    size_t ld_scores;
    int32_t *argmax;
    size_t ld_argmax;
    void *workspace;
    size_t workspace_bytes;
    int32_t *device_status;
    void *stream;
} cli_maxsim_t;

cli_status_t maxsim_scores(const cli_maxsim_t *args);
size_t maxsim_workspace_bytes(size_t query_count, size_t document_count, size_t query_rows,
                              size_t document_rows, size_t width);

/*
 * maxsim_scores_named -- hard MaxSim of each query against the documents it
 * names only ("Training", `uform_late_interaction_side_t`: a query's tokens
 * score the documents it attracts and repels, a document is scored by the
 * queries naming it).  S(q, d) and the argmax of every named pair are those of
 * maxsim_scores; for a pair no query names, S(q, d) = 0 and its argmax
 * entries are row indices of the document (0 where its work item was skipped;
 * after more than 2^18 float64 argmax recomputations in one call, possibly the
 * true argmax row instead), so maxsim_backward runs on the same outputs (with
 * dS = 0 there, as the
 * named-negatives loss over S gives).  Work items (1024 document rows by 128
 * query rows) that hold no named pair are not computed.
 *
 *   base      every field as in cli_maxsim_t; the workspace must hold
 *             maxsim_named_workspace_bytes(...)
 *   pairs     device CSR over the queries: offsets [count + 1], the documents
 *             each query scores, strictly ascending, below documents.count
 *             (CLI_MALFORMED in the device status otherwise); weights unread
 */
typedef struct {
    cli_maxsim_t base;
    cli_edges_t pairs;
} cli_maxsim_named_t;

cli_status_t maxsim_scores_named(const cli_maxsim_named_t *args);
size_t maxsim_named_workspace_bytes(size_t query_count, size_t document_count, size_t query_rows,
                                    size_t document_rows, size_t width);

/*
 * maxsim_backward -- the gradient through the argmax: with
 * c = dS[q][d] (divided by |q| when mean), for every query token t of q,
 *     dQ[t]      += c * D[offsets_d + argmax[d][t]]
 *     dD[offsets_d + argmax[d][t]] += c * Q[t].
 *
 *   argmax        device int32, the layout maxsim_scores writes; an entry of a
 *                 pair with c = 0 is not read (nor checked)
 *   d_scores      device fp32 [queries.count x ld_d_scores]
 *   d_queries     device fp32 [queries.rows x width] (written)
 *   d_documents   device fp32 [documents.rows x width] (written)
 *   workspace     device, >= maxsim_backward_workspace_bytes(...), 256-byte
 *                 aligned: the row -> query map, one flag per query and per
 *                 document (whether some c is nonzero: the rows of a query or
 *                 document with c = 0 throughout are written as zeros without
 *                 gathering), and the list of active documents; contents
 *                 on entry are ignored
 */
typedef struct {
    cli_tape_t queries, documents;
    size_t width;
    int mean;
    const int32_t *argmax;
    size_t ld_argmax;
    const float *d_scores;
    size_t ld_d_scores;
    float *d_queries;
    float *d_documents;
    void *workspace;
    size_t workspace_bytes;
    int32_t *device_status;
    void *stream;
} cli_maxsim_backward_t;

cli_status_t maxsim_backward(const cli_maxsim_backward_t *args);
size_t maxsim_backward_workspace_bytes(size_t query_count, size_t document_count, size_t query_rows,
                                       size_t document_rows, size_t width);

/*
 * maxsim_backward_named -- the MaxSim backward over the named pairs only (the
 * pairs of maxsim_scores_named): dQ and dD receive c(q, d) Q/D rows through the
 * argmax of every named pair, and a pair no query names contributes nothing,
 * whatever dS holds there.  One warp per named pair adds its rows into dQ and
 * dD with vector L2 reductions, so dQ and dD reproduce to rounding, not bit
 * for bit.  The workspace is not used (base.workspace may be NULL).
 *
 *   base      every other field as in cli_maxsim_backward_t
 *   pairs     as in cli_maxsim_named_t
 */
typedef struct {
    cli_maxsim_backward_t base;
    cli_edges_t pairs;
} cli_maxsim_backward_named_t;

cli_status_t maxsim_backward_named(const cli_maxsim_backward_named_t *args);

/*
 * maxsim_backward_no_alloc -- maxsim_backward for callers that cannot allocate
 * device memory and have no buffer to lend as workspace: code running where an
 * allocation is not allowed or would stall the device, or a runtime whose
 * device memory is all reserved by its own allocator.  The pages have no
 * counterpart; this entry point exists only for such callers.
 *
 * Same arguments and results as maxsim_backward; `workspace` and
 * `workspace_bytes` are not read.  Its one piece of scratch (the query of every
 * query-tape row) lives in a fixed device array of
 * CLI_MAXSIM_NO_ALLOC_MAX_QUERY_ROWS int32 entries (1 MiB) that every GPU
 * loading the library holds until the process exits.  A query tape of more
 * rows returns CLI_UNSUPPORTED.  Every call shares that array: calls whose
 * kernels overlap on the GPU (other streams or host threads) race on it.  The
 * first call on each device looks the array's address up and caches it with
 * the device's current context; make that call before any stream capture.  A
 * call in another context (after cudaDeviceReset) looks it up again.  Nothing
 * here calls cudaMalloc, cudaFree or any allocating routine.
 */
#define CLI_MAXSIM_NO_ALLOC_MAX_QUERY_ROWS 262144
cli_status_t maxsim_backward_no_alloc(const cli_maxsim_backward_t *args);

/*
 * cli_selftest_bounded_wait -- runs the failure path of the kernels' bounded
 * waits, faulting nothing.  Every wait of the tensor-core kernels gives up
 * after a time limit (2 s in the verbs above): the waiter writes CLI_INTERNAL
 * to the device status and raises its CTA's abort flag, the CTA's other
 * waiters give up too, and the kernel returns with the context usable.  This
 * call enqueues one CTA of 64 threads that wait on an mbarrier nothing arrives
 * at, with a limit of `limit_us` microseconds.
 *
 *   device_status   device int32 (written: CLI_INTERNAL once the wait gives up)
 *   gave_up         device int32, or NULL (written: the number of threads
 *                   whose wait gave up, 64)
 *   limit_us        1 .. 2,000,000; anything else is CLI_INVALID_ARGUMENT, as
 *                   is a NULL device_status
 *   stream          cudaStream_t
 */
cli_status_t cli_selftest_bounded_wait(int32_t *device_status, int32_t *gave_up, uint32_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* CLI_H */
