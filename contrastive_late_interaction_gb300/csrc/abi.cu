// The C ABI of include/cli.h: host-side argument checks, workspace carve-up,
// TMA descriptors and kernel launches.  Nothing here allocates device memory.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <cmath>

#include "../../include/cli.h"
#include "cli_internal.h"

namespace cli {
namespace {

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void *p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}

bool overlaps(const Range &a, const Range &b) {
    if (a.lo == a.hi || b.lo == b.hi || a.lo == 0 || b.lo == 0) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

// True when any output range overlaps any input range or another output.
bool any_overlap(const Range *in, int nin, const Range *out, int nout) {
    for (int o = 0; o < nout; ++o) {
        for (int i = 0; i < nin; ++i)
            if (overlaps(out[o], in[i])) return true;
        for (int p = o + 1; p < nout; ++p)
            if (overlaps(out[o], out[p])) return true;
    }
    return false;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// bf16 [rows x cols] with row stride ld (elements), boxes of 64 x 128 with the
// 128-byte swizzle; out-of-range elements read as zero.
bool encode_bf16_rows(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t ld) {
    return encode_bf16_tiles(map, base, cols, rows, ld, 64, 128, true);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool edges_ok(const cli_edges_t &e) {
    if (!e.offsets) return e.edges == 0;
    if (e.edges > 0 && !e.ids) return false;
    return e.edges < (1ull << 31);
}

size_t edge_bytes(const cli_edges_t &e, size_t count) {
    return e.offsets ? (count + 1) * sizeof(uint64_t) : 0;
}

EdgeSet to_set(const cli_edges_t &e) { return {e.offsets, e.ids, e.weights, e.offsets ? e.edges : 0}; }

}  // namespace
}  // namespace cli

using namespace cli;

extern "C" {

const char *cli_status_name(int status) {
    switch (status) {
        case CLI_OK: return "ok";
        case CLI_INVALID_ARGUMENT: return "invalid-argument";
        case CLI_SHAPE_MISMATCH: return "shape-mismatch";
        case CLI_UNSUPPORTED: return "unsupported";
        case CLI_DEVICE: return "device";
        case CLI_MALFORMED: return "malformed";
        case CLI_INTERNAL: return "internal";
        default: return "unknown";
    }
}

// ----------------------------------------------------------------------------
// pooled sigmoid pair loss
// ----------------------------------------------------------------------------

size_t pair_loss_sigmoid_workspace_bytes(size_t count, size_t width, size_t edges) {
    return carve_pooled_workspace(nullptr, count, width, edges).bytes;
}

}  // extern "C"

namespace cli {
namespace {

// Host checks of a pooled call that need no workspace layout; `edges` receives
// the total size of the three edge sets.
cli_status_t pooled_checks(const cli_pair_loss_sigmoid_t *a, size_t &edges) {
    const cli_relations_t &rel = a->relations;
    if (!a->embeddings || !a->inverse_temperature || !a->bias || !a->loss || !a->d_embeddings ||
        !a->d_inverse_temperature || !a->d_bias || !a->device_status || !a->workspace)
        return CLI_INVALID_ARGUMENT;
    if (a->count < 2 || a->count >= (1ull << 31)) return CLI_SHAPE_MISMATCH;
    if (a->width == 0 || a->width % 8 != 0 || a->ld < a->width || a->ld % 8 != 0) return CLI_SHAPE_MISMATCH;
    if (a->width > 4096) return CLI_UNSUPPORTED;
    if (a->row_begin > a->count || a->row_count > a->count - a->row_begin) return CLI_SHAPE_MISMATCH;
    if (a->row_count == 0 && a->row_begin != 0) return CLI_SHAPE_MISMATCH;
    if (a->ld_d_embeddings < a->width || a->ld_d_embeddings % 4 != 0) return CLI_SHAPE_MISMATCH;
    if (!aligned(a->embeddings, 16) || !aligned(a->d_embeddings, 16) || !aligned(a->workspace, 256))
        return CLI_INVALID_ARGUMENT;
    if (!edges_ok(rel.attract) || !edges_ok(rel.repel) || !edges_ok(rel.ignore)) return CLI_INVALID_ARGUMENT;
    // "a contrastive step naming no attract edge" is refused (Training, uform_trainer_step).
    if (!rel.attract.offsets || rel.attract.edges == 0) return CLI_INVALID_ARGUMENT;
    if (!(rel.ambient_weight >= 0.0f) || std::isinf(rel.ambient_weight)) return CLI_INVALID_ARGUMENT;
    edges = rel.attract.edges + (rel.repel.offsets ? rel.repel.edges : 0) + (rel.ignore.offsets ? rel.ignore.edges : 0);
    if (edges >= (1ull << 30)) return CLI_UNSUPPORTED;
    return CLI_OK;
}

// True when an output of a pooled call (the workspace taken as ws_bytes, plus
// an optional extra output range) overlaps an input or another output; `pairs`
// is the number of (t, b) pairs (and of their gradients), `extra_in` an
// optional extra input range.
bool pooled_overlap(const cli_pair_loss_sigmoid_t *a, size_t ws_bytes, Range extra, size_t pairs = 1,
                    Range extra_in = Range{0, 0}) {
    const cli_relations_t &rel = a->relations;
    const size_t n = a->count;
    const Range inputs[] = {
        range_of(a->embeddings, ((n - 1) * a->ld + a->width) * 2),
        range_of(a->inverse_temperature, 4 * pairs),
        range_of(a->bias, 4 * pairs),
        extra_in,
        range_of(rel.attract.offsets, edge_bytes(rel.attract, n)),
        range_of(rel.attract.ids, rel.attract.offsets ? rel.attract.edges * 4 : 0),
        range_of(rel.attract.weights, rel.attract.offsets && rel.attract.weights ? rel.attract.edges * 4 : 0),
        range_of(rel.repel.offsets, edge_bytes(rel.repel, n)),
        range_of(rel.repel.ids, rel.repel.offsets ? rel.repel.edges * 4 : 0),
        range_of(rel.repel.weights, rel.repel.offsets && rel.repel.weights ? rel.repel.edges * 4 : 0),
        range_of(rel.ignore.offsets, edge_bytes(rel.ignore, n)),
        range_of(rel.ignore.ids, rel.ignore.offsets ? rel.ignore.edges * 4 : 0),
    };
    const Range outputs[] = {
        range_of(a->loss, 4),
        range_of(a->d_embeddings, ((n - 1) * a->ld_d_embeddings + a->width) * 4),
        range_of(a->d_inverse_temperature, 4 * pairs),
        range_of(a->d_bias, 4 * pairs),
        range_of(a->workspace, ws_bytes),
        range_of(a->device_status, 4),
        extra,
    };
    return any_overlap(inputs, sizeof(inputs) / sizeof(inputs[0]), outputs, sizeof(outputs) / sizeof(outputs[0]));
}

// The pooled kernel's launch record for embeddings `e` of width `width`
// (written dE d_e with row stride ld_de) and scalar outputs loss, dt, db.
PooledLaunch pooled_launch_record(const cli_pair_loss_sigmoid_t *a, const PooledWorkspace &ws, int width, float *d_e,
                                  long long ld_de, float *loss, float *dt, float *db, int sms) {
    PooledLaunch L;
    L.n = static_cast<int>(a->count);
    L.width = width;
    L.t_ptr = a->inverse_temperature;
    L.b_ptr = a->bias;
    L.ambient = a->relations.ambient_weight;
    L.named = a->relations.negatives_named ? 1 : 0;
    L.rel_off = ws.rel_off;
    L.rel = ws.rel;
    L.d_e = d_e;
    L.ld_de = ld_de;
    L.partials = ws.partials;
    L.sums = ws.sums;
    L.loss = loss;
    L.dt = dt;
    L.db = db;
    L.status = a->device_status;
    L.sm_count = sms;
    L.row_lo = static_cast<int>(a->row_begin);
    L.row_hi = a->row_count ? static_cast<int>(a->row_begin + a->row_count) : 0;
    return L;
}

}  // namespace
}  // namespace cli

extern "C" {

cli_status_t pair_loss_sigmoid_fwd_bwd(const cli_pair_loss_sigmoid_t *a) {
    if (!a) return CLI_INVALID_ARGUMENT;
    const cli_relations_t &rel = a->relations;
    size_t edges = 0;
    const cli_status_t st = pooled_checks(a, edges);
    if (st != CLI_OK) return st;
    const PooledWorkspace ws = carve_pooled_workspace(a->workspace, a->count, a->width, edges);
    if (a->workspace_bytes < ws.bytes) return CLI_INVALID_ARGUMENT;
    if (pooled_overlap(a, ws.bytes, Range{0, 0})) return CLI_INVALID_ARGUMENT;
    const size_t n = a->count;

    const int sms = sm_count();
    if (sms <= 0) return CLI_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    CUtensorMap tmap;
    if (!encode_bf16_rows(&tmap, a->embeddings, a->width, n, a->ld)) return CLI_DEVICE;

    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    const EdgeSet sets[3] = {to_set(rel.attract), to_set(rel.repel), to_set(rel.ignore)};
    if (launch_relation_prep(sets, static_cast<int>(n), rel.negatives_named, rel.ambient_weight, ws, a->device_status,
                             stream) != cudaSuccess)
        return CLI_DEVICE;
    if (cudaMemset2DAsync(a->d_embeddings, a->ld_d_embeddings * 4, 0, a->width * 4, n, stream) != cudaSuccess)
        return CLI_DEVICE;
    const PooledLaunch L = pooled_launch_record(a, ws, static_cast<int>(a->width), a->d_embeddings,
                                                static_cast<long long>(a->ld_d_embeddings), a->loss,
                                                a->d_inverse_temperature, a->d_bias, sms);
    if (launch_pooled_fused(tmap, L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}

// ----------------------------------------------------------------------------
// temperature groups of the pooled sigmoid pair loss
// ----------------------------------------------------------------------------

cli_status_t pair_loss_sigmoid_groups_fwd_bwd(const cli_pair_loss_groups_t *g) {
    if (!g) return CLI_INVALID_ARGUMENT;
    const cli_pair_loss_sigmoid_t *a = &g->base;
    const cli_relations_t &rel = a->relations;
    size_t edges = 0;
    const cli_status_t st = pooled_checks(a, edges);
    if (st != CLI_OK) return st;
    if (!g->groups || !aligned(g->groups, 4)) return CLI_INVALID_ARGUMENT;
    if (g->group_count == 0 || g->group_count >= (1ull << 31)) return CLI_SHAPE_MISMATCH;
    const PooledWorkspace ws = carve_pooled_workspace(a->workspace, a->count, a->width, edges);
    if (a->workspace_bytes < ws.bytes) return CLI_INVALID_ARGUMENT;
    if (pooled_overlap(a, ws.bytes, Range{0, 0}, g->group_count, range_of(g->groups, a->count * 4)))
        return CLI_INVALID_ARGUMENT;

    const int sms = sm_count();
    if (sms <= 0) return CLI_DEVICE;
    const size_t n = a->count;
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    CUtensorMap tmap;
    if (!encode_bf16_rows(&tmap, a->embeddings, a->width, n, a->ld)) return CLI_DEVICE;
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    if (launch_validate_groups(g->groups, static_cast<int>(n), static_cast<int>(g->group_count), a->device_status,
                               stream) != cudaSuccess)
        return CLI_DEVICE;
    const EdgeSet sets[3] = {to_set(rel.attract), to_set(rel.repel), to_set(rel.ignore)};
    if (launch_relation_prep(sets, static_cast<int>(n), rel.negatives_named, rel.ambient_weight, ws, a->device_status,
                             stream) != cudaSuccess)
        return CLI_DEVICE;
    if (cudaMemset2DAsync(a->d_embeddings, a->ld_d_embeddings * 4, 0, a->width * 4, n, stream) != cudaSuccess)
        return CLI_DEVICE;
    PooledLaunch L = pooled_launch_record(a, ws, static_cast<int>(a->width), a->d_embeddings,
                                          static_cast<long long>(a->ld_d_embeddings), a->loss,
                                          a->d_inverse_temperature, a->d_bias, sms);
    if (g->group_count > 1) {   // one group is the symmetric call
        if (cudaMemsetAsync(a->d_inverse_temperature, 0, g->group_count * 4, stream) != cudaSuccess ||
            cudaMemsetAsync(a->d_bias, 0, g->group_count * 4, stream) != cudaSuccess)
            return CLI_DEVICE;
        L.group = g->groups;
    }
    if (launch_pooled_fused(tmap, L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}

// ----------------------------------------------------------------------------
// Matryoshka prefixes of the pooled sigmoid pair loss
// ----------------------------------------------------------------------------

size_t pair_loss_sigmoid_matryoshka_workspace_bytes(size_t count, size_t width, size_t edges) {
    return carve_matryoshka_workspace(nullptr, count, width, edges).bytes;
}

cli_status_t pair_loss_sigmoid_matryoshka_fwd_bwd(const cli_pair_loss_matryoshka_t *m) {
    if (!m) return CLI_INVALID_ARGUMENT;
    const cli_pair_loss_sigmoid_t *a = &m->base;
    const cli_relations_t &rel = a->relations;
    size_t edges = 0;
    const cli_status_t st = pooled_checks(a, edges);
    if (st != CLI_OK) return st;
    if (!m->prefix_widths) return CLI_INVALID_ARGUMENT;
    if (m->prefix_count == 0 || m->prefix_count > CLI_MATRYOSHKA_MAX_PREFIXES) return CLI_SHAPE_MISMATCH;
    for (size_t k = 0; k < m->prefix_count; ++k) {
        const size_t p = m->prefix_widths[k];
        if (p == 0 || p % 8 != 0 || p > a->width) return CLI_SHAPE_MISMATCH;
        if (k > 0 && p <= m->prefix_widths[k - 1]) return CLI_SHAPE_MISMATCH;
    }
    if (m->prefix_loss && !aligned(m->prefix_loss, 4)) return CLI_INVALID_ARGUMENT;
    const MatryoshkaWorkspace ws = carve_matryoshka_workspace(a->workspace, a->count, a->width, edges);
    if (a->workspace_bytes < ws.bytes) return CLI_INVALID_ARGUMENT;
    if (pooled_overlap(a, ws.bytes, range_of(m->prefix_loss, m->prefix_loss ? m->prefix_count * 4 : 0)))
        return CLI_INVALID_ARGUMENT;

    const int sms = sm_count();
    if (sms <= 0) return CLI_DEVICE;
    const size_t n = a->count;
    const int ni = static_cast<int>(n);
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    const uint16_t *e = static_cast<const uint16_t *>(static_cast<const void *>(a->embeddings));
    const long long ld = static_cast<long long>(a->ld);
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    const EdgeSet sets[3] = {to_set(rel.attract), to_set(rel.repel), to_set(rel.ignore)};
    if (launch_relation_prep(sets, ni, rel.negatives_named, rel.ambient_weight, ws.pooled, a->device_status, stream) !=
        cudaSuccess)
        return CLI_DEVICE;
    if (cudaMemset2DAsync(a->d_embeddings, a->ld_d_embeddings * 4, 0, a->width * 4, n, stream) != cudaSuccess)
        return CLI_DEVICE;
    for (size_t k = 0; k < m->prefix_count; ++k) {
        const int p = static_cast<int>(m->prefix_widths[k]);
        CUtensorMap tmap;
        if (!encode_bf16_rows(&tmap, ws.u, static_cast<uint64_t>(p), n, static_cast<uint64_t>(p))) return CLI_DEVICE;
        if (launch_prefix_normalize(e, ld, ni, p, ws, a->device_status, stream) != cudaSuccess) return CLI_DEVICE;
        if (cudaMemsetAsync(ws.de_p, 0, n * static_cast<size_t>(p) * 4, stream) != cudaSuccess) return CLI_DEVICE;
        float *sc = ws.scalars + 3 * k;
        const PooledLaunch L = pooled_launch_record(a, ws.pooled, p, ws.de_p, p, sc, sc + 1, sc + 2, sms);
        if (launch_pooled_fused(tmap, L, stream) != cudaSuccess) return CLI_DEVICE;
        if (launch_prefix_backprop(e, ld, ni, p, ws, a->d_embeddings, static_cast<long long>(a->ld_d_embeddings),
                                   a->device_status, stream) != cudaSuccess)
            return CLI_DEVICE;
    }
    if (launch_matryoshka_finish(ws, static_cast<int>(m->prefix_count), a->loss, a->d_inverse_temperature, a->d_bias,
                                 m->prefix_loss, a->device_status, stream) != cudaSuccess)
        return CLI_DEVICE;
    return CLI_OK;
}

// ----------------------------------------------------------------------------
// sigmoid pair loss over a score matrix
// ----------------------------------------------------------------------------

size_t pair_loss_sigmoid_scores_workspace_bytes(size_t rows, size_t cols) {
    return align256(static_cast<size_t>(score_loss_blocks(rows, cols)) * 4 * sizeof(float));
}

cli_status_t pair_loss_sigmoid_scores_fwd_bwd(const cli_pair_loss_sigmoid_scores_t *a) {
    if (!a) return CLI_INVALID_ARGUMENT;
    const cli_relations_t &rel = a->relations;
    if (!a->scores || !a->inverse_temperature || !a->bias || !a->loss || !a->d_scores || !a->d_inverse_temperature ||
        !a->d_bias || !a->device_status || !a->workspace)
        return CLI_INVALID_ARGUMENT;
    if (a->rows == 0 || a->cols == 0 || a->rows >= (1ull << 31) || a->cols >= (1ull << 31)) return CLI_SHAPE_MISMATCH;
    if (a->ld < a->cols || a->ld_d_scores < a->cols) return CLI_SHAPE_MISMATCH;
    if (a->sides && a->rows != a->cols) return CLI_SHAPE_MISMATCH;
    if (!edges_ok(rel.attract) || !edges_ok(rel.repel) || !edges_ok(rel.ignore)) return CLI_INVALID_ARGUMENT;
    if (!rel.attract.offsets || rel.attract.edges == 0) return CLI_INVALID_ARGUMENT;
    if (!(rel.ambient_weight >= 0.0f) || std::isinf(rel.ambient_weight)) return CLI_INVALID_ARGUMENT;
    if (a->workspace_bytes < pair_loss_sigmoid_scores_workspace_bytes(a->rows, a->cols)) return CLI_INVALID_ARGUMENT;
    const size_t r = a->rows;
    const Range inputs[] = {
        range_of(a->scores, ((r - 1) * a->ld + a->cols) * 4),
        range_of(a->inverse_temperature, 4),
        range_of(a->bias, 4),
        range_of(a->sides, a->sides ? r : 0),
        range_of(rel.attract.offsets, edge_bytes(rel.attract, r)),
        range_of(rel.attract.ids, rel.attract.offsets ? rel.attract.edges * 4 : 0),
        range_of(rel.repel.offsets, edge_bytes(rel.repel, r)),
        range_of(rel.repel.ids, rel.repel.offsets ? rel.repel.edges * 4 : 0),
        range_of(rel.ignore.offsets, edge_bytes(rel.ignore, r)),
        range_of(rel.ignore.ids, rel.ignore.offsets ? rel.ignore.edges * 4 : 0),
    };
    const Range outputs[] = {
        range_of(a->loss, 4),
        range_of(a->d_scores, ((r - 1) * a->ld_d_scores + a->cols) * 4),
        range_of(a->d_inverse_temperature, 4),
        range_of(a->d_bias, 4),
        range_of(a->workspace, pair_loss_sigmoid_scores_workspace_bytes(a->rows, a->cols)),
        range_of(a->device_status, 4),
    };
    if (any_overlap(inputs, sizeof(inputs) / sizeof(inputs[0]), outputs, sizeof(outputs) / sizeof(outputs[0])))
        return CLI_INVALID_ARGUMENT;
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    ScoreLossLaunch L;
    L.rows = static_cast<int>(a->rows);
    L.cols = static_cast<int>(a->cols);
    L.ld = static_cast<long long>(a->ld);
    L.ld_ds = static_cast<long long>(a->ld_d_scores);
    L.scores = a->scores;
    L.t_ptr = a->inverse_temperature;
    L.b_ptr = a->bias;
    L.sets[0] = to_set(rel.attract);
    L.sets[1] = to_set(rel.repel);
    L.sets[2] = to_set(rel.ignore);
    L.named = rel.negatives_named ? 1 : 0;
    L.ambient = rel.ambient_weight;
    L.sides = a->sides;
    L.loss = a->loss;
    L.d_scores = a->d_scores;
    L.dt = a->d_inverse_temperature;
    L.db = a->d_bias;
    L.partials = static_cast<float *>(a->workspace);
    L.blocks = score_loss_blocks(a->rows, a->cols);
    L.status = a->device_status;
    if (launch_score_loss(L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}

size_t pair_loss_scores_workspace_bytes(int form, size_t rows, size_t cols) {
    if (form == CLI_FORM_SIGMOID) return pair_loss_sigmoid_scores_workspace_bytes(rows, cols);
    return align256(rows * 4 * sizeof(float));
}

cli_status_t pair_loss_scores_fwd_bwd(const cli_pair_loss_scores_t *f) {
    if (!f) return CLI_INVALID_ARGUMENT;
    if (f->form == CLI_FORM_SIGMOID) return pair_loss_sigmoid_scores_fwd_bwd(&f->args);
    if (f->form != CLI_FORM_BALANCED && f->form != CLI_FORM_RANKED) return CLI_INVALID_ARGUMENT;
    const cli_pair_loss_sigmoid_scores_t *a = &f->args;
    const cli_relations_t &rel = a->relations;
    if (!a->scores || !a->inverse_temperature || !a->bias || !a->loss || !a->d_scores || !a->d_inverse_temperature ||
        !a->d_bias || !a->device_status || !a->workspace)
        return CLI_INVALID_ARGUMENT;
    if (a->rows == 0 || a->cols == 0 || a->rows >= (1ull << 31) || a->cols >= (1ull << 31)) return CLI_SHAPE_MISMATCH;
    if (a->ld < a->cols || a->ld_d_scores < a->cols) return CLI_SHAPE_MISMATCH;
    if (a->sides && a->rows != a->cols) return CLI_SHAPE_MISMATCH;
    if (!edges_ok(rel.attract) || !edges_ok(rel.repel) || !edges_ok(rel.ignore)) return CLI_INVALID_ARGUMENT;
    if (!rel.attract.offsets || rel.attract.edges == 0) return CLI_INVALID_ARGUMENT;
    if (!(rel.ambient_weight >= 0.0f) || std::isinf(rel.ambient_weight)) return CLI_INVALID_ARGUMENT;
    const size_t wsb = pair_loss_scores_workspace_bytes(f->form, a->rows, a->cols);
    if (a->workspace_bytes < wsb) return CLI_INVALID_ARGUMENT;
    const size_t r = a->rows;
    const Range inputs[] = {
        range_of(a->scores, ((r - 1) * a->ld + a->cols) * 4),
        range_of(a->inverse_temperature, 4),
        range_of(a->bias, 4),
        range_of(a->sides, a->sides ? r : 0),
        range_of(rel.attract.offsets, edge_bytes(rel.attract, r)),
        range_of(rel.attract.ids, rel.attract.offsets ? rel.attract.edges * 4 : 0),
        range_of(rel.repel.offsets, edge_bytes(rel.repel, r)),
        range_of(rel.repel.ids, rel.repel.offsets ? rel.repel.edges * 4 : 0),
        range_of(rel.ignore.offsets, edge_bytes(rel.ignore, r)),
        range_of(rel.ignore.ids, rel.ignore.offsets ? rel.ignore.edges * 4 : 0),
    };
    const Range outputs[] = {
        range_of(a->loss, 4),
        range_of(a->d_scores, ((r - 1) * a->ld_d_scores + a->cols) * 4),
        range_of(a->d_inverse_temperature, 4),
        range_of(a->d_bias, 4),
        range_of(a->workspace, wsb),
        range_of(a->device_status, 4),
    };
    if (any_overlap(inputs, sizeof(inputs) / sizeof(inputs[0]), outputs, sizeof(outputs) / sizeof(outputs[0])))
        return CLI_INVALID_ARGUMENT;
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    ScoreLossLaunch L;
    L.rows = static_cast<int>(a->rows);
    L.cols = static_cast<int>(a->cols);
    L.ld = static_cast<long long>(a->ld);
    L.ld_ds = static_cast<long long>(a->ld_d_scores);
    L.scores = a->scores;
    L.t_ptr = a->inverse_temperature;
    L.b_ptr = a->bias;
    L.sets[0] = to_set(rel.attract);
    L.sets[1] = to_set(rel.repel);
    L.sets[2] = to_set(rel.ignore);
    L.named = rel.negatives_named ? 1 : 0;
    L.ambient = rel.ambient_weight;
    L.sides = a->sides;
    L.loss = a->loss;
    L.d_scores = a->d_scores;
    L.dt = a->d_inverse_temperature;
    L.db = a->d_bias;
    L.partials = static_cast<float *>(a->workspace);
    L.blocks = static_cast<int>(a->rows);
    L.status = a->device_status;
    if (launch_score_forms(f->form, L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}

// ----------------------------------------------------------------------------
// MaxSim
// ----------------------------------------------------------------------------

namespace {

bool tape_ok(const cli_tape_t &t) {
    return t.data && t.offsets && t.count > 0 && t.rows >= t.count && t.rows < (1ull << 31) &&
           t.count < (1ull << 31) && aligned(t.data, 16);
}

int chunk_rows_for(size_t rows_d, size_t rows_q, int sms) {
    const long long mblocks = static_cast<long long>((rows_q + 127) / 128);
    const long long target_items = 16LL * sms;
    long long r = static_cast<long long>((static_cast<long double>(rows_d) * mblocks) / target_items);
    if (r < 1024) r = 1024;
    if (r > 16384) r = 16384;
    return static_cast<int>((r + 127) / 128 * 128);
}

struct MaxSimWs {
    float *mval;
    uint32_t *chunk_doc;
    unsigned long long *fix_list;
    uint32_t *fix_count;
    uint32_t fix_cap;
    size_t bytes;
    int n_chunks, chunk_rows;
};

// Argmax entries the forward lists for the float64 fix-up (rows whose maximum
// over a document is <= 0 or subnormal); past this many it scans its whole table.
size_t fix_capacity(size_t nd, size_t rows_q) {
    const size_t all = nd * rows_q;
    return all < (size_t{1} << 18) ? all : (size_t{1} << 18);
}

// Named pairs run on the finest chunks (1024 document rows), so that items
// holding no named pair are skipped at a fine grain.
constexpr int kNamedChunkRows = 1024;

MaxSimWs carve_maxsim(void *base, size_t nd, size_t rows_q, size_t rows_d, int sms, bool named = false) {
    MaxSimWs w;
    uint8_t *p = static_cast<uint8_t *>(base);
    size_t off = 0;
    w.mval = reinterpret_cast<float *>(p ? p + off : nullptr);
    off += align256(nd * rows_q * sizeof(float));
    w.chunk_rows = named ? kNamedChunkRows : chunk_rows_for(rows_d, rows_q, sms > 0 ? sms : 148);
    w.n_chunks = static_cast<int>((rows_d + w.chunk_rows - 1) / w.chunk_rows);
    w.chunk_doc = reinterpret_cast<uint32_t *>(p ? p + off : nullptr);
    off += align256((static_cast<size_t>(w.n_chunks) + 1) * sizeof(uint32_t));
    w.fix_cap = static_cast<uint32_t>(fix_capacity(nd, rows_q));
    w.fix_list = reinterpret_cast<unsigned long long *>(p ? p + off : nullptr);
    off += align256(static_cast<size_t>(w.fix_cap) * sizeof(unsigned long long));
    w.fix_count = reinterpret_cast<uint32_t *>(p ? p + off : nullptr);
    off += align256(2 * sizeof(uint32_t));
    w.bytes = off;
    return w;
}

}  // namespace

size_t maxsim_workspace_bytes(size_t query_count, size_t document_count, size_t query_rows, size_t document_rows,
                              size_t width) {
    (void)query_count;
    (void)width;
    // The chunking depends on the SM count; size for the smallest chunks (most chunks).
    const size_t chunks = (document_rows + 1023) / 1024 + 1;
    return align256(document_count * query_rows * sizeof(float)) + align256((chunks + 1) * sizeof(uint32_t)) +
           align256(fix_capacity(document_count, query_rows) * sizeof(unsigned long long)) +
           align256(2 * sizeof(uint32_t));
}

}  // extern "C"

namespace cli {
namespace {

// Work items of the named-pair schedule at most: chunks of kNamedChunkRows rows
// times 128-row query blocks.
size_t named_items_max(size_t query_rows, size_t document_rows) {
    return ((document_rows + kNamedChunkRows - 1) / kNamedChunkRows + 1) * ((query_rows + 127) / 128);
}

// maxsim_scores, over every pair (pairs null) or the named ones.
cli_status_t maxsim_forward_call(const cli_maxsim_t *a, const cli_edges_t *pairs) {
    if (!a) return CLI_INVALID_ARGUMENT;
    if (!a->scores || !a->argmax || !a->device_status || !a->workspace) return CLI_INVALID_ARGUMENT;
    if (!tape_ok(a->queries) || !tape_ok(a->documents)) return CLI_INVALID_ARGUMENT;
    if (a->width == 0 || a->width % 8 != 0) return CLI_SHAPE_MISMATCH;
    if (a->width > 256) return CLI_UNSUPPORTED;
    const size_t nq = a->queries.count, nd = a->documents.count, rq = a->queries.rows, rd = a->documents.rows;
    if (a->ld_scores < nd || a->ld_argmax < rq) return CLI_SHAPE_MISMATCH;
    if (pairs && (!pairs->offsets || !edges_ok(*pairs))) return CLI_INVALID_ARGUMENT;
    const size_t wsb = pairs ? maxsim_named_workspace_bytes(nq, nd, rq, rd, a->width)
                             : maxsim_workspace_bytes(nq, nd, rq, rd, a->width);
    if (a->workspace_bytes < wsb || !aligned(a->workspace, 256)) return CLI_INVALID_ARGUMENT;
    const Range inputs[] = {
        range_of(a->queries.data, rq * a->width * 2), range_of(a->queries.offsets, (nq + 1) * 8),
        range_of(a->documents.data, rd * a->width * 2), range_of(a->documents.offsets, (nd + 1) * 8),
        pairs ? range_of(pairs->offsets, (nq + 1) * 8) : Range{0, 0},
        pairs ? range_of(pairs->ids, pairs->edges * 4) : Range{0, 0},
    };
    const Range outputs[] = {
        range_of(a->scores, ((nq - 1) * a->ld_scores + nd) * 4),
        range_of(a->argmax, ((nd - 1) * a->ld_argmax + rq) * 4),
        range_of(a->workspace, wsb),
        range_of(a->device_status, 4),
    };
    if (any_overlap(inputs, 6, outputs, 4)) return CLI_INVALID_ARGUMENT;
    const int sms = sm_count();
    if (sms <= 0) return CLI_DEVICE;
    const MaxSimWs ws = carve_maxsim(a->workspace, nd, rq, rd, sms, pairs != nullptr);
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    CUtensorMap tq, td;
    if (!encode_bf16_rows(&tq, a->queries.data, a->width, rq, a->width) ||
        !encode_bf16_rows(&td, a->documents.data, a->width, rd, a->width))
        return CLI_DEVICE;
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    if (launch_validate_tape(a->queries.offsets, static_cast<int>(nq), rq, a->device_status, stream) != cudaSuccess ||
        launch_validate_tape(a->documents.offsets, static_cast<int>(nd), rd, a->device_status, stream) != cudaSuccess)
        return CLI_DEVICE;
    MaxSimLaunch L;
    L.nq = static_cast<int>(nq);
    L.nd = static_cast<int>(nd);
    L.rows_q = static_cast<int>(rq);
    L.rows_d = static_cast<int>(rd);
    L.width = static_cast<int>(a->width);
    L.mean = a->mean ? 1 : 0;
    L.q_off = a->queries.offsets;
    L.d_off = a->documents.offsets;
    L.scores = a->scores;
    L.ld_scores = static_cast<long long>(a->ld_scores);
    L.argmax = a->argmax;
    L.ld_argmax = static_cast<long long>(a->ld_argmax);
    L.mval = ws.mval;
    L.chunk_doc = ws.chunk_doc;
    L.n_chunks = ws.n_chunks;
    L.chunk_rows = ws.chunk_rows;
    L.q = static_cast<const uint16_t *>(a->queries.data);
    L.d = static_cast<const uint16_t *>(a->documents.data);
    L.fix_list = ws.fix_list;
    L.fix_count = ws.fix_count;
    L.fix_cap = ws.fix_cap;
    L.status = a->device_status;
    L.sm_count = sms;
    if (pairs) {
        // Pairs index documents; an argmax entry of a pair no query names is 0.
        if (launch_validate_edges(to_set(*pairs), static_cast<int>(nq), static_cast<int>(nd), a->device_status,
                                  stream) != cudaSuccess)
            return CLI_DEVICE;
        if (cudaMemset2DAsync(a->argmax, a->ld_argmax * 4, 0, rq * 4, nd, stream) != cudaSuccess) return CLI_DEVICE;
        const size_t items = named_items_max(rq, rd);
        uint8_t *q = static_cast<uint8_t *>(a->workspace) + ws.bytes;
        L.pair_off = pairs->offsets;
        L.pair_ids = pairs->ids;
        L.item_flags = reinterpret_cast<uint32_t *>(q);
        L.item_list = reinterpret_cast<uint32_t *>(q + align256(items * 4));
        L.item_count = reinterpret_cast<uint32_t *>(q + 2 * align256(items * 4));
    }
    if (launch_maxsim_forward(tq, td, L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}

}  // namespace
}  // namespace cli

extern "C" {

cli_status_t maxsim_scores(const cli_maxsim_t *a) { return maxsim_forward_call(a, nullptr); }

size_t maxsim_named_workspace_bytes(size_t query_count, size_t document_count, size_t query_rows,
                                    size_t document_rows, size_t width) {
    return maxsim_workspace_bytes(query_count, document_count, query_rows, document_rows, width) +
           2 * align256(named_items_max(query_rows, document_rows) * 4) + 256;
}

cli_status_t maxsim_scores_named(const cli_maxsim_named_t *a) {
    if (!a) return CLI_INVALID_ARGUMENT;
    return maxsim_forward_call(&a->base, &a->pairs);
}

size_t maxsim_backward_workspace_bytes(size_t query_count, size_t document_count, size_t query_rows,
                                       size_t document_rows, size_t width) {
    (void)document_rows;
    (void)width;
    // the row -> query map, one activity flag per query and per document, the list of active documents
    // and its length
    return align256(query_rows * sizeof(int32_t)) + align256(query_count) + align256(document_count) +
           align256(document_count * sizeof(uint32_t)) + 256;
}

}  // extern "C"

namespace cli {
namespace {

// maxsim_backward over every pair (pairs null) or the named ones only.
cli_status_t maxsim_backward_call(const cli_maxsim_backward_t *a, const cli_edges_t *pairs) {
    if (!a) return CLI_INVALID_ARGUMENT;
    if (!a->argmax || !a->d_scores || !a->d_queries || !a->d_documents || !a->device_status) return CLI_INVALID_ARGUMENT;
    if (!pairs && !a->workspace) return CLI_INVALID_ARGUMENT;
    if (!tape_ok(a->queries) || !tape_ok(a->documents)) return CLI_INVALID_ARGUMENT;
    if (a->width == 0 || a->width % 8 != 0) return CLI_SHAPE_MISMATCH;
    if (a->width > 256) return CLI_UNSUPPORTED;
    const size_t nq = a->queries.count, nd = a->documents.count, rq = a->queries.rows, rd = a->documents.rows;
    if (a->ld_d_scores < nd || a->ld_argmax < rq) return CLI_SHAPE_MISMATCH;
    if (!aligned(a->d_queries, 16) || !aligned(a->d_documents, 16)) return CLI_INVALID_ARGUMENT;
    if (pairs && (!pairs->offsets || !edges_ok(*pairs))) return CLI_INVALID_ARGUMENT;
    const size_t wsb = pairs ? 0 : maxsim_backward_workspace_bytes(nq, nd, rq, rd, a->width);
    if (!pairs && (a->workspace_bytes < wsb || !aligned(a->workspace, 256))) return CLI_INVALID_ARGUMENT;
    const Range inputs[] = {
        range_of(a->queries.data, rq * a->width * 2), range_of(a->queries.offsets, (nq + 1) * 8),
        range_of(a->documents.data, rd * a->width * 2), range_of(a->documents.offsets, (nd + 1) * 8),
        range_of(a->argmax, ((nd - 1) * a->ld_argmax + rq) * 4),
        range_of(a->d_scores, ((nq - 1) * a->ld_d_scores + nd) * 4),
        pairs ? range_of(pairs->offsets, (nq + 1) * 8) : Range{0, 0},
        pairs ? range_of(pairs->ids, pairs->edges * 4) : Range{0, 0},
    };
    const Range outputs[] = {
        range_of(a->d_queries, rq * a->width * 4),
        range_of(a->d_documents, rd * a->width * 4),
        range_of(a->workspace, wsb),
        range_of(a->device_status, 4),
    };
    if (any_overlap(inputs, 8, outputs, 4)) return CLI_INVALID_ARGUMENT;
    const int sms = sm_count();
    if (sms <= 0) return CLI_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    if (launch_validate_tape(a->queries.offsets, static_cast<int>(nq), rq, a->device_status, stream) != cudaSuccess ||
        launch_validate_tape(a->documents.offsets, static_cast<int>(nd), rd, a->device_status, stream) != cudaSuccess)
        return CLI_DEVICE;
    MaxSimBwdLaunch L;
    L.nq = static_cast<int>(nq);
    L.nd = static_cast<int>(nd);
    L.rows_q = static_cast<int>(rq);
    L.rows_d = static_cast<int>(rd);
    L.width = static_cast<int>(a->width);
    L.mean = a->mean ? 1 : 0;
    L.q_off = a->queries.offsets;
    L.d_off = a->documents.offsets;
    L.q = static_cast<const uint16_t *>(a->queries.data);
    L.d = static_cast<const uint16_t *>(a->documents.data);
    L.argmax = a->argmax;
    L.ld_argmax = static_cast<long long>(a->ld_argmax);
    L.d_scores = a->d_scores;
    L.ld_ds = static_cast<long long>(a->ld_d_scores);
    L.dq = a->d_queries;
    L.dd = a->d_documents;
    L.qmap = static_cast<int32_t *>(a->workspace);
    if (!pairs) {
        uint8_t *w = static_cast<uint8_t *>(a->workspace) + align256(rq * sizeof(int32_t));
        L.q_active = w;
        L.d_active = w + align256(nq);
        L.d_list = reinterpret_cast<uint32_t *>(L.d_active + align256(nd));
        L.d_count = L.d_list + align256(nd * sizeof(uint32_t)) / sizeof(uint32_t);
    }
    L.status = a->device_status;
    L.sm_count = sms;
    if (pairs) {
        if (launch_validate_edges(to_set(*pairs), static_cast<int>(nq), static_cast<int>(nd), a->device_status,
                                  stream) != cudaSuccess)
            return CLI_DEVICE;
        if (cudaMemsetAsync(a->d_queries, 0, rq * a->width * 4, stream) != cudaSuccess ||
            cudaMemsetAsync(a->d_documents, 0, rd * a->width * 4, stream) != cudaSuccess)
            return CLI_DEVICE;
        if (launch_maxsim_backward_named(L, pairs->offsets, pairs->ids, static_cast<long long>(pairs->edges), stream) !=
            cudaSuccess)
            return CLI_DEVICE;
        return CLI_OK;
    }
    if (launch_maxsim_backward(L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}

}  // namespace
}  // namespace cli

extern "C" {

cli_status_t maxsim_backward(const cli_maxsim_backward_t *a) { return maxsim_backward_call(a, nullptr); }

cli_status_t maxsim_backward_named(const cli_maxsim_backward_named_t *a) {
    if (!a) return CLI_INVALID_ARGUMENT;
    return maxsim_backward_call(&a->base, &a->pairs);
}

}  // extern "C"
