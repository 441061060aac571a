// Internal interfaces between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/cli.h"

namespace cli {

// One resolved "special" column of an anchor row: both directions of the pair
// (row -> col and col -> row) with their weights (0 = skipped) and whether each
// direction attracts (flags bit 0: row -> col, bit 1: col -> row).
struct RelEntry {
    uint32_t col;
    float w_out;
    float w_in;
    uint32_t flags;
};

// Device view of one CSR edge set.
struct EdgeSet {
    const uint64_t *offsets;  // NULL = no edges
    const uint32_t *ids;
    const float *weights;     // NULL = weight one
    uint64_t edges;
};

// Workspace carve-up for the pooled loss.
struct PooledWorkspace {
    uint32_t *indeg;       // [3][n]  in-degree counters, then fill cursors
    uint32_t *tin_off;     // [3][n+1] transposed offsets
    uint32_t *tin_ids;     // [E_total]  (set s at tin_base[s])
    float *tin_w;          // [E_total]
    uint32_t *rel_off;     // [n+1]
    RelEntry *rel;         // [2 E_total + n]
    float *partials;       // [pooled_partial_slots(n)][4]
    double *sums;          // [pooled_finish_blocks()][3]
    size_t bytes;
};

PooledWorkspace carve_pooled_workspace(void *base, size_t n, size_t width, size_t edges_total);
size_t align256(size_t x);

struct PooledLaunch {
    int n, width;
    const float *t_ptr, *b_ptr;
    float ambient;
    int named;
    const uint32_t *rel_off;
    const RelEntry *rel;
    float *d_e;
    long long ld_de;
    float *partials;
    double *sums;
    float *loss, *dt, *db;
    int32_t *status;
    int sm_count;
    // Temperature groups: item i's group (device, validated), or null for one
    // (t, b).  With groups, t_ptr and b_ptr index by group and dt, db are
    // per-group arrays that the kernel adds into (zeroed by the caller).
    const int32_t *group = nullptr;
    // Anchor band: only cells whose row (anchor) lies in row_lo .. row_hi - 1
    // are scored (row_hi = 0: every row).
    int row_lo = 0, row_hi = 0;
};

// Relation preparation: validation, transposition and merged special lists.
cudaError_t launch_relation_prep(const EdgeSet sets[3], int n, int named, float ambient, const PooledWorkspace &ws,
                                 int32_t *status, cudaStream_t stream);

cudaError_t launch_pooled_fused(const CUtensorMap &tmap_e, const PooledLaunch &L, cudaStream_t stream);
size_t pooled_fused_smem_bytes();
long long pooled_partial_slots(int n);
int pooled_finish_blocks();

// Matryoshka prefixes: the pooled workspace, then a bf16 copy of the
// normalised prefix rows, their inverse norms, the prefix's dE and the
// per-prefix (loss, dt, db).
constexpr int kMaxMatryoshkaPrefixes = 8;
struct MatryoshkaWorkspace {
    PooledWorkspace pooled;
    uint16_t *u;           // [n][width] bf16 (a prefix of width p uses row stride p)
    float *inv_norm;       // [n]
    float *de_p;           // [n][width] fp32 (row stride p)
    float *scalars;        // [kMaxMatryoshkaPrefixes][3]
    size_t bytes;
};
MatryoshkaWorkspace carve_matryoshka_workspace(void *base, size_t n, size_t width, size_t edges_total);
cudaError_t launch_prefix_normalize(const uint16_t *e, long long ld, int n, int p, const MatryoshkaWorkspace &ws,
                                    const int32_t *status, cudaStream_t stream);
cudaError_t launch_prefix_backprop(const uint16_t *e, long long ld, int n, int p, const MatryoshkaWorkspace &ws,
                                   float *de, long long ld_de, const int32_t *status, cudaStream_t stream);
cudaError_t launch_matryoshka_finish(const MatryoshkaWorkspace &ws, int count, float *loss, float *dt, float *db,
                                     float *prefix_loss, const int32_t *status, cudaStream_t stream);

// Score-matrix loss.
struct ScoreLossLaunch {
    int rows, cols;
    long long ld, ld_ds;
    const float *scores;
    const float *t_ptr, *b_ptr;
    EdgeSet sets[3];
    int named;
    float ambient;
    const uint8_t *sides;
    float *loss, *d_scores, *dt, *db;
    float *partials;       // [blocks][4]
    int blocks;
    int32_t *status;
};
cudaError_t launch_score_loss(const ScoreLossLaunch &L, cudaStream_t stream);
// balanced (form 1) and ranked (form 2); L.partials holds rows x 4 floats.
cudaError_t launch_score_forms(int form, const ScoreLossLaunch &L, cudaStream_t stream);
int score_loss_blocks(size_t rows, size_t cols);

// MaxSim.
struct MaxSimLaunch {
    int nq, nd, rows_q, rows_d, width, mean;
    const uint64_t *q_off, *d_off;
    float *scores;
    long long ld_scores;
    int32_t *argmax;
    long long ld_argmax;
    float *mval;              // workspace [nd][rows_q]
    uint32_t *chunk_doc;      // workspace [n_chunks + 1]
    int n_chunks, chunk_rows;
    int32_t *status;
    int sm_count;
    // Named pairs (pair_off null: every pair): the documents each query scores
    // (CSR over the queries, validated), and workspace for the item schedule.
    const uint64_t *pair_off = nullptr;
    const uint32_t *pair_ids = nullptr;
    uint32_t *item_flags = nullptr;   // [n_chunks * n_mblocks]
    uint32_t *item_list = nullptr;    // [n_chunks * n_mblocks]
    uint32_t *item_count = nullptr;   // [1]
    // The tapes (bf16 rows) for the float64 argmax fix-up, and its workspace: the
    // listed entries (document << 32 | row), [count, overflow flag], capacity.
    const uint16_t *q = nullptr, *d = nullptr;
    unsigned long long *fix_list = nullptr;
    uint32_t *fix_count = nullptr;
    uint32_t fix_cap = 0;
};
cudaError_t launch_maxsim_forward(const CUtensorMap &tmap_q, const CUtensorMap &tmap_d, const MaxSimLaunch &L,
                                  cudaStream_t stream);
size_t maxsim_forward_smem_bytes(int width);

struct MaxSimBwdLaunch {
    int nq, nd, rows_q, rows_d, width, mean;
    const uint64_t *q_off, *d_off;
    const uint16_t *q, *d;
    const int32_t *argmax;
    long long ld_argmax;
    const float *d_scores;
    long long ld_ds;
    float *dq, *dd;
    int32_t *qmap;            // workspace [rows_q]
    int32_t *status;
    int sm_count;
    // Workspace flags (null: every query and document active): whether some c(q, d) of query q, of
    // document d, is nonzero.  The backward skips the rows of inactive ones.
    uint8_t *q_active = nullptr;   // [nq]
    uint8_t *d_active = nullptr;   // [nd]
    uint32_t *d_list = nullptr;    // [nd]: the active documents in order (dQ walks these only)
    uint32_t *d_count = nullptr;   // [1]: their number
};
cudaError_t launch_maxsim_backward(const MaxSimBwdLaunch &L, cudaStream_t stream);
// The backward over named pairs only (dQ and dD zeroed by the caller).
cudaError_t launch_maxsim_backward_named(const MaxSimBwdLaunch &L, const uint64_t *pair_off, const uint32_t *pair_ids,
                                         long long pairs, cudaStream_t stream);

// bf16 [rows x cols] (row stride ld elements) as a TMA map with boxes of
// box_cols x box_rows, optionally with the 128-byte swizzle; out-of-range
// elements read as zero.
bool encode_bf16_tiles(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_cols,
                       uint32_t box_rows, bool swizzle128);

// Shared validation kernels.
cudaError_t launch_validate_edges(const EdgeSet &set, int n, int id_limit, int32_t *status, cudaStream_t stream);
cudaError_t launch_validate_groups(const int32_t *group, int n, int groups, int32_t *status, cudaStream_t stream);
cudaError_t launch_validate_tape(const uint64_t *offsets, int count, uint64_t rows, int32_t *status,
                                 cudaStream_t stream);

}  // namespace cli
