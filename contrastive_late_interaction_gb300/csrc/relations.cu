// Relation resolution for the pooled loss ("Training", `uform_edges_view_t`,
// `uform_relations_view_t`, `uform_negatives_t`), done once per call on the
// device:
//   1. validate each CSR edge set (offsets non-decreasing from 0 to `edges`,
//      ids below N and strictly ascending per row, weights finite and >= 0);
//   2. transpose each set (counting sort by target, then a per-row sort), so
//      the direction j -> i of a pair can be read from row i;
//   3. merge, for every anchor row i, the three out-lists (i -> *), the three
//      in-lists (* -> i) and the diagonal into one sorted list of "special"
//      columns, each carrying the resolved (attract?, weight) of both
//      directions.  Resolution order per direction: the diagonal is never
//      scored, then ignore, attract, repel, and otherwise the run's negatives
//      (ambient: repel at `ambient_weight`; named: skipped).
// Every other cell of row i resolves to the default in both directions, which
// is what the fused tile kernel assumes for columns not in the list.

#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {

namespace {

constexpr uint32_t kNone = 0xFFFFFFFFu;

// Rows 0..n-1 of one edge set; ids must lie below id_limit.
__global__ void validate_edges_kernel(EdgeSet s, int n, int id_limit, int32_t *status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (!s.offsets) return;
    if (i == 0 && (s.offsets[0] != 0 || s.offsets[n] != s.edges)) report(status, CLI_MALFORMED);
    if (i >= n) return;
    const uint64_t a = s.offsets[i], b = s.offsets[i + 1];
    if (a > b || b > s.edges) {
        report(status, CLI_MALFORMED);
        return;
    }
    uint32_t prev = 0;
    for (uint64_t k = a; k < b; ++k) {
        const uint32_t id = s.ids[k];
        if (id >= static_cast<uint32_t>(id_limit) || (k > a && id <= prev)) {
            report(status, CLI_MALFORMED);
            return;
        }
        prev = id;
        if (s.weights) {
            const float w = s.weights[k];
            if (!(w >= 0.0f) || isinf(w)) {
                report(status, CLI_MALFORMED);
                return;
            }
        }
    }
}

__global__ void validate_tape_kernel(const uint64_t *off, int count, uint64_t rows, int32_t *status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0 && (off[0] != 0 || off[count] != rows)) report(status, CLI_MALFORMED);
    if (i >= count) return;
    const uint64_t a = off[i], b = off[i + 1];
    if (a > b || b > rows) report(status, CLI_MALFORMED);
    else if (a == b) report(status, CLI_INVALID_ARGUMENT);  // an empty query or document has no max
}

// Every item's temperature group lies in [0, groups).
__global__ void validate_groups_kernel(const int32_t *group, int n, int groups, int32_t *status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n && (group[i] < 0 || group[i] >= groups)) report(status, CLI_MALFORMED);
}

__global__ void count_indegree_kernel(EdgeSet a, EdgeSet r, EdgeSet g, int n, uint32_t *indeg, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const EdgeSet sets[3] = {a, r, g};
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (!sets[s].offsets) continue;
        for (uint64_t k = sets[s].offsets[i]; k < sets[s].offsets[i + 1]; ++k)
            atomicAdd(&indeg[static_cast<size_t>(s) * n + sets[s].ids[k]], 1u);
    }
}

// Exclusive scan of `count` values into out[0..count], starting at `base`;
// one block of 1024 threads.  Each warp scans a contiguous range in coalesced
// 32-value steps (shuffles and a running carry, no block barrier), the warp
// totals are scanned once, and a second coalesced pass adds each warp's offset.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const uint32_t *in, uint32_t *out, int count,
                                                            uint32_t base, const int32_t *status) {
    if (read_status(status) != 0) return;
    constexpr int kWarps = kScanThreads / 32;
    __shared__ uint32_t warp_off[kWarps];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int per = ((count + kWarps - 1) / kWarps + 31) & ~31;
    const int lo = min(count, w * per), hi = min(count, lo + per);
    uint32_t carry = 0;
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const uint32_t v = i < hi ? in[i] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (i < hi) out[i] = carry + x - v;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) warp_off[w] = carry;
    __syncthreads();
    if (w == 0) {
        const uint32_t t = warp_off[lane];
        uint32_t x = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        warp_off[lane] = x - t;   // exclusive
        if (lane == 31) out[count] = base + x;
    }
    __syncthreads();
    const uint32_t add = base + warp_off[w];
    for (int i = lo + lane; i < hi; i += 32) out[i] += add;
}

__global__ void fill_transpose_kernel(EdgeSet a, EdgeSet r, EdgeSet g, int n, const uint32_t *tin_off,
                                      uint32_t *cursor, uint32_t *tin_ids, float *tin_w, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const EdgeSet sets[3] = {a, r, g};
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (!sets[s].offsets) continue;
        for (uint64_t k = sets[s].offsets[i]; k < sets[s].offsets[i + 1]; ++k) {
            const uint32_t j = sets[s].ids[k];
            const uint32_t pos = tin_off[static_cast<size_t>(s) * (n + 1) + j] +
                                 atomicAdd(&cursor[static_cast<size_t>(s) * n + j], 1u);
            tin_ids[pos] = static_cast<uint32_t>(i);
            tin_w[pos] = sets[s].weights ? sets[s].weights[k] : 1.0f;
        }
    }
}

// Sorts every transposed row by source id (rows are short: insertion sort).
// `present`: bit s set when edge set s was given (the others have no rows).
__global__ void sort_rows_kernel(const uint32_t *tin_off, uint32_t *tin_ids, float *tin_w, int n, int present,
                                 const int32_t *status) {
    if (read_status(status) != 0) return;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= 3 * n) return;
    const int s = idx / n, j = idx % n;
    if (!((present >> s) & 1)) return;
    const uint32_t a = tin_off[static_cast<size_t>(s) * (n + 1) + j];
    const uint32_t b = tin_off[static_cast<size_t>(s) * (n + 1) + j + 1];
    for (uint32_t k = a + 1; k < b; ++k) {
        const uint32_t id = tin_ids[k];
        const float w = tin_w[k];
        uint32_t m = k;
        while (m > a && tin_ids[m - 1] > id) {
            tin_ids[m] = tin_ids[m - 1];
            tin_w[m] = tin_w[m - 1];
            --m;
        }
        tin_ids[m] = id;
        tin_w[m] = w;
    }
}

struct Cursor {
    const uint32_t *ids;
    const float *w;
    uint32_t k, end;
    __device__ uint32_t head() const { return k < end ? ids[k] : kNone; }
};

// Merges row i's lists.  emit = false: count the distinct columns; emit = true:
// write the resolved entries at out.
template <bool emit>
__device__ uint32_t merge_row(int i, EdgeSet a, EdgeSet r, EdgeSet g, int n, const uint32_t *tin_off,
                              const uint32_t *tin_ids, const float *tin_w, int named, float ambient, RelEntry *out) {
    const EdgeSet sets[3] = {a, r, g};
    Cursor outc[3], inc[3];
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (sets[s].offsets) {
            outc[s] = {sets[s].ids, sets[s].weights, static_cast<uint32_t>(sets[s].offsets[i]),
                       static_cast<uint32_t>(sets[s].offsets[i + 1])};
            const size_t o = static_cast<size_t>(s) * (n + 1);
            inc[s] = {tin_ids, tin_w, tin_off[o + i], tin_off[o + i + 1]};
        } else {
            outc[s] = {nullptr, nullptr, 0u, 0u};
            inc[s] = {nullptr, nullptr, 0u, 0u};
        }
    }
    bool diag_left = true;
    uint32_t count = 0;
    const float w_def = named ? 0.0f : ambient;
    for (;;) {
        uint32_t c = diag_left ? static_cast<uint32_t>(i) : kNone;
#pragma unroll
        for (int s = 0; s < 3; ++s) {
            c = min(c, outc[s].head());
            c = min(c, inc[s].head());
        }
        if (c == kNone) break;
        bool o_in[3] = {false, false, false}, i_in[3] = {false, false, false};
        float o_w[3] = {1.f, 1.f, 1.f}, i_w[3] = {1.f, 1.f, 1.f};
#pragma unroll
        for (int s = 0; s < 3; ++s) {
            if (outc[s].head() == c) {
                o_in[s] = true;
                o_w[s] = outc[s].w ? outc[s].w[outc[s].k] : 1.0f;
                ++outc[s].k;
            }
            if (inc[s].head() == c) {
                i_in[s] = true;
                i_w[s] = inc[s].w[inc[s].k];
                ++inc[s].k;
            }
        }
        if (c == static_cast<uint32_t>(i)) diag_left = false;
        if (emit) {
            RelEntry e;
            e.col = c;
            e.flags = 0;
            // row -> col
            if (c == static_cast<uint32_t>(i) || o_in[2]) e.w_out = 0.f;
            else if (o_in[0]) { e.w_out = o_w[0]; e.flags |= 1u; }
            else if (o_in[1]) e.w_out = o_w[1];
            else e.w_out = w_def;
            // col -> row
            if (c == static_cast<uint32_t>(i) || i_in[2]) e.w_in = 0.f;
            else if (i_in[0]) { e.w_in = i_w[0]; e.flags |= 2u; }
            else if (i_in[1]) e.w_in = i_w[1];
            else e.w_in = w_def;
            out[count] = e;
        }
        ++count;
    }
    return count;
}

// Row i's merged list is written at rel_off[i] = the number of list slots of
// the rows before it, where row i has one slot per edge it is the source or the
// target of (in any set) plus one for the diagonal: an upper bound on its
// distinct columns, so no counting pass is needed.  Slots past the row's
// distinct columns hold sentinel entries (column 0xFFFFFFFF, past every real
// column), which the tile kernel never reaches.  rel_off[i] follows from the
// edge sets' offsets and the transposed offsets, both prefix sums already.
__device__ __forceinline__ uint32_t rel_slots_before(EdgeSet a, EdgeSet r, EdgeSet g, int n, const uint32_t *tin_off,
                                                     const uint32_t *tin_base, int i) {
    const EdgeSet sets[3] = {a, r, g};
    uint32_t before = static_cast<uint32_t>(i);
#pragma unroll
    for (int s = 0; s < 3; ++s)
        if (sets[s].offsets)
            before += static_cast<uint32_t>(sets[s].offsets[i]) +
                      (tin_off[static_cast<size_t>(s) * (n + 1) + i] - tin_base[s]);
    return before;
}

struct TinBase {
    uint32_t v[3];   // where each set's transposed ids start in the shared id array
};

__global__ void merge_emit_kernel(EdgeSet a, EdgeSet r, EdgeSet g, int n, const uint32_t *tin_off,
                                  const uint32_t *tin_ids, const float *tin_w, TinBase tb, uint32_t *rel_off,
                                  RelEntry *rel, int named, float ambient, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint32_t o0 = rel_slots_before(a, r, g, n, tin_off, tb.v, i);
    const uint32_t o1 = rel_slots_before(a, r, g, n, tin_off, tb.v, i + 1);
    rel_off[i] = o0;
    if (i == n - 1) rel_off[n] = o1;
    const uint32_t used = merge_row<true>(i, a, r, g, n, tin_off, tin_ids, tin_w, named, ambient, rel + o0);
    RelEntry sentinel;
    sentinel.col = kNone;
    sentinel.flags = 0;
    sentinel.w_out = 0.f;
    sentinel.w_in = 0.f;
    for (uint32_t k = o0 + used; k < o1; ++k) rel[k] = sentinel;
}

inline unsigned blocks_for(long long n, int threads) { return static_cast<unsigned>((n + threads - 1) / threads); }

}  // namespace

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

PooledWorkspace carve_pooled_workspace(void *base, size_t n, size_t width, size_t edges_total) {
    (void)width;
    PooledWorkspace w;
    uint8_t *p = static_cast<uint8_t *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *q = p ? p + off : nullptr;
        off += align256(bytes);
        return q;
    };
    w.indeg = reinterpret_cast<uint32_t *>(take(3 * n * sizeof(uint32_t)));
    w.tin_off = reinterpret_cast<uint32_t *>(take(3 * (n + 1) * sizeof(uint32_t)));
    w.tin_ids = reinterpret_cast<uint32_t *>(take((edges_total + 1) * sizeof(uint32_t)));
    w.tin_w = reinterpret_cast<float *>(take((edges_total + 1) * sizeof(float)));
    w.rel_off = reinterpret_cast<uint32_t *>(take((n + 1) * sizeof(uint32_t)));
    w.rel = reinterpret_cast<RelEntry *>(take((2 * edges_total + n) * sizeof(RelEntry)));
    w.partials = reinterpret_cast<float *>(
        take(static_cast<size_t>(pooled_partial_slots(static_cast<int>(n))) * 4 * sizeof(float)));
    w.sums = reinterpret_cast<double *>(take(static_cast<size_t>(pooled_finish_blocks()) * 3 * sizeof(double)));
    w.bytes = off;
    return w;
}

cudaError_t launch_validate_edges(const EdgeSet &set, int n, int id_limit, int32_t *status, cudaStream_t stream) {
    if (!set.offsets) return cudaSuccess;
    validate_edges_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(set, n, id_limit, status);
    return cudaGetLastError();
}

cudaError_t launch_validate_tape(const uint64_t *offsets, int count, uint64_t rows, int32_t *status,
                                 cudaStream_t stream) {
    validate_tape_kernel<<<blocks_for(count, 256), 256, 0, stream>>>(offsets, count, rows, status);
    return cudaGetLastError();
}

cudaError_t launch_validate_groups(const int32_t *group, int n, int groups, int32_t *status, cudaStream_t stream) {
    validate_groups_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(group, n, groups, status);
    return cudaGetLastError();
}

cudaError_t launch_relation_prep(const EdgeSet sets[3], int n, int named, float ambient, const PooledWorkspace &ws,
                                 int32_t *status, cudaStream_t stream) {
    cudaError_t err;
    for (int s = 0; s < 3; ++s)
        if ((err = launch_validate_edges(sets[s], n, n, status, stream)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(ws.indeg, 0, 3 * static_cast<size_t>(n) * sizeof(uint32_t), stream)) != cudaSuccess)
        return err;
    count_indegree_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(sets[0], sets[1], sets[2], n, ws.indeg, status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    // Transposed offsets of set s index one shared id array, after the sets before it (absent sets have
    // no transposed rows and are never read).
    uint64_t base = 0;
    TinBase tb;
    for (int s = 0; s < 3; ++s) {
        tb.v[s] = static_cast<uint32_t>(base);
        if (!sets[s].offsets) continue;
        scan_kernel<<<1, kScanThreads, 0, stream>>>(ws.indeg + static_cast<size_t>(s) * n,
                                                    ws.tin_off + static_cast<size_t>(s) * (n + 1), n,
                                                    static_cast<uint32_t>(base), status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        base += sets[s].edges;
    }
    if ((err = cudaMemsetAsync(ws.indeg, 0, 3 * static_cast<size_t>(n) * sizeof(uint32_t), stream)) != cudaSuccess)
        return err;
    fill_transpose_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(sets[0], sets[1], sets[2], n, ws.tin_off, ws.indeg,
                                                                   ws.tin_ids, ws.tin_w, status);
    const int present = (sets[0].offsets ? 1 : 0) | (sets[1].offsets ? 2 : 0) | (sets[2].offsets ? 4 : 0);
    sort_rows_kernel<<<blocks_for(3LL * n, 256), 256, 0, stream>>>(ws.tin_off, ws.tin_ids, ws.tin_w, n, present,
                                                                    status);
    merge_emit_kernel<<<blocks_for(n, 128), 128, 0, stream>>>(sets[0], sets[1], sets[2], n, ws.tin_off, ws.tin_ids,
                                                               ws.tin_w, tb, ws.rel_off, ws.rel, named, ambient,
                                                               status);
    return cudaGetLastError();
}

}  // namespace cli
