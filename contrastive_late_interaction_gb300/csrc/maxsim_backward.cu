// Hard MaxSim backward ("UForm", section "ColBERT-Style Late-Interaction
// Rerankers": each query token's gradient flows through its best match alone):
//     dQ[t] = sum_d c(q(t), d) D[d, a(t, d)],   dD[d, s] = sum_{t: a(t, d) = s} c(q(t), d) Q[t],
// with c = dS[q, d] (/ |q| for the mean form) and a the forward's argmax.
//
// GB300 design.  Both sums are gathers of bf16 rows that the L2 holds (the
// tapes), so neither needs a floating-point atomic: dQ walks the documents per
// query row (8 threads per row, document resolutions shared by shuffles), and
// dD sorts each document's query rows by their argmax target in shared memory
// (histogram, scan, scatter) and then sums each target's bucket.  Queries and
// documents no pair with c != 0 reaches are flagged first and skipped.  dD runs
// first; dQ, which reads nothing dD writes, is its programmatic dependent and
// starts on the SMs that dD's last wave leaves.

#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"
#include "compact.cuh"

namespace cli {
namespace ms {

// q_active[q] = 1 when some c(q, d) is nonzero, d_active[d] = 1 when some
// c(q, d) is (one block per query; both zeroed beforehand, every writer
// writes 1); the block also maps its query's rows to the query.
__global__ void active_kernel(const float *d_scores, long long ld_ds, int nd, const uint64_t *q_off, int32_t *qmap,
                              uint8_t *q_active, uint8_t *d_active, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int q = blockIdx.x;
    for (uint64_t t = q_off[q] + threadIdx.x; t < q_off[q + 1]; t += blockDim.x) qmap[t] = q;
    const float *row = d_scores + static_cast<long long>(q) * ld_ds;
    int any = 0;
    for (int d = threadIdx.x; d < nd; d += blockDim.x)
        if (row[d] != 0.0f) {
            any = 1;
            d_active[d] = 1;
        }
    if (__syncthreads_or(any) && threadIdx.x == 0) q_active[q] = 1;
}

// The map from query row to query, when there are no activity flags to compute
// (active_kernel writes it otherwise).
__global__ void qmap_kernel(const uint64_t *q_off, int nq, int32_t *qmap, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= nq) return;
    for (uint64_t t = q_off[q]; t < q_off[q + 1]; ++t) qmap[t] = q;
}

// A row of zeros as wide as the widest token (256 bf16): the gather source of
// a pair that adds nothing, so the gathers need neither branches nor masks.
__device__ const uint4 kZeroRow[32] = {};

// acc[i] += c * (the 8 bf16 of u), as four packed fp32 pair FMAs; u holds
// features 2i (low half of word i) and 2i + 1 (high half).
__device__ __forceinline__ void fma_bf16x8(float2 (&acc)[4], const uint4 u, float c) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = __ffma2_rn(make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u)), c2, acc[i]);
}

// dQ[t] = sum_d c(q(t), d) * D[d_off[d] + argmax[d][t]]: 8 threads per query
// row, each owning 8 features of every 64-feature block.  Documents go in
// steps of 8: thread `sub` of the row's group resolves document d0 + sub (its
// argmax entry, range check, row address and c) and the group shares the eight
// results by shuffles, so each thread then spends its instructions on the
// 16-byte gathers and packed FMAs.  The loads that resolve the next step are
// issued before this step's gathers, so a step waits on one round trip to L2,
// not two.  Only the step's documents with c != 0 for some row of the warp are
// gathered (a ballot over the group lanes; a loss that ignores pairs leaves
// many c = 0), and a pair that adds nothing reads a row of zeros, so no load or
// FMA is masked.
constexpr int kDqRows = 32;
constexpr int kDqUnroll = 8;
template <int NBLK>   // 64-feature blocks of the width (1..4)
// Up to width 128, at most 64 registers, so four blocks (32 warps) share an SM: the gathers are
// latency-bound.
__global__ void __launch_bounds__(256, NBLK <= 2 ? 4 : 2) dq_kernel(MaxSimBwdLaunch L) {
    if (read_status(L.status) != 0) return;
    const int t = blockIdx.x * kDqRows + (threadIdx.x >> 3);
    const int sub = threadIdx.x & 7;
    const bool row_ok = t < L.rows_q;      // rows past the tape still shuffle with their group
    const int tc = row_ok ? t : L.rows_q - 1;
    const int q = L.qmap[tc];
    const float scale = L.mean ? 1.0f / static_cast<float>(L.q_off[q + 1] - L.q_off[q]) : 1.0f;
    float2 acc[NBLK][4];
#pragma unroll
    for (int k = 0; k < NBLK; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[k][i] = make_float2(0.f, 0.f);
    const float *dsrow = L.d_scores + static_cast<long long>(q) * L.ld_ds;
    const int32_t *amcol = L.argmax + tc;
    // A warp whose rows all belong to queries no document scores with c != 0 stores zeros.
    const bool warp_idle = __all_sync(0xffffffffu, L.q_active != nullptr && L.q_active[q] == 0);
    // The documents in turn: the active ones from the list when some are not (every other document has
    // c = 0 for every query), else all of them in order (no list indirection in the loads).
    const int n_docs = L.d_list ? static_cast<int>(*L.d_count) : L.nd;
    const bool use_list = n_docs < L.nd;
    // The i-th document's id: from the list (a load, issued a step before the id is used, so that the
    // loads it addresses never wait on it) or i itself.
    auto id_at = [&](int i) { return use_list && i < n_docs ? static_cast<int>(__ldg(L.d_list + i)) : i; };
    // The loads that resolve the i-th document (its argmax entry and c, given its id) ...
    int a_n = 0, d_n = 0;
    float c_n = 0.f;
    auto fetch = [&](int i, int id) {
        if (i < n_docs) {
            d_n = id;
            a_n = __ldg(amcol + static_cast<long long>(d_n) * L.ld_argmax);
            c_n = __ldg(dsrow + d_n);
        }
    };
    // ... and their use, with the document's offsets (a small, cache-resident table): the gathered row
    // (the zero row past the last document, for a rejected entry or for c = 0) and c.
    const unsigned long long zero_row = reinterpret_cast<unsigned long long>(kZeroRow);
    auto finish = [&](int i, unsigned long long &src, float &c) {
        src = zero_row;
        c = 0.f;
        if (i < n_docs) {
            const int d = use_list ? d_n : i;   // in order, the offsets' addresses need no loaded value
            const uint64_t o = __ldg(L.d_off + d), e = __ldg(L.d_off + d + 1);
            if (c_n != 0.0f) {   // a pair with c = 0 (one a loss ignores) gathers nothing, nor is checked
                if (a_n < 0 || static_cast<uint64_t>(a_n) >= e - o) {
                    if (row_ok) report(L.status, CLI_MALFORMED);
                } else {
                    src = reinterpret_cast<unsigned long long>(L.d + (o + static_cast<uint64_t>(a_n)) * L.width);
                    c = c_n * scale;
                }
            }
        }
    };
    // This thread's features of every 64-feature block (a block past the width reads the row's last 8
    // features: they land in accumulators that are never stored).
    int fo[NBLK];
#pragma unroll
    for (int k = 0; k < NBLK; ++k) fo[k] = min(k * 64 + sub * 8, L.width - 8);
    // One step: this lane's group holds document d0 + u's row address and c in lane u of the group.
    auto step = [&](unsigned long long src, float c) {
        // The step's documents with c != 0 for some row of the warp, in order: the warp's rows usually
        // belong to one query, so this is the step's active set, and a pair with c = 0 costs no gather.
        const unsigned act = __ballot_sync(0xffffffffu, c != 0.0f);
        unsigned mm = (act | (act >> 8) | (act >> 16) | (act >> 24)) & 0xFFu;
        const int n_act = __popc(mm);
        if (n_act == kDqUnroll) {
            // Every document of the step: all eight rows' loads in flight together, then the FMAs (a row
            // with c = 0 for a document reads the zero row).
            uint4 x[kDqUnroll][NBLK];
            float cu[kDqUnroll];
#pragma unroll
            for (int u = 0; u < kDqUnroll; ++u) {
                const uint16_t *row = reinterpret_cast<const uint16_t *>(__shfl_sync(0xffffffffu, src, u, 8));
                cu[u] = __shfl_sync(0xffffffffu, c, u, 8);
#pragma unroll
                for (int k = 0; k < NBLK; ++k) x[u][k] = __ldg(reinterpret_cast<const uint4 *>(row + fo[k]));
            }
#pragma unroll
            for (int u = 0; u < kDqUnroll; ++u)
#pragma unroll
                for (int k = 0; k < NBLK; ++k) fma_bf16x8(acc[k], x[u][k], cu[u]);
            return;
        }
        // The active documents four at a time, the same way (a slot past the last one reads the zero
        // row with c = 0).
        for (int u0 = 0; u0 < n_act; u0 += 4) {
            uint4 x[4][NBLK];
            float cu[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = mm != 0 ? __ffs(mm) - 1 : 0;
                mm &= mm - 1;
                unsigned long long sp = __shfl_sync(0xffffffffu, src, p, 8);
                cu[u] = __shfl_sync(0xffffffffu, c, p, 8);
                if (u0 + u >= n_act) {
                    sp = zero_row;
                    cu[u] = 0.f;
                }
                const uint16_t *row = reinterpret_cast<const uint16_t *>(sp);
#pragma unroll
                for (int k = 0; k < NBLK; ++k) x[u][k] = __ldg(reinterpret_cast<const uint4 *>(row + fo[k]));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int k = 0; k < NBLK; ++k) fma_bf16x8(acc[k], x[u][k], cu[u]);
        }
    };
    unsigned long long src;
    float c;
    fetch(sub, id_at(sub));
    finish(sub, src, c);
    int id_next = id_at(kDqUnroll + sub);
    for (int d0 = 0; d0 < (warp_idle ? 0 : n_docs); d0 += kDqUnroll) {
        const int id_after = id_at(d0 + 2 * kDqUnroll + sub);   // the id two steps on, in flight meanwhile
        fetch(d0 + kDqUnroll + sub, id_next);   // the next step's resolution, in flight during this step
        step(src, c);
        finish(d0 + kDqUnroll + sub, src, c);
        id_next = id_after;
    }
    if (!row_ok) return;
    float *dst = L.dq + static_cast<long long>(t) * L.width;
#pragma unroll
    for (int k = 0; k < NBLK; ++k) {
        const int f = k * 64 + sub * 8;
        if (f < L.width) {
            reinterpret_cast<float4 *>(dst + f)[0] = make_float4(acc[k][0].x, acc[k][0].y, acc[k][1].x, acc[k][1].y);
            reinterpret_cast<float4 *>(dst + f)[1] = make_float4(acc[k][2].x, acc[k][2].y, acc[k][3].x, acc[k][3].y);
        }
    }
}

// dD rows of one document by sort-then-gather.  For a window of up to
// kDsMaxRows document rows and a chunk of up to kDsChunk query rows:
//   1. count, per document row s, the query rows whose argmax names it
//      (shared-memory histogram), and scan the counts into bucket offsets;
//   2. scatter the query rows into their buckets (a shared list of the row's
//      offset in the chunk and, in the high half, its query, so that step 3
//      reads c(q, d) from the shared table without a global lookup);
//   3. 8-lane groups take document rows in turn and sum c(q(t), d) * Q[t] over
//      the row's bucket in registers, lanes as features (whole-sector row
//      gathers from the L2-resident query tape), then write the row once (the
//      first chunk stores, later chunks add; the CTA owns the document, so no
//      atomics touch dD).
// No floating-point atomics; results do not depend on scheduling order within
// a bucket because each bucket is summed by one group in list order, and the
// list order is the scatter order (atomic slot claims), which may vary between
// runs: dD is reproducible to rounding, not bit for bit.
// One CTA of 1024 threads per SM, so the list holds 32800 query rows (160 KB of
// shared memory in all): two chunks cover 65600 query rows, and every chunk past
// the first pays its sort passes again and a read-modify-write of the rows (with
// two CTAs of 512 threads and 16384-row chunks the config-5 backward took 3.28
// ms, with this 2.91 ms; one chunk over every row whose c is nonzero, in a
// 49152-entry list, measured 2.90 ms at config 5 and slower at config 3).
constexpr int kDsThreads = 1024;
constexpr int kDsMaxRows = 2048;
constexpr int kDsChunk = 32800;
constexpr int kDsMaxTable = 4096;
constexpr int kDsBatch = 8;   // argmax entries per thread in flight in the histogram and scatter passes

__host__ __device__ inline size_t ds_smem_bytes() {
    return static_cast<size_t>(kDsMaxRows) * 4 + (kDsMaxRows + 1) * 4 + kDsChunk * 4 + kDsMaxTable * 4 + 64;
}

// A 16-byte block of zeros in device memory: the load address of a lane with
// nothing to gather, so the gathers need neither branches nor masks.
__device__ const uint4 kZero16 = {0u, 0u, 0u, 0u};

// Adds c(q(t), d) * Q[t] over the bucket entries [b0, b1) into this lane's
// accumulators (features 16 part .. 16 part + 15 of every 128-feature block;
// acc[k][h][i] holds features 16 part + 8h + 2i, + 1 of block k), kUnroll entries
// in flight.  kFast: the list entries name the query and c comes from the
// shared table; otherwise the query and c come from device memory.
template <int NB, int kUnroll, bool kFast>
__device__ __forceinline__ void dd_row_sum(const MaxSimBwdLaunch &L, const uint32_t *list, const float *ctab, int d,
                                           int c0, uint32_t b0, uint32_t b1, int part, float2 (&acc)[NB][2][4]) {
    for (uint32_t e = b0; e < b1; e += kUnroll) {
        uint4 x[kUnroll][NB][2];
        float c[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const bool v = e + u < b1;
            const uint32_t ent = list[v ? e + u : b0];
            const int t = c0 + static_cast<int>(ent & 0xFFFFu);
            float cc;
            if (kFast) {
                cc = ctab[ent >> 16];
            } else {
                const int q = __ldg(L.qmap + t);
                cc = __ldg(L.d_scores + static_cast<long long>(q) * L.ld_ds + d);
                if (L.mean) cc /= static_cast<float>(L.q_off[q + 1] - L.q_off[q]);
            }
            c[u] = v ? cc : 0.f;
            const uint16_t *src = L.q + static_cast<long long>(t) * L.width;
#pragma unroll
            for (int k = 0; k < NB; ++k)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int f = k * 128 + part * 16 + h * 8;
                    x[u][k][h] = __ldg((v && f < L.width) ? reinterpret_cast<const uint4 *>(src + f) : &kZero16);
                }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                fma_bf16x8(acc[k][0], x[u][k][0], c[u]);
                fma_bf16x8(acc[k][1], x[u][k][1], c[u]);
            }
    }
}

// NB: 128-feature blocks of the width (ceil(width / 128)); kDsUnroll: bucket
// entries in flight per 8-lane group.
template <int NB, int kDsUnroll>
__global__ void __launch_bounds__(kDsThreads, 1) dd_sort_kernel(MaxSimBwdLaunch L) {
    extern __shared__ uint8_t ds_raw[];
    // dQ (launched next) reads nothing dD writes: let its CTAs start on the SMs this grid's last wave leaves.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    uint32_t *cnt = reinterpret_cast<uint32_t *>(ds_raw);            // [kDsMaxRows] counts, then cursors
    uint32_t *off = cnt + kDsMaxRows;                                  // [kDsMaxRows + 1] bucket starts
    uint32_t *list = off + kDsMaxRows + 1;                             // [kDsChunk] (q << 16) | row offset
    float *ctab = reinterpret_cast<float *>(list + kDsChunk);          // [kDsMaxTable]
    __shared__ uint32_t warp_sums[kDsThreads / 32];
    if (read_status(L.status) != 0) return;
    const int d = blockIdx.x;
    if (L.d_active && !L.d_active[d]) {   // no query scores it: its rows are zero (its argmax entries are not read)
        const uint64_t z0 = L.d_off[d];
        float4 *dst = reinterpret_cast<float4 *>(L.dd + static_cast<long long>(z0) * L.width);
        const long long n4 = static_cast<long long>(L.d_off[d + 1] - z0) * L.width / 4;
        for (long long i = threadIdx.x; i < n4; i += kDsThreads) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t o0 = L.d_off[d];
    const int dl = static_cast<int>(L.d_off[d + 1] - o0);
    const int32_t *am = L.argmax + static_cast<long long>(d) * L.ld_argmax;
    const bool use_table = L.nq <= kDsMaxTable;
    const bool packed = L.nq <= 65536;   // list entries carry the query as well as the row
    // With c(q, d) in the shared table, rows whose c is zero (pairs a named loss does not score) are left out
    // of the buckets: they add nothing.
    const bool skip_zero = use_table && packed;
    if (use_table)
        for (int q = threadIdx.x; q < L.nq; q += kDsThreads) {
            float c = L.d_scores[static_cast<long long>(q) * L.ld_ds + d];
            if (L.mean) c /= static_cast<float>(L.q_off[q + 1] - L.q_off[q]);
            ctab[q] = c;
        }
    for (int w0 = 0; w0 < dl; w0 += kDsMaxRows) {
        const int wrows = min(kDsMaxRows, dl - w0);
        // Chunks of equal size (none a small remainder: every chunk pays a pass over the buckets).
        const int n_chunks = (L.rows_q + kDsChunk - 1) / kDsChunk;
        const int chunk_rows = (L.rows_q + n_chunks - 1) / n_chunks;
        for (int c0 = 0; c0 < L.rows_q; c0 += chunk_rows) {
            const int crows = min(chunk_rows, L.rows_q - c0);
            for (int r = threadIdx.x; r < wrows; r += kDsThreads) cnt[r] = 0;
            __syncthreads();
            // 1. histogram of the chunk's targets inside the window (eight loads in flight per thread)
            for (int k0 = threadIdx.x; k0 < crows; k0 += kDsBatch * kDsThreads) {
                int a[kDsBatch], qv[kDsBatch];
#pragma unroll
                for (int i = 0; i < kDsBatch; ++i) {
                    const int k = k0 + i * kDsThreads;
                    a[i] = k < crows ? __ldg(am + c0 + k) : 0;
                    qv[i] = (skip_zero && k < crows) ? __ldg(L.qmap + c0 + k) : 0;
                }
#pragma unroll
                for (int i = 0; i < kDsBatch; ++i) {
                    if (k0 + i * kDsThreads >= crows) break;
                    if (skip_zero && ctab[qv[i]] == 0.0f) continue;   // adds nothing to dD, and is not read
                    if (a[i] < 0 || a[i] >= dl) {
                        report(L.status, CLI_MALFORMED);
                        continue;
                    }
                    const int r = a[i] - w0;
                    if (r >= 0 && r < wrows) atomicAdd(&cnt[r], 1u);
                }
            }
            __syncthreads();
            // exclusive scan of cnt[0..wrows) into off[], then cnt[] becomes the cursor
            {
                constexpr int kPer = kDsMaxRows / kDsThreads;   // entries per thread
                uint32_t v[kPer], sum = 0;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int r = threadIdx.x * kPer + i;
                    v[i] = r < wrows ? cnt[r] : 0u;
                    sum += v[i];
                }
                uint32_t x = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane == 31) warp_sums[warp] = x;
                __syncthreads();
                uint32_t before = 0;
                for (int w = 0; w < warp; ++w) before += warp_sums[w];
                uint32_t run = before + x - sum;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int r = threadIdx.x * kPer + i;
                    if (r < wrows) {
                        off[r] = run;
                        cnt[r] = run;
                    }
                    run += v[i];
                }
                if (threadIdx.x == kDsThreads - 1) off[wrows] = run;
            }
            __syncthreads();
            // 2. scatter the chunk's rows into their buckets (eight rows per thread at a time)
            for (int k0 = threadIdx.x; k0 < crows; k0 += kDsBatch * kDsThreads) {
                int a[kDsBatch];
                uint32_t qk[kDsBatch];
#pragma unroll
                for (int i = 0; i < kDsBatch; ++i) {
                    const int k = k0 + i * kDsThreads;
                    a[i] = k < crows ? __ldg(am + c0 + k) : -1;
                    qk[i] = (packed && k < crows) ? static_cast<uint32_t>(__ldg(L.qmap + c0 + k)) << 16 : 0u;
                }
#pragma unroll
                for (int i = 0; i < kDsBatch; ++i) {
                    const int r = a[i] - w0;
                    if (skip_zero && a[i] >= 0 && ctab[qk[i] >> 16] == 0.0f) continue;   // as in the histogram
                    if (a[i] >= 0 && a[i] < dl && r >= 0 && r < wrows)
                        list[atomicAdd(&cnt[r], 1u)] = qk[i] | static_cast<uint32_t>(k0 + i * kDsThreads);
                }
            }
            __syncthreads();
            // 3. one 8-lane group per document row (bucket): sum c * Q[t] over its entries,
            //    lane `part` owning features 16 part .. 16 part + 15 of every 128-feature block.
            //    The first chunk stores the row, later chunks add to it.
            const int part = lane & 7;
            for (int r = warp * 4 + (lane >> 3); r < wrows; r += kDsThreads / 8) {
                float2 acc[NB][2][4];
#pragma unroll
                for (int k = 0; k < NB; ++k)
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) acc[k][i2 >> 2][i2 & 3] = make_float2(0.f, 0.f);
                const uint32_t b0 = off[r], b1 = off[r + 1];
                if (use_table && packed)
                    dd_row_sum<NB, kDsUnroll, true>(L, list, ctab, d, c0, b0, b1, part, acc);
                else
                    dd_row_sum<NB, kDsUnroll, false>(L, list, ctab, d, c0, b0, b1, part, acc);
                float *dst = L.dd + (static_cast<long long>(o0) + w0 + r) * L.width;
#pragma unroll
                for (int k = 0; k < NB; ++k)
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int f = k * 128 + part * 16 + h * 4;
                        if (f < L.width) {
                            const float2 p0 = acc[k][h >> 1][2 * (h & 1)], p1 = acc[k][h >> 1][2 * (h & 1) + 1];
                            float4 v4 = make_float4(p0.x, p0.y, p1.x, p1.y);
                            if (c0 > 0) {
                                const float4 o4 = *reinterpret_cast<const float4 *>(dst + f);
                                v4.x += o4.x; v4.y += o4.y; v4.z += o4.z; v4.w += o4.w;
                            }
                            *reinterpret_cast<float4 *>(dst + f) = v4;
                        }
                    }
            }
            __syncthreads();
        }
    }
}

// Backward over named pairs only: one warp per named (query, document) pair,
// rows of the query in turn; lanes own 4 features of each 128-feature block.
// dQ[t] += c D[argmax], dD[argmax] += c Q[t] with vector L2 reductions (dQ and
// dD zeroed before): the sums reproduce to rounding, not bit for bit.
__global__ void __launch_bounds__(256) named_backward_kernel(MaxSimBwdLaunch L, const uint64_t *pair_off,
                                                             const uint32_t *pair_ids, long long pairs) {
    if (read_status(L.status) != 0) return;
    const long long k = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (k >= pairs) return;
    int lo = 0, hi = L.nq;   // the query q with pair_off[q] <= k < pair_off[q + 1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pair_off[mid] <= static_cast<uint64_t>(k)) lo = mid; else hi = mid;
    }
    const int q = lo, d = static_cast<int>(pair_ids[k]);
    const uint64_t t0 = L.q_off[q], t1 = L.q_off[q + 1], o = L.d_off[d], len = L.d_off[d + 1] - o;
    float c = L.d_scores[static_cast<long long>(q) * L.ld_ds + d];
    if (L.mean) c /= static_cast<float>(t1 - t0);
    if (c == 0.0f) return;
    for (uint64_t t = t0; t < t1; ++t) {
        const int a = __ldg(L.argmax + static_cast<long long>(d) * L.ld_argmax + static_cast<long long>(t));
        if (a < 0 || static_cast<uint64_t>(a) >= len) {
            if (lane == 0) report(L.status, CLI_MALFORMED);
            continue;
        }
        const uint16_t *dr = L.d + (o + static_cast<uint64_t>(a)) * L.width, *qr = L.q + t * L.width;
        float *dq = L.dq + t * L.width, *dd = L.dd + (o + static_cast<uint64_t>(a)) * L.width;
        for (int f = lane * 4; f < L.width; f += 128) {
            const uint2 xd = *reinterpret_cast<const uint2 *>(dr + f), xq = *reinterpret_cast<const uint2 *>(qr + f);
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dq + f),
                         "f"(c * __uint_as_float(xd.x << 16)), "f"(c * __uint_as_float(xd.x & 0xFFFF0000u)),
                         "f"(c * __uint_as_float(xd.y << 16)), "f"(c * __uint_as_float(xd.y & 0xFFFF0000u))
                         : "memory");
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dd + f),
                         "f"(c * __uint_as_float(xq.x << 16)), "f"(c * __uint_as_float(xq.x & 0xFFFF0000u)),
                         "f"(c * __uint_as_float(xq.y << 16)), "f"(c * __uint_as_float(xq.y & 0xFFFF0000u))
                         : "memory");
        }
    }
}

}  // namespace ms

// dQ as a programmatic dependent of the dD grid launched just before it on the
// same stream: its CTAs may start once every dD CTA has started (dD signals at
// its start), filling the SMs that dD's last wave (one long CTA per SM, one
// document each) leaves idle.  dQ reads only what the kernels before dD wrote
// (they completed before dD began), never dD's output, so it needs no wait on
// the dD grid; the stream's later work still waits for both.
template <typename K>
cudaError_t launch_after_dd(K kernel, const MaxSimBwdLaunch &L, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((L.rows_q + ms::kDqRows - 1) / ms::kDqRows));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, L);
}

cudaError_t launch_maxsim_backward(const MaxSimBwdLaunch &L, cudaStream_t stream) {
    using namespace ms;
    cudaError_t err;
    if (L.q_active) {   // the activity flags (and the row -> query map), then the list of active documents
        if ((err = cudaMemsetAsync(L.q_active, 0, L.nq, stream)) != cudaSuccess ||
            (err = cudaMemsetAsync(L.d_active, 0, L.nd, stream)) != cudaSuccess)
            return err;
        active_kernel<<<L.nq, 256, 0, stream>>>(L.d_scores, L.ld_ds, L.nd, L.q_off, L.qmap, L.q_active, L.d_active,
                                               L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        compact_items_kernel<uint8_t><<<1, kCompactThreads, 0, stream>>>(L.d_active, L.nd, L.d_list, L.d_count,
                                                                         L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    } else {
        qmap_kernel<<<(L.nq + 255) / 256, 256, 0, stream>>>(L.q_off, L.nq, L.qmap, L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    const size_t ds_smem = ds_smem_bytes();
    if ((L.width + 127) / 128 == 1) {
        if ((err = cudaFuncSetAttribute(dd_sort_kernel<1, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(ds_smem))) != cudaSuccess)
            return err;
        dd_sort_kernel<1, 4><<<L.nd, kDsThreads, ds_smem, stream>>>(L);
    } else {
        if ((err = cudaFuncSetAttribute(dd_sort_kernel<2, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(ds_smem))) != cudaSuccess)
            return err;
        dd_sort_kernel<2, 1><<<L.nd, kDsThreads, ds_smem, stream>>>(L);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    switch ((L.width + 63) / 64) {
        case 1: err = launch_after_dd(dq_kernel<1>, L, stream); break;
        case 2: err = launch_after_dd(dq_kernel<2>, L, stream); break;
        case 3: err = launch_after_dd(dq_kernel<3>, L, stream); break;
        default: err = launch_after_dd(dq_kernel<4>, L, stream); break;
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}


cudaError_t launch_maxsim_backward_named(const MaxSimBwdLaunch &L, const uint64_t *pair_off, const uint32_t *pair_ids,
                                         long long pairs, cudaStream_t stream) {
    if (pairs == 0) return cudaSuccess;
    ms::named_backward_kernel<<<static_cast<unsigned>((pairs + 7) / 8), 256, 0, stream>>>(L, pair_off, pair_ids,
                                                                                        pairs);
    return cudaGetLastError();
}

}  // namespace cli
