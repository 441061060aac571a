// Hard MaxSim late interaction over ragged token tapes ("UForm", section
// "ColBERT-Style Late-Interaction Rerankers"; tapes as in "Arenas", "Rows and
// Tapes"):
//     S(q, d) = sum_{t in q} max_{s in d} <q_t, d_s>   (optionally / |q|)
// forward with the argmax, backward routed through it.
//
// GB300 design of the forward.  The whole query tape times the whole document
// tape is one dense contraction with K = width, so it runs on tcgen05: a CTA
// keeps a 128-row block of the query tape resident in shared memory and
// streams 128-row tiles of the document tape through a TMA ring; each tile
// product lands in one of two TMEM buffers.  Four epilogue warps read the
// tiles back, one query row per thread, and keep a running (max, argmax) per
// row across the tiles of the current document; the boundaries between
// documents are the same for every row, so the segment logic is warp-uniform.
// Per 32-column chunk each score becomes a key that carries the column in the
// 5 low mantissa bits (31 - column, so among equal positive values the largest
// key names the lowest column; one ALU instruction per cell).  For a chunk
// inside one document the keys go back into TMEM and a reducing TMEM load
// returns their maximum; a chunk holding a document boundary masks its keys per
// segment and reduces them with a tree of three-input max operations.  The
// reported value is truncated by less than 2^-18 relative.  A row whose
// maximum over a document is not a positive normal number (every score of the
// document negative, whose keys order equal values the other way, or zero, or
// subnormal) is listed by the per-query sums, which read every maximum anyway,
// and `argmax_fixup_kernel` finds its argmax again in float64 from the tapes,
// the lowest row among equal scores; the tile kernel does nothing for it.
//
// The ragged schedule: the document tape is cut into chunks of whole
// documents of about `chunk_rows` rows (a binary search over the offsets per
// chunk), and a work item is (chunk, query block).  Items run chunk-major, so
// the CTAs running at the same time share one chunk of the document tape in L2.
//
// Per-row maxima go to a document-major workspace m[d][t]; a second kernel sums
// them per query in a fixed order.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace ms {

constexpr int BM = 128;   // query rows per block
constexpr int BN = 128;   // document rows per tile
constexpr int BK = 64;    // K extent of one TMA box
constexpr int STAGES = 2;
constexpr uint32_t BOX_BYTES = 128 * BK * 2;   // 16 KB
constexpr int kThreads = 192;
constexpr uint32_t TMEM_COLS = 256;            // two 128-column score buffers

struct Barriers {
    uint64_t q_full, q_free, full[STAGES], empty[STAGES], s_full[2], s_free[2], mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

// Dynamic shared memory: [Q: nk boxes][ring: STAGES x nk boxes][Barriers].
__host__ __device__ inline size_t smem_bytes_for(int nk) {
    return 1024 + static_cast<size_t>(nk) * BOX_BYTES * (1 + STAGES) + sizeof(Barriers);
}

struct Params {
    int nq, nd, rows_q, rows_d, width, nk, mean;
    int n_mblocks, n_chunks;
    long long items;
    const uint64_t *q_off, *d_off;
    const uint32_t *chunk_doc;
    int32_t *argmax;
    long long ld_argmax;
    float *mval;
    int32_t *status;
    // Named pairs: the work items to run (chunk * n_mblocks + mblock, in
    // chunk-major order) and their count on the device; null runs every item.
    const uint32_t *item_list, *item_count;
};

// The number of work items and the w-th one as (chunk, query block).
__device__ __forceinline__ long long item_total(const Params &P) {
    return P.item_list ? static_cast<long long>(*P.item_count) : P.items;
}
__device__ __forceinline__ void item_at(const Params &P, long long w, int &chunk, int &mb) {
    const long long it = P.item_list ? static_cast<long long>(P.item_list[w]) : w;
    chunk = static_cast<int>(it / P.n_mblocks);
    mb = static_cast<int>(it % P.n_mblocks);
}

// Keys: each score's bits with the 5 low mantissa bits replaced by 31 - column
// (one lop3, the mask ~31 held in a register so the two-constant form does not
// split into two operations).  The largest key is the largest score truncated
// by less than 2^-18 relative.  Among equal truncated scores that are positive
// it names the lowest column.  Among negative ones a larger low field makes a
// smaller float, so it names the highest column, and a zero or subnormal
// maximum may be flushed by a reducing load: a key that is not a positive
// normal number does not decode to the lowest column.  A document maximum that
// is a positive normal number came from a key that does (truncation keeps a
// positive normal value positive and normal), so a row whose maximum over the
// document is anything else goes to the float64 fix-up.

// Running (max, argmax) update from the largest key of a chunk's columns of the
// current document; `base` is the chunk's first row relative to the document.
__device__ __forceinline__ void update_best(float key, int base, float &best, int &best_col) {
    const int bits = __float_as_int(key);
    const float val = __int_as_float(bits & ~31);
    if (val > best) {
        best = val;
        best_col = base + (31 - (bits & 31));
    }
}

// The keys of a chunk into TMEM (over its scores, which are not read again).
__device__ __forceinline__ void chunk_keys_to_tmem(uint32_t taddr, uint32_t hi_mask) {
    uint32_t r[32];
    tmem_ld32_async(taddr, r);
    tmem_wait_ld();
    tmem_regs_ready(r);
#pragma unroll
    for (int i = 0; i < 32; ++i)
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r[i]) : "r"(r[i]), "r"(hi_mask), "r"(31 - i));
    tmem_st32(taddr, r);
    tmem_wait_st();
    tmem_regs_ready(r);   // the store's registers stay reserved until it has completed
}

// The update from a chunk wholly inside the current document: its keys go to
// TMEM and a reducing TMEM load returns their maximum, so no max tree runs on
// the ALU.
__device__ __forceinline__ void chunk_max_tmem(uint32_t taddr, int base, float &best, int &best_col,
                                               uint32_t hi_mask) {
    chunk_keys_to_tmem(taddr, hi_mask);
    uint32_t x[32];
    float m;
    tmem_ld32_max_async(taddr, x, m);
    tmem_wait_ld();
    tmem_regs_ready(x, m);
    update_best(m, base, best, best_col);
}

// Largest keys of a chunk's columns [0, p) and [p, 32) (0 < p < 32, warp-uniform)
// from keys already in TMEM.  Each range is a run of aligned power-of-two
// pieces (the prefix by the bits of p from the top, the suffix by the bits of
// p from the bottom).  Every piece slot is loaded, an absent one from the
// chunk's first columns, and dropped afterwards, so no register written by an
// asynchronous load is merged across a branch; all loads are in flight
// together, and the TMEM loads reduce the pieces of four columns and more.
struct SplitLoads {
    uint32_t r16[16], r8[8], r4[4], r2[2], r1;
    float m16, m8, m4;
    unsigned present;   // bit s: the piece of 2^s columns is part of the range
};

__device__ __forceinline__ void split_issue(uint32_t ta, int lo_of[5], SplitLoads &x) {
    auto at = [&](int s) { return ta + static_cast<uint32_t>((x.present >> s) & 1u ? lo_of[s] : 0); };
    tmem_ld16_max_async(at(4), x.r16, x.m16);
    tmem_ld8_max_async(at(3), x.r8, x.m8);
    tmem_ld4_max_async(at(2), x.r4, x.m4);
    tmem_ld2_async(at(1), x.r2);
    tmem_ld1_async(at(0), x.r1);
}

__device__ __forceinline__ float split_result(SplitLoads &x) {
    tmem_regs_ready_n(x.r16);
    tmem_regs_ready_n(x.r8);
    tmem_regs_ready_n(x.r4);
    tmem_regs_ready_n(x.r2);
    asm volatile("" : "+r"(x.r1), "+f"(x.m16), "+f"(x.m8), "+f"(x.m4)::"memory");
    const float ninf = -INFINITY;
    const unsigned pr = x.present;
    const float m2 = fmaxf(__uint_as_float(x.r2[0]), __uint_as_float(x.r2[1]));
    return fmaxf(fmax3(pr & 16u ? x.m16 : ninf, pr & 8u ? x.m8 : ninf, pr & 4u ? x.m4 : ninf),
                 fmaxf(pr & 2u ? m2 : ninf, pr & 1u ? __uint_as_float(x.r1) : ninf));
}

// `two`: whether the suffix is wanted.
__device__ __forceinline__ void split_max(uint32_t ta, int p, bool two, float &ma, float &mb) {
    SplitLoads a, b;
    int lo_a[5], lo_b[5];
    a.present = static_cast<unsigned>(p) & 31u;   // prefix: pieces from the largest down
    int lo = 0;
#pragma unroll
    for (int s = 4; s >= 0; --s) {
        lo_a[s] = lo;
        if (a.present & (1u << s)) lo += 1 << s;
    }
    b.present = two ? (32u - static_cast<unsigned>(p)) & 31u : 0u;   // suffix: from the smallest up
    lo = p;
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        lo_b[s] = lo;
        if (b.present & (1u << s)) lo += 1 << s;
    }
    split_issue(ta, lo_a, a);
    split_issue(ta, lo_b, b);
    tmem_wait_ld();
    ma = split_result(a);
    mb = split_result(b);
}

// The update from 32 scores of a chunk restricted to its columns [lo, hi)
// (a chunk holding a document boundary or the end of the work item): keys
// outside the range become -inf and a tree of three-input max operations
// (16 instructions) picks the largest.
__device__ __forceinline__ void chunk_max(const float (&v)[32], int lo, int hi, int base, float &best, int &best_col,
                                          uint32_t hi_mask) {
    float key[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        uint32_t kb;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(kb) : "r"(__float_as_uint(v[r])), "r"(hi_mask), "r"(31 - r));
        key[r] = (r >= lo && r < hi) ? __uint_as_float(kb) : -INFINITY;
    }
    float m[12];
#pragma unroll
    for (int i = 0; i < 10; ++i) m[i] = fmax3(key[3 * i], key[3 * i + 1], key[3 * i + 2]);
    m[10] = key[30];
    m[11] = key[31];
    const float n0 = fmax3(m[0], m[1], m[2]), n1 = fmax3(m[3], m[4], m[5]);
    const float n2 = fmax3(m[6], m[7], m[8]), n3 = fmax3(m[9], m[10], m[11]);
    update_best(fmaxf(fmax3(n0, n1, n2), n3), base, best, best_col);
}

__global__ void __launch_bounds__(kThreads, 2)
    forward_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_d, Params P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *q_smem = base;
    uint8_t *ring = base + static_cast<size_t>(P.nk) * BOX_BYTES;
    Barriers &bar = *reinterpret_cast<Barriers *>(ring + static_cast<size_t>(STAGES) * P.nk * BOX_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (read_status(P.status) != 0) return;

    if (threadIdx.x == 0) {
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_free, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bar.full[s], 1);
            mbar_init(&bar.empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.s_full[s], 1);
            mbar_init(&bar.s_free[s], 4);
        }
        mbar_init(&bar.mma_done, 1);
        bar.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_d);
    }
    if (warp == 1) tmem_alloc(&bar.tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;
    volatile int *abort_flag = &bar.abort_flag;
    const uint32_t stage_bytes = static_cast<uint32_t>(P.nk) * BOX_BYTES;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, it = 0;
            bool ok = true;
            const long long items = item_total(P);
            for (long long w = blockIdx.x; w < items && ok; w += gridDim.x) {
                int chunk, mb;
                item_at(P, w, chunk, mb);
                const uint32_t d0 = P.chunk_doc[chunk], d1 = P.chunk_doc[chunk + 1];
                if (d0 == d1) continue;
                const long long r_lo = static_cast<long long>(P.d_off[d0]), r_hi = static_cast<long long>(P.d_off[d1]);
                if (!mbar_wait(&bar.q_free, (it & 1) ^ 1, abort_flag, P.status, kSleepProducer)) break;
                ++it;
                mbar_arrive_expect_tx(&bar.q_full, stage_bytes);
                for (int kc = 0; kc < P.nk; ++kc)
                    tma_load_2d(q_smem + kc * BOX_BYTES, &tmap_q, &bar.q_full, kc * BK, mb * BM);
                for (long long r0 = r_lo; r0 < r_hi; r0 += BN) {
                    if (!mbar_wait(&bar.empty[stage], phase ^ 1, abort_flag, P.status, kSleepProducer)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar.full[stage], stage_bytes);
                    uint8_t *dst = ring + static_cast<size_t>(stage) * stage_bytes;
                    for (int kc = 0; kc < P.nk; ++kc)
                        tma_load_2d(dst + kc * BOX_BYTES, &tmap_d, &bar.full[stage], kc * BK, static_cast<int>(r0));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                mbar_wait(&bar.empty[stage], phase ^ 1, abort_flag, P.status);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            mbar_wait(&bar.q_free, (it & 1) ^ 1, abort_flag, P.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, 128, 0, 0);
            const uint32_t qa = smem_u32(q_smem), ra = smem_u32(ring);
            int stage = 0;
            uint32_t phase = 0, it = 0, tc = 0;
            bool ok = true;
            const long long items = item_total(P);
            for (long long w = blockIdx.x; w < items && ok; w += gridDim.x) {
                int chunk, mb;
                item_at(P, w, chunk, mb);
                (void)mb;
                const uint32_t d0 = P.chunk_doc[chunk], d1 = P.chunk_doc[chunk + 1];
                if (d0 == d1) continue;
                const long long r_lo = static_cast<long long>(P.d_off[d0]), r_hi = static_cast<long long>(P.d_off[d1]);
                if (!mbar_wait(&bar.q_full, it & 1, abort_flag, P.status, kSleepIssuer)) break;
                ++it;
                for (long long r0 = r_lo; r0 < r_hi; r0 += BN, ++tc) {
                    const uint32_t buf = tc & 1;
                    if (!mbar_wait(&bar.full[stage], phase, abort_flag, P.status, kSleepIssuer)) { ok = false; break; }
                    if (!mbar_wait(&bar.s_free[buf], ((tc >> 1) & 1) ^ 1, abort_flag, P.status, kSleepIssuer)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t da = ra + stage * stage_bytes;
                    for (int kc = 0; kc < P.nk; ++kc) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t a = sdesc_sw128(qa + kc * BOX_BYTES + kk * 32, 16, 1024);
                            const uint64_t b = sdesc_sw128(da + kc * BOX_BYTES + kk * 32, 16, 1024);
                            mma_bf16(tmem + buf * BN, a, b, idesc, (kc | kk) != 0);
                        }
                    }
                    mma_commit(&bar.empty[stage]);
                    mma_commit(&bar.s_full[buf]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                mma_commit(&bar.q_free);
            }
            mma_commit(&bar.mma_done);
            mbar_wait(&bar.mma_done, 0, abort_flag, P.status);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t hi_mask;
        asm volatile("mov.b32 %0, 0xFFFFFFE0;" : "=r"(hi_mask));   // opaque to constant folding
        uint32_t tc = 0;
        bool ok = true;
        const long long items = item_total(P);
        for (long long w = blockIdx.x; w < items && ok; w += gridDim.x) {
            int chunk, mb;
            item_at(P, w, chunk, mb);
            const uint32_t d0 = P.chunk_doc[chunk], d1 = P.chunk_doc[chunk + 1];
            if (d0 == d1) continue;
            // Positions below are 32-bit offsets from the item's first row.
            const long long r_lo = static_cast<long long>(P.d_off[d0]);
            const int span = static_cast<int>(static_cast<long long>(P.d_off[d1]) - r_lo);
            const int t = mb * BM + row;
            const bool t_ok = t < P.rows_q;
            uint32_t cur = d0;
            int cur_beg = 0, cur_end = static_cast<int>(static_cast<long long>(P.d_off[d0 + 1]) - r_lo);
            float best = -INFINITY;
            int best_col = 0;
            // The current document is complete: its row maximum and argmax out, the next one begins.
            auto close_doc = [&]() {
                if (t_ok) {
                    P.argmax[static_cast<long long>(cur) * P.ld_argmax + t] = best_col;
                    P.mval[static_cast<long long>(cur) * P.rows_q + t] = best;
                }
                ++cur;
                best = -INFINITY;
                best_col = 0;
                if (cur < d1) {
                    cur_beg = cur_end;
                    cur_end = static_cast<int>(static_cast<long long>(P.d_off[cur + 1]) - r_lo);
                }
            };
            for (int r0 = 0; r0 < span; r0 += BN, ++tc) {
                const uint32_t buf = tc & 1;
                if (!mbar_wait(&bar.s_full[buf], (tc >> 1) & 1, abort_flag, P.status, kSleepEpilogue)) { ok = false; break; }
                tc_fence_after();
                if (r0 + BN <= span && cur_end >= r0 + BN) {
                    // the whole tile lies inside the current document
#pragma unroll 1
                    for (int ch = 0; ch < BN / 32; ++ch)
                        chunk_max_tmem(tmem + lane_base + buf * BN + ch * 32, r0 + ch * 32 - cur_beg, best, best_col,
                                       hi_mask);
                    if (cur_end == r0 + BN) close_doc();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.s_free[buf]);
                    continue;
                }
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) {
                    const int c0 = r0 + ch * 32;
                    if (c0 >= span) break;
                    const uint32_t ta = tmem + lane_base + buf * BN + ch * 32;
                    const int hi_chunk = min(c0 + 32, span);
                    if (hi_chunk == c0 + 32 && cur_end >= c0 + 32) {
                        // the whole chunk lies inside the current document
                        chunk_max_tmem(ta, c0 - cur_beg, best, best_col, hi_mask);
                        if (cur_end == c0 + 32) close_doc();
                        continue;
                    }
                    // The current document ends inside the chunk (warp-uniform: document boundaries are
                    // shared by all rows).  With one boundary whose next document covers the rest of the
                    // chunk, or at the end of the work item, the prefix and suffix maxima come from TMEM;
                    // chunks holding more boundaries take the masked register tree per segment.
                    const bool tail = hi_chunk < c0 + 32 && cur_end == hi_chunk;
                    const bool split = hi_chunk == c0 + 32 && cur + 1 < d1 &&
                                       static_cast<long long>(P.d_off[cur + 2]) - r_lo >= c0 + 32;
                    if (tail || split) {
                        chunk_keys_to_tmem(ta, hi_mask);
                        float ma, mb;
                        split_max(ta, cur_end - c0, split, ma, mb);
                        update_best(ma, c0 - cur_beg, best, best_col);
                        close_doc();
                        if (split) update_best(mb, c0 - cur_beg, best, best_col);
                        continue;
                    }
                    float v[32];
                    tmem_ld32(ta, v);
                    int lo = c0;
                    while (lo < hi_chunk) {
                        const int seg_hi = min(hi_chunk, cur_end);
                        chunk_max(v, lo - c0, seg_hi - c0, c0 - cur_beg, best, best_col, hi_mask);
                        if (seg_hi == cur_end) close_doc();
                        lo = seg_hi;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.s_free[buf]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Named pairs: flags[chunk * n_mblocks + mb] = 1 for every work item holding a
// (query, document) pair that some query names (one thread per query).
__global__ void mark_items_kernel(const uint64_t *q_off, const uint64_t *pair_off, const uint32_t *pair_ids, int nq,
                                  const uint32_t *chunk_doc, int n_chunks, int n_mblocks, uint32_t *flags,
                                  const int32_t *status) {
    if (read_status(status) != 0) return;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= nq) return;
    const int mb0 = static_cast<int>(q_off[q] / 128), mb1 = static_cast<int>((q_off[q + 1] - 1) / 128);
    for (uint64_t k = pair_off[q]; k < pair_off[q + 1]; ++k) {
        const uint32_t d = pair_ids[k];
        int lo = 0, hi = n_chunks;   // the chunk c with chunk_doc[c] <= d < chunk_doc[c + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (chunk_doc[mid] <= d) lo = mid; else hi = mid;
        }
        for (int mb = mb0; mb <= mb1; ++mb) flags[static_cast<long long>(lo) * n_mblocks + mb] = 1u;
    }
}

// The flagged items in index order (chunk-major) and their count: one block,
// each thread compacting a contiguous segment after a scan of the counts.
constexpr int kCompactThreads = 1024;
template <typename F>
__global__ void __launch_bounds__(kCompactThreads) compact_items_kernel(const F *flags, long long n, uint32_t *list,
                                                                        uint32_t *count, const int32_t *status) {
    __shared__ uint32_t part[kCompactThreads];
    if (read_status(status) != 0) return;
    const long long per = (n + kCompactThreads - 1) / kCompactThreads;
    const long long lo = threadIdx.x * per, hi = lo + per < n ? lo + per : n;
    uint32_t c = 0;
    for (long long i = lo; i < hi; ++i) c += flags[i] ? 1u : 0u;
    part[threadIdx.x] = c;
    __syncthreads();
    for (int o = 1; o < kCompactThreads; o <<= 1) {   // inclusive scan (Hillis-Steele)
        const uint32_t v = threadIdx.x >= o ? part[threadIdx.x - o] : 0u;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    uint32_t at = part[threadIdx.x] - c;
    for (long long i = lo; i < hi; ++i)
        if (flags[i]) list[at++] = static_cast<uint32_t>(i);
    if (threadIdx.x == kCompactThreads - 1) *count = part[threadIdx.x];
}

// chunk_doc[k] = first document starting at or after row k * chunk_rows;
// chunk_doc[n_chunks] = nd.
__global__ void schedule_kernel(const uint64_t *d_off, int nd, int n_chunks, long long chunk_rows,
                                uint32_t *chunk_doc, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k > n_chunks) return;
    if (k == n_chunks) {
        chunk_doc[k] = static_cast<uint32_t>(nd);
        return;
    }
    const uint64_t target = static_cast<uint64_t>(k) * static_cast<uint64_t>(chunk_rows);
    int lo = 0, hi = nd;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (d_off[mid] < target) lo = mid + 1; else hi = mid;
    }
    chunk_doc[k] = static_cast<uint32_t>(lo);
}

// S[q][d] = sum over the query's rows of m[d][t], in row order (/ |q| if mean).
// A maximum that is not a positive normal number (its argmax came from a key
// that need not name the lowest row) is listed for `argmax_fixup_kernel`:
// (document << 32 | row) in list[0 .. cap), count[0] the number found, count[1]
// set when they do not fit.  With named pairs (pair_off not null) a pair no
// query names scores 0 and lists nothing (its items may not have run).
__global__ void query_sum_kernel(const float *mval, const uint64_t *q_off, int nq, int nd, int rows_q, int mean,
                                 float *scores, long long ld, unsigned long long *list, uint32_t *count, uint32_t cap,
                                 const uint64_t *pair_off, const uint32_t *pair_ids, const int32_t *status) {
    if (read_status(status) != 0) return;
    const long long total = static_cast<long long>(nq) * nd;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int d = static_cast<int>(idx / nq), q = static_cast<int>(idx % nq);
        if (pair_off) {
            uint64_t lo = pair_off[q], hi = pair_off[q + 1];
            while (lo < hi) {
                const uint64_t mid = (lo + hi) >> 1;
                if (pair_ids[mid] < static_cast<uint32_t>(d)) lo = mid + 1; else hi = mid;
            }
            if (!(lo < pair_off[q + 1] && pair_ids[lo] == static_cast<uint32_t>(d))) {
                scores[static_cast<long long>(q) * ld + d] = 0.0f;
                continue;
            }
        }
        const uint64_t a = q_off[q], b = q_off[q + 1];
        const float *m = mval + static_cast<long long>(d) * rows_q;
        float s = 0.f, lowest = INFINITY;
        for (uint64_t t = a; t < b; ++t) {
            const float v = m[t];
            s += v;
            lowest = fminf(lowest, v);
        }
        if (!(lowest >= 1.17549435e-38f)) {   // rare: some row's scores all <= 0 over the document, or subnormal
            for (uint64_t t = a; t < b; ++t) {
                if (m[t] >= 1.17549435e-38f) continue;
                const uint32_t k = atomicAdd(count, 1u);
                if (k < cap)
                    list[k] = (static_cast<unsigned long long>(d) << 32) | static_cast<uint32_t>(t);
                else
                    atomicOr(count + 1, 1u);
            }
        }
        if (mean) s /= static_cast<float>(b - a);
        scores[static_cast<long long>(q) * ld + d] = s;
    }
}

// The argmax entries whose row maximum over the document is not a positive
// normal number (every score of the document <= 0 for that row, or a subnormal
// maximum): their key's column need not be the lowest among equal scores.  One
// warp per entry finds the argmax again from the tapes: every document row's
// score in float64 (each bf16 product is exact in float64, and so, far below any
// difference a float32 score could show, is their sum), keeping the lowest row
// among equal scores, and writes it.  The warps take the entries the per-query
// sums listed; after an overflow of the list they scan the maxima for such
// entries instead.
struct FixupArgs {
    const uint16_t *q, *d;
    const uint64_t *d_off;
    int width, nd, rows_q;
    int32_t *argmax;
    long long ld_argmax;
    const float *mval;
    const unsigned long long *list;
    const uint32_t *count;   // [0] entries found, [1] overflow flag
    uint32_t cap;
    const int32_t *status;
};

__device__ __forceinline__ double bf16_to_f64(uint16_t b) {
    return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

__device__ void fix_entry(const FixupArgs &A, int d, int t, int lane) {
    const long long r0 = static_cast<long long>(A.d_off[d]);
    const long long len = static_cast<long long>(A.d_off[d + 1]) - r0;
    const uint16_t *qr = A.q + static_cast<long long>(t) * A.width;
    double bv = -INFINITY;
    long long bi = 0;
    for (long long s = lane; s < len; s += 32) {   // ascending: a strict comparison keeps the lowest row
        const uint16_t *dr = A.d + (r0 + s) * A.width;
        double acc = 0.0;
        for (int k = 0; k < A.width; ++k) acc += bf16_to_f64(qr[k]) * bf16_to_f64(dr[k]);
        if (acc > bv) {
            bv = acc;
            bi = s;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const long long oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if (lane == 0) A.argmax[static_cast<long long>(d) * A.ld_argmax + t] = static_cast<int32_t>(bi);
}

__global__ void __launch_bounds__(256) argmax_fixup_kernel(FixupArgs A) {
    if (read_status(A.status) != 0) return;
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    if (A.count[1] == 0) {
        const long long n = min(static_cast<long long>(A.count[0]), static_cast<long long>(A.cap));
        for (long long e = warp; e < n; e += warps) {
            const unsigned long long v = A.list[e];
            fix_entry(A, static_cast<int>(v >> 32), static_cast<int>(v & 0xFFFFFFFFu), lane);
        }
        return;
    }
    const long long total = static_cast<long long>(A.nd) * A.rows_q;
    for (long long b = warp * 32; b < total; b += warps * 32) {   // warp-uniform trip count
        const long long i = b + lane;
        const int d = static_cast<int>(i / A.rows_q), t = static_cast<int>(i % A.rows_q);
        const bool marked = i < total && !(A.mval[i] >= 1.17549435e-38f);
        unsigned m = __ballot_sync(0xffffffffu, marked);
        while (m) {
            const int l = __ffs(m) - 1;
            m &= m - 1;
            fix_entry(A, __shfl_sync(0xffffffffu, d, l), __shfl_sync(0xffffffffu, t, l), lane);
        }
    }
}

// ----------------------------------------------------------------------------
// backward
// ----------------------------------------------------------------------------

// q_active[q] = 1 when some c(q, d) is nonzero, d_active[d] = 1 when some
// c(q, d) is (one block per query; both zeroed beforehand, every writer
// writes 1).
__global__ void active_kernel(const float *d_scores, long long ld_ds, int nd, uint8_t *q_active, uint8_t *d_active,
                              const int32_t *status) {
    if (read_status(status) != 0) return;
    const int q = blockIdx.x;
    const float *row = d_scores + static_cast<long long>(q) * ld_ds;
    int any = 0;
    for (int d = threadIdx.x; d < nd; d += blockDim.x)
        if (row[d] != 0.0f) {
            any = 1;
            d_active[d] = 1;
        }
    if (__syncthreads_or(any) && threadIdx.x == 0) q_active[q] = 1;
}

// The dD rows of a document no query scores are zero (its argmax entries are
// not read).
__global__ void dd_zero_kernel(MaxSimBwdLaunch L) {
    if (read_status(L.status) != 0) return;
    const int d = blockIdx.x;
    if (L.d_active[d]) return;
    const uint64_t o0 = L.d_off[d];
    const int dl = static_cast<int>(L.d_off[d + 1] - o0);
    float4 *dst = reinterpret_cast<float4 *>(L.dd + static_cast<long long>(o0) * L.width);
    const long long n4 = static_cast<long long>(dl) * L.width / 4;
    for (long long i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

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
    // The loads that resolve the i-th document (its id, argmax entry and c) ...
    int a_n = 0, d_n = 0;
    float c_n = 0.f;
    auto fetch = [&](int i) {
        if (i < n_docs) {
            d_n = use_list ? static_cast<int>(__ldg(L.d_list + i)) : i;
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
    fetch(sub);
    finish(sub, src, c);
    for (int d0 = 0; d0 < (warp_idle ? 0 : n_docs); d0 += kDqUnroll) {
        fetch(d0 + kDqUnroll + sub);   // the next step's resolution, in flight during this step
        step(src, c);
        finish(d0 + kDqUnroll + sub, src, c);
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
constexpr int kDsThreads = 512;
constexpr int kDsMaxRows = 4096;
constexpr int kDsChunk = 16384;
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
__global__ void __launch_bounds__(kDsThreads, 2) dd_sort_kernel(MaxSimBwdLaunch L) {
    extern __shared__ uint8_t ds_raw[];
    uint32_t *cnt = reinterpret_cast<uint32_t *>(ds_raw);            // [kDsMaxRows] counts, then cursors
    uint32_t *off = cnt + kDsMaxRows;                                  // [kDsMaxRows + 1] bucket starts
    uint32_t *list = off + kDsMaxRows + 1;                             // [kDsChunk] (q << 16) | row offset
    float *ctab = reinterpret_cast<float *>(list + kDsChunk);          // [kDsMaxTable]
    __shared__ uint32_t warp_sums[kDsThreads / 32];
    if (read_status(L.status) != 0) return;
    const int d = blockIdx.x;
    if (L.d_active && !L.d_active[d]) return;   // dd_zero_kernel writes its rows
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
                constexpr int kPer = kDsMaxRows / kDsThreads;   // 8 entries per thread
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

size_t maxsim_forward_smem_bytes(int width) { return ms::smem_bytes_for((width + ms::BK - 1) / ms::BK); }

cudaError_t launch_maxsim_forward(const CUtensorMap &tmap_q, const CUtensorMap &tmap_d, const MaxSimLaunch &L,
                                  cudaStream_t stream) {
    using namespace ms;
    cudaError_t err;
    schedule_kernel<<<(L.n_chunks + 1 + 255) / 256, 256, 0, stream>>>(L.d_off, L.nd, L.n_chunks, L.chunk_rows,
                                                                     L.chunk_doc, L.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    Params P;
    P.nq = L.nq;
    P.nd = L.nd;
    P.rows_q = L.rows_q;
    P.rows_d = L.rows_d;
    P.width = L.width;
    P.nk = (L.width + BK - 1) / BK;
    P.mean = L.mean;
    P.n_mblocks = (L.rows_q + BM - 1) / BM;
    P.n_chunks = L.n_chunks;
    P.items = static_cast<long long>(P.n_mblocks) * L.n_chunks;
    P.q_off = L.q_off;
    P.d_off = L.d_off;
    P.chunk_doc = L.chunk_doc;
    P.argmax = L.argmax;
    P.ld_argmax = L.ld_argmax;
    P.mval = L.mval;
    P.status = L.status;
    P.item_list = nullptr;
    P.item_count = nullptr;
    if ((err = cudaMemsetAsync(L.fix_count, 0, 2 * sizeof(uint32_t), stream)) != cudaSuccess) return err;
    if (L.pair_off) {   // named pairs: run only the items that hold one
        const long long n_items = P.items;
        if ((err = cudaMemsetAsync(L.item_flags, 0, static_cast<size_t>(n_items) * 4, stream)) != cudaSuccess) return err;
        mark_items_kernel<<<(L.nq + 255) / 256, 256, 0, stream>>>(L.q_off, L.pair_off, L.pair_ids, L.nq, L.chunk_doc,
                                                                 L.n_chunks, P.n_mblocks, L.item_flags, L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        compact_items_kernel<<<1, kCompactThreads, 0, stream>>>(L.item_flags, n_items, L.item_list, L.item_count,
                                                                L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        P.item_list = L.item_list;
        P.item_count = L.item_count;
    }
    // At least 80 KB so that no more than two CTAs (2 x 256 TMEM columns) share an SM.
    size_t smem = smem_bytes_for(P.nk);
    if (smem < 80 * 1024) smem = 80 * 1024;
    static size_t configured = 0;
    if (configured < smem) {
        if ((err = cudaFuncSetAttribute(forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem))) != cudaSuccess)
            return err;
        configured = smem;
    }
    const int per_sm = smem * 2 + 2048 <= 233472 ? 2 : 1;
    long long grid = static_cast<long long>(L.sm_count) * per_sm;
    if (grid > P.items) grid = P.items;
    forward_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tmap_q, tmap_d, P);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    query_sum_kernel<<<L.sm_count * 8, 256, 0, stream>>>(L.mval, L.q_off, L.nq, L.nd, L.rows_q, L.mean, L.scores,
                                                          L.ld_scores, L.fix_list, L.fix_count, L.fix_cap, L.pair_off,
                                                          L.pair_ids, L.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    FixupArgs F;
    F.q = L.q;
    F.d = L.d;
    F.d_off = L.d_off;
    F.width = L.width;
    F.nd = L.nd;
    F.rows_q = L.rows_q;
    F.argmax = L.argmax;
    F.ld_argmax = L.ld_argmax;
    F.mval = L.mval;
    F.list = L.fix_list;
    F.count = L.fix_count;
    F.cap = L.fix_cap;
    F.status = L.status;
    argmax_fixup_kernel<<<L.sm_count * 2, 256, 0, stream>>>(F);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    return cudaSuccess;
}

cudaError_t launch_maxsim_backward(const MaxSimBwdLaunch &L, cudaStream_t stream) {
    using namespace ms;
    cudaError_t err;
    qmap_kernel<<<(L.nq + 255) / 256, 256, 0, stream>>>(L.q_off, L.nq, L.qmap, L.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (L.q_active) {
        if ((err = cudaMemsetAsync(L.q_active, 0, L.nq, stream)) != cudaSuccess ||
            (err = cudaMemsetAsync(L.d_active, 0, L.nd, stream)) != cudaSuccess)
            return err;
        active_kernel<<<L.nq, 256, 0, stream>>>(L.d_scores, L.ld_ds, L.nd, L.q_active, L.d_active, L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        compact_items_kernel<uint8_t><<<1, kCompactThreads, 0, stream>>>(L.d_active, L.nd, L.d_list, L.d_count,
                                                                         L.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        dd_zero_kernel<<<L.nd, 512, 0, stream>>>(L);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    const unsigned dq_grid = (L.rows_q + kDqRows - 1) / kDqRows;
    switch ((L.width + 63) / 64) {
        case 1: dq_kernel<1><<<dq_grid, 256, 0, stream>>>(L); break;
        case 2: dq_kernel<2><<<dq_grid, 256, 0, stream>>>(L); break;
        case 3: dq_kernel<3><<<dq_grid, 256, 0, stream>>>(L); break;
        default: dq_kernel<4><<<dq_grid, 256, 0, stream>>>(L); break;
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
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
    return cudaGetLastError();
}

}  // namespace cli

namespace cli {

cudaError_t launch_maxsim_backward_named(const MaxSimBwdLaunch &L, const uint64_t *pair_off, const uint32_t *pair_ids,
                                         long long pairs, cudaStream_t stream) {
    if (pairs == 0) return cudaSuccess;
    ms::named_backward_kernel<<<static_cast<unsigned>((pairs + 7) / 8), 256, 0, stream>>>(L, pair_off, pair_ids,
                                                                                        pairs);
    return cudaGetLastError();
}

}  // namespace cli
