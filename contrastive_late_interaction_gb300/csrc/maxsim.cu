// Hard MaxSim late interaction over ragged token tapes ("UForm", section
// "ColBERT-Style Late-Interaction Rerankers"; tapes as in "Arenas", "Rows and
// Tapes"):
//     S(q, d) = sum_{t in q} max_{s in d} <q_t, d_s>   (optionally / |q|)
// with the argmax; the backward routed through it is in maxsim_backward.cu.
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
#include "compact.cuh"

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
        auto add = [&](float v) {
            s += v;
            lowest = fminf(lowest, v);
        };
        // In row order: single maxima up to a 16-byte boundary of the workspace, then 16-byte loads (two
        // in flight), then the rest.
        uint64_t t = a;
        const uint64_t at = static_cast<uint64_t>(d) * static_cast<uint64_t>(rows_q);   // m[t] is mval[at + t]
        for (; t < b && ((at + t) & 3u) != 0; ++t) add(m[t]);
        for (; t + 8 <= b; t += 8) {
            const float4 u = *reinterpret_cast<const float4 *>(m + t), w = *reinterpret_cast<const float4 *>(m + t + 4);
            add(u.x); add(u.y); add(u.z); add(u.w);
            add(w.x); add(w.y); add(w.z); add(w.w);
        }
        for (; t + 4 <= b; t += 4) {
            const float4 u = *reinterpret_cast<const float4 *>(m + t);
            add(u.x); add(u.y); add(u.z); add(u.w);
        }
        for (; t < b; ++t) add(m[t]);
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

}  // namespace cli
