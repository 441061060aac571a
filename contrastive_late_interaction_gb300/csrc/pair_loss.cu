// Pooled sigmoid pair loss, forward and backward, fused over 128 x 128 tiles.
//
// What is computed ("UForm", section "Matryoshka-Like Multi-Scale Embedders",
// the SigLIP loss; "Training", `uform_pair_loss_form_t` = sigmoid,
// `uform_relations_view_t`, `uform_negatives_t`):
//     z_ij = t <e_i, e_j> + b,   l_ij = w_ij * softplus(-y_ij z_ij),
//     L = (1/N) sum_{i != j} l_ij,  dE, dt, db.
//
// GB300 design.  The score matrix is symmetric (s_ij = s_ji) and, with one
// temperature group, so is z.  The kernel therefore visits only tile pairs
// (I, J) with I <= J.  For each one:
//   1. tcgen05 computes S_IJ = E_I E_J^T into TMEM (bf16 operands staged by TMA
//      in 128-byte-swizzled 128 x 64 boxes, fp32 accumulation);
//   2. four epilogue warps read S_IJ from TMEM, one row per thread, and for
//      every cell evaluate one sigmoid and one softplus that serve both ordered
//      pairs (i, j) and (j, i): p = sigma(z), sp = softplus(z).  With each
//      direction's resolved (attract?, weight) the gradient of the two pairs
//      is G_ij = sum_dir w (p - [attract]) and the loss w (sp - [attract] z).
//      H_IJ = (t/N) G_IJ is written as bf16 into shared memory; partial sums
//      of the loss, G*s (for dt) and G (for db) go to a fixed slot per warp;
//   3. tcgen05 computes the two gradient contractions from shared memory,
//      dE_I += H_IJ E_J and (I != J) dE_J += H_IJ^T E_I, in 64-column chunks,
//      reading H and the E tiles in both K-major and MN-major form from the
//      same bytes; the epilogue warps add each chunk into dE (fp32) with
//      vector reductions.
// Neither S nor H ever reaches device memory.  Relations are resolved once
// per call into a per-row sorted list of "special" columns (both directions
// of every pair some edge set names, plus the diagonal); every other cell
// takes the run's default.
//
// Two CTAs share an SM (about 97 KB of shared memory and 256 TMEM columns
// each), so one CTA's epilogue overlaps the other's tensor-core work.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace pooled {

constexpr int BM = 128;                 // tile rows and columns
constexpr int BK = 64;                  // K extent of one TMA box (128 bytes of bf16)
constexpr int STAGES = 2;
constexpr uint32_t BOX_BYTES = BM * BK * 2;   // 16 KB
constexpr int kThreads = 192;           // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t TM_S = 0, TM_DEI = 128, TM_DEJ = 192;

struct SharedStorage {
    alignas(1024) uint8_t ring[STAGES][2][BOX_BYTES];
    alignas(1024) uint8_t h[2][BOX_BYTES];     // H tile, two 64-column K blocks
    alignas(16) float stage_t[4][32 * 16];     // per epilogue warp: 32 rows x 16 fp32, transposed drain
    uint64_t full[STAGES], empty[STAGES];
    uint64_t s_full, s_free, h_ready, h_free, de_full, de_free, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = sizeof(SharedStorage) + 1024;  // + alignment slack

struct Params {
    int n, width, nk, nb;
    long long tile_pairs;
    const float *t_ptr, *b_ptr;
    float ambient;
    int named;
    const uint32_t *rel_off;
    const RelEntry *rel;
    float *d_e;
    long long ld_de;
    float *partials;   // [tile_pairs][4 warps][4]
    int32_t *status;
};

// Tile pair p -> (I, J), I <= J.  The upper triangle of tile pairs is walked in
// super-blocks of kSuper x kSuper tiles (row-major over super-blocks I' <= J',
// then row-major inside a super-block, keeping I <= J on the diagonal ones),
// so the CTAs running at the same time read and reduce into the rows of a few
// super-blocks only: their E rows and dE rows stay resident in L2.
constexpr int kSuper = 8;

// Row-major enumeration of the upper triangle of an n x n grid: index -> (i, j).
__device__ __forceinline__ void tri_decode(long long p, int n, int &i, int &j) {
    // start(i) = i*n - i*(i-1)/2; invert approximately, then correct.
    const double fn = static_cast<double>(n) + 0.5;
    int r = static_cast<int>(fn - sqrt(fn * fn - 2.0 * static_cast<double>(p)));
    if (r < 0) r = 0;
    if (r > n - 1) r = n - 1;
    auto start = [n](long long x) { return x * n - x * (x - 1) / 2; };
    while (r > 0 && start(r) > p) --r;
    while (r < n - 1 && start(r + 1) <= p) ++r;
    i = r;
    j = r + static_cast<int>(p - start(r));
}

__device__ __forceinline__ void decode_pair(long long p, int nb, int &I, int &J) {
    const int ns = (nb + kSuper - 1) / kSuper;          // super-blocks per side
    const int last = nb - (ns - 1) * kSuper;            // tiles in the last super-block row/column
    // walk super-blocks (si, sj), si <= sj, counting the tile pairs each holds
    long long before = 0;
    for (int si = 0; si < ns; ++si) {
        const int hi = si == ns - 1 ? last : kSuper;
        // off-diagonal super-blocks of this row: (ns - 1 - si) of them, the last one narrower
        const long long diag = static_cast<long long>(hi) * (hi + 1) / 2;
        const long long full_off = si < ns - 1 ? static_cast<long long>(ns - 2 - si) * hi * kSuper + static_cast<long long>(hi) * last : 0;
        if (p < before + diag + full_off) {
            long long q = p - before;
            if (q < diag) {   // diagonal super-block: upper triangle of hi x hi
                int i, j;
                tri_decode(q, hi, i, j);
                I = si * kSuper + i;
                J = si * kSuper + j;
                return;
            }
            q -= diag;
            // off-diagonal super-blocks sj = si+1 .. ns-1, each hi x width(sj), row-major
            for (int sj = si + 1; sj < ns; ++sj) {
                const int w = sj == ns - 1 ? last : kSuper;
                const long long cnt = static_cast<long long>(hi) * w;
                if (q < cnt) {
                    I = si * kSuper + static_cast<int>(q / w);
                    J = sj * kSuper + static_cast<int>(q % w);
                    return;
                }
                q -= cnt;
            }
        }
        before += diag + full_off;
    }
    I = J = nb - 1;   // not reached for p < tile_pairs
}

__device__ __forceinline__ float fast_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigma(z), sigma(-z) and softplus(z) from one exp(-|z|):
//   e = exp(-|z|), sigma(z) = 1/(1+e) for z >= 0 and e/(1+e) otherwise,
//   softplus(z) = max(z, 0) + log1p(e); log1p(e) uses e(1 - e/2) for e < 2^-7
//   (relative error below e^2/3) and ln2 * log2(1 + e) otherwise.
struct CellFn {
    float p, pc, sp;
};
__device__ __forceinline__ CellFn cell_fn(float z) {
    const float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
    float e = fast_ex2(-fabsf(z) * kLog2e);
    float q = 1.0f + e;
    float r = fast_rcp(q);
    float er = e * r;
    bool pos = z >= 0.0f;
    CellFn c;
    c.p = pos ? r : er;
    c.pc = pos ? er : r;
    float l1p = (e < 0.0078125f) ? e * (1.0f - 0.5f * e) : kLn2 * fast_lg2(q);
    c.sp = fmaxf(z, 0.0f) + l1p;
    return c;
}

__device__ __forceinline__ void red_add_v4(float *gptr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gptr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 2)
    fused_tiles_kernel(const __grid_constant__ CUtensorMap tmap_e, Params P) {
    extern __shared__ uint8_t smem_raw[];
    SharedStorage &sm = *reinterpret_cast<SharedStorage *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (read_status(P.status) != 0) return;  // an earlier stage of the call failed

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, 4);
        mbar_init(&sm.h_ready, 4);
        mbar_init(&sm.h_free, 1);
        mbar_init(&sm.de_full, 1);
        mbar_init(&sm.de_free, 4);
        mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_e);
    }
    if (warp == 1) tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (long long p = blockIdx.x; p < P.tile_pairs && ok; p += gridDim.x) {
                int I, J;
                decode_pair(p, P.nb, I, J);
                const bool diag = I == J;
                for (int pass = 0; pass < 2 && ok; ++pass) {   // S pass, then the dE pass
                    for (int kc = 0; kc < P.nk; ++kc) {
                        if (!mbar_wait(&sm.empty[stage], phase ^ 1, abort_flag, P.status, kSleepProducer)) { ok = false; break; }
                        mbar_arrive_expect_tx(&sm.full[stage], diag ? BOX_BYTES : 2 * BOX_BYTES);
                        tma_load_2d(sm.ring[stage][0], &tmap_e, &sm.full[stage], kc * BK, I * BM);
                        if (!diag) tma_load_2d(sm.ring[stage][1], &tmap_e, &sm.full[stage], kc * BK, J * BM);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // Let in-flight loads land before the CTA can exit.
            for (int s = 0; s < STAGES; ++s) mbar_wait(&sm.empty[stage], phase ^ 1, abort_flag, P.status),
                                              (++stage == STAGES ? (stage = 0, phase ^= 1) : 0);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            const uint32_t idesc_di = idesc_bf16(128, 64, 0, 1);   // A = H (K-major), B = E_J (MN-major)
            const uint32_t idesc_dj = idesc_bf16(128, 64, 1, 1);   // A = H^T (MN-major), B = E_I (MN-major)
            const uint32_t h0 = smem_u32(sm.h[0]);
            int stage = 0;
            uint32_t phase = 0, k = 0, chunk = 0;
            bool ok = true;
            for (long long p = blockIdx.x; p < P.tile_pairs && ok; p += gridDim.x, ++k) {
                int I, J;
                decode_pair(p, P.nb, I, J);
                const bool diag = I == J;
                // S = E_I E_J^T
                if (!mbar_wait(&sm.s_free, (k & 1) ^ 1, abort_flag, P.status, kSleepIssuer)) break;
                tc_fence_after();
                for (int kc = 0; kc < P.nk; ++kc) {
                    if (!mbar_wait(&sm.full[stage], phase, abort_flag, P.status, kSleepIssuer)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a = smem_u32(sm.ring[stage][0]);
                    const uint32_t b = diag ? a : smem_u32(sm.ring[stage][1]);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16(tmem + TM_S, sdesc_sw128(a + kk * 32, 16, 1024), sdesc_sw128(b + kk * 32, 16, 1024),
                                 idesc_s, (kc | kk) != 0);
                    mma_commit(&sm.empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(&sm.s_full);
                // dE_I += H E_J, dE_J += H^T E_I, 64 columns of D at a time
                if (!mbar_wait(&sm.h_ready, k & 1, abort_flag, P.status, kSleepIssuer)) break;
                tc_fence_after();
                for (int dc = 0; dc < P.nk; ++dc, ++chunk) {
                    if (!mbar_wait(&sm.full[stage], phase, abort_flag, P.status, kSleepIssuer)) { ok = false; break; }
                    if (!mbar_wait(&sm.de_free, (chunk & 1) ^ 1, abort_flag, P.status, kSleepIssuer)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ei = smem_u32(sm.ring[stage][0]);
                    const uint32_t ej = diag ? ei : smem_u32(sm.ring[stage][1]);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk) {
                        // A: H rows i, K = j (16 per step) inside 64-wide K blocks.
                        const uint64_t a = sdesc_sw128(h0 + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024);
                        // B: E_J box viewed as [N = 64 features] x [K = j]; 16 rows of j = 2048 bytes.
                        const uint64_t b = sdesc_sw128(ej + kk * 2048, 1024, 1024);
                        mma_bf16(tmem + TM_DEI, a, b, idesc_di, kk != 0);
                    }
                    if (!diag) {
#pragma unroll
                        for (int kk = 0; kk < BM / 16; ++kk) {
                            // A: H viewed as [M = j] x [K = i]: j contiguous within a 64-wide block
                            // (blocks BOX_BYTES apart), 8 rows of i per 1024 bytes.
                            const uint64_t a = sdesc_sw128(h0 + kk * 2048, BOX_BYTES, 1024);
                            const uint64_t b = sdesc_sw128(ei + kk * 2048, 1024, 1024);
                            mma_bf16(tmem + TM_DEJ, a, b, idesc_dj, kk != 0);
                        }
                    }
                    mma_commit(&sm.empty[stage]);
                    mma_commit(&sm.de_full);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(&sm.h_free);
            }
            mma_commit(&sm.mma_done);
            mbar_wait(&sm.mma_done, 0, abort_flag, P.status);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;        // row of the tile this thread owns
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float t = *P.t_ptr, b = *P.b_ptr;
        const float inv_n = 1.0f / static_cast<float>(P.n);
        const float c_h = t * inv_n;             // H = (t/N) G
        const float w_d = P.named ? 0.0f : P.ambient;
        const uint32_t h0 = smem_u32(sm.h[0]);
        const uint32_t stage_s = smem_u32(sm.stage_t[quad]);
        uint32_t k = 0, chunk = 0;
        for (long long p = blockIdx.x; p < P.tile_pairs; p += gridDim.x, ++k) {
            int I, J;
            decode_pair(p, P.nb, I, J);
            const bool diag = I == J;
            const int gi = I * BM + row;          // this thread's item (anchor)
            const bool row_ok = gi < P.n;
            const int j0 = J * BM;
            // This row's special columns inside [j0, j0 + 128).
            uint32_t e_beg = 0, e_end = 0;
            if (row_ok) {
                uint32_t lo = P.rel_off[gi], hi = P.rel_off[gi + 1];
                e_end = hi;
                while (lo < hi) {
                    uint32_t mid = (lo + hi) >> 1;
                    if (P.rel[mid].col < static_cast<uint32_t>(j0)) lo = mid + 1; else hi = mid;
                }
                e_beg = lo;
            }
            if (!mbar_wait(&sm.s_full, k & 1, abort_flag, P.status, kSleepEpilogue)) break;
            if (!mbar_wait(&sm.h_free, (k & 1) ^ 1, abort_flag, P.status, kSleepEpilogue)) break;
            tc_fence_after();

            float acc_sp = 0.f, acc_p = 0.f, acc_ps = 0.f;     // default cells (times 2 w_d later)
            float fix_l = 0.f, fix_g = 0.f, fix_gs = 0.f;     // corrections for special cells
            uint32_t e = e_beg;
#pragma unroll 1
            for (int ch = 0; ch < BM / 32; ++ch) {
                float v[32];
                tmem_ld32(tmem + lane_base + TM_S + ch * 32, v);
                const int c0 = j0 + ch * 32;
                const int valid = min(32, P.n - c0);     // columns of this chunk inside the batch
                float hv[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float s = v[r];
                    const float z = fmaf(t, s, b);
                    const CellFn f = cell_fn(z);
                    const bool ok_col = row_ok && r < valid;
                    acc_sp += ok_col ? f.sp : 0.f;
                    acc_p += ok_col ? f.p : 0.f;
                    acc_ps += ok_col ? f.p * s : 0.f;
                    hv[r] = ok_col ? c_h * 2.0f * w_d * f.p : 0.f;
                }
                // Special cells: replace the default by the resolved pair of directions.
                while (e < e_end) {
                    const RelEntry en = P.rel[e];
                    if (en.col >= static_cast<uint32_t>(c0 + 32)) break;
                    ++e;
                    const int r = static_cast<int>(en.col) - c0;
                    float s = 0.f;
#pragma unroll
                    for (int q = 0; q < 32; ++q) s = (q == r) ? v[q] : s;
                    const float z = fmaf(t, s, b);
                    const CellFn f = cell_fn(z);
                    const bool ao = en.flags & 1u, ai = en.flags & 2u;
                    const float g = en.w_out * (ao ? -f.pc : f.p) + en.w_in * (ai ? -f.pc : f.p);
                    const float l = en.w_out * (ao ? f.sp - z : f.sp) + en.w_in * (ai ? f.sp - z : f.sp);
                    const float g_def = 2.0f * w_d * f.p;
                    fix_l += l - 2.0f * w_d * f.sp;
                    fix_g += g - g_def;
                    fix_gs += (g - g_def) * s;
                    const float hnew = c_h * g;
#pragma unroll
                    for (int q = 0; q < 32; ++q) hv[q] = (q == r) ? hnew : hv[q];
                }
                // bf16 H row segment into the swizzled K-major tile.
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t col = ch * 32 + q * 8;
                    st_shared_v4(h0 + sw128_bf16_offset(row, col, BM), pack_bf16x2(hv[q * 8 + 0], hv[q * 8 + 1]),
                                 pack_bf16x2(hv[q * 8 + 2], hv[q * 8 + 3]), pack_bf16x2(hv[q * 8 + 4], hv[q * 8 + 5]),
                                 pack_bf16x2(hv[q * 8 + 6], hv[q * 8 + 7]));
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.s_free);
                mbar_arrive(&sm.h_ready);
            }
            // Per-warp partial sums of this tile pair (diagonal tiles see every pair twice).
            float l_sum = 2.0f * w_d * acc_sp + fix_l;
            float g_sum = 2.0f * w_d * acc_p + fix_g;
            float gs_sum = 2.0f * w_d * acc_ps + fix_gs;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                l_sum += __shfl_xor_sync(0xffffffffu, l_sum, o);
                g_sum += __shfl_xor_sync(0xffffffffu, g_sum, o);
                gs_sum += __shfl_xor_sync(0xffffffffu, gs_sum, o);
            }
            if (lane == 0) {
                const float scale = diag ? 0.5f : 1.0f;
                float *slot = P.partials + (p * 4 + quad) * 4;
                slot[0] = l_sum * scale;
                slot[1] = gs_sum * scale;
                slot[2] = g_sum * scale;
                slot[3] = 0.f;
            }
            // Drain the gradient chunks into dE.
            bool ok = true;
            for (int dc = 0; dc < P.nk; ++dc, ++chunk) {
                if (!mbar_wait(&sm.de_full, chunk & 1, abort_flag, P.status, kSleepEpilogue)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int side = 0; side < (diag ? 1 : 2); ++side) {
                    const int row0 = (side == 0 ? I : J) * BM + quad * 32;   // first row of this warp's 32
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float v[32];
                        tmem_ld32(tmem + lane_base + (side == 0 ? TM_DEI : TM_DEJ) + half * 32, v);
                        const int col0 = dc * BK + half * 32;
#pragma unroll
                        for (int h16 = 0; h16 < 2; ++h16) {
                            // lane = row: write 16 values (4 x 16 B, chunk index swizzled by row)
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int kk = k ^ ((lane >> 1) & 3);
                                st_shared_v4(stage_s + (lane * 16 + kk * 4) * 4, __float_as_uint(v[h16 * 16 + k * 4]),
                                             __float_as_uint(v[h16 * 16 + k * 4 + 1]), __float_as_uint(v[h16 * 16 + k * 4 + 2]),
                                             __float_as_uint(v[h16 * 16 + k * 4 + 3]));
                            }
                            __syncwarp();
                            // read back: instruction m covers rows 8m .. 8m+7, 4 lanes x 16 B per row
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const int r = m * 8 + (lane >> 2), k = lane & 3;
                                const int kk = k ^ ((r >> 1) & 3);
                                const float4 x = *reinterpret_cast<const float4 *>(&sm.stage_t[quad][r * 16 + kk * 4]);
                                const int grow = row0 + r, gcol = col0 + h16 * 16 + k * 4;
                                if (grow < P.n && gcol < P.width)
                                    red_add_v4(P.d_e + static_cast<long long>(grow) * P.ld_de + gcol, x.x, x.y, x.z, x.w);
                            }
                            __syncwarp();
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.de_free);
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
// final scalar reduction: fixed order, float64
// ----------------------------------------------------------------------------

__global__ void finish_kernel(const float *partials, long long slots, int n, float *loss, float *dt, float *db,
                              int32_t *status) {
    if (read_status(status) != 0) return;
    __shared__ double red[3][256];
    double l = 0, gs = 0, g = 0;
    for (long long s = threadIdx.x; s < slots; s += blockDim.x) {
        l += partials[s * 4 + 0];
        gs += partials[s * 4 + 1];
        g += partials[s * 4 + 2];
    }
    red[0][threadIdx.x] = l;
    red[1][threadIdx.x] = gs;
    red[2][threadIdx.x] = g;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w)
            for (int c = 0; c < 3; ++c) red[c][threadIdx.x] += red[c][threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double inv_n = 1.0 / static_cast<double>(n);
        *loss = static_cast<float>(red[0][0] * inv_n);
        *dt = static_cast<float>(red[1][0] * inv_n);
        *db = static_cast<float>(red[2][0] * inv_n);
    }
}

}  // namespace pooled

size_t pooled_fused_smem_bytes() { return pooled::kSmemBytes; }

cudaError_t launch_pooled_fused(const CUtensorMap &tmap_e, const PooledLaunch &L, cudaStream_t stream) {
    using namespace pooled;
    static bool configured = false;
    if (!configured) {
        cudaError_t err = cudaFuncSetAttribute(fused_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kSmemBytes));
        if (err != cudaSuccess) return err;
        configured = true;
    }
    Params P;
    P.n = L.n;
    P.width = L.width;
    P.nk = (L.width + BK - 1) / BK;
    P.nb = (L.n + BM - 1) / BM;
    P.tile_pairs = static_cast<long long>(P.nb) * (P.nb + 1) / 2;
    P.t_ptr = L.t_ptr;
    P.b_ptr = L.b_ptr;
    P.ambient = L.ambient;
    P.named = L.named;
    P.rel_off = L.rel_off;
    P.rel = L.rel;
    P.d_e = L.d_e;
    P.ld_de = L.ld_de;
    P.partials = L.partials;
    P.status = L.status;
    long long grid = static_cast<long long>(L.sm_count) * 2;
    if (grid > P.tile_pairs) grid = P.tile_pairs;
    fused_tiles_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tmap_e, P);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    finish_kernel<<<1, 256, 0, stream>>>(L.partials, P.tile_pairs * 4, L.n, L.loss, L.dt, L.db, L.status);
    return cudaGetLastError();
}

long long pooled_tile_pairs(int n) {
    long long nb = (n + pooled::BM - 1) / pooled::BM;
    return nb * (nb + 1) / 2;
}

}  // namespace cli
