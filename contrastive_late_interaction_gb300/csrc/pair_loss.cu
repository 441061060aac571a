// Pooled sigmoid pair loss, forward and backward, fused over 256 x 256 blocks
// of the score matrix.
//
// What is computed ("UForm", section "Matryoshka-Like Multi-Scale Embedders",
// the SigLIP loss; "Training", `uform_pair_loss_form_t` = sigmoid,
// `uform_relations_view_t`, `uform_negatives_t`):
//     z_ij = t <e_i, e_j> + b,   l_ij = w_ij * softplus(-y_ij z_ij),
//     L = (1/N) sum_{i != j} l_ij,  dE, dt, db.
//
// GB300 design.  The score matrix is symmetric (s_ij = s_ji) and, with one
// temperature group, so is z.  The kernel visits the upper triangle of 2 x 2
// blocks of 128 x 128 tiles: rows I0, I1 = I0 + 1 against columns J0, J1 =
// J0 + 1 (on a diagonal block the columns are the rows, and the mirrored tile
// (I1, I0) is skipped).  One persistent CTA per SM; for each block:
//   1. S pass.  tcgen05 computes the four tiles S_xy = E_Ix E_Jy^T into the
//      512 TMEM columns, as one M = 128, N = 256 product per tile row (bf16
//      operands staged by TMA in 128-byte-swizzled 128 x 64 boxes, fp32
//      accumulation).  The four boxes of one K step fill
//      a stage; the shared memory that holds H later is lent to the pass as
//      two more stages.
//   2. Epilogue.  Eight warps read S from TMEM, one row per thread (two warps
//      per TMEM lane quarter, one per tile row), and for every cell evaluate
//      one sigmoid and one softplus that serve both ordered pairs (i, j) and
//      (j, i): with each direction's resolved (attract?, weight) the gradient
//      of the two pairs is G_ij = sum_dir w (p - [attract]) and the loss
//      w (sp - [attract] z).  H_xy = (t/N) G_xy goes to shared memory as bf16;
//      partial sums of the loss, G*s (for dt) and G (for db) go to a fixed
//      slot per warp.
//   3. Gradient passes.  Per 128 columns of D, tcgen05 accumulates
//          dE_Ix += sum_y H_xy E_Jy    (pass 0, the row side)
//          dE_Jy += sum_x H_xy^T E_Ix  (pass 1, the column side; none on a
//                                        diagonal block, where pass 0 takes
//                                        the one mirrored product)
//      in two TMEM accumulators of 128 columns, double-buffered, reading H
//      and the E boxes in both K-major and MN-major form from the same bytes
//      (N = 128 products: per product the H operand is read once for 128
//      features, not 64, which is what the shared-memory bandwidth of this
//      pass pays for); the epilogue warps add each chunk into dE (fp32) while
//      the next chunk's MMAs run, each vector reduction covering 128
//      contiguous bytes of four rows after a transpose through shared memory
//      (the L2 reductions cost per request, not per byte).
// Each accumulator sums the contributions of two tiles before it leaves the
// SM, so per FLOP half as many fp32 partials reach L2 as with single tile
// pairs: L2 reductions of dE are what bound this kernel.  Neither S nor H ever
// reaches device memory.  Relations are resolved once per call into a per-row
// sorted list of "special" columns (both directions of every pair some edge
// set names, plus the diagonal); every other cell takes the run's default.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace pooled {

constexpr int BM = 128;                 // tile rows and columns
constexpr int BK = 64;                  // K extent of one TMA box (128 bytes of bf16)
constexpr uint32_t BOX_BYTES = BM * BK * 2;   // 16 KB
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2..9 epilogue
constexpr uint32_t TMEM_COLS = 512;
constexpr int kStages = 3;              // stage 0: the box ring (two halves); stages 1, 2: the H region, lent to the S pass
constexpr int kPartialsPerBlock = kEpiWarps;
constexpr int kFinishBlocks = 256;

struct SharedStorage {
    alignas(1024) uint8_t ring[4][BOX_BYTES];   // stage 0: boxes of I0, I1, J0, J1
    alignas(1024) uint8_t hreg[8][BOX_BYTES];   // H tiles 0..3 (two boxes each); stages 1 and 2 of the S pass
    alignas(16) float stage_t[kEpiWarps][32 * 32];   // per epilogue warp: 32 rows x 32 fp32, transposed drain
    uint64_t full[kStages], empty[kStages];   // H-region stages 1 and 2 (index 0 unused)
    uint64_t ring_full[2], ring_empty[2];     // ring halves: 0 = boxes of I0, I1; 1 = of J0, J1
    uint64_t s_full, h_ready, h_free, de_full[2], de_free[2], mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = sizeof(SharedStorage) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

struct Params {
    int n, width, nk, nb, nbb;
    long long blocks;
    const float *t_ptr, *b_ptr;
    float ambient;
    int named;
    const uint32_t *rel_off;
    const RelEntry *rel;
    float *d_e;
    long long ld_de;
    float *partials;   // [blocks][kEpiWarps][4]
    int32_t *status;
    // Temperature groups (null when one pair serves every cell): item i's group,
    // the per-group gradients (accumulated), and the mode's full grid of blocks.
    const int32_t *group;
    float *dt_g, *db_g;
    // Ordered traversal (groups, or an anchor band): every block (I, J) of block
    // rows bi0 .. bi0 + blocks / nbb - 1, each cell scored for its row's anchor
    // only, and only anchors in rows row_lo .. row_hi - 1.
    int ordered, bi0, row_lo, row_hi;
};

// Pair p -> (I, J), I <= J, over an n x n grid.  The upper triangle is walked
// in super-blocks of kSuper x kSuper (row-major over super-blocks I' <= J',
// then row-major inside a super-block, keeping I <= J on the diagonal ones),
// so the CTAs running at the same time read and reduce into the rows of a few
// super-blocks only: their E rows and dE rows stay resident in L2.
constexpr int kSuper = 4;

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
    const int last = nb - (ns - 1) * kSuper;            // entries in the last super-block row/column
    long long before = 0;
    for (int si = 0; si < ns; ++si) {
        const int hi = si == ns - 1 ? last : kSuper;
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
    I = J = nb - 1;   // not reached for p < nb (nb + 1) / 2
}

// One 2 x 2 block of tiles.  Slot (x, y) is the tile pair (I0 + x, J0 + y);
// box position 0..3 holds the E rows of I0, I1, J0, J1; accumulator 0..3
// collects dE of the same four tile rows (on a diagonal block J = I, so the
// column side lands in accumulators 0 and 1 and positions 2, 3 are unused).
struct Block {
    int I0, J0;
    bool diag, i1, j1;
};

__device__ __forceinline__ Block decode_block(long long p, const Params &P) {
    int bi, bj;
    if (P.ordered) {   // every ordered block, each cell scored for its row's anchor only
        bi = P.bi0 + static_cast<int>(p / P.nbb);
        bj = static_cast<int>(p % P.nbb);
    } else {
        decode_pair(p, P.nbb, bi, bj);
    }
    Block b;
    b.I0 = 2 * bi;
    b.J0 = 2 * bj;
    b.diag = bi == bj && !P.ordered;
    b.i1 = b.I0 + 1 < P.nb;
    b.j1 = b.J0 + 1 < P.nb;
    return b;
}
__device__ __forceinline__ bool slot_on(const Block &b, int x, int y) {
    return (x == 0 || b.i1) && (y == 0 || b.j1) && !(b.diag && x == 1 && y == 0);
}
__device__ __forceinline__ bool box_on(const Block &b, int pos) {
    return pos == 0 || (pos == 1 ? b.i1 : (!b.diag && (pos == 2 || b.j1)));
}
__device__ __forceinline__ int col_pos(const Block &b, int y) { return b.diag ? y : 2 + y; }
__device__ __forceinline__ int box_tile(const Block &b, int pos) { return pos < 2 ? b.I0 + pos : b.J0 + pos - 2; }

// Gradient schedule of a block.  Pass 0 is the row side (dE of I0, I1) and,
// off the diagonal, pass 1 the column side (dE of J0, J1); each runs over
// chunks of 128 features (two 64-feature boxes per tile).  In pass 0 ring half
// h holds the two feature boxes of tile J_h (of I_h on a diagonal block, whose
// column tiles are its rows); in pass 1 those of I_h.
__device__ __forceinline__ int grad_passes(const Block &b) { return b.diag ? 1 : 2; }
__device__ __forceinline__ int grad_half_tile(const Block &b, int pass, int h) {   // -1: absent
    if (pass == 0 && !b.diag) return (h == 0 || b.j1) ? b.J0 + h : -1;
    return (h == 0 || b.i1) ? b.I0 + h : -1;
}
// The tile row whose dE accumulator a (0, 1) collects in pass `pass` (-1: none).
__device__ __forceinline__ int grad_acc_tile(const Block &b, int pass, int a) {
    if (pass == 0) return (a == 0 || b.i1) ? b.I0 + a : -1;
    return (a == 0 || b.j1) ? b.J0 + a : -1;
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
// Three-input minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// sigma(z), sigma(-z) and softplus(z) from one exp(-|z|):
//   e = exp(-|z|), sigma(z) = 1/(1+e) for z >= 0 and e/(1+e) otherwise,
//   softplus(z) = max(z, 0) + log1p(e); log1p(e) uses e(1 - e/2) for e < 2^-7
//   (relative error below e^2/3) and ln2 * log2(1 + e) otherwise.
struct CellFn {
    float p, pc, sp;
};
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
__device__ __forceinline__ CellFn cell_fn(float z) {
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
// The same where |z| >= kFarZ, so e < 2^-7: 1/(1+e) = 1 - e + e^2 with
// relative error below e^3 < 2^-21, and log1p(e) = e(1 - e/2).  One MUFU op.
constexpr float kFarZ = 4.86f;   // > 7 ln 2
__device__ __forceinline__ CellFn cell_fn_far(float z) {
    const float e = fast_ex2(-fabsf(z) * kLog2e);
    const float r = fmaf(e, e - 1.0f, 1.0f);
    const float er = e * r;
    const bool pos = z >= 0.0f;
    CellFn c;
    c.p = pos ? r : er;
    c.pc = pos ? er : r;
    c.sp = fmaxf(z, 0.0f) + fmaf(-0.5f * e, e, e);
    return c;
}

__device__ __forceinline__ void red_add_v4(float *gptr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gptr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Default cells of one 32-column chunk: accumulate the sums and write H.
// kFull: every row and column of the warp's chunk lies inside the batch.
template <bool kFar, bool kFull>
__device__ __forceinline__ void default_cells(const float (&v)[32], float t, float b, bool row_ok, int valid,
                                              float hscale, float &acc_sp, float &acc_p, float &acc_ps,
                                              float (&hv)[32]) {
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float s = v[r];
        const float z = fmaf(t, s, b);
        const CellFn f = kFar ? cell_fn_far(z) : cell_fn(z);
        if (kFull) {
            acc_sp += f.sp;
            acc_p += f.p;
            acc_ps = fmaf(f.p, s, acc_ps);
            hv[r] = hscale * f.p;
        } else {
            const bool ok_col = row_ok && r < valid;
            acc_sp += ok_col ? f.sp : 0.f;
            acc_p += ok_col ? f.p : 0.f;
            acc_ps += ok_col ? f.p * s : 0.f;
            hv[r] = ok_col ? hscale * f.p : 0.f;
        }
    }
}

// Default cells of a full chunk where every z <= -kFarZ (the common repel
// cell): e = exp(z) < 2^-7, sigma(z) = e - e^2 and softplus(z) = e - e^2/2,
// each to relative error below e^2 < 2^-14.  The chunk's sums of e and e^2
// give those of sigma and softplus; one MUFU op per cell.
__device__ __forceinline__ void default_cells_negfar(const float (&v)[32], float t2, float b2, float hscale,
                                                     float &acc_sp, float &acc_p, float &acc_ps, float (&hv)[32]) {
    float se = 0.f, se2 = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float s = v[r];
        const float e = fast_ex2(fmaf(t2, s, b2));   // exp(z) with t2 = t log2(e), b2 = b log2(e)
        const float p = fmaf(-e, e, e);
        se += e;
        se2 = fmaf(e, e, se2);
        acc_ps = fmaf(p, s, acc_ps);
        hv[r] = hscale * p;
    }
    acc_sp += fmaf(-0.5f, se2, se);
    acc_p += se - se2;
}

__global__ void __launch_bounds__(kThreads, 1)
    fused_blocks_kernel(const __grid_constant__ CUtensorMap tmap_e, Params P) {
    extern __shared__ uint8_t smem_raw[];
    SharedStorage &sm = *reinterpret_cast<SharedStorage *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (read_status(P.status) != 0) return;  // an earlier stage of the call failed

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&sm.ring_full[h], 1);
            mbar_init(&sm.ring_empty[h], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.h_ready, kEpiWarps);
        mbar_init(&sm.h_free, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.de_full[b], 1);
            mbar_init(&sm.de_free[b], kEpiWarps);
        }
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
    // Box `pos` of stage `s`: stage 0 is the ring, stages 1 and 2 the two halves of the H region.
    auto box_ptr = [&](int s, int pos) -> uint8_t * { return s == 0 ? sm.ring[pos] : sm.hreg[(s - 1) * 4 + pos]; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t ph = 0;   // bit s (1, 2): parity of H-region stage s's next use; bit 3 + h: of ring half h
            uint32_t kblk = 0;
            bool ok = true;
            // Ring half h holds the boxes of positions 2h and 2h + 1 (h = 0: I0, I1; h = 1: J0, J1).
            auto load_half = [&](const Block &bk, int h, int k0) -> bool {
                const int bit = 3 + h;
                if (!mbar_wait(&sm.ring_empty[h], ((ph >> bit) & 1) ^ 1, abort_flag, P.status, kSleepProducer)) return false;
                const int nbox = (box_on(bk, 2 * h) ? 1 : 0) + (box_on(bk, 2 * h + 1) ? 1 : 0);
                mbar_arrive_expect_tx(&sm.ring_full[h], nbox * BOX_BYTES);   // none on a diagonal block's J half
                for (int pos = 2 * h; pos < 2 * h + 2; ++pos)
                    if (box_on(bk, pos)) tma_load_2d(sm.ring[pos], &tmap_e, &sm.ring_full[h], k0, box_tile(bk, pos) * BM);
                ph ^= 1u << bit;
                return true;
            };
            // Ring half h: the two 64-feature boxes of `tile` from feature k0 (none when the tile is absent;
            // a box past the width reads zeros).
            const int nc = (P.nk + 1) / 2;
            auto load_grad_half = [&](int h, int tile, int k0) -> bool {
                const int bit = 3 + h;
                if (!mbar_wait(&sm.ring_empty[h], ((ph >> bit) & 1) ^ 1, abort_flag, P.status, kSleepProducer)) return false;
                mbar_arrive_expect_tx(&sm.ring_full[h], tile >= 0 ? 2 * BOX_BYTES : 0u);
                if (tile >= 0) {
                    tma_load_2d(sm.ring[2 * h], &tmap_e, &sm.ring_full[h], k0, tile * BM);
                    tma_load_2d(sm.ring[2 * h + 1], &tmap_e, &sm.ring_full[h], k0 + BK, tile * BM);
                }
                ph ^= 1u << bit;
                return true;
            };
            for (long long p = blockIdx.x; p < P.blocks && ok; p += gridDim.x, ++kblk) {
                const Block bk = decode_block(p, P);
                int nbox = 0;
                for (int pos = 0; pos < 4; ++pos) nbox += box_on(bk, pos) ? 1 : 0;
                bool h_owned = false;
                // S pass: stage kc % 3, stage 0 being both ring halves.
                for (int kc = 0; kc < P.nk && ok; ++kc) {
                    const int s = kc % kStages;
                    if (s == 0) {
                        ok = load_half(bk, 0, kc * BK) && load_half(bk, 1, kc * BK);
                        continue;
                    }
                    if (!h_owned) {
                        // The H region holds the previous block's H until its gradient MMAs are done.
                        if (!mbar_wait(&sm.h_free, (kblk & 1) ^ 1, abort_flag, P.status, kSleepProducer)) { ok = false; break; }
                        h_owned = true;
                    }
                    if (!mbar_wait(&sm.empty[s], ((ph >> s) & 1) ^ 1, abort_flag, P.status, kSleepProducer)) { ok = false; break; }
                    mbar_arrive_expect_tx(&sm.full[s], nbox * BOX_BYTES);
                    for (int pos = 0; pos < 4; ++pos)
                        if (box_on(bk, pos))
                            tma_load_2d(box_ptr(s, pos), &tmap_e, &sm.full[s], kc * BK, box_tile(bk, pos) * BM);
                    ph ^= 1u << s;
                }
                // Gradient passes: per 128-feature chunk ring half 0, then half 1, so that each half loads
                // while the other half's products run.
                for (int pass = 0; pass < grad_passes(bk) && ok; ++pass)
                    for (int c = 0; c < nc && ok; ++c)
                        for (int h = 0; h < 2 && ok; ++h) ok = load_grad_half(h, grad_half_tile(bk, pass, h), c * 2 * BK);
            }
            // Let in-flight loads land before the CTA can exit.
            for (int s = 1; s < kStages; ++s) mbar_wait(&sm.empty[s], ((ph >> s) & 1) ^ 1, abort_flag, P.status);
            for (int h = 0; h < 2; ++h) mbar_wait(&sm.ring_empty[h], ((ph >> (3 + h)) & 1) ^ 1, abort_flag, P.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, 256, 0, 0);
            const uint32_t idesc_row = idesc_bf16(128, 128, 0, 1);   // A = H (K-major), B = E (MN-major)
            const uint32_t idesc_col = idesc_bf16(128, 128, 1, 1);   // A = H^T (MN-major), B = E (MN-major)
            uint32_t ph = 0;   // bit s (1, 2): parity of H-region stage s's next use; bit 3 + h: of ring half h
            uint32_t kblk = 0, chunk = 0;
            bool ok = true;
            auto wait_half = [&](int h) -> bool {
                return mbar_wait(&sm.ring_full[h], (ph >> (3 + h)) & 1, abort_flag, P.status, kSleepIssuer);
            };
            auto free_half = [&](int h) {
                mma_commit(&sm.ring_empty[h]);
                ph ^= 1u << (3 + h);
            };
            for (long long p = blockIdx.x; p < P.blocks && ok; p += gridDim.x, ++kblk) {
                const Block bk = decode_block(p, P);
                // S takes every TMEM column: wait until the last gradient chunk has been drained.
                if (chunk > 0 && !mbar_wait(&sm.de_free[(chunk - 1) & 1], ((chunk - 1) >> 1) & 1, abort_flag, P.status,
                                            kSleepIssuer))
                    break;
                tc_fence_after();
                for (int kc = 0; kc < P.nk; ++kc) {
                    const int s = kc % kStages;
                    if (s == 0 ? !(wait_half(0) && wait_half(1))
                               : !mbar_wait(&sm.full[s], (ph >> s) & 1, abort_flag, P.status, kSleepIssuer)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // One N = 256 MMA per tile row: the boxes of J0 and J1 (I0 and I1 on a diagonal
                    // block) are adjacent, so together they are one 256-row K-major operand whose
                    // product fills the TMEM columns of slots (x, 0) and (x, 1).  A slot that is
                    // off (an absent J1, or (1, 0) on a diagonal block) is computed from whatever
                    // the unloaded box holds and never read.
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (x == 1 && !bk.i1) continue;
                        const uint32_t a = smem_u32(box_ptr(s, x)), b = smem_u32(box_ptr(s, col_pos(bk, 0)));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_bf16(tmem + x * 2 * BM, sdesc_sw128(a + kk * 32, 16, 1024), sdesc_sw128(b + kk * 32, 16, 1024),
                                     idesc_s, (kc | kk) != 0);
                    }
                    if (s == 0) {
                        free_half(0);
                        free_half(1);
                    } else {
                        mma_commit(&sm.empty[s]);
                        ph ^= 1u << s;
                    }
                }
                if (!ok) break;
                mma_commit(&sm.s_full);
                // Gradient passes, 128 features at a time, into TMEM buffer (chunk & 1): accumulator a of
                // the pass at columns a * 128.  Products are M = 128, N = 128, K = 16; the B operand is a
                // tile's two feature boxes of ring half h, adjacent in shared memory, viewed as
                // [N = 128 features] x [K = rows] (MN-major, the boxes BOX_BYTES apart).
                if (!mbar_wait(&sm.h_ready, kblk & 1, abort_flag, P.status, kSleepIssuer)) break;
                tc_fence_after();
                const int nc = (P.nk + 1) / 2;
                for (int pass = 0; pass < grad_passes(bk) && ok; ++pass)
                    for (int c = 0; c < nc; ++c, ++chunk) {
                        const uint32_t buf = chunk & 1;
                        if (!mbar_wait(&sm.de_free[buf], ((chunk >> 1) & 1) ^ 1, abort_flag, P.status, kSleepIssuer)) { ok = false; break; }
                        const uint32_t acc0 = tmem + buf * 256;
                        uint32_t started = 0;   // bit a: accumulator a holds this chunk's first product
                        // acc[a] += H_xy E (A: H rows i, K = j, K-major) or H_xy^T E (A: H viewed as [M = j] x
                        // [K = i], MN-major, j contiguous within a 64-wide block, blocks BOX_BYTES apart).
                        auto product = [&](int a, int x, int y, bool transposed, uint32_t eb) {
                            const uint32_t h = smem_u32(sm.hreg[2 * (2 * x + y)]);
#pragma unroll
                            for (int kk = 0; kk < BM / 16; ++kk) {
                                const uint64_t ad = transposed ? sdesc_sw128(h + kk * 2048, BOX_BYTES, 1024)
                                                               : sdesc_sw128(h + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024);
                                mma_bf16(acc0 + a * 128, ad, sdesc_sw128(eb + kk * 2048, BOX_BYTES, 1024),
                                         transposed ? idesc_col : idesc_row, ((started >> a) & 1) || kk != 0);
                            }
                            started |= 1u << a;
                        };
                        for (int h = 0; h < 2; ++h) {
                            if (!wait_half(h)) { ok = false; break; }
                            tc_fence_after();
                            if (grad_half_tile(bk, pass, h) >= 0) {
                                const uint32_t eb = smem_u32(sm.ring[2 * h]);
                                if (bk.diag) {
                                    // E of I_h: row side of the slots (x, h), and the column side of (0, 1)
                                    // into I1 (a diagonal tile's H is symmetric: its row side is all of it).
                                    for (int x = 0; x < 2; ++x)
                                        if (slot_on(bk, x, h)) product(x, x, h, false, eb);
                                    if (h == 0 && slot_on(bk, 0, 1)) product(1, 0, 1, true, eb);
                                } else if (pass == 0) {   // E of J_h: dE_Ix += H_xh E_Jh
                                    for (int x = 0; x < 2; ++x)
                                        if (slot_on(bk, x, h)) product(x, x, h, false, eb);
                                } else {                  // E of I_h: dE_Jy += H_hy^T E_Ih
                                    for (int y = 0; y < 2; ++y)
                                        if (slot_on(bk, h, y)) product(y, h, y, true, eb);
                                }
                            }
                            free_half(h);
                        }
                        if (!ok) break;
                        mma_commit(&sm.de_full[buf]);
                    }
                if (!ok) break;
                mma_commit(&sm.h_free);
            }
            mma_commit(&sm.mma_done);
            mbar_wait(&sm.mma_done, 0, abort_flag, P.status);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int ew = warp - 2;                 // 0..7
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int x = ew >> 2;                   // tile row of the block this warp reads (and drains)
        const int row = quad * 32 + lane;        // row of the tile this thread owns
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float inv_n = 1.0f / static_cast<float>(P.n);
        const float w_d = P.named ? 0.0f : P.ambient;
        // A visited cell serves both ordered pairs, or (with groups) its row's anchor only.
        const float dirs = P.ordered ? 1.0f : 2.0f;
        const float w_dd = dirs * w_d;
        const uint32_t stage_s = smem_u32(sm.stage_t[ew]);
        uint32_t kblk = 0, chunk = 0;
        for (long long p = blockIdx.x; p < P.blocks; p += gridDim.x, ++kblk) {
            const Block bk = decode_block(p, P);
            const bool x_on = x == 0 || bk.i1;
            const int gi = (bk.I0 + x) * BM + row;   // this thread's item (anchor)
            const bool row_ok = x_on && gi >= P.row_lo && gi < P.row_hi;
            const int y_first = (bk.diag && x == 1) ? 1 : 0;
            // This row's (t, b): the run's pair, or its anchor's group's.
            const int grp = (P.group && row_ok) ? P.group[gi] : 0;
            const float t = P.t_ptr[grp], b = P.b_ptr[grp];
            const float t2 = t * kLog2e, b2 = b * kLog2e;
            const float c_h = t * inv_n;             // H = (t/N) G
            // This row's special columns from the first tile column it reads on.
            uint32_t e = 0, e_end = 0;
            if (row_ok) {
                const uint32_t jfirst = static_cast<uint32_t>((bk.J0 + y_first) * BM);
                uint32_t lo = P.rel_off[gi], hi = P.rel_off[gi + 1];
                e_end = hi;
                while (lo < hi) {
                    const uint32_t mid = (lo + hi) >> 1;
                    if (P.rel[mid].col < jfirst) lo = mid + 1; else hi = mid;
                }
                e = lo;
            }
            if (!mbar_wait(&sm.s_full, kblk & 1, abort_flag, P.status, kSleepEpilogue)) break;
            tc_fence_after();

            float l_sum = 0.f, g_sum = 0.f, gs_sum = 0.f;
            for (int y = y_first; y < 2; ++y) {
                if (!slot_on(bk, x, y)) continue;   // warp-uniform
                const int slot = 2 * x + y;
                const int j0 = (bk.J0 + y) * BM;
                const uint32_t hbase = smem_u32(sm.hreg[2 * slot]);
                float acc_sp = 0.f, acc_p = 0.f, acc_ps = 0.f;   // default cells (times dirs w_d later)
                float fix_l = 0.f, fix_g = 0.f, fix_gs = 0.f;   // corrections for special cells
#pragma unroll 1
                for (int ch = 0; ch < BM / 32; ++ch) {
                    // The chunk's scores and their maximum (a reducing TMEM load), and their minimum (a
                    // tree of three-input min operations): the chunk's range of z (t may be negative)
                    // picks the cheapest exact-enough path.
                    float v[32], smax;
                    {
                        uint32_t r[32];
                        tmem_ld32_max_async(tmem + lane_base + slot * BM + ch * 32, r, smax);
                        tmem_wait_ld();
                        tmem_regs_ready(r, smax);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    }
                    float m3[11];
#pragma unroll
                    for (int i = 0; i < 10; ++i) m3[i] = fmin3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
                    m3[10] = fminf(v[30], v[31]);
                    const float smin = fminf(fmin3(fmin3(m3[0], m3[1], m3[2]), fmin3(m3[3], m3[4], m3[5]),
                                                   fmin3(m3[6], m3[7], m3[8])),
                                             fmin3(m3[9], m3[10], m3[10]));
                    const int c0 = j0 + ch * 32;
                    const int valid = min(32, P.n - c0);   // columns of this chunk inside the batch
                    const float za = fmaf(t, smin, b), zb = fmaf(t, smax, b);
                    const float zlo = fminf(za, zb), zhi = fmaxf(za, zb);
                    float hv[32];
                    const float hscale = c_h * w_dd;
                    const bool full = __all_sync(0xffffffffu, row_ok && valid == 32);
                    const bool negfar = __all_sync(0xffffffffu, zhi <= -kFarZ);
                    const bool far = __all_sync(0xffffffffu, zhi <= -kFarZ || zlo >= kFarZ);
                    if (negfar && full)
                        default_cells_negfar(v, t2, b2, hscale, acc_sp, acc_p, acc_ps, hv);
                    else if (far && full)
                        default_cells<true, true>(v, t, b, row_ok, valid, hscale, acc_sp, acc_p, acc_ps, hv);
                    else if (far)
                        default_cells<true, false>(v, t, b, row_ok, valid, hscale, acc_sp, acc_p, acc_ps, hv);
                    else if (full)
                        default_cells<false, true>(v, t, b, row_ok, valid, hscale, acc_sp, acc_p, acc_ps, hv);
                    else
                        default_cells<false, false>(v, t, b, row_ok, valid, hscale, acc_sp, acc_p, acc_ps, hv);
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
                        const float w_in = P.ordered ? 0.0f : en.w_in;   // (j, i) is its own visit when ordered
                        const float g = en.w_out * (ao ? -f.pc : f.p) + w_in * (ai ? -f.pc : f.p);
                        const float l = en.w_out * (ao ? f.sp - z : f.sp) + w_in * (ai ? f.sp - z : f.sp);
                        const float g_def = w_dd * f.p;
                        fix_l += l - w_dd * f.sp;
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
                        st_shared_v4(hbase + sw128_bf16_offset(row, col, BM), pack_bf16x2(hv[q * 8 + 0], hv[q * 8 + 1]),
                                     pack_bf16x2(hv[q * 8 + 2], hv[q * 8 + 3]), pack_bf16x2(hv[q * 8 + 4], hv[q * 8 + 5]),
                                     pack_bf16x2(hv[q * 8 + 6], hv[q * 8 + 7]));
                    }
                }
                // A diagonal tile sees every unordered pair twice.
                const float scale = (bk.diag && x == y) ? 0.5f : 1.0f;
                l_sum += scale * (w_dd * acc_sp + fix_l);
                g_sum += scale * (w_dd * acc_p + fix_g);
                gs_sum += scale * (w_dd * acc_ps + fix_gs);
            }
            if (P.group) {   // this row's cells belong to its group's (t, b)
                if (row_ok && (g_sum != 0.f || gs_sum != 0.f)) {
                    atomicAdd(P.dt_g + grp, gs_sum * inv_n);
                    atomicAdd(P.db_g + grp, g_sum * inv_n);
                }
                g_sum = gs_sum = 0.f;
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.h_ready);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                l_sum += __shfl_xor_sync(0xffffffffu, l_sum, o);
                g_sum += __shfl_xor_sync(0xffffffffu, g_sum, o);
                gs_sum += __shfl_xor_sync(0xffffffffu, gs_sum, o);
            }
            if (lane == 0) {
                float *slot = P.partials + (p * kPartialsPerBlock + ew) * 4;
                slot[0] = l_sum;
                slot[1] = gs_sum;
                slot[2] = g_sum;
                slot[3] = 0.f;
            }
            // Drain the gradient chunks into dE: this warp takes accumulator x of each pass.
            bool ok = true;
            const int nc = (P.nk + 1) / 2;
            for (int pass = 0; pass < grad_passes(bk) && ok; ++pass)
                for (int c = 0; c < nc; ++c, ++chunk) {
                    const uint32_t buf = chunk & 1;
                    if (!mbar_wait(&sm.de_full[buf], (chunk >> 1) & 1, abort_flag, P.status, kSleepEpilogue)) { ok = false; break; }
                    tc_fence_after();
                    const int tile = grad_acc_tile(bk, pass, x);   // warp-uniform; -1: an absent tile row
                    if (tile >= 0) {
                        const int row0 = tile * BM + quad * 32;     // first row of this warp's 32
#pragma unroll 1
                        for (int piece = 0; piece < 4; ++piece) {
                            const int c0 = c * 128 + piece * 32;
                            if (c0 >= P.width) break;
                            float v[32];
                            tmem_ld32(tmem + lane_base + buf * 256 + x * 128 + piece * 32, v);
                            // lane = row: its 32 values as 8 x 16 B, chunk index swizzled by row
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                st_shared_v4(stage_s + (lane * 32 + ((k ^ (lane & 7)) * 4)) * 4, __float_as_uint(v[k * 4]),
                                             __float_as_uint(v[k * 4 + 1]), __float_as_uint(v[k * 4 + 2]),
                                             __float_as_uint(v[k * 4 + 3]));
                            __syncwarp();
                            // read back: instruction m covers rows 4m .. 4m+3, 8 lanes x 16 B = 128 B per row
                            const int col = c0 + (lane & 7) * 4;
#pragma unroll
                            for (int m = 0; m < 8; ++m) {
                                const int r = m * 4 + (lane >> 3);
                                const float4 xv = *reinterpret_cast<const float4 *>(&sm.stage_t[ew][r * 32 + (((lane & 7) ^ (r & 7)) * 4)]);
                                const int grow = row0 + r;
                                if (grow < P.n && col < P.width)
                                    red_add_v4(P.d_e + static_cast<long long>(grow) * P.ld_de + col, xv.x, xv.y, xv.z, xv.w);
                            }
                            __syncwarp();
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.de_free[buf]);
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
// final scalar reduction: fixed order, float64, two levels
// ----------------------------------------------------------------------------

// Block g sums the slots of its contiguous range (thread k adds k, k + 256, ...
// of the range, then a fixed-shape tree).
__global__ void finish_partial_kernel(const float *partials, long long slots, double *sums, const int32_t *status) {
    if (read_status(status) != 0) return;
    __shared__ double red[3][256];
    const long long per = (slots + gridDim.x - 1) / gridDim.x;
    const long long lo = blockIdx.x * per, hi = min(slots, lo + per);
    double l = 0, gs = 0, g = 0;
    for (long long s = lo + threadIdx.x; s < hi; s += blockDim.x) {
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
    if (threadIdx.x == 0)
        for (int c = 0; c < 3; ++c) sums[blockIdx.x * 3 + c] = red[c][0];
}

__global__ void finish_kernel(const double *sums, int n, float *loss, float *dt, float *db, const int32_t *status) {
    if (read_status(status) != 0) return;
    __shared__ double red[3][kFinishBlocks];
    for (int c = 0; c < 3; ++c) red[c][threadIdx.x] = sums[threadIdx.x * 3 + c];
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w)
            for (int c = 0; c < 3; ++c) red[c][threadIdx.x] += red[c][threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double inv_n = 1.0 / static_cast<double>(n);
        *loss = static_cast<float>(red[0][0] * inv_n);
        if (dt) *dt = static_cast<float>(red[1][0] * inv_n);   // with groups the kernel sums them per group
        if (db) *db = static_cast<float>(red[2][0] * inv_n);
    }
}

// Blocks of one call: the upper triangle, or every ordered block (groups, or an
// anchor band covering the whole batch at most).
long long block_count(int n, bool groups) {
    const long long nb = (n + BM - 1) / BM, nbb = (nb + 1) / 2;
    return groups ? nbb * nbb : nbb * (nbb + 1) / 2;
}

}  // namespace pooled

size_t pooled_fused_smem_bytes() { return pooled::kSmemBytes; }

long long pooled_partial_slots(int n) { return pooled::block_count(n, true) * pooled::kPartialsPerBlock; }
int pooled_finish_blocks() { return pooled::kFinishBlocks; }

cudaError_t launch_pooled_fused(const CUtensorMap &tmap_e, const PooledLaunch &L, cudaStream_t stream) {
    using namespace pooled;
    static bool configured = false;
    if (!configured) {
        cudaError_t err = cudaFuncSetAttribute(fused_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kSmemBytes));
        if (err != cudaSuccess) return err;
        configured = true;
    }
    Params P;
    P.n = L.n;
    P.width = L.width;
    P.nk = (L.width + BK - 1) / BK;
    P.nb = (L.n + BM - 1) / BM;
    P.nbb = (P.nb + 1) / 2;
    // An anchor band narrower than the batch takes the ordered traversal over the block rows it touches.
    P.row_lo = L.row_lo;
    P.row_hi = L.row_hi > 0 ? L.row_hi : L.n;
    const bool band = P.row_lo > 0 || P.row_hi < L.n;
    P.ordered = (L.group != nullptr || band) ? 1 : 0;
    P.bi0 = P.ordered ? P.row_lo / (2 * BM) : 0;
    const long long bi_end = P.ordered ? (P.row_hi + 2 * BM - 1) / (2 * BM) : 0;
    P.blocks = P.ordered ? (bi_end - P.bi0) * P.nbb : block_count(L.n, false);
    P.group = L.group;
    P.dt_g = L.group ? L.dt : nullptr;
    P.db_g = L.group ? L.db : nullptr;
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
    if (P.blocks <= 0) return cudaErrorInvalidValue;   // the host checks keep the band inside the batch
    long long grid = static_cast<long long>(L.sm_count);
    if (grid > P.blocks) grid = P.blocks;
    fused_blocks_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tmap_e, P);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    finish_partial_kernel<<<kFinishBlocks, 256, 0, stream>>>(L.partials, P.blocks * kPartialsPerBlock, L.sums, L.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    finish_kernel<<<1, kFinishBlocks, 0, stream>>>(L.sums, L.n, L.loss, L.group ? nullptr : L.dt,
                                                   L.group ? nullptr : L.db, L.status);
    return cudaGetLastError();
}

}  // namespace cli
