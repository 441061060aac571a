// The `balanced` and `ranked` pair-loss forms over a rows x cols score matrix
// ("Training", `uform_pair_loss_form_t`: balanced -- the sigmoid cross-entropy
// of every cell, its attract and repel halves normalized apart; ranked -- the
// sigmoid cross-entropy of every positive's score over every negative's, where
// the bias cancels; "UForm", "ColBERT-Style Late-Interaction Rerankers": ranked
// is the default for the rows of hard MaxSim scores).
//
// Readings (the pages give words only):
//   balanced: l_p = sum_attract w l / sum_attract w + sum_repel w l / sum_repel w
//   ranked:   l_p = sum_{i in P, j in N} w_i w_j softplus(-t (S_pi - S_pj)) / (W_P W_N)
//   L = (1/rows) sum_p l_p, cells resolved as in the sigmoid form (relations,
//   sides, negatives).
//
// One CTA per row: a first pass resolves every column of the row and sums the
// weights of its attract and repel cells (and, for ranked, gathers the
// positives into shared memory); a second pass writes the row of dS and the
// row's loss, dt and db partials (block reductions in a fixed order), which a
// final kernel sums over rows in order.

#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPos = 16;   // positives held per pass of the ranked form

__device__ bool find_in_row(const EdgeSet &s, int i, uint32_t j, float *w) {
    if (!s.offsets) return false;
    uint64_t lo = s.offsets[i], hi = s.offsets[i + 1];
    while (lo < hi) {
        const uint64_t mid = (lo + hi) >> 1;
        const uint32_t v = s.ids[mid];
        if (v == j) {
            if (w) *w = s.weights ? s.weights[mid] : 1.0f;
            return true;
        }
        if (v < j) lo = mid + 1; else hi = mid;
    }
    return false;
}

// Resolves cell (i, j): returns +1 attract, -1 repel, 0 skipped; *w its weight.
__device__ int resolve_cell(const ScoreLossLaunch &L, int i, int j, float *w) {
    if (L.sides && (!(L.sides[i] & 1) || !(L.sides[j] & 2))) return 0;
    if (find_in_row(L.sets[2], i, static_cast<uint32_t>(j), nullptr)) return 0;
    if (find_in_row(L.sets[0], i, static_cast<uint32_t>(j), w)) return 1;
    if (find_in_row(L.sets[1], i, static_cast<uint32_t>(j), w)) return -1;
    if (L.named) return 0;
    *w = L.ambient;
    return -1;
}

__device__ float block_sum(float v, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float s = 0.f;
    for (int k = 0; k < kThreads / 32; ++k) s += scratch[k];
    return s;
}

__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }
__device__ __forceinline__ float sigmoid_f(float x) {
    return x >= 0.f ? 1.f / (1.f + expf(-x)) : expf(x) / (1.f + expf(x));
}

__global__ void __launch_bounds__(kThreads) balanced_kernel(ScoreLossLaunch L) {
    __shared__ float scratch[kThreads / 32];
    if (read_status(L.status) != 0) return;
    const int i = blockIdx.x;
    const float t = *L.t_ptr, b = *L.b_ptr;
    float wa = 0.f, wr = 0.f;
    for (int j = threadIdx.x; j < L.cols; j += kThreads) {
        float w = 0.f;
        const int y = resolve_cell(L, i, j, &w);
        if (y > 0) wa += w;
        else if (y < 0) wr += w;
    }
    const float WA = block_sum(wa, scratch), WR = block_sum(wr, scratch);
    const float inv_r = 1.0f / static_cast<float>(L.rows);
    float acc_l = 0.f, acc_gs = 0.f, acc_g = 0.f;
    const float *srow = L.scores + static_cast<long long>(i) * L.ld;
    float *drow = L.d_scores + static_cast<long long>(i) * L.ld_ds;
    for (int j = threadIdx.x; j < L.cols; j += kThreads) {
        float w = 0.f;
        const int y = resolve_cell(L, i, j, &w);
        float g = 0.f;
        if (y != 0) {
            const float s = srow[j];
            const float m = -static_cast<float>(y) * fmaf(t, s, b);
            const float norm = y > 0 ? WA : WR;
            const float wn = w / norm;
            g = -wn * static_cast<float>(y) * sigmoid_f(m);   // dl/dz of the normalised cell
            acc_l += wn * softplus_f(m);
            acc_gs += g * s;
            acc_g += g;
        }
        drow[j] = t * g * inv_r;
    }
    const float l = block_sum(acc_l, scratch), gs = block_sum(acc_gs, scratch), gg = block_sum(acc_g, scratch);
    if (threadIdx.x == 0) {
        float *slot = L.partials + static_cast<long long>(i) * 4;
        slot[0] = l * inv_r;
        slot[1] = gs * inv_r;
        slot[2] = gg * inv_r;
        slot[3] = 0.f;
    }
}

__global__ void __launch_bounds__(kThreads) ranked_kernel(ScoreLossLaunch L) {
    __shared__ float scratch[kThreads / 32];
    __shared__ float pos_s[kMaxPos], pos_w[kMaxPos], pos_g[kMaxPos];
    __shared__ int pos_j[kMaxPos];
    __shared__ int npos_s;
    if (read_status(L.status) != 0) return;
    const int i = blockIdx.x;
    const float t = *L.t_ptr;
    const float *srow = L.scores + static_cast<long long>(i) * L.ld;
    float *drow = L.d_scores + static_cast<long long>(i) * L.ld_ds;
    // pass 1: weight sums of the positives (attract) and negatives (repel)
    float wp = 0.f, wn = 0.f;
    for (int j = threadIdx.x; j < L.cols; j += kThreads) {
        float w = 0.f;
        const int y = resolve_cell(L, i, j, &w);
        if (y > 0) wp += w;
        else if (y < 0) wn += w;
        drow[j] = 0.f;
    }
    const float WP = block_sum(wp, scratch), WN = block_sum(wn, scratch);
    float acc_l = 0.f, acc_dt = 0.f;
    const bool any = WP > 0.f && WN > 0.f;
    const float inv = any ? 1.0f / (WP * WN * static_cast<float>(L.rows)) : 0.f;
    // pass 2: positives in groups of kMaxPos (in column order), every negative against each
    for (int start = 0; any && start < L.cols;) {
        __syncthreads();
        if (threadIdx.x == 0) {
            int n = 0, j = start;
            for (; j < L.cols && n < kMaxPos; ++j) {
                float w = 0.f;
                if (resolve_cell(L, i, j, &w) > 0) {
                    pos_j[n] = j;
                    pos_s[n] = srow[j];
                    pos_w[n] = w;
                    ++n;
                }
            }
            npos_s = n;
            scratch[0] = __int_as_float(j);   // where the next group starts
        }
        __syncthreads();
        const int npos = npos_s;
        const int next = __float_as_int(scratch[0]);
        float gpos[kMaxPos];
#pragma unroll
        for (int k = 0; k < kMaxPos; ++k) gpos[k] = 0.f;
        for (int j = threadIdx.x; j < L.cols; j += kThreads) {
            float w = 0.f;
            if (resolve_cell(L, i, j, &w) >= 0) continue;   // not a negative
            const float sj = srow[j];
            float dj = 0.f;
#pragma unroll
            for (int k = 0; k < kMaxPos; ++k) {
                if (k < npos) {
                    const float pw = pos_w[k] * w * inv;
                    const float m = t * (pos_s[k] - sj);
                    const float sg = sigmoid_f(-m);
                    acc_l += pw * softplus_f(-m);
                    acc_dt -= pw * sg * (pos_s[k] - sj);
                    gpos[k] -= pw * sg * t;
                    dj += pw * sg * t;
                }
            }
            drow[j] += dj;
        }
        for (int k = 0; k < npos; ++k) {
            const float g = block_sum(gpos[k], scratch);
            if (threadIdx.x == 0) pos_g[k] = g;
        }
        __syncthreads();
        if (threadIdx.x == 0)
            for (int k = 0; k < npos; ++k) drow[pos_j[k]] = pos_g[k];
        start = next;
        if (npos < kMaxPos) break;
    }
    const float l = block_sum(acc_l, scratch), dt = block_sum(acc_dt, scratch);
    if (threadIdx.x == 0) {
        float *slot = L.partials + static_cast<long long>(i) * 4;
        slot[0] = l;
        slot[1] = dt;
        slot[2] = 0.f;
        slot[3] = 0.f;
    }
}

// Row partials summed in row order (fp64): thread k adds rows k, k+256, ...,
// then a fixed-shape tree.
__global__ void forms_finish_kernel(const float *partials, int rows, float *loss, float *dt, float *db,
                                    const int32_t *status) {
    if (read_status(status) != 0) return;
    __shared__ double red[3][256];
    double l = 0, gs = 0, g = 0;
    for (int k = threadIdx.x; k < rows; k += blockDim.x) {
        l += partials[k * 4 + 0];
        gs += partials[k * 4 + 1];
        g += partials[k * 4 + 2];
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
        *loss = static_cast<float>(red[0][0]);
        *dt = static_cast<float>(red[1][0]);
        *db = static_cast<float>(red[2][0]);
    }
}

}  // namespace

cudaError_t launch_score_forms(int form, const ScoreLossLaunch &L, cudaStream_t stream) {
    cudaError_t err;
    for (int s = 0; s < 3; ++s)
        if ((err = launch_validate_edges(L.sets[s], L.rows, L.cols, L.status, stream)) != cudaSuccess) return err;
    if (form == 1) balanced_kernel<<<L.rows, kThreads, 0, stream>>>(L);
    else ranked_kernel<<<L.rows, kThreads, 0, stream>>>(L);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    forms_finish_kernel<<<1, 256, 0, stream>>>(L.partials, L.rows, L.loss, L.dt, L.db, L.status);
    return cudaGetLastError();
}

}  // namespace cli
