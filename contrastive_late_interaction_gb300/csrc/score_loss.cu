// The sigmoid pair loss over a given rows x cols score matrix ("UForm", section
// "ColBERT-Style Late-Interaction Rerankers": MaxSim scores fill the same band
// the pooled embedder builds, scored by a selectable pair-loss form; this is
// the `sigmoid` form of "Training", `uform_pair_loss_form_t`):
//     l_ij = w_ij softplus(-y_ij (t S_ij + b)),  L = (1/rows) sum l_ij,
// with dS, dt, db.  Elementwise and bandwidth-bound: one pass reading S and
// writing dS, relation lookups by binary search in each row's CSR slice, and
// per-block partial sums reduced in a fixed order.

#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace {

__device__ bool find_edge(const EdgeSet &s, int i, uint32_t j, float *w) {
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

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) score_loss_kernel(ScoreLossLaunch L) {
    __shared__ float red[3][kThreads / 32];
    if (read_status(L.status) != 0) return;
    const float t = *L.t_ptr, b = *L.b_ptr;
    const float inv_r = 1.0f / static_cast<float>(L.rows);
    const long long total = static_cast<long long>(L.rows) * L.cols;
    float acc_l = 0.f, acc_gs = 0.f, acc_g = 0.f;
    for (long long idx = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * kThreads) {
        const int i = static_cast<int>(idx / L.cols), j = static_cast<int>(idx % L.cols);
        const float s = L.scores[static_cast<long long>(i) * L.ld + j];
        float y = 0.f, w = 0.f;
        bool scored = true;
        if (L.sides && (!(L.sides[i] & 1) || !(L.sides[j] & 2))) scored = false;
        if (scored && find_edge(L.sets[2], i, static_cast<uint32_t>(j), nullptr)) scored = false;
        if (scored) {
            if (find_edge(L.sets[0], i, static_cast<uint32_t>(j), &w)) y = 1.f;
            else if (find_edge(L.sets[1], i, static_cast<uint32_t>(j), &w)) y = -1.f;
            else if (!L.named) { y = -1.f; w = L.ambient; }
            else scored = false;
        }
        float g = 0.f;
        if (scored) {
            const float z = fmaf(t, s, b);
            const float m = -y * z;                                       // loss = w softplus(m)
            const float sp = fmaxf(m, 0.f) + log1pf(expf(-fabsf(m)));
            const float sig = m >= 0.f ? 1.f / (1.f + expf(-m)) : expf(m) / (1.f + expf(m));  // sigma(m)
            g = -w * y * sig;                                             // dl/dz
            acc_l += w * sp;
            acc_gs += g * s;
            acc_g += g;
        }
        L.d_scores[static_cast<long long>(i) * L.ld_ds + j] = t * g * inv_r;
    }
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc_l += __shfl_xor_sync(0xffffffffu, acc_l, o);
        acc_gs += __shfl_xor_sync(0xffffffffu, acc_gs, o);
        acc_g += __shfl_xor_sync(0xffffffffu, acc_g, o);
    }
    if (lane == 0) {
        red[0][wp] = acc_l;
        red[1][wp] = acc_gs;
        red[2][wp] = acc_g;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float l = 0.f, gs = 0.f, g = 0.f;
        for (int k = 0; k < kThreads / 32; ++k) {
            l += red[0][k];
            gs += red[1][k];
            g += red[2][k];
        }
        float *slot = L.partials + static_cast<long long>(blockIdx.x) * 4;
        slot[0] = l;
        slot[1] = gs;
        slot[2] = g;
        slot[3] = 0.f;
    }
}

// Sums the per-block partials in a fixed order: thread k adds blocks k, k+256,
// ... in order, then a fixed-shape tree over the 256 threads.
__global__ void score_finish_kernel(const float *partials, int blocks, int rows, float *loss, float *dt, float *db,
                                    const int32_t *status) {
    if (read_status(status) != 0) return;
    __shared__ double red[3][256];
    double l = 0, gs = 0, g = 0;
    for (int k = threadIdx.x; k < blocks; k += blockDim.x) {
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
        const double inv = 1.0 / static_cast<double>(rows);
        *loss = static_cast<float>(red[0][0] * inv);
        *dt = static_cast<float>(red[1][0] * inv);
        *db = static_cast<float>(red[2][0] * inv);
    }
}

}  // namespace

int score_loss_blocks(size_t rows, size_t cols) {
    const long long cells = static_cast<long long>(rows) * static_cast<long long>(cols);
    long long b = (cells + kThreads * 8 - 1) / (kThreads * 8);
    if (b < 1) b = 1;
    if (b > 4096) b = 4096;
    return static_cast<int>(b);
}

cudaError_t launch_score_loss(const ScoreLossLaunch &L, cudaStream_t stream) {
    cudaError_t err;
    for (int s = 0; s < 3; ++s)
        if ((err = launch_validate_edges(L.sets[s], L.rows, L.cols, L.status, stream)) != cudaSuccess) return err;
    score_loss_kernel<<<L.blocks, kThreads, 0, stream>>>(L);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    score_finish_kernel<<<1, 256, 0, stream>>>(L.partials, L.blocks, L.rows, L.loss, L.dt, L.db, L.status);
    return cudaGetLastError();
}

}  // namespace cli
