// Matryoshka prefixes under the pooled sigmoid pair loss ("Training",
// `uform_contrastive_t`, `matryoshka_dimensions`: ascending prefix widths,
// every one scored; "UForm", section "Matryoshka-Like Multi-Scale Embedders":
// each prefix trained under the SigLIP loss on cosine similarities):
//     L = sum_p L_sigmoid(u_p),  u_p,i = e_i[:p] / |e_i[:p]|,
//     dE_i[:p] += (g_i - (g_i . u_i) u_i) / |e_i[:p]|,  g = dL_p / du_p.
//
// Per prefix the call normalises the prefix rows into a bf16 copy (one warp per
// row), runs the fused pooled kernel on that copy, and sends its dE back
// through the normalisation into dE (one warp per row).  The relations are
// resolved once for all prefixes; the per-prefix (loss, dt, db) land in the
// workspace and a last kernel sums them in prefix order.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace {

constexpr int kRowsPerBlock = 8;   // one warp per row

__device__ __forceinline__ void bf16x8_unpack(const uint4 u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// u[i][0..p) = bf16(e_i[:p] / |e_i[:p]|) (nearest even), inv_norm[i] = 1 / |e_i[:p]|,
// both zero for a prefix of zero norm.  p and ld are multiples of 8.
__global__ void __launch_bounds__(256) prefix_normalize_kernel(const uint16_t *e, long long ld, int n, int p,
                                                               uint16_t *u, float *inv_norm, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int i = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (i >= n) return;
    const uint16_t *row = e + static_cast<long long>(i) * ld;
    float ss = 0.f;
    for (int k = lane * 8; k < p; k += 256) {
        float x[8];
        bf16x8_unpack(*reinterpret_cast<const uint4 *>(row + k), x);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
    }
    ss = warp_sum(ss);
    const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
    uint16_t *dst = u + static_cast<long long>(i) * p;
    for (int k = lane * 8; k < p; k += 256) {
        float x[8];
        bf16x8_unpack(*reinterpret_cast<const uint4 *>(row + k), x);
        uint4 o;
        uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * j] * inv, x[2 * j + 1] * inv);
            ow[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(dst + k) = o;
    }
    if (lane == 0) inv_norm[i] = inv;
}

// dE[i][0..p) += (g - (g . u) u) * inv_norm[i] with g = de_p[i][0..p) and
// u = e_i[:p] * inv_norm[i] in fp32.
__global__ void __launch_bounds__(256) prefix_backprop_kernel(const uint16_t *e, long long ld, int n, int p,
                                                              const float *inv_norm, const float *de_p, float *de,
                                                              long long ld_de, const int32_t *status) {
    if (read_status(status) != 0) return;
    const int i = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (i >= n) return;
    const float inv = inv_norm[i];
    const uint16_t *row = e + static_cast<long long>(i) * ld;
    const float *g = de_p + static_cast<long long>(i) * p;
    float dot = 0.f;
    for (int k = lane * 8; k < p; k += 256) {
        float x[8];
        bf16x8_unpack(*reinterpret_cast<const uint4 *>(row + k), x);
        const float4 g0 = *reinterpret_cast<const float4 *>(g + k), g1 = *reinterpret_cast<const float4 *>(g + k + 4);
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) dot = fmaf(gv[j], x[j] * inv, dot);
    }
    dot = warp_sum(dot);
    float *out = de + static_cast<long long>(i) * ld_de;
    for (int k = lane * 8; k < p; k += 256) {
        float x[8];
        bf16x8_unpack(*reinterpret_cast<const uint4 *>(row + k), x);
        const float4 g0 = *reinterpret_cast<const float4 *>(g + k), g1 = *reinterpret_cast<const float4 *>(g + k + 4);
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float4 o0 = *reinterpret_cast<float4 *>(out + k), o1 = *reinterpret_cast<float4 *>(out + k + 4);
        float ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) ov[j] = fmaf(gv[j] - dot * (x[j] * inv), inv, ov[j]);
        *reinterpret_cast<float4 *>(out + k) = make_float4(ov[0], ov[1], ov[2], ov[3]);
        *reinterpret_cast<float4 *>(out + k + 4) = make_float4(ov[4], ov[5], ov[6], ov[7]);
    }
}

// loss, dt, db = the per-prefix values summed in prefix order; prefix_loss (if
// given) receives each prefix's loss.
__global__ void matryoshka_finish_kernel(const float *scalars, int count, float *loss, float *dt, float *db,
                                         float *prefix_loss, const int32_t *status) {
    if (read_status(status) != 0 || threadIdx.x != 0) return;
    double l = 0, t = 0, b = 0;
    for (int k = 0; k < count; ++k) {
        l += scalars[3 * k];
        t += scalars[3 * k + 1];
        b += scalars[3 * k + 2];
        if (prefix_loss) prefix_loss[k] = scalars[3 * k];
    }
    *loss = static_cast<float>(l);
    *dt = static_cast<float>(t);
    *db = static_cast<float>(b);
}

inline unsigned row_blocks(int n) { return static_cast<unsigned>((n + kRowsPerBlock - 1) / kRowsPerBlock); }

}  // namespace

MatryoshkaWorkspace carve_matryoshka_workspace(void *base, size_t n, size_t width, size_t edges_total) {
    MatryoshkaWorkspace w;
    w.pooled = carve_pooled_workspace(base, n, width, edges_total);
    uint8_t *p = static_cast<uint8_t *>(base);
    size_t off = w.pooled.bytes;
    auto take = [&](size_t bytes) {
        uint8_t *q = p ? p + off : nullptr;
        off += align256(bytes);
        return q;
    };
    w.u = reinterpret_cast<uint16_t *>(take(n * width * 2));
    w.inv_norm = reinterpret_cast<float *>(take(n * 4));
    w.de_p = reinterpret_cast<float *>(take(n * width * 4));
    w.scalars = reinterpret_cast<float *>(take(kMaxMatryoshkaPrefixes * 3 * 4));
    w.bytes = off;
    return w;
}

cudaError_t launch_prefix_normalize(const uint16_t *e, long long ld, int n, int p, const MatryoshkaWorkspace &ws,
                                    const int32_t *status, cudaStream_t stream) {
    prefix_normalize_kernel<<<row_blocks(n), 256, 0, stream>>>(e, ld, n, p, ws.u, ws.inv_norm, status);
    return cudaGetLastError();
}

cudaError_t launch_prefix_backprop(const uint16_t *e, long long ld, int n, int p, const MatryoshkaWorkspace &ws,
                                   float *de, long long ld_de, const int32_t *status, cudaStream_t stream) {
    prefix_backprop_kernel<<<row_blocks(n), 256, 0, stream>>>(e, ld, n, p, ws.inv_norm, ws.de_p, de, ld_de, status);
    return cudaGetLastError();
}

cudaError_t launch_matryoshka_finish(const MatryoshkaWorkspace &ws, int count, float *loss, float *dt, float *db,
                                     float *prefix_loss, const int32_t *status, cudaStream_t stream) {
    matryoshka_finish_kernel<<<1, 32, 0, stream>>>(ws.scalars, count, loss, dt, db, prefix_loss, status);
    return cudaGetLastError();
}

}  // namespace cli
