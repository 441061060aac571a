// Ordered compaction of a flag array into an index list (one block): shared by
// the named-pair MaxSim schedule and the backward's list of active documents.
#pragma once

#include <stdint.h>

#include "cli_device.cuh"

namespace cli {
namespace ms {

// The flagged entries in index order and their count: one block, each thread
// compacting a contiguous segment after a scan of the counts.
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

}  // namespace ms
}  // namespace cli
