// maxsim_backward_no_alloc: the MaxSim backward for callers that cannot
// allocate device memory and have no buffer to lend as workspace.
//
// Some callers cannot call cudaMalloc: code running where an allocation is not
// allowed or would stall the device (cudaMalloc may wait for the GPU to go
// idle), or a runtime whose device memory is all reserved up front by its own
// allocator with nothing left to lend as scratch.  For them this entry point
// keeps the only scratch the backward needs -- the map from query-tape row to
// query -- in a file-scope device array of fixed size.  The caller still
// passes every input and output.
//
// The array costs kNoAllocMaxQueryRows * 4 bytes (1 MiB) on every GPU that
// loads the library, until the process exits.  All calls share it and it keeps
// the last call's contents; this path fully rewrites every entry it reads
// before reading it, so nothing needs clearing, but two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// it.  The first call on each device looks the array's device address up (with
// that device current) and caches it with the device's current context; make
// that first call before any stream capture.  After cudaDeviceReset the
// context, and with it the array's address, changes: a call in the new
// context looks the address up again.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/cli.h"
#include "cli_internal.h"

namespace cli {
namespace {

constexpr size_t kNoAllocMaxQueryRows = CLI_MAXSIM_NO_ALLOC_MAX_QUERY_ROWS;
static __device__ __align__(256) int32_t g_query_of_row[kNoAllocMaxQueryRows];

constexpr int kMaxDevices = 64;
struct Scratch {
    int32_t *ptr;
    CUcontext ctx;   // the context the address belongs to
};
Scratch g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// The calling thread's current context (NULL before the runtime has made one
// current), through the driver entry point, so the library needs no libcuda link.
CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p)
                   : nullptr;
    }();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// Device address of g_query_of_row on the current device, looked up once per
// device and context; NULL on failure.
int32_t *scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    Scratch &s = g_scratch[dev];
    if (!s.ptr || !ctx || ctx != s.ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_query_of_row) != cudaSuccess || !p) return nullptr;
        s.ptr = static_cast<int32_t *>(p);
        s.ctx = current_context();   // current now that the runtime has set the device up
    }
    return s.ptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool tape_valid(const cli_tape_t &t) {
    return t.data && t.offsets && t.count > 0 && t.rows >= t.count && t.rows < (1ull << 31) &&
           t.count < (1ull << 31) && aligned16(t.data);
}

}  // namespace
}  // namespace cli

extern "C" cli_status_t maxsim_backward_no_alloc(const cli_maxsim_backward_t *a) {
    using namespace cli;
    if (!a) return CLI_INVALID_ARGUMENT;
    if (!a->argmax || !a->d_scores || !a->d_queries || !a->d_documents || !a->device_status)
        return CLI_INVALID_ARGUMENT;
    if (!tape_valid(a->queries) || !tape_valid(a->documents)) return CLI_INVALID_ARGUMENT;
    if (a->width == 0 || a->width % 8 != 0) return CLI_SHAPE_MISMATCH;
    if (a->width > 256) return CLI_UNSUPPORTED;
    const size_t nq = a->queries.count, nd = a->documents.count, rq = a->queries.rows, rd = a->documents.rows;
    if (rq > kNoAllocMaxQueryRows) return CLI_UNSUPPORTED;   // beyond the fixed scratch
    if (a->ld_d_scores < nd || a->ld_argmax < rq) return CLI_SHAPE_MISMATCH;
    if (!aligned16(a->d_queries) || !aligned16(a->d_documents)) return CLI_INVALID_ARGUMENT;
    // outputs may not overlap inputs or each other
    struct R { uintptr_t lo, hi; };
    auto r = [](const void *p, size_t n) { return R{reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + n}; };
    const R in[] = {r(a->queries.data, rq * a->width * 2), r(a->queries.offsets, (nq + 1) * 8),
                    r(a->documents.data, rd * a->width * 2), r(a->documents.offsets, (nd + 1) * 8),
                    r(a->argmax, ((nd - 1) * a->ld_argmax + rq) * 4), r(a->d_scores, ((nq - 1) * a->ld_d_scores + nd) * 4)};
    const R out[] = {r(a->d_queries, rq * a->width * 4), r(a->d_documents, rd * a->width * 4), r(a->device_status, 4)};
    for (const R &o : out) {
        for (const R &i : in)
            if (o.lo < i.hi && i.lo < o.hi) return CLI_INVALID_ARGUMENT;
        for (const R &p : out)
            if (&p != &o && o.lo < p.hi && p.lo < o.hi) return CLI_INVALID_ARGUMENT;
    }
    int32_t *qmap = scratch_for_current_device();
    if (!qmap) return CLI_DEVICE;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return CLI_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(a->stream);
    if (cudaMemsetAsync(a->device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return CLI_DEVICE;
    if (launch_validate_tape(a->queries.offsets, static_cast<int>(nq), rq, a->device_status, stream) != cudaSuccess ||
        launch_validate_tape(a->documents.offsets, static_cast<int>(nd), rd, a->device_status, stream) != cudaSuccess)
        return CLI_DEVICE;
    MaxSimBwdLaunch L;
    L.nq = static_cast<int>(nq);
    L.nd = static_cast<int>(nd);
    L.rows_q = static_cast<int>(rq);
    L.rows_d = static_cast<int>(rd);
    L.width = static_cast<int>(a->width);
    L.mean = a->mean ? 1 : 0;
    L.q_off = a->queries.offsets;
    L.d_off = a->documents.offsets;
    L.q = static_cast<const uint16_t *>(a->queries.data);
    L.d = static_cast<const uint16_t *>(a->documents.data);
    L.argmax = a->argmax;
    L.ld_argmax = static_cast<long long>(a->ld_argmax);
    L.d_scores = a->d_scores;
    L.ld_ds = static_cast<long long>(a->ld_d_scores);
    L.dq = a->d_queries;
    L.dd = a->d_documents;
    L.qmap = qmap;
    L.status = a->device_status;
    L.sm_count = sms;
    if (launch_maxsim_backward(L, stream) != cudaSuccess) return CLI_DEVICE;
    return CLI_OK;
}
