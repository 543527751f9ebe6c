// moe_route_permute_noalloc: the routing / grouping of moe_route_permute with
// its scratch in a fixed device array owned by this library, for callers that
// must not allocate device memory themselves.
//
// Who cannot allocate: code running inside a CUDA stream capture in the global
// capture mode (cudaMalloc is an unsafe call there), plug-ins or callbacks of
// another runtime that owns every byte of device memory, and latency-critical
// loops where a cudaMalloc / cudaFree could synchronise the device.  They still
// pass their inputs and outputs; only the per-chunk counting scratch moves here.
#include <cstdio>
#include <mutex>

#include "../../include/qmm.h"
#include "qmm_internal.h"

namespace qmm {
namespace {

// Scratch of the per-chunk expert counts: chunks * E int32, chunks = ceil(T / 256).
// 1 MiB, held by every GPU that loads the library until the process exits.
constexpr size_t kNoAllocScratchInts = QMM_NOALLOC_SCRATCH_BYTES / 4;
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

// Device address of the scratch array, resolved once per device (with that
// device current).  In host code the array's name is only a host-side
// stand-in, never a device address.
constexpr int kMaxDev = 64;
int32_t* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;
qmm_status noalloc_fail(qmm_status st, const char* msg, const char* detail = "") {
    char buf[384];
    snprintf(buf, sizeof buf, "moe_route_permute_noalloc: %s%s", msg, detail);
    set_last_error(buf);
    return st;
}

qmm_status scratch_for_current_device(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(QMM_ERR_CUDA, "cudaGetDevice: ", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDev) return noalloc_fail(QMM_ERR_UNSUPPORTED_DEVICE, "device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return noalloc_fail(QMM_ERR_UNSUPPORTED_DEVICE, "this library is built for sm_103a only");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess)
            return noalloc_fail(QMM_ERR_CUDA, "cudaGetSymbolAddress(scratch): ", cudaGetErrorString(e));
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return QMM_OK;
}

}  // namespace
}  // namespace qmm

extern "C" qmm_status moe_route_permute_noalloc(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                                int32_t* counts, int32_t* offsets, int32_t* src, int32_t* row,
                                                cudaStream_t stream) {
    using namespace qmm;
    if (T < 0 || k < 1 || k > 16 || E < k || E > 512)
        return noalloc_fail(QMM_ERR_UNSUPPORTED_SHAPE, "need T >= 0, 1 <= k <= 16, k <= E <= 512");
    if (!counts || !offsets || (T > 0 && (!logits || !ids || !w || !src || !row)))
        return noalloc_fail(QMM_ERR_INVALID_ARG, "null pointer");
    const size_t chunks = ((size_t)T + kRouteChunk - 1) / kRouteChunk;
    if (chunks * (size_t)E > kNoAllocScratchInts) {
        char d[160];
        snprintf(d, sizeof d, " (ceil(T/256) * E = %zu counters, the built-in scratch holds %zu)", chunks * (size_t)E,
                 kNoAllocScratchInts);
        return noalloc_fail(QMM_ERR_UNSUPPORTED_SHAPE, "T * E too large for the fixed scratch", d);
    }
    int32_t* scratch = nullptr;
    qmm_status st = scratch_for_current_device(&scratch);
    if (st != QMM_OK) return st;
    cudaError_t e;
    if (T == 0) {
        if ((e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream)) != cudaSuccess)
            return noalloc_fail(QMM_ERR_CUDA, "cudaMemsetAsync: ", cudaGetErrorString(e));
        return QMM_OK;
    }
    // Every counter the kernels read is written first by this call (each chunk
    // stores all E of its counts), so the scratch needs no clearing.
    RouteBufs b{ids, w, counts, offsets, src, row, scratch, nullptr, nullptr, 0};
    e = launch_route(logits, T, E, k, b, stream);
    if (e != cudaSuccess) return noalloc_fail(QMM_ERR_CUDA, "launch: ", cudaGetErrorString(e));
    return QMM_OK;
}
