// C ABI (include/qmm.h): argument checks, tensor-map encoding, workspace
// layout and the launch sequence of each entry point.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/qmm.h"
#include "ptx.cuh"
#include "qmm_internal.h"

namespace qmm {

__device__ uint32_t g_qmm_err;   // device error word (first kernel-side failure code)

namespace {

thread_local std::string t_last_error;

qmm_status fail(qmm_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

qmm_status cuda_fail(cudaError_t e, const char* what) {
    return fail(QMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    bool profile = false;
    long calls = 0;                                   // profiled calls since profiling was enabled
    int slot = 0;                                     // ring slot of the call being recorded
    bool slot_ready[QMM_PROFILE_RING] = {};
    cudaEvent_t ev[QMM_PROFILE_RING][QMM_PROFILE_PHASES + 1];
    qmm_status status = QMM_OK;
    std::string why;
    int sms = 0;
    uint32_t* err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

// Per-device one-time set-up: architecture check, SM count, error word address.
qmm_status device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(QMM_ERR_UNSUPPORTED_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (major != 10 || minor != 3) {
            d.status = QMM_ERR_UNSUPPORTED_DEVICE;
            char buf[128];
            snprintf(buf, sizeof buf, "compute capability %d.%d; this library is built for sm_103a only", major,
                     minor);
            d.why = buf;
        } else {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_qmm_err);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
            d.err = static_cast<uint32_t*>(p);
            e = cudaMemset(d.err, 0, sizeof(uint32_t));
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
            if (!g_encode) {
                cudaDriverEntryPointQueryResult q;
                void* fn = nullptr;
                e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
                if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                    return fail(QMM_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
            }
        }
        d.ready = true;
    }
    if (d.status != QMM_OK) return fail(d.status, "%s", d.why.c_str());
    *out = &d;
    return QMM_OK;
}

// The dense GEMMs' K-split scratch: the caller's workspace (none: no splits).
static qmm_status split_workspace(const char* who, void* ws, size_t ws_bytes, GemmParams* p) {
    p->split_part = nullptr;
    p->split_part_cap = 0;
    if (!ws || ws_bytes == 0) return QMM_OK;
    if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return fail(QMM_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
    p->split_part = static_cast<float*>(ws);
    p->split_part_cap = (long)(ws_bytes / sizeof(float));
    return QMM_OK;
}

// 2-D tiled tensor map over a row-major [outer][inner] matrix.
qmm_status make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(QMM_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu map", (int)r,
                    (unsigned long long)outer, (unsigned long long)inner);
    return QMM_OK;
}

// Record phase boundary i of a profiled expert-stage call, into the ring slot of
// this call (the last QMM_PROFILE_RING calls stay readable without a host sync
// in between).
cudaError_t mark(DeviceState* d, int i, cudaStream_t s) {
    if (!d->profile) return cudaSuccess;
    if (i == 0) {
        d->slot = (int)(d->calls % QMM_PROFILE_RING);
        if (!d->slot_ready[d->slot]) {
            for (int j = 0; j <= QMM_PROFILE_PHASES; ++j) {
                cudaError_t e = cudaEventCreate(&d->ev[d->slot][j]);
                if (e != cudaSuccess) return e;
            }
            d->slot_ready[d->slot] = true;
        }
    }
    cudaError_t e = cudaEventRecord(d->ev[d->slot][i], s);
    if (i == QMM_PROFILE_PHASES) ++d->calls;
    return e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int route_chunks(int T) { return (T + kRouteChunk - 1) / kRouteChunk; }
int max_tile_entries(int T, int E, int k) { return (int)(((long)T * k + 127) / 128) + E; }
int max_tile_entries256(int T, int E, int k) { return (int)(((long)T * k + 255) / 256) + E; }

// Workspace regions of the expert stage, in the order of the QMM_WS_FIELDS list.
void stage_layout(int T, int D, int F, int E, int k, size_t* off) {
    const size_t P = (size_t)T * k;
    size_t sz[QMM_WS_FIELDS - 1] = {
        P * 4,                                      // ids
        P * 4,                                      // w
        (size_t)E * 4,                              // counts
        (size_t)(E + 1) * 4,                        // offsets
        P * 4,                                      // src
        P * 4,                                      // row
        (size_t)route_chunks(T) * E * 4,            // chunk counts
        (size_t)max_tile_entries(T, E, k) * 16,     // tile list, 128-row entries
        16,                                         // tile count
        (size_t)max_tile_entries256(T, E, k) * 16,  // tile list, 256-row entries
        16,                                         // tile count
        P * D * 2,                                  // X_perm
        P * F * 2,                                  // Hq (f16 codes)
        P * (F / 32) * 2,                           // Hd
        P * (F / 32) * 2,                           // Hs
        (size_t)max_tile_entries(T, E, k) * (F / 32) * 128 * 4,   // Hd32: fp32 d per tile entry
        P * D * 4,                                  // Yslot
        P * 4,                                      // wrow: routing weight per routed row
    };
    size_t o = 0;
    for (int i = 0; i < QMM_WS_FIELDS - 1; ++i) {
        off[i] = o;
        o = align_up(o + sz[i], 256);
    }
    off[QMM_WS_FIELDS - 1] = o;
}

}  // namespace

void set_last_error(const char* msg) { t_last_error = msg; }

}  // namespace qmm

using namespace qmm;

extern "C" {

const char* qmm_last_error(void) { return t_last_error.c_str(); }

qmm_status qmm_check_status(cudaStream_t stream) {
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t code = 0;
    e = cudaMemcpy(&code, d->err, sizeof code, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (code != 0) {
        cudaMemset(d->err, 0, sizeof code);
        if (code == DEV_BAD_OFFSETS)
            return fail(QMM_ERR_INVALID_ARG, "expert offsets must satisfy 0 = o[0] <= ... <= o[E] = P (device check)");
        if (code == DEV_BAD_ROW) return fail(QMM_ERR_INVALID_ARG, "combine row index outside [0, P) (device check)");
        return fail(QMM_ERR_TIMEOUT, "a kernel wait timed out (device code %u)", code);
    }
    return QMM_OK;
}

size_t qmm_dense_workspace_size(int M, int K, int N) {
    // partial tiles of at most 256 x 256 fp32 for at most one work item per SM
    if (M < 1 || N < 1 || K < 256 || K % 256) return 0;
    DeviceState* d = nullptr;
    if (device_state(&d) != QMM_OK) return 0;
    return sizeof(float) * 65536 * (size_t)d->sms;
}

qmm_status qmm_w4a16(const uint16_t* X, int M, int K, int N, const uint8_t* Wc, const uint8_t* Ws, float scale2,
                     void* Y, qmm_dtype ydt, cudaStream_t stream) {
    return qmm_w4a16_ws(X, M, K, N, Wc, Ws, scale2, Y, ydt, nullptr, 0, stream);
}

qmm_status qmm_w4a16_ws(const uint16_t* X, int M, int K, int N, const uint8_t* Wc, const uint8_t* Ws, float scale2,
                        void* Y, qmm_dtype ydt, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!X || !Wc || !Ws || !Y) return fail(QMM_ERR_INVALID_ARG, "qmm_w4a16: null pointer");
    if (!aligned16(X) || !aligned16(Wc) || !aligned16(Ws) || !aligned16(Y))
        return fail(QMM_ERR_INVALID_ARG, "qmm_w4a16: buffers must be 16-byte aligned");
    if (ydt != QMM_F32 && ydt != QMM_BF16) return fail(QMM_ERR_INVALID_ARG, "qmm_w4a16: bad output type");
    if (M < 1 || K < 32 || N < 32 || K % 32 || N % 32)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE, "qmm_w4a16: need M >= 1, K %% 32 == 0, N %% 32 == 0 (M=%d K=%d N=%d)",
                    M, K, N);
    GemmParams p{};
    qmm_status st = split_workspace("qmm_w4a16", ws, ws_bytes, &p);
    if (st != QMM_OK) return st;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != QMM_OK) return st;
    // sh.rows x sh.bn tiles; clusters of cn CTAs share the activation rows
    const TileShape sh = w4_dense_shape(M, N, d->sms);
    const int n_tiles = (N + sh.bn - 1) / sh.bn;
    const int cn = cluster_for(n_tiles);
    CUtensorMap ta, tb;
    if ((st = make_tmap(&ta, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, (uint64_t)K * 2, 64, sh.rows / cn,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != QMM_OK)
        return st;
    if ((st = make_tmap(&tb, Wc, CU_TENSOR_MAP_DATA_TYPE_UINT8, K / 2, N, K / 2, 32, sh.bn,
                        CU_TENSOR_MAP_SWIZZLE_32B)) != QMM_OK)
        return st;
    p.M = M;
    p.N = N;
    p.K = K;
    p.m_tiles = (M + sh.rows - 1) / sh.rows;
    p.n_tiles = n_tiles;
    p.n_step = sh.bn;
    p.w_scale = Ws;
    p.scale2_dense = scale2;
    p.Y = Y;
    p.ydt = (ydt == QMM_BF16) ? 1 : 0;
    p.ldy = N;
    p.err = d->err;
    cudaError_t e = launch_w4a16_dense(ta, tb, p, cn, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_w4a16 launch");
    return QMM_OK;
}

qmm_status qmm_fp8_blk128(const uint16_t* X, int M, int K, int N, const uint8_t* W, const float* S, uint16_t* Y,
                          cudaStream_t stream) {
    return qmm_fp8_blk128_ws(X, M, K, N, W, S, Y, nullptr, 0, stream);
}

qmm_status qmm_fp8_blk128_ws(const uint16_t* X, int M, int K, int N, const uint8_t* W, const float* S, uint16_t* Y,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!X || !W || !S || !Y) return fail(QMM_ERR_INVALID_ARG, "qmm_fp8_blk128: null pointer");
    if (!aligned16(X) || !aligned16(W) || !aligned16(S) || !aligned16(Y))
        return fail(QMM_ERR_INVALID_ARG, "qmm_fp8_blk128: buffers must be 16-byte aligned");
    if (M < 1 || K < 128 || N < 128 || K % 128 || N % 128)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE,
                    "qmm_fp8_blk128: need M >= 1, K %% 128 == 0, N %% 128 == 0 (M=%d K=%d N=%d)", M, K, N);
    GemmParams p{};
    qmm_status st = split_workspace("qmm_fp8_blk128", ws, ws_bytes, &p);
    if (st != QMM_OK) return st;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != QMM_OK) return st;
    const int cn = cluster_for(N / 128);
    CUtensorMap ta, tb;
    const int bm = fp8_tile_rows();
    if ((st = make_tmap(&ta, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, (uint64_t)K * 2, 64, bm / cn,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != QMM_OK)
        return st;
    if ((st = make_tmap(&tb, W, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)) != QMM_OK)
        return st;
    p.M = M;
    p.N = N;
    p.K = K;
    p.m_tiles = (M + bm - 1) / bm;
    p.n_tiles = N / 128;
    p.n_step = 128;
    p.blk_scale = S;
    p.Y = Y;
    p.ydt = 1;
    p.ldy = N;
    p.err = d->err;
    cudaError_t e = launch_fp8_blk128(ta, tb, p, cn, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_fp8_blk128 launch");
    return QMM_OK;
}

// ---------------------------------------------------------------- dense Q8_0 x q8_1

// Workspace of qmm_q8_0_q8_1: f16 activation codes [M][K], the activations' d per
// 128-row tile [entries][K/32][128] fp32, the tile list and its count, and the
// weight codes as f16 [N][K] (the kernel reads both operands expanded).
static void q8_layout(int M, int K, int N, size_t* off) {
    const int entries = (M + 127) / 128;
    const size_t sz[5] = {(size_t)M * K * 2, (size_t)entries * (K / 32) * 128 * 4, (size_t)entries * 16, 16,
                          q8_weights_f16() ? (size_t)N * K * 2 : 0};
    size_t o = 0;
    for (int i = 0; i < 5; ++i) {
        off[i] = o;
        o = align_up(o + sz[i], 256);
    }
    off[5] = o;
}

size_t qmm_q8_0_q8_1_workspace_size(int M, int K, int N) {
    if (M < 1 || K < 256 || K % 256 || N < 128 || N % 128) return 0;
    size_t off[6];
    q8_layout(M, K, N, off);
    return off[5];
}

qmm_status qmm_q8_0_q8_1(const int8_t* Xq, const uint16_t* Xd, int M, int K, int N, const int8_t* Wq,
                         const uint16_t* Wd, int8_t* Yq, uint16_t* Yd, uint16_t* Ys, float* Y, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
    if (M < 1 || K < 256 || K % 256 || N < 128 || N % 128)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE, "qmm_q8_0_q8_1: need M >= 1, K %% 256 == 0, N %% 128 == 0 (M=%d K=%d N=%d)",
                    M, K, N);
    if (!Xq || !Xd || !Wq || !Wd || !Yq || !Yd || !Ys || !ws)
        return fail(QMM_ERR_INVALID_ARG, "qmm_q8_0_q8_1: null pointer");
    if (!aligned16(Xq) || !aligned16(Xd) || !aligned16(Wq) || !aligned16(Wd) || !aligned16(Yq) || !aligned16(Yd) ||
        !aligned16(Ys) || (Y && !aligned16(Y)) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return fail(QMM_ERR_INVALID_ARG, "qmm_q8_0_q8_1: buffers must be 16-byte aligned (workspace 256-byte aligned)");
    const size_t need = qmm_q8_0_q8_1_workspace_size(M, K, N);
    if (ws_bytes < need) return fail(QMM_ERR_WORKSPACE, "qmm_q8_0_q8_1: workspace %zu < %zu bytes", ws_bytes, need);
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    size_t off[6];
    q8_layout(M, K, N, off);
    uint8_t* base = static_cast<uint8_t*>(ws);
    __half* X16 = reinterpret_cast<__half*>(base + off[0]);
    float* dX32 = reinterpret_cast<float*>(base + off[1]);
    int4* tiles = reinterpret_cast<int4*>(base + off[2]);
    int32_t* count = reinterpret_cast<int32_t*>(base + off[3]);
    __half* W16 = reinterpret_cast<__half*>(base + off[4]);
    const int entries = (M + 127) / 128;
    const bool wf16 = q8_weights_f16();
    cudaError_t e = launch_dense_tiles(M, tiles, count, stream);
    if (e == cudaSuccess) e = launch_codes_i8_to_f16(Xq, X16, (long)M * K, stream);
    if (e == cudaSuccess && wf16) e = launch_codes_i8_to_f16(Wq, W16, (long)N * K, stream);
    if (e == cudaSuccess)
        e = launch_hd_to_entries(reinterpret_cast<const __half*>(Xd), tiles, count, entries, K / 32, dX32, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_q8_0_q8_1: operand layout");
    CUtensorMap ta, tb, tw;
    if ((st = wf16 ? make_tmap(&ta, W16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, N, (uint64_t)K * 2, 64, 128,
                               CU_TENSOR_MAP_SWIZZLE_128B)
                    : make_tmap(&ta, Wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)) !=
        QMM_OK)
        return st;
    if ((st = make_tmap(&tb, X16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, M, (uint64_t)K * 2, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != QMM_OK)
        return st;
    if ((st = make_tmap(&tw, Wd, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K / 32, N, K / 16, 8, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != QMM_OK)
        return st;
    GemmParams p{};
    p.N = N;
    p.K = K;
    p.n_tiles = N / 128;
    p.n_step = 128;
    p.tiles = tiles;
    p.num_entries = count;
    p.max_entries = entries;
    p.dH32 = dX32;
    p.err = d->err;
    e = launch_q8_dense(ta, tb, tw, p, Yq, reinterpret_cast<__half*>(Yd), reinterpret_cast<__half*>(Ys), Y, M, d->sms,
                        stream);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_q8_0_q8_1 launch");
    return QMM_OK;
}

size_t moe_route_workspace_size(int T, int E, int k) {
    (void)k;
    if (T < 0 || E < 1) return 0;
    return align_up((size_t)route_chunks(T) * E * 4, 256);
}

static qmm_status check_route_shape(const char* who, int T, int E, int k) {
    if (T < 0 || k < 1 || k > 16 || E < k || E > 512)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE, "%s: need T >= 0, 1 <= k <= 16, k <= E <= 512 (T=%d E=%d k=%d)", who,
                    T, E, k);
    return QMM_OK;
}

qmm_status moe_route_permute(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                             int32_t* offsets, int32_t* src, int32_t* row, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
    qmm_status st = check_route_shape("moe_route_permute", T, E, k);
    if (st != QMM_OK) return st;
    if (!counts || !offsets || (T > 0 && (!logits || !ids || !w || !src || !row || !ws)))
        return fail(QMM_ERR_INVALID_ARG, "moe_route_permute: null pointer");
    if (ws_bytes < moe_route_workspace_size(T, E, k))
        return fail(QMM_ERR_WORKSPACE, "moe_route_permute: workspace %zu < %zu bytes", ws_bytes,
                    moe_route_workspace_size(T, E, k));
    DeviceState* d = nullptr;
    if ((st = device_state(&d)) != QMM_OK) return st;
    cudaError_t e;
    if (T == 0) {
        if ((e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream)) != cudaSuccess)
            return cuda_fail(e, "moe_route_permute");
        return QMM_OK;
    }
    RouteBufs b{ids, w, counts, offsets, src, row, static_cast<int32_t*>(ws), nullptr, nullptr, 0};
    e = launch_route(logits, T, E, k, b, stream);
    if (e != cudaSuccess) return cuda_fail(e, "moe_route_permute launch");
    return QMM_OK;
}

// Gate/up + SwiGLU + q8_1 over permuted rows Xp [P][D], grouped by the 256-row
// tile list: 256 token rows x (64 gate + 64 up weight rows) per tile, clusters
// of CTAs sharing the token rows.  Writes Hq (f16 codes), Hd, Hs, Hd32.
// Pointer-table form of the expert weights (moe_expert_table_build): E tensor
// maps of the gate/up codes, E of the down indices, then the E gate/up scale and
// E down scale pointers.
struct TableView {
    const CUtensorMap* gu_maps;
    const CUtensorMap* dn_maps;
    const uint8_t* const* gu_scales;
    const __half* const* dn_scales;
};
static size_t table_bytes(int E) { return align_up((size_t)E * (2 * sizeof(CUtensorMap) + 2 * sizeof(void*)), 256); }
static TableView table_view(const void* table, int E) {
    const uint8_t* b = static_cast<const uint8_t*>(table);
    TableView v;
    v.gu_maps = reinterpret_cast<const CUtensorMap*>(b);
    v.dn_maps = v.gu_maps + E;
    v.gu_scales = reinterpret_cast<const uint8_t* const*>(b + (size_t)2 * E * sizeof(CUtensorMap));
    v.dn_scales = reinterpret_cast<const __half* const*>(v.gu_scales + E);
    return v;
}

static qmm_status run_gate_up(DeviceState* d, const uint16_t* Xp, int P, int D, int F, int E, const uint8_t* Wgu_c,
                              const uint8_t* Wgu_s, const TableView* tab, const float* gu_scale2, const RouteBufs& rb,
                              __half* Hq, __half* Hd, __half* Hs, float* Hd32, cudaStream_t stream) {
    qmm_status st;
    // sh.rows token rows x (sh.bn / 2 gate + sh.bn / 2 up) weight rows per tile
    const TileShape sh = w4_gate_up_shape();
    const int hstep = sh.bn / 2;
    if (F % hstep) return fail(QMM_ERR_UNSUPPORTED_SHAPE, "expert stage: F %% %d != 0 (F=%d)", hstep, F);
    const int gu_cn = gate_up_cluster(F / hstep);
    CUtensorMap ta, tb;
    if ((st = make_tmap(&ta, Xp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, P, (uint64_t)D * 2, 64, sh.rows / gu_cn,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != QMM_OK)
        return st;
    if (tab) {
        memset(&tb, 0, sizeof tb);   // not read: every expert has its own map in the table
    } else if ((st = make_tmap(&tb, Wgu_c, CU_TENSOR_MAP_DATA_TYPE_UINT8, D / 2, (uint64_t)E * 2 * F, D / 2, 32,
                               hstep, CU_TENSOR_MAP_SWIZZLE_32B)) != QMM_OK) {
        return st;
    }
    GemmParams g{};
    if (tab) {
        g.wmaps = tab->gu_maps;
        g.wscale_tab = tab->gu_scales;
    }
    g.K = D;
    g.F = F;
    g.n_tiles = F / hstep;
    g.n_step = hstep;
    g.tiles = sh.rows == 256 ? rb.tiles2 : rb.tiles;
    g.num_entries = sh.rows == 256 ? rb.num_entries2 : rb.num_entries;
    g.max_entries = sh.rows == 256 ? rb.max_entries2 : rb.max_entries;
    g.w_scale = Wgu_s;
    g.scale2 = gu_scale2;
    g.Hq = Hq;
    g.Hd = Hd;
    g.Hs = Hs;
    g.Hd32 = Hd32;
    g.err = d->err;
    cudaError_t e = launch_w4_gate_up_swiglu(ta, tb, g, gu_cn, stream);
    if (e != cudaSuccess) return cuda_fail(e, "expert stage: gate/up launch");
    return QMM_OK;
}

// Down product over IQ4_NL weights x q8_1 H (f16 codes Hq, fp32 d in the
// per-128-row-entry layout Hd32), grouped by the 128-row tile list.  Without a
// combine: Yslot [P][D] per routed row.  With one (src, wrow given): the weighted
// combine is fused in, Y [T][D] += wrow[r] * y_r at token src[r] (Y zeroed first).
static qmm_status run_down(DeviceState* d, const __half* Hq, const float* Hd32, int P, int D, int F, int E,
                           const uint8_t* Wd_idx, const uint16_t* Wd_s, const TableView* tab, const int4* tiles,
                           const int32_t* num_entries, int max_entries, float* out, const int32_t* src,
                           const float* wrow, cudaStream_t stream) {
    qmm_status st;
    CUtensorMap ta, tb;
    if (tab) {
        memset(&ta, 0, sizeof ta);   // not read: every expert has its own map in the table
    } else if ((st = make_tmap(&ta, Wd_idx, CU_TENSOR_MAP_DATA_TYPE_UINT8, F / 2, (uint64_t)E * D, F / 2, 32, 128,
                               CU_TENSOR_MAP_SWIZZLE_32B)) != QMM_OK) {
        return st;
    }
    if ((st = make_tmap(&tb, Hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, F, P, (uint64_t)F * 2, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != QMM_OK)
        return st;
    GemmParams q{};
    q.N = D;
    q.K = F;
    q.n_tiles = D / 128;
    q.n_step = 128;
    q.tiles = tiles;
    q.num_entries = num_entries;
    q.max_entries = max_entries;
    q.dH32 = Hd32;
    q.dW = reinterpret_cast<const __half*>(Wd_s);
    if (tab) {
        q.wmaps = tab->dn_maps;
        q.dW_tab = tab->dn_scales;
    }
    q.src = src;
    q.wrow = wrow;
    q.Y = out;
    q.ydt = 0;
    q.ldy = D;
    q.err = d->err;
    cudaError_t e = launch_iq4_down(ta, tb, q, d->sms, src != nullptr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "expert stage: down launch");
    return QMM_OK;
}

static qmm_status check_stage_shape(int T, int D, int F, int E, int k) {
    qmm_status st = check_route_shape("moe_expert_stage_w4_iq4", T, E, k);
    if (st != QMM_OK) return st;
    if (D < 128 || D % 128 || F < 128 || F % 128 || F > 1024)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE,
                    "moe_expert_stage_w4_iq4: need D %% 128 == 0, F %% 128 == 0, F <= 1024 (D=%d F=%d)", D, F);
    return QMM_OK;
}

size_t moe_expert_stage_workspace_size(int T, int D, int F, int E, int k) {
    if (T < 0 || D < 0 || F < 32 || E < 1 || k < 1) return 0;
    size_t off[QMM_WS_FIELDS];
    stage_layout(T, D, F, E, k, off);
    return off[QMM_WS_FIELDS - 1];
}

qmm_status moe_expert_stage_workspace_layout(int T, int D, int F, int E, int k, size_t* offsets_out) {
    if (!offsets_out) return fail(QMM_ERR_INVALID_ARG, "moe_expert_stage_workspace_layout: null pointer");
    qmm_status st = check_stage_shape(T, D, F, E, k);
    if (st != QMM_OK) return st;
    stage_layout(T, D, F, E, k, offsets_out);
    return QMM_OK;
}

static qmm_status expert_stage(const uint16_t* X, const float* logits, int T, int D, int F, int E, int k,
                               const uint8_t* Wgu_c, const uint8_t* Wgu_s, const float* gu_scale2, const uint8_t* Wd_idx,
                               const uint16_t* Wd_s, const TableView* tab, float* Y, void* ws, size_t ws_bytes,
                               unsigned flags, cudaStream_t stream);

qmm_status moe_expert_stage_w4_iq4(const uint16_t* X, const float* logits, int T, int D, int F, int E, int k,
                                   const uint8_t* Wgu_c, const uint8_t* Wgu_s, const float* gu_scale2,
                                   const uint8_t* Wd_idx, const uint16_t* Wd_s, float* Y, void* ws, size_t ws_bytes,
                                   cudaStream_t stream) {
    return expert_stage(X, logits, T, D, F, E, k, Wgu_c, Wgu_s, gu_scale2, Wd_idx, Wd_s, nullptr, Y, ws, ws_bytes, 0u,
                        stream);
}

// The expert stage over contiguous [E][...] weights (tab == nullptr) or over a
// pointer table of per-expert weights.
static qmm_status expert_stage(const uint16_t* X, const float* logits, int T, int D, int F, int E, int k,
                               const uint8_t* Wgu_c, const uint8_t* Wgu_s, const float* gu_scale2, const uint8_t* Wd_idx,
                               const uint16_t* Wd_s, const TableView* tab, float* Y, void* ws, size_t ws_bytes,
                               unsigned flags, cudaStream_t stream) {
    qmm_status st = check_stage_shape(T, D, F, E, k);
    if (st != QMM_OK) return st;
    if (flags & ~(unsigned)QMM_STAGE_SLOTS) return fail(QMM_ERR_INVALID_ARG, "moe_expert_stage_w4_iq4_ex: unknown flags");
    if (!gu_scale2 || (!tab && (!Wgu_c || !Wgu_s || !Wd_idx || !Wd_s)) || (T > 0 && (!X || !logits || !Y || !ws)))
        return fail(QMM_ERR_INVALID_ARG, "moe_expert_stage_w4_iq4: null pointer");
    if (!aligned16(X) || !aligned16(logits) || !aligned16(Wgu_c) || !aligned16(Wgu_s) || !aligned16(Wd_idx) ||
        !aligned16(Wd_s) || !aligned16(Y) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return fail(QMM_ERR_INVALID_ARG,
                    "moe_expert_stage_w4_iq4: buffers must be 16-byte aligned (workspace 256-byte aligned)");
    const size_t need = moe_expert_stage_workspace_size(T, D, F, E, k);
    if (ws_bytes < need) return fail(QMM_ERR_WORKSPACE, "moe_expert_stage_w4_iq4: workspace %zu < %zu bytes", ws_bytes, need);
    DeviceState* d = nullptr;
    if ((st = device_state(&d)) != QMM_OK) return st;
    if (T == 0) return QMM_OK;
    const bool slots = (flags & QMM_STAGE_SLOTS) != 0;

    size_t off[QMM_WS_FIELDS];
    stage_layout(T, D, F, E, k, off);
    uint8_t* base = static_cast<uint8_t*>(ws);
    auto at = [&](int i) { return static_cast<void*>(base + off[i]); };
    const int P = T * k;
    const int max_entries = max_tile_entries(T, E, k);

    cudaError_t e;
    if ((e = mark(d, 0, stream)) != cudaSuccess) return cuda_fail(e, "profiling event");
    const int max_entries2 = max_tile_entries256(T, E, k);
    RouteBufs rb{static_cast<int32_t*>(at(0)), static_cast<float*>(at(1)), static_cast<int32_t*>(at(2)),
                 static_cast<int32_t*>(at(3)), static_cast<int32_t*>(at(4)), static_cast<int32_t*>(at(5)),
                 static_cast<int32_t*>(at(6)), static_cast<int4*>(at(7)), static_cast<int32_t*>(at(8)),
                 max_entries, static_cast<int4*>(at(9)), static_cast<int32_t*>(at(10)), max_entries2};
    float* wrow = static_cast<float*>(at(17));
    if (!slots) {
        // the fused combine accumulates into Y: the top-k kernel zeroes it, the
        // permutation records each routed row's weight
        rb.wrow = wrow;
        rb.yzero = Y;
        rb.yzero_D = D;
    }
    e = launch_route(logits, T, E, k, rb, stream);
    if (e != cudaSuccess) return cuda_fail(e, "expert stage: routing");
    if ((e = mark(d, 1, stream)) != cudaSuccess) return cuda_fail(e, "profiling event");
    uint16_t* Xp = static_cast<uint16_t*>(at(11));
    e = launch_gather_rows(X, rb.src, P, D, Xp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "expert stage: gather");
    if ((e = mark(d, 2, stream)) != cudaSuccess) return cuda_fail(e, "profiling event");

    __half* Hq = static_cast<__half*>(at(12));
    __half* Hd = static_cast<__half*>(at(13));
    __half* Hs = static_cast<__half*>(at(14));
    float* Hd32 = static_cast<float*>(at(15));
    float* Yslot = static_cast<float*>(at(16));

    // gate/up + SwiGLU + q8_1
    if ((st = run_gate_up(d, Xp, P, D, F, E, Wgu_c, Wgu_s, tab, gu_scale2, rb, Hq, Hd, Hs, Hd32, stream)) != QMM_OK)
        return st;
    if ((e = mark(d, 3, stream)) != cudaSuccess) return cuda_fail(e, "profiling event");

    // down (IQ4_NL weights on the MMA's M side, q8_1 H codes on its N side), with the
    // weighted combine fused in, or to per-slot rows followed by the combine kernel
    if ((st = run_down(d, Hq, Hd32, P, D, F, E, Wd_idx, Wd_s, tab, rb.tiles, rb.num_entries, max_entries,
                       slots ? Yslot : Y, slots ? nullptr : rb.src, slots ? nullptr : wrow, stream)) != QMM_OK)
        return st;
    if ((e = mark(d, 4, stream)) != cudaSuccess) return cuda_fail(e, "profiling event");

    if (slots) {
        e = launch_combine(Yslot, P, rb.row, rb.w, T, k, D, Y, d->err, stream);
        if (e != cudaSuccess) return cuda_fail(e, "expert stage: combine");
    }
    if ((e = mark(d, 5, stream)) != cudaSuccess) return cuda_fail(e, "profiling event");
    return QMM_OK;
}

qmm_status moe_expert_stage_w4_iq4_ex(const uint16_t* X, const float* logits, int T, int D, int F, int E, int k,
                                      const uint8_t* Wgu_c, const uint8_t* Wgu_s, const float* gu_scale2,
                                      const uint8_t* Wd_idx, const uint16_t* Wd_s, float* Y, void* ws, size_t ws_bytes,
                                      unsigned flags, cudaStream_t stream) {
    return expert_stage(X, logits, T, D, F, E, k, Wgu_c, Wgu_s, gu_scale2, Wd_idx, Wd_s, nullptr, Y, ws, ws_bytes, flags,
                        stream);
}

// ---------------------------------------------------------------- per-expert pointer tables

size_t moe_expert_table_size(int E) {
    if (E < 1 || E > 512) return 0;
    return table_bytes(E);
}

qmm_status moe_expert_table_build(int D, int F, int E, const uint8_t* const* Wgu_c, const uint8_t* const* Wgu_s,
                                  const uint8_t* const* Wd_idx, const uint16_t* const* Wd_s, void* table,
                                  size_t table_size, cudaStream_t stream) {
    if (E < 1 || E > 512 || D < 128 || D % 128 || F < 128 || F % 128 || F > 1024)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE,
                    "moe_expert_table_build: need 1 <= E <= 512, D %% 128 == 0, F %% 128 == 0, F <= 1024");
    if (!Wgu_c || !Wgu_s || !Wd_idx || !Wd_s || !table)
        return fail(QMM_ERR_INVALID_ARG, "moe_expert_table_build: null pointer");
    if (reinterpret_cast<uintptr_t>(table) & 255u)
        return fail(QMM_ERR_INVALID_ARG, "moe_expert_table_build: table must be 256-byte aligned");
    if (table_size < table_bytes(E))
        return fail(QMM_ERR_WORKSPACE, "moe_expert_table_build: table %zu < %zu bytes", table_size, table_bytes(E));
    for (int e = 0; e < E; ++e) {
        if (!Wgu_c[e] || !Wgu_s[e] || !Wd_idx[e] || !Wd_s[e])
            return fail(QMM_ERR_INVALID_ARG, "moe_expert_table_build: null pointer for expert %d", e);
        if (!aligned16(Wgu_c[e]) || !aligned16(Wgu_s[e]) || !aligned16(Wd_idx[e]) || !aligned16(Wd_s[e]))
            return fail(QMM_ERR_INVALID_ARG, "moe_expert_table_build: expert %d's buffers must be 16-byte aligned", e);
    }
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    // the table on the host, then one copy into the caller's device buffer
    std::vector<uint8_t> host(table_bytes(E), 0);
    CUtensorMap* gu = reinterpret_cast<CUtensorMap*>(host.data());
    CUtensorMap* dn = gu + E;
    const void** gus = reinterpret_cast<const void**>(host.data() + (size_t)2 * E * sizeof(CUtensorMap));
    const void** dns = gus + E;
    const int hstep = w4_gate_up_shape().bn / 2;
    for (int e = 0; e < E; ++e) {
        // the expert's gate/up codes [2F][D/2] and down indices [D][F/2], boxes as in the
        // contiguous form
        if ((st = make_tmap(&gu[e], Wgu_c[e], CU_TENSOR_MAP_DATA_TYPE_UINT8, D / 2, (uint64_t)2 * F, D / 2, 32, hstep,
                            CU_TENSOR_MAP_SWIZZLE_32B)) != QMM_OK)
            return st;
        if ((st = make_tmap(&dn[e], Wd_idx[e], CU_TENSOR_MAP_DATA_TYPE_UINT8, F / 2, (uint64_t)D, F / 2, 32, 128,
                            CU_TENSOR_MAP_SWIZZLE_32B)) != QMM_OK)
            return st;
        gus[e] = Wgu_s[e];
        dns[e] = Wd_s[e];
    }
    cudaError_t e = cudaMemcpyAsync(table, host.data(), host.size(), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "moe_expert_table_build: copy");
    return QMM_OK;
}

qmm_status moe_expert_stage_w4_iq4_table(const uint16_t* X, const float* logits, int T, int D, int F, int E, int k,
                                         const float* gu_scale2, const void* table, float* Y, void* ws,
                                         size_t ws_bytes, unsigned flags, cudaStream_t stream) {
    if (!table || (reinterpret_cast<uintptr_t>(table) & 255u))
        return fail(QMM_ERR_INVALID_ARG, "moe_expert_stage_w4_iq4_table: table null or not 256-byte aligned");
    const TableView tab = table_view(table, E);
    return expert_stage(X, logits, T, D, F, E, k, nullptr, nullptr, gu_scale2, nullptr, nullptr, &tab, Y, ws, ws_bytes,
                        flags, stream);
}

// ---------------------------------------------------------------- sub-step entry points

// Workspace of the qmm_dbg_* calls: 128-row tile list + count, 256-row tile list
// + count, f16 H codes [P][F], fp32 d of H per 128-row entry.
static void dbg_layout(int P, int F, int E, size_t* off) {
    const int me = (P + 127) / 128 + E, me2 = (P + 255) / 256 + E;
    const size_t sz[6] = {(size_t)me * 16, 16, (size_t)me2 * 16, 16, (size_t)P * F * 2,
                          (size_t)me * (F / 32) * 128 * 4};
    size_t o = 0;
    for (int i = 0; i < 6; ++i) {
        off[i] = o;
        o = align_up(o + sz[i], 256);
    }
    off[6] = o;
}

size_t qmm_dbg_workspace_size(int P, int D, int F, int E) {
    if (P < 0 || D < 0 || F < 32 || E < 1) return 0;
    size_t off[7];
    dbg_layout(P, F, E, off);
    return off[6];
}

static qmm_status dbg_common(const char* who, int P, int D, int F, int E, const void* const* bufs, int nbufs,
                             void* ws, size_t ws_bytes, DeviceState** d) {
    if (P < 0 || E < 1 || E > 512 || D < 128 || D % 128 || F < 128 || F % 128 || F > 1024)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE, "%s: need P >= 0, 1 <= E <= 512, D %% 128 == 0, F %% 128 == 0, F <= 1024",
                    who);
    for (int i = 0; i < nbufs; ++i) {
        if (!bufs[i] && P > 0) return fail(QMM_ERR_INVALID_ARG, "%s: null pointer", who);
        if (!aligned16(bufs[i])) return fail(QMM_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", who);
    }
    if (P > 0 && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return fail(QMM_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
    const size_t need = qmm_dbg_workspace_size(P, D, F, E);
    if (ws_bytes < need) return fail(QMM_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", who, ws_bytes, need);
    return device_state(d);
}

// Tile lists from the caller's offsets into the dbg workspace.
static qmm_status dbg_tiles(DeviceState* d, const int32_t* offsets, int P, int E, uint8_t* base, const size_t* off,
                            RouteBufs* rb, cudaStream_t stream) {
    *rb = RouteBufs{};
    rb->tiles = reinterpret_cast<int4*>(base + off[0]);
    rb->num_entries = reinterpret_cast<int32_t*>(base + off[1]);
    rb->max_entries = (P + 127) / 128 + E;
    rb->tiles2 = reinterpret_cast<int4*>(base + off[2]);
    rb->num_entries2 = reinterpret_cast<int32_t*>(base + off[3]);
    rb->max_entries2 = (P + 255) / 256 + E;
    cudaError_t e = launch_tiles_from_offsets(offsets, E, P, d->err, *rb, stream);
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "tile lists from offsets");
}

qmm_status qmm_dbg_gate_up_q8_1(const uint16_t* X_perm, const int32_t* offsets, int P, int D, int F, int E,
                                const uint8_t* Wgu_c, const uint8_t* Wgu_s, const float* gu_scale2, int8_t* Hq,
                                uint16_t* Hd, uint16_t* Hs, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const void* bufs[] = {X_perm, offsets, Wgu_c, Wgu_s, gu_scale2, Hq, Hd, Hs};
    DeviceState* d = nullptr;
    qmm_status st = dbg_common("qmm_dbg_gate_up_q8_1", P, D, F, E, bufs, 8, ws, ws_bytes, &d);
    if (st != QMM_OK || P == 0) return st;
    size_t off[7];
    dbg_layout(P, F, E, off);
    uint8_t* base = static_cast<uint8_t*>(ws);
    RouteBufs rb;
    if ((st = dbg_tiles(d, offsets, P, E, base, off, &rb, stream)) != QMM_OK) return st;
    __half* Hq16 = reinterpret_cast<__half*>(base + off[4]);
    float* Hd32 = reinterpret_cast<float*>(base + off[5]);
    if ((st = run_gate_up(d, X_perm, P, D, F, E, Wgu_c, Wgu_s, nullptr, gu_scale2, rb, Hq16, reinterpret_cast<__half*>(Hd),
                          reinterpret_cast<__half*>(Hs), Hd32, stream)) != QMM_OK)
        return st;
    cudaError_t e = launch_codes_f16_to_i8(Hq16, Hq, (long)P * F, stream);
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "qmm_dbg_gate_up_q8_1: code conversion");
}

qmm_status qmm_dbg_down_iq4(const int8_t* Hq, const uint16_t* Hd, const int32_t* offsets, int P, int D, int F, int E,
                            const uint8_t* Wd_idx, const uint16_t* Wd_s, float* Yslot, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
    const void* bufs[] = {Hq, Hd, offsets, Wd_idx, Wd_s, Yslot};
    DeviceState* d = nullptr;
    qmm_status st = dbg_common("qmm_dbg_down_iq4", P, D, F, E, bufs, 6, ws, ws_bytes, &d);
    if (st != QMM_OK || P == 0) return st;
    size_t off[7];
    dbg_layout(P, F, E, off);
    uint8_t* base = static_cast<uint8_t*>(ws);
    RouteBufs rb;
    if ((st = dbg_tiles(d, offsets, P, E, base, off, &rb, stream)) != QMM_OK) return st;
    __half* Hq16 = reinterpret_cast<__half*>(base + off[4]);
    float* Hd32 = reinterpret_cast<float*>(base + off[5]);
    cudaError_t e = launch_codes_i8_to_f16(Hq, Hq16, (long)P * F, stream);
    if (e == cudaSuccess)
        e = launch_hd_to_entries(reinterpret_cast<const __half*>(Hd), rb.tiles, rb.num_entries, rb.max_entries, F / 32,
                                 Hd32, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_dbg_down_iq4: operand layout");
    return run_down(d, Hq16, Hd32, P, D, F, E, Wd_idx, Wd_s, nullptr, rb.tiles, rb.num_entries, rb.max_entries, Yslot,
                    nullptr, nullptr, stream);
}

qmm_status qmm_dbg_combine(const float* Yslot, int P, const int32_t* row, const float* w, int T, int k, int D,
                           float* Y, cudaStream_t stream) {
    if (T < 0 || P < 0 || k < 1 || k > 16 || D < 4 || D % 4)
        return fail(QMM_ERR_UNSUPPORTED_SHAPE, "qmm_dbg_combine: need T, P >= 0, 1 <= k <= 16, D %% 4 == 0");
    if (T > 0 && (!Yslot || !row || !w || !Y)) return fail(QMM_ERR_INVALID_ARG, "qmm_dbg_combine: null pointer");
    if (!aligned16(Yslot) || !aligned16(Y)) return fail(QMM_ERR_INVALID_ARG, "qmm_dbg_combine: Yslot, Y 16-byte aligned");
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK || T == 0) return st;
    cudaError_t e = launch_combine(Yslot, P, row, w, T, k, D, Y, d->err, stream);
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "qmm_dbg_combine launch");
}

qmm_status qmm_dbg_wait_timeout(unsigned timeout_us, cudaStream_t stream) {
    if (timeout_us < 1 || timeout_us > 2000000u)
        return fail(QMM_ERR_INVALID_ARG, "qmm_dbg_wait_timeout: need 1 <= timeout_us <= 2000000");
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    cudaError_t e = launch_wait_timeout_probe(d->err, (uint64_t)timeout_us * 1000u, stream);
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "qmm_dbg_wait_timeout launch");
}

qmm_status qmm_profile_enable(int on) {
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    if (on && !d->profile) d->calls = 0;
    d->profile = on != 0;
    return QMM_OK;
}

qmm_status qmm_profile_read_call(long i, float* ms_out) {
    if (!ms_out) return fail(QMM_ERR_INVALID_ARG, "qmm_profile_read_call: null pointer");
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    if (i < 0 || i >= d->calls || i < d->calls - QMM_PROFILE_RING)
        return fail(QMM_ERR_INVALID_ARG, "qmm_profile_read_call: call %ld is not among the last %d of %ld profiled calls",
                    i, QMM_PROFILE_RING, d->calls);
    cudaEvent_t* ev = d->ev[i % QMM_PROFILE_RING];
    cudaError_t e = cudaEventSynchronize(ev[QMM_PROFILE_PHASES]);
    if (e != cudaSuccess) return cuda_fail(e, "qmm_profile_read_call");
    for (int j = 0; j < QMM_PROFILE_PHASES; ++j) {
        e = cudaEventElapsedTime(&ms_out[j], ev[j], ev[j + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "qmm_profile_read_call");
    }
    return QMM_OK;
}

qmm_status qmm_profile_read(float* ms_out) {
    if (!ms_out) return fail(QMM_ERR_INVALID_ARG, "qmm_profile_read: null pointer");
    DeviceState* d = nullptr;
    qmm_status st = device_state(&d);
    if (st != QMM_OK) return st;
    if (d->calls == 0) return fail(QMM_ERR_INVALID_ARG, "qmm_profile_read: no profiled call yet");
    return qmm_profile_read_call(d->calls - 1, ms_out);
}

}  // extern "C"
