// Routed-MoE data movement: top-k routing with renormalised weights, per-expert
// grouping (histogram, prefix scan, stable permutation), the 128-row tile list
// the grouped GEMMs walk, the row gather of X, and the weighted combine.
//
// Routing follows "AMD_HIP.md", RDNA4 speed switches (router_top10: top-k ids
// and renormalised weights); grouping tokens per expert for grouped GEMMs over
// a 64/128-row M tile follows "perf: strix-hip BF16 GEMMs via hipBLASLt"
// (routed-MoE prefill twins, per-expert pointer tables and max_m_tiles).
//
// Grouping is deterministic: the pairs (t, j) of expert e take rows
// offsets[e] + 0, 1, ... in ascending token order (a token picks an expert at
// most once), computed with per-chunk counts and bit masks, never with atomic
// slot claims.
#include <cfloat>
#include <climits>

#include "ptx.cuh"
#include "qmm_internal.h"

namespace qmm {

constexpr int kMaxK = 16;

// One warp per token.  Lane l holds logits l, l+32, ...; k rounds of a warp
// arg-max (ties to the lower expert index) pick the experts in descending order.
// With yz, the warp also sets row t of yz [T][D] fp32 to zero (the output the
// down product then accumulates into, when the combine is fused into it).
template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ w,
                                                         float* __restrict__ yz, int D) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
        if (yz) {
            float4* row = reinterpret_cast<float4*>(yz + (long)t * D);
            for (int i = lane; i < D / 4; i += 32) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float v[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? __ldg(logits + (long)t * E + e) : -FLT_MAX;
        }
        uint32_t taken = 0;
        float vals[kMaxK];
        int sel[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                float bv = -FLT_MAX;
                int bi = -1;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !((taken >> i) & 1u) && (bi < 0 || v[i] > bv)) {
                        bv = v[i];
                        bi = e;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
                vals[j] = bv;
                sel[j] = bi;
            }
        }
        // w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k chosen experts
        float ex[kMaxK];
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                ex[j] = expf(vals[j] - vals[0]);
                den += ex[j];
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k && lane == j) {
                ids[(long)t * k + j] = sel[j];
                w[(long)t * k + j] = ex[j] / den;
            }
        }
    }
}

// Per chunk of kRouteChunk tokens: how many of its pairs chose each expert.
__global__ void __launch_bounds__(256) route_hist_kernel(const int32_t* __restrict__ ids, int T, int E, int k,
                                                         int32_t* __restrict__ chunk_hist) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const long p0 = (long)blockIdx.x * kRouteChunk * k;
    const long p1 = min((long)T * k, p0 + (long)kRouteChunk * k);
    for (long p = p0 + threadIdx.x; p < p1; p += blockDim.x) atomicAdd(&hist[ids[p]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(long)blockIdx.x * E + e] = hist[e];
}

// Exclusive block-wide scan of one int per thread (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* total) {
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        warp_sums[lane] = s;   // inclusive
    }
    __syncthreads();
    const int base = wid ? warp_sums[wid - 1] : 0;
    *total = warp_sums[31];
    __syncthreads();
    return base + x - v;
}

// Tile lists of the grouped GEMMs, for expert e = threadIdx.x with `cnt` rows
// starting at row `off` (every thread of the 1024-thread block calls this):
// 128-row entries {expert, first row, rows, 0} and 256-row entries
// {expert, first row, rows, index of its first 128-row entry}.
__device__ void build_tile_lists(int E, int cnt, int off, int4* __restrict__ tiles, int32_t* __restrict__ num_entries,
                                 int max_entries, int4* __restrict__ tiles2, int32_t* __restrict__ num_entries2,
                                 int max_entries2) {
    const int e = threadIdx.x;
    const int mt = (e < E) ? (cnt + 127) / 128 : 0;
    int ntiles;
    const int tbase = block_exclusive_scan(mt, &ntiles);
    for (int i = 0; i < mt; ++i) {
        const int idx = tbase + i;
        if (idx < max_entries) tiles[idx] = make_int4(e, off + 128 * i, min(128, cnt - 128 * i), 0);
    }
    if (e == 0) *num_entries = min(ntiles, max_entries);
    if (tiles2) {
        const int mt2 = (e < E) ? (cnt + 255) / 256 : 0;
        int ntiles2;
        const int tbase2 = block_exclusive_scan(mt2, &ntiles2);
        for (int i = 0; i < mt2; ++i) {
            const int idx = tbase2 + i;
            if (idx < max_entries2) tiles2[idx] = make_int4(e, off + 256 * i, min(256, cnt - 256 * i), tbase + 2 * i);
        }
        if (e == 0) *num_entries2 = min(ntiles2, max_entries2);
    }
}

// One CTA of 1024 threads (E <= 1024): per-expert counts and the exclusive
// per-chunk bases (in place in chunk_hist), offsets, and the tile lists.
__global__ void __launch_bounds__(1024) route_scan_kernel(int chunks, int E, int32_t* __restrict__ chunk_hist,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int4* __restrict__ tiles, int32_t* __restrict__ num_entries,
                                                          int max_entries, int4* __restrict__ tiles2,
                                                          int32_t* __restrict__ num_entries2, int max_entries2) {
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < E) {
        // exclusive running sum over the chunks, 8 independent loads at a time
        int c = 0;
        for (; c + 8 <= chunks; c += 8) {
            int h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = chunk_hist[(long)(c + i) * E + e];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                chunk_hist[(long)(c + i) * E + e] = cnt;
                cnt += h[i];
            }
        }
        for (; c < chunks; ++c) {
            const int h = chunk_hist[(long)c * E + e];
            chunk_hist[(long)c * E + e] = cnt;
            cnt += h;
        }
        counts[e] = cnt;
    }
    int total;
    const int off = block_exclusive_scan(e < E ? cnt : 0, &total);
    if (e < E) offsets[e] = off;
    if (e == 0) offsets[E] = total;
    if (tiles) build_tile_lists(E, cnt, off, tiles, num_entries, max_entries, tiles2, num_entries2, max_entries2);
}

// One CTA per chunk (blockDim == kRouteChunk, one token per thread): the rank of
// a pair among its expert's pairs inside the chunk is the number of earlier
// tokens of the chunk whose bit is set in that expert's mask.
// With wrow, also the routing weight of each routed row: wrow[row] = w[t][j].
__global__ void __launch_bounds__(kRouteChunk) route_permute_kernel(const int32_t* __restrict__ ids, int T, int E,
                                                                    int k, const int32_t* __restrict__ chunk_base,
                                                                    const int32_t* __restrict__ offsets,
                                                                    int32_t* __restrict__ src,
                                                                    int32_t* __restrict__ row,
                                                                    const float* __restrict__ w,
                                                                    float* __restrict__ wrow) {
    constexpr int WORDS = kRouteChunk / 32;
    extern __shared__ uint32_t masks[];   // [E][WORDS]
    for (int i = threadIdx.x; i < E * WORDS; i += blockDim.x) masks[i] = 0;
    __syncthreads();
    const int tl = threadIdx.x;
    const long t = (long)blockIdx.x * kRouteChunk + tl;
    const bool live = t < T;
    int my[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k && live) {
            my[j] = ids[t * k + j];
            atomicOr(&masks[my[j] * WORDS + (tl >> 5)], 1u << (tl & 31));
        }
    }
    __syncthreads();
    if (live) {
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                const int e = my[j];
                const uint32_t* m = masks + e * WORDS;
                int rank = __popc(m[tl >> 5] & ((1u << (tl & 31)) - 1u));
                for (int wd = 0; wd < (tl >> 5); ++wd) rank += __popc(m[wd]);
                const int r = offsets[e] + chunk_base[(long)blockIdx.x * E + e] + rank;
                row[t * k + j] = r;
                src[r] = (int32_t)t;
                if (wrow) wrow[r] = w[t * k + j];
            }
        }
    }
}

cudaError_t launch_route(const float* logits, int T, int E, int k, const RouteBufs& b, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int warps_needed = T;
    const int grid_topk = (warps_needed + 7) / 8;
    const int epl = (E + 31) / 32;
    switch (epl) {
#define QMM_TOPK_CASE(N)                                                                    \
    case N:                                                                                 \
        route_topk_kernel<N><<<grid_topk, 256, 0, s>>>(logits, T, E, k, b.ids, b.w, b.yzero, b.yzero_D); \
        break;
        QMM_TOPK_CASE(1) QMM_TOPK_CASE(2) QMM_TOPK_CASE(3) QMM_TOPK_CASE(4) QMM_TOPK_CASE(5) QMM_TOPK_CASE(6)
        QMM_TOPK_CASE(7) QMM_TOPK_CASE(8) QMM_TOPK_CASE(9) QMM_TOPK_CASE(10) QMM_TOPK_CASE(11) QMM_TOPK_CASE(12)
        QMM_TOPK_CASE(13) QMM_TOPK_CASE(14) QMM_TOPK_CASE(15) QMM_TOPK_CASE(16)
#undef QMM_TOPK_CASE
        default:
            return cudaErrorInvalidValue;
    }
    const int chunks = (T + kRouteChunk - 1) / kRouteChunk;
    route_hist_kernel<<<chunks, 256, E * sizeof(int32_t), s>>>(b.ids, T, E, k, b.chunk_hist);
    route_scan_kernel<<<1, 1024, 0, s>>>(chunks, E, b.chunk_hist, b.counts, b.offsets, b.tiles, b.num_entries,
                                         b.max_entries, b.tiles2, b.num_entries2, b.max_entries2);
    const size_t msmem = (size_t)E * (kRouteChunk / 32) * sizeof(uint32_t);
    route_permute_kernel<<<chunks, kRouteChunk, msmem, s>>>(b.ids, T, E, k, b.chunk_hist, b.offsets, b.src, b.row, b.w,
                                                            b.wrow);
    return cudaGetLastError();
}

// X_perm[r, :] = X[src[r], :], one warp per row, 16-byte vectors (D % 8 == 0).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ X, const int32_t* __restrict__ src,
                                                          int rows, int vec_per_row, uint4* __restrict__ Xp) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const uint4* in = X + (long)src[r] * vec_per_row;
        uint4* out = Xp + (long)r * vec_per_row;
        int i = lane;
        for (; i + 96 < vec_per_row; i += 128) {           // four 16-byte loads in flight per lane
            const uint4 a0 = __ldg(in + i), a1 = __ldg(in + i + 32), a2 = __ldg(in + i + 64), a3 = __ldg(in + i + 96);
            out[i] = a0;
            out[i + 32] = a1;
            out[i + 64] = a2;
            out[i + 96] = a3;
        }
        for (; i < vec_per_row; i += 32) out[i] = __ldg(in + i);
    }
}

cudaError_t launch_gather_rows(const uint16_t* X, const int32_t* src, int rows, int D, uint16_t* Xp, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    int sms = 148;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = min((rows + 7) / 8, sms * 8);
    gather_rows_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(X), src, rows, D / 8,
                                           reinterpret_cast<uint4*>(Xp));
    return cudaGetLastError();
}

// Y[t, :] = sum_j w[t, j] * Yslot[row[t, j], :], j ascending; one CTA of NT
// threads per token, so that each slot row is read as one contiguous run (two
// 16-byte vectors per thread per slot, 2k loads in flight per thread).
// A row index outside [0, P) contributes nothing and raises DEV_BAD_ROW.
template <int NT>
__global__ void __launch_bounds__(NT) combine_kernel(const float4* __restrict__ Yslot, int P,
                                                      const int32_t* __restrict__ row, const float* __restrict__ w,
                                                      int k, int vec_per_row, float4* __restrict__ Y, uint32_t* err) {
    const long t = blockIdx.x;
    int rr[kMaxK];
    float ww[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
            rr[j] = __ldg(row + t * k + j);
            ww[j] = __ldg(w + t * k + j);
            if ((unsigned)rr[j] >= (unsigned)P) {   // the same for every thread of the CTA
                if (threadIdx.x == 0) atomicCAS(err, 0u, (uint32_t)DEV_BAD_ROW);
                rr[j] = 0;
                ww[j] = 0.f;
            }
        }
    }
    for (int i = threadIdx.x; i < vec_per_row; i += 2 * NT) {
        const bool two = i + NT < vec_per_row;
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                const float4* src = Yslot + (long)rr[j] * vec_per_row + i;
                const float4 v0 = __ldcs(src);
                const float4 v1 = two ? __ldcs(src + NT) : make_float4(0.f, 0.f, 0.f, 0.f);
                acc0.x = fmaf(ww[j], v0.x, acc0.x);
                acc0.y = fmaf(ww[j], v0.y, acc0.y);
                acc0.z = fmaf(ww[j], v0.z, acc0.z);
                acc0.w = fmaf(ww[j], v0.w, acc0.w);
                acc1.x = fmaf(ww[j], v1.x, acc1.x);
                acc1.y = fmaf(ww[j], v1.y, acc1.y);
                acc1.z = fmaf(ww[j], v1.z, acc1.z);
                acc1.w = fmaf(ww[j], v1.w, acc1.w);
            }
        }
        Y[t * vec_per_row + i] = acc0;
        if (two) Y[t * vec_per_row + i + NT] = acc1;
    }
}

cudaError_t launch_combine(const float* Yslot, int P, const int32_t* row, const float* w, int T, int k, int D,
                           float* Y, uint32_t* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    // one pass over the row where a CTA size fits it exactly (D = 2560: 320 threads)
    const int vec = D / 4;
    const float4* ys = reinterpret_cast<const float4*>(Yslot);
    float4* y = reinterpret_cast<float4*>(Y);
    if (vec == 640)
        combine_kernel<320><<<T, 320, 0, s>>>(ys, P, row, w, k, vec, y, err);
    else
        combine_kernel<256><<<T, 256, 0, s>>>(ys, P, row, w, k, vec, y, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- sub-step entry points
// (the qmm_dbg_* calls run one step of the expert stage on caller buffers)

// Tile lists from caller-given expert offsets [E+1] (one CTA of 1024 threads).
// Offsets that are not 0 = o[0] <= o[1] <= ... <= o[E] = P give empty lists and
// raise DEV_BAD_OFFSETS in the device error word.
__global__ void __launch_bounds__(1024) tiles_from_offsets_kernel(const int32_t* __restrict__ offsets, int E, int P,
                                                                  uint32_t* err, int4* __restrict__ tiles,
                                                                  int32_t* __restrict__ num_entries, int max_entries,
                                                                  int4* __restrict__ tiles2,
                                                                  int32_t* __restrict__ num_entries2, int max_entries2) {
    const int e = threadIdx.x;
    int off = 0, cnt = 0;
    bool bad = false;
    if (e < E) {
        off = offsets[e];
        const int next = offsets[e + 1];
        bad = off < 0 || next < off || next > P;
        cnt = bad ? 0 : next - off;
    }
    if (e == 0) bad = bad || offsets[0] != 0 || offsets[E] != P;
    if (__syncthreads_or(bad)) {
        if (e == 0) {
            atomicCAS(err, 0u, (uint32_t)DEV_BAD_OFFSETS);
            *num_entries = 0;
            *num_entries2 = 0;
        }
        return;
    }
    build_tile_lists(E, cnt, off, tiles, num_entries, max_entries, tiles2, num_entries2, max_entries2);
}

// q8_1 codes: f16 (exact integers) <-> int8, 8 per thread (n8 = P * F / 8).
__global__ void __launch_bounds__(256) codes_f16_to_i8_kernel(const uint4* __restrict__ src, uint2* __restrict__ dst,
                                                             long n8) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
        const int lo = (int)__low2float(h), hi = (int)__high2float(h);
        o[j >> 1] |= (((uint32_t)lo & 0xFFu) | (((uint32_t)hi & 0xFFu) << 8)) << (16 * (j & 1));
    }
    dst[i] = make_uint2(o[0], o[1]);
}

__global__ void __launch_bounds__(256) codes_i8_to_f16_kernel(const uint2* __restrict__ src, uint4* __restrict__ dst,
                                                             long n8) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const uint2 v = src[i];
    const uint32_t w[2] = {v.x, v.y};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b = w[j >> 1] >> (16 * (j & 1));
        const __half2 h = __floats2half2_rn((float)(int8_t)(b & 0xFFu), (float)(int8_t)((b >> 8) & 0xFFu));
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

// fp32 d of H in the per-128-row-entry layout [entry][F/32][128] the down kernel
// reads (rows past an entry's end are 0); one CTA per entry.
__global__ void __launch_bounds__(256) hd_to_entries_kernel(const __half* __restrict__ Hd, const int4* __restrict__ tiles,
                                                           const int32_t* __restrict__ num_entries, int groups,
                                                           float* __restrict__ Hd32) {
    const int entry = blockIdx.x;
    if (entry >= *num_entries) return;
    const int4 t = tiles[entry];
    for (int i = threadIdx.x; i < groups * 128; i += blockDim.x) {
        const int b = i >> 7, r = i & 127;
        Hd32[(long)entry * groups * 128 + i] = r < t.z ? __half2float(Hd[((long)t.y + r) * groups + b]) : 0.f;
    }
}

cudaError_t launch_tiles_from_offsets(const int32_t* offsets, int E, int P, uint32_t* err, const RouteBufs& b,
                                      cudaStream_t s) {
    tiles_from_offsets_kernel<<<1, 1024, 0, s>>>(offsets, E, P, err, b.tiles, b.num_entries, b.max_entries, b.tiles2,
                                                 b.num_entries2, b.max_entries2);
    return cudaGetLastError();
}

cudaError_t launch_codes_f16_to_i8(const __half* src, int8_t* dst, long n, cudaStream_t s) {
    const long n8 = n / 8;
    if (n8 == 0) return cudaSuccess;
    codes_f16_to_i8_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                                                       reinterpret_cast<uint2*>(dst), n8);
    return cudaGetLastError();
}

cudaError_t launch_codes_i8_to_f16(const int8_t* src, __half* dst, long n, cudaStream_t s) {
    const long n8 = n / 8;
    if (n8 == 0) return cudaSuccess;
    codes_i8_to_f16_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(reinterpret_cast<const uint2*>(src),
                                                                       reinterpret_cast<uint4*>(dst), n8);
    return cudaGetLastError();
}

cudaError_t launch_hd_to_entries(const __half* Hd, const int4* tiles, const int32_t* num_entries, int max_entries,
                                 int groups, float* Hd32, cudaStream_t s) {
    if (max_entries == 0) return cudaSuccess;
    hd_to_entries_kernel<<<max_entries, 256, 0, s>>>(Hd, tiles, num_entries, groups, Hd32);
    return cudaGetLastError();
}

}  // namespace qmm
