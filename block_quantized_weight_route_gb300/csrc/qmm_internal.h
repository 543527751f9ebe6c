// Internal declarations shared by the library's translation units (not installed).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qmm {

// Parameters of one launch of the block-quantised GEMM kernel family.
struct GemmParams {
    int M, N, K;            // dense: output rows, columns; all: reduction length
    int F;                  // gate/up: rows of each half (gate, up) per expert
    int m_tiles, n_tiles;   // dense: tile grid; grouped: n_tiles per row-tile entry
    int n_step;             // output columns advanced per column tile
    const int4* tiles;      // grouped: {expert, first row, rows, 0} per 128-row entry
    const int* num_entries; // grouped: device count of valid entries
    int max_entries;        // grouped: capacity of `tiles`
    const uint8_t* w_scale; // W4: E4M3 scale bytes, one per 16 K per weight row
    const float* scale2;    // gate/up: fp32 scale2 per expert
    float scale2_dense;     // dense W4: fp32 scale2
    const float* blk_scale; // FP8: [N/128][K/128] block scales
    const float* dH32;      // down: fp32 d of H per 128-row tile entry, [entry][K/32][128]
    const __half* dW;       // down: IQ4_NL block scales, [E][N][K/32]
    // per-expert weights (pointer-table form of the expert stage; null: the
    // contiguous [E][...] arrays through tmB / tmA, w_scale and dW above)
    const CUtensorMap* wmaps;          // [E] tensor maps of each expert's weight codes
    const uint8_t* const* wscale_tab;  // gate/up: [E] E4M3 scale matrices [2F][D/16]
    const __half* const* dW_tab;       // down: [E] IQ4_NL scale matrices [D][F/32]
    const int32_t* src;     // down with the combine fused: token of each routed row [P]
    const float* wrow;      // down with the combine fused: routing weight of each routed row [P]
    void* Y;                // output (fp32 or bf16)
    int ydt;                // 0: fp32, 1: bf16
    long ldy;               // output row pitch in elements
    __half* Hq;             // gate/up: q8_1 codes of H [rows][F], exact f16 integers
    __half* Hd;             // gate/up: q8_1 d per 32-block [rows][F/32]
    __half* Hs;             // gate/up: q8_1 s per 32-block [rows][F/32]
    float* Hd32;            // gate/up: fp32 value of the fp16 d, [entry][F/32][128 rows]
    uint32_t* err;          // device error word
    // dense only: K splits of the last, partly filled wave of tiles.  Work items
    // [split_from, ...) are split_S consecutive K ranges of the tiles (items)
    // split_from, split_from + 1, ...; each split writes its fp32 partial tile
    // to split_part, and a reduction kernel launched after the GEMM adds them in
    // split order and writes the output.  split_S == 1: no splits.
    int split_from;
    int split_S;
    float* split_part;      // [split tile][cluster rank][split][BM][BN] fp32 (null: never split)
    long split_part_cap;    // floats available at split_part
};

// Launchers (return a cudaError_t from the launch).  Each takes two encoded
// tensor maps: tmA for the activation operand (box rows 128 / cn: each CTA of a
// cluster of cn loads that slice and multicasts it), tmB for the raw weight
// codes; cn must divide p.n_tiles (cluster_for picks it).
int cluster_for(int n_tiles);
int gate_up_cluster(int n_tiles);   // the same choice for the gate/up GEMM
cudaError_t launch_w4a16_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                               cudaStream_t s);
cudaError_t launch_w4_gate_up_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                                     cudaStream_t s);
// token rows and weight rows (gate + up for the gate/up product) of one W4 tile
struct TileShape {
    int rows, bn;
};
TileShape w4_dense_shape(int M, int N, int sms);   // the launch picks the kernel by n_step (128 or 256)
TileShape w4_gate_up_shape();
// token rows of one FP8 tile (the activation box height before the cluster split)
int fp8_tile_rows();
cudaError_t launch_fp8_blk128(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int cn,
                              cudaStream_t s);
// combine = false: per-slot rows p.Y [P][N] fp32; true: Y[src[r]] += wrow[r] * y_r
// accumulated into p.Y [T][N] fp32 (which must start at zero).
cudaError_t launch_iq4_down(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid, bool combine,
                            cudaStream_t s);

int smem_iq4_down();

// Dense Q8_0 x q8_1 projection re-quantised to q8_1 (gemm_q8.cu): tmA Q8_0 codes
// [N][K] int8 (or, when q8_weights_f16(), the same codes as f16, 128-byte swizzle),
// tmB activation codes [M][K] f16, tmW weight scales [N][K/32] fp16;
// p.tiles / num_entries: 128-row tiles of M (launch_dense_tiles), p.dH32: the
// activations' d per tile [entry][K/32][128] fp32.
bool q8_weights_f16();
cudaError_t launch_dense_tiles(int M, int4* tiles, int32_t* num_entries, cudaStream_t s);
cudaError_t launch_q8_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmW, const GemmParams& p,
                            int8_t* Yq, __half* Yd, __half* Ys, float* Y, int M, int grid, cudaStream_t s);

// Routing and data-movement kernels (route.cu).
struct RouteBufs {
    int32_t* ids;         // [T][k]
    float* w;             // [T][k]
    int32_t* counts;      // [E]
    int32_t* offsets;     // [E+1]
    int32_t* src;         // [T*k]
    int32_t* row;         // [T][k]
    int32_t* chunk_hist;  // [chunks][E]  (scratch)
    int4* tiles;          // [max_entries] 128-row entries (optional)
    int32_t* num_entries; // [1]            (optional)
    int max_entries;
    int4* tiles2;         // [max_entries2] 256-row entries (optional, needs tiles)
    int32_t* num_entries2;
    int max_entries2;
    float* wrow = nullptr;    // [T*k] weight of the pair at each routed row (optional)
    float* yzero = nullptr;   // [T][yzero_D] fp32 rows set to zero by the top-k kernel (optional)
    int yzero_D = 0;
};
constexpr int kRouteChunk = 256;   // tokens per grouping chunk
cudaError_t launch_route(const float* logits, int T, int E, int k, const RouteBufs& b, cudaStream_t s);
cudaError_t launch_gather_rows(const uint16_t* X, const int32_t* src, int rows, int D, uint16_t* Xp, cudaStream_t s);
cudaError_t launch_tiles_from_offsets(const int32_t* offsets, int E, int P, uint32_t* err, const RouteBufs& b,
                                      cudaStream_t s);
cudaError_t launch_codes_f16_to_i8(const __half* src, int8_t* dst, long n, cudaStream_t s);
cudaError_t launch_codes_i8_to_f16(const int8_t* src, __half* dst, long n, cudaStream_t s);
cudaError_t launch_hd_to_entries(const __half* Hd, const int4* tiles, const int32_t* num_entries, int max_entries,
                                 int groups, float* Hd32, cudaStream_t s);
cudaError_t launch_wait_timeout_probe(uint32_t* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_combine(const float* Yslot, int P, const int32_t* row, const float* w, int T, int k, int D,
                           float* Y, uint32_t* err, cudaStream_t s);

// Set the calling thread's message returned by qmm_last_error().
void set_last_error(const char* msg);
}  // namespace qmm
