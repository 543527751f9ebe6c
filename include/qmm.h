/*
 * qmm.h -- C ABI of the block-quantised prefill GEMM and routed-MoE expert-stage
 * library for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates, frees or keeps a pointer past the call.  Buffers must be
 *    16-byte aligned.  All matrices are row-major with K (the reduction
 *    dimension) fastest for weights.
 *  - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t).
 *  - 4-bit codes are packed two per byte: element 2j of a row is the low nibble
 *    of byte j, element 2j+1 the high nibble.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream).  Calls are asynchronous and never synchronise the host.
 *  - Argument checks happen before anything is enqueued; a failed check returns
 *    QMM_ERR_INVALID_ARG / QMM_ERR_UNSUPPORTED_SHAPE / QMM_ERR_WORKSPACE and
 *    enqueues nothing.  Launch failures return QMM_ERR_CUDA.  qmm_last_error()
 *    gives a message for the calling thread's last failure.
 *  - Kernel-side waits are bounded; a wait that runs out records a code in a
 *    device error word, and qmm_check_status() (which synchronises `stream`)
 *    returns QMM_ERR_TIMEOUT for it.
 *  - The library runs only on compute capability 10.3 (GB300); any other device
 *    gives QMM_ERR_UNSUPPORTED_DEVICE.  There is no fallback path.
 *  - Device addresses the library looks up once per device (its device error
 *    word, the fixed scratch of moe_route_permute_noalloc) are kept for the
 *    life of the process: they do not survive cudaDeviceReset, after which the
 *    library must not be called again in that process.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1,
    QMM_ERR_UNSUPPORTED_SHAPE = 2,
    QMM_ERR_UNSUPPORTED_DEVICE = 3,
    QMM_ERR_WORKSPACE = 4,
    QMM_ERR_CUDA = 5,
    QMM_ERR_TIMEOUT = 6
} qmm_status;

typedef enum { QMM_F32 = 0, QMM_BF16 = 1 } qmm_dtype;

/* Message describing the calling thread's most recent failed call ("" if none). */
const char *qmm_last_error(void);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: QMM_OK, QMM_ERR_TIMEOUT (a kernel wait ran out; the code is
 * in the message), or QMM_ERR_CUDA if the synchronisation itself failed. */
qmm_status qmm_check_status(cudaStream_t stream);

/*
 * qmm_w4a16 -- dense prefill product with 4-bit weights.
 *   Y[m,n] = scale2 * sum_k X[m,k] * e2m1(Wc[n,k]) * e4m3(Ws[n, k/16])
 * Format: "perf: strix-hip BF16 GEMMs via hipBLASLt", commit "f16a twins for the
 * dense M128 and routed-MoE kernels" (e2m1 codes, one E4M3 scale per 16 K, an
 * fp32 per-tensor scale2 applied once in the epilogue; e2m1 x E4M3 is exact).
 *   X   [M][K]    bf16 activations
 *   Wc  [N][K/2]  packed e2m1 codes (bit 3 sign, bits 0-2 index {0,.5,1,1.5,2,3,4,6})
 *   Ws  [N][K/16] OCP E4M3 scale bytes
 *   Y   [M][N]    fp32 (ydt = QMM_F32) or bf16 rounded to nearest even (QMM_BF16)
 * fp32 accumulation.  Shapes: M >= 1, K % 32 == 0, N % 32 == 0.
 */
qmm_status qmm_w4a16(const uint16_t *X, int M, int K, int N, const uint8_t *Wc, const uint8_t *Ws, float scale2,
                     void *Y, qmm_dtype ydt, cudaStream_t stream);

/*
 * qmm_w4a16_ws / qmm_fp8_blk128_ws -- the same products with a caller-owned
 * device workspace `ws` (256-byte aligned; NULL or 0 bytes: as the calls
 * without it).  When the last wave of tiles would leave at least half the SMs
 * idle (few tiles, or a ragged last wave) and K % 256 == 0, its tiles are split
 * along K over several CTAs: each split writes its fp32 partial tile to ws and
 * a second kernel on the same stream adds the partials in split order, scales,
 * rounds and writes Y (deterministic for a given GPU).  A workspace smaller than
 * a split needs only turns the split off.  ws must not be used by another call
 * until this one has finished on `stream`.
 * qmm_dense_workspace_size: bytes that always suffice for an M x K x N call on
 * the current device (256 KB per SM), 0 when the shape never splits (or no
 * device is usable).
 */
size_t qmm_dense_workspace_size(int M, int K, int N);
qmm_status qmm_w4a16_ws(const uint16_t *X, int M, int K, int N, const uint8_t *Wc, const uint8_t *Ws, float scale2,
                        void *Y, qmm_dtype ydt, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * qmm_fp8_blk128 -- dense prefill product with FP8 weights and 128x128 block scales.
 *   Y[m,n] = sum_kb S[n/128][kb] * sum_{k in block kb} X[m,k] * e4m3(W[n,k])
 * Each 128-K block is summed unscaled and folded once with its fp32 scale:
 * "perf: strix-hip BF16 GEMMs via hipBLASLt", FP8 block-scaling twin commit.
 *   X [M][K] bf16;  W [N][K] OCP E4M3 bytes;  S [N/128][K/128] fp32;  Y [M][N] bf16 (RNE).
 * fp32 accumulation.  Shapes: M >= 1, K % 128 == 0, N % 128 == 0.
 * qmm_fp8_blk128_ws: with a workspace as qmm_w4a16_ws (a split adds the folded
 * partials of its K range).
 */
qmm_status qmm_fp8_blk128(const uint16_t *X, int M, int K, int N, const uint8_t *W, const float *S, uint16_t *Y,
                          cudaStream_t stream);
qmm_status qmm_fp8_blk128_ws(const uint16_t *X, int M, int K, int N, const uint8_t *W, const float *S, uint16_t *Y,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * qmm_q8_0_q8_1 -- dense projection with Q8_0 weights and q8_1 activations,
 * the output rounded to q8_1 blocks ("Run Edge0-145B Q3_K on AMD HIP (Linux,
 * gfx1100)", commit 17c02cd: the D and U projections of a latent layer as
 * Q8_0 x q8_1 integer dots, D re-quantising its products to q8_1 and writing the
 * fp32 rows too when asked):
 *   y[m,n] = sum_b fp16(Xd[m][b]) * fp16(Wd[n][b]) * sum_{k in block b} Xq[m][k] * Wq[n][k]
 *   (one exact integer dot per block of 32, folded in fp32), then per row m and
 *   32 consecutive n: d = max|y|/127, q = round-half-away(y/d) in [-127, 127],
 *   Yq = q, Yd = fp16(d), Ys = fp16(d * sum q)  (all zero for an all-zero block).
 *   Xq [M][K] int8, Xd [M][K/32] fp16 (the q8_1 activations' d);
 *   Wq [N][K] int8, Wd [N][K/32] fp16 (Q8_0: 32 codes and one scale per block);
 *   Yq [M][N] int8, Yd / Ys [M][N/32] fp16; Y [M][N] fp32 before the rounding, or NULL.
 *   ws: device scratch of at least qmm_q8_0_q8_1_workspace_size(M, K, N) bytes,
 *   256-byte aligned (both operands' codes as f16 -- 2 (M + N) K bytes -- and
 *   per-tile d tables); qmm_q8_0_q8_1_workspace_size returns 0 for a shape it
 *   does not take.
 * Shapes: M >= 1, K % 256 == 0, N % 128 == 0.
 */
size_t qmm_q8_0_q8_1_workspace_size(int M, int K, int N);
qmm_status qmm_q8_0_q8_1(const int8_t *Xq, const uint16_t *Xd, int M, int K, int N, const int8_t *Wq,
                         const uint16_t *Wd, int8_t *Yq, uint16_t *Yd, uint16_t *Ys, float *Y, void *ws,
                         size_t ws_bytes, cudaStream_t stream);

/*
 * moe_route_permute -- top-k routing and per-expert grouping of T tokens.
 * For each token t: ids[t][0..k) are the k largest logits (descending; a tie
 * goes to the lower expert index) and w[t][j] = exp(l_j - l_max) / sum over the
 * k chosen of exp(l_i - l_max), which equals softmax followed by renormalising
 * the chosen weights ("AMD_HIP.md", RDNA4 speed switches, router_top10).
 * Grouping: counts[e] = pairs (t,j) that chose e; offsets = exclusive prefix sum
 * of counts (offsets[E] = T*k); the pairs of expert e take rows offsets[e],
 * offsets[e]+1, ... in ascending token order; row[t][j] is the row of pair
 * (t,j) and src[row] its token.  Integer outputs are deterministic.
 *   logits [T][E] fp32; ids [T][k] int32; w [T][k] fp32; counts [E] int32;
 *   offsets [E+1] int32; src [T*k] int32; row [T][k] int32.
 *   ws: device scratch of at least moe_route_workspace_size(T, E, k) bytes.
 * Shapes: T >= 0, 1 <= k <= 16, k <= E <= 512.
 */
size_t moe_route_workspace_size(int T, int E, int k);
qmm_status moe_route_permute(const float *logits, int T, int E, int k, int32_t *ids, float *w, int32_t *counts,
                             int32_t *offsets, int32_t *src, int32_t *row, void *ws, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * moe_expert_stage_w4_iq4 -- the routed expert stage of a prompt.
 * "Run Edge0-145B Q3_K on AMD HIP (Linux, gfx1100)", commit 4cb5224: gate/up,
 * SwiGLU, H rounded to q8_1, down over IQ4_NL, for every expert's tokens; with
 * this library's gate/up format (W4 as in qmm_w4a16, per-expert scale2):
 *   route + group as moe_route_permute;
 *   for each routed row r (token t, expert e):
 *     g[n] = scale2[e] * X[t] . Wgu[e][n],  u[n] = scale2[e] * X[t] . Wgu[e][F+n]
 *     h = silu(g) * u;   H = q8_1(h) per 32 columns:
 *       d = max|h|/127, q = round-half-away(h/d) in [-127,127], s = d * sum(q)
 *     y_r[n] = sum_b d_H[b] * d_W[e][n][b] * sum_{k in b} q[k] * CB[idx[e][n][k]]
 *       (CB = IQ4_NL codebook {-127,-104,-83,-65,-49,-35,-22,-10,1,13,25,38,53,69,89,113})
 *   Y[t] = sum_j w[t][j] * y_{row[t][j]}     (j ascending)
 *   X [T][D] bf16; logits [T][E] fp32;
 *   Wgu_c [E][2F][D/2] packed e2m1 (rows 0..F-1 gate, F..2F-1 up); Wgu_s [E][2F][D/16] E4M3;
 *   gu_scale2 [E] fp32; Wd_idx [E][D][F/2] packed IQ4_NL indices; Wd_s [E][D][F/32] fp16;
 *   Y [T][D] fp32.
 *   ws: device scratch of at least moe_expert_stage_workspace_size(...) bytes;
 *   its regions (routing outputs, permuted X, H codes/scales, per-row down
 *   outputs) are listed by moe_expert_stage_workspace_layout().
 * Shapes: D % 128 == 0, F % 128 == 0, F <= 1024, 1 <= k <= 16, k <= E <= 512, T >= 0.
 * The weighted combine is fused into the down product: each routed row's
 * outputs are added, times its weight, into Y with fp32 atomic adds (Y is
 * zeroed by the routing step), so the order in which a token's k terms are
 * summed is not fixed and Y may differ between calls in the last bits (well
 * inside the stage tolerance); moe_expert_stage_w4_iq4_ex with QMM_STAGE_SLOTS
 * gives the j-ordered, reproducible sum instead.
 */
size_t moe_expert_stage_workspace_size(int T, int D, int F, int E, int k);
qmm_status moe_expert_stage_w4_iq4(const uint16_t *X, const float *logits, int T, int D, int F, int E, int k,
                                   const uint8_t *Wgu_c, const uint8_t *Wgu_s, const float *gu_scale2,
                                   const uint8_t *Wd_idx, const uint16_t *Wd_s, float *Y, void *ws, size_t ws_bytes,
                                   cudaStream_t stream);

/*
 * moe_expert_stage_w4_iq4_ex -- moe_expert_stage_w4_iq4 with options.
 *   flags = 0: as moe_expert_stage_w4_iq4 (combine fused into the down product).
 *   flags = QMM_STAGE_SLOTS: the down product writes every routed row's outputs to
 *     the workspace region Yslot [T*k][D] fp32, and a separate combine kernel
 *     forms Y[t] = sum_j w[t][j] * Yslot[row[t][j]] in ascending j: the same
 *     result every call, and the per-row down outputs stay inspectable.
 * Other flag bits: QMM_ERR_INVALID_ARG.
 */
#define QMM_STAGE_SLOTS 1u
qmm_status moe_expert_stage_w4_iq4_ex(const uint16_t *X, const float *logits, int T, int D, int F, int E, int k,
                                      const uint8_t *Wgu_c, const uint8_t *Wgu_s, const float *gu_scale2,
                                      const uint8_t *Wd_idx, const uint16_t *Wd_s, float *Y, void *ws, size_t ws_bytes,
                                      unsigned flags, cudaStream_t stream);

/*
 * Per-expert pointer tables: the expert stage over weights held in one
 * allocation per expert, as the routed-MoE grouped GEMMs of "perf: strix-hip
 * BF16 GEMMs via hipBLASLt" take them (per-expert pointer tables), with no
 * copy of the weights.
 * moe_expert_table_size(E): bytes of the table for E experts (0 if E is not in 1..512).
 * moe_expert_table_build: Wgu_c, Wgu_s, Wd_idx, Wd_s are HOST arrays of E DEVICE
 *   pointers, expert e's matrices in the layouts of moe_expert_stage_w4_iq4
 *   without the leading [E]: Wgu_c[e] [2F][D/2], Wgu_s[e] [2F][D/16],
 *   Wd_idx[e] [D][F/2], Wd_s[e] [D][F/32] fp16; each 16-byte aligned.  Writes
 *   into the caller's device buffer `table` (256-byte aligned, at least
 *   moe_expert_table_size(E) bytes) one TMA tensor map per expert for its
 *   gate/up codes and one for its down indices, and the scale pointers; this is
 *   a set-up call: it copies from the host and synchronises `stream`.  The
 *   table stays valid as long as the experts' buffers do.
 *   Shapes: 1 <= E <= 512, D % 128 == 0, F % 128 == 0, F <= 1024.
 * moe_expert_stage_w4_iq4_table: moe_expert_stage_w4_iq4_ex with each expert's
 *   weights taken from the table (same results, bit for bit with
 *   QMM_STAGE_SLOTS, as the contiguous call on the same values); the kernels
 *   read the expert's tensor map from the table when a tile of that expert starts.
 */
size_t moe_expert_table_size(int E);
qmm_status moe_expert_table_build(int D, int F, int E, const uint8_t *const *Wgu_c, const uint8_t *const *Wgu_s,
                                  const uint8_t *const *Wd_idx, const uint16_t *const *Wd_s, void *table,
                                  size_t table_size, cudaStream_t stream);
qmm_status moe_expert_stage_w4_iq4_table(const uint16_t *X, const float *logits, int T, int D, int F, int E, int k,
                                         const float *gu_scale2, const void *table, float *Y, void *ws,
                                         size_t ws_bytes, unsigned flags, cudaStream_t stream);

/* Byte offsets, inside the expert-stage workspace, of its regions (for callers
 * that inspect intermediate results).  Writes QMM_WS_FIELDS offsets in this order:
 *   0 ids [T*k] i32     1 w [T*k] f32       2 counts [E] i32    3 offsets [E+1] i32
 *   4 src [T*k] i32     5 row [T*k] i32     6 chunk counts
 *   7 tile list, 128-row entries   8 its count   9 tile list, 256-row entries   10 its count
 *  11 X_perm [T*k][D] bf16   12 Hq [T*k][F] fp16: the q8_1 codes (integers in [-127, 127]) held
 *     exactly as f16, the operand type of the down product's tensor-core MMA
 *  13 Hd [T*k][F/32] fp16   14 Hs [T*k][F/32] fp16
 *  15 d of H as fp32 per 128-row tile (internal)
 *  16 Yslot [T*k][D] fp32 (written with QMM_STAGE_SLOTS only)
 *  17 wrow [T*k] fp32: the routing weight of each routed row (fused combine)
 *  18 total size */
#define QMM_WS_FIELDS 19
qmm_status moe_expert_stage_workspace_layout(int T, int D, int F, int E, int k, size_t *offsets_out);

/*
 * Sub-steps of moe_expert_stage_w4_iq4 on caller-provided buffers, one step per
 * call, so that each can be checked on its own inputs (same kernels as the
 * stage).  P routed rows, grouped by expert: rows offsets[e] .. offsets[e+1]-1
 * belong to expert e (offsets [E+1] int32 on the device, 0 = offsets[0] <= ...
 * <= offsets[E] = P; other offsets compute nothing and make qmm_check_status
 * return QMM_ERR_INVALID_ARG).  All pointers are device pointers owned by the
 * caller; ws is device scratch of at least qmm_dbg_workspace_size(P, D, F, E)
 * bytes, 256-byte aligned; other buffers 16-byte aligned.
 * Shapes: P >= 0, 1 <= E <= 512, D % 128 == 0, F % 128 == 0, F <= 1024.
 *
 * qmm_dbg_gate_up_q8_1 -- the gate/up product, SwiGLU and the q8_1 rounding of H
 * ("Run Edge0-145B Q3_K on AMD HIP (Linux, gfx1100)", commit 4cb5224):
 *   for row r of expert e: g, u, h as in moe_expert_stage_w4_iq4 with
 *   X[t] replaced by X_perm[r]; Hq [P][F] int8 codes, Hd, Hs [P][F/32] fp16.
 * qmm_dbg_down_iq4 -- the down product over IQ4_NL weights (same page):
 *   Yslot[r][n] = sum_b d_H[r][b] * d_W[e][n][b] * sum_{k in b} Hq[r][k] * CB[idx[e][n][k]]
 *   Hq [P][F] int8, Hd [P][F/32] fp16, Yslot [P][D] fp32.
 * qmm_dbg_combine -- the weighted combine: Y[t] = sum_j w[t][j] * Yslot[row[t][j]]
 *   (j ascending); Yslot [P][D] fp32, row/w [T][k], Y [T][D] fp32.  A row index
 *   outside [0, P) adds nothing and makes qmm_check_status return
 *   QMM_ERR_INVALID_ARG.  Shapes: 1 <= k <= 16, D % 4 == 0.
 */
size_t qmm_dbg_workspace_size(int P, int D, int F, int E);
qmm_status qmm_dbg_gate_up_q8_1(const uint16_t *X_perm, const int32_t *offsets, int P, int D, int F, int E,
                                const uint8_t *Wgu_c, const uint8_t *Wgu_s, const float *gu_scale2, int8_t *Hq,
                                uint16_t *Hd, uint16_t *Hs, void *ws, size_t ws_bytes, cudaStream_t stream);
qmm_status qmm_dbg_down_iq4(const int8_t *Hq, const uint16_t *Hd, const int32_t *offsets, int P, int D, int F, int E,
                            const uint8_t *Wd_idx, const uint16_t *Wd_s, float *Yslot, void *ws, size_t ws_bytes,
                            cudaStream_t stream);
qmm_status qmm_dbg_combine(const float *Yslot, int P, const int32_t *row, const float *w, int T, int k, int D, float *Y,
                           cudaStream_t stream);

/*
 * qmm_dbg_wait_timeout -- test hook for failure detection (no counterpart on
 * the pages).  Launches one warp that waits, with the same bounded mbarrier
 * wait every kernel of the library uses, on a barrier that nothing arrives on;
 * after timeout_us microseconds (1 .. 2,000,000) the wait gives up, records a
 * code in the device error word and the kernel returns normally.  The next
 * qmm_check_status on the stream then returns QMM_ERR_TIMEOUT (and clears the
 * word); the CUDA context stays usable.
 */
qmm_status qmm_dbg_wait_timeout(unsigned timeout_us, cudaStream_t stream);

/*
 * moe_route_permute_noalloc -- moe_route_permute for callers that cannot
 * allocate device memory (no counterpart on the pages: a library convenience).
 * Same inputs, outputs, results and shape rules as moe_route_permute, without
 * the ws / ws_bytes arguments.  Such callers are, for example, code running in
 * a CUDA stream capture under the global capture mode (where cudaMalloc is not
 * allowed), plug-ins of another runtime that owns all device memory, and
 * latency-critical loops where cudaMalloc / cudaFree would synchronise.
 * The per-chunk counting scratch lives instead in a fixed device array inside
 * this library: QMM_NOALLOC_SCRATCH_BYTES (1 MiB) on every GPU that loads the
 * library, kept until the process exits.  The limit: ceil(T / 256) * E counters
 * of 4 bytes must fit in it (with E = 512, T <= 131072; with E = 256,
 * T <= 262144; with E = 128, T <= 524288); larger shapes return
 * QMM_ERR_UNSUPPORTED_SHAPE with the sizes in qmm_last_error().
 * The first call on a device looks up the array's device address (a host-side
 * set-up step, no allocation); make that first call before any stream capture.
 * The function itself calls no cudaMalloc, cudaFree or allocating routine.
 * Every call shares the one array: calls whose work overlaps on the GPU (on
 * different streams, or in different host threads) race on it, so serialise
 * them.  Every counter is written before it is read, so nothing needs clearing.
 */
#define QMM_NOALLOC_SCRATCH_BYTES (1u << 20)
qmm_status moe_route_permute_noalloc(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                                     int32_t *counts, int32_t *offsets, int32_t *src, int32_t *row,
                                     cudaStream_t stream);

/*
 * Phase timing of the expert stage (for benchmarks).  With profiling on, each
 * moe_expert_stage_w4_iq4 call records CUDA events on its stream between its
 * phases: 0 routing (top-k, counts, scan, permutation), 1 row gather of X,
 * 2 gate/up + SwiGLU + q8_1, 3 down (with the fused combine), 4 the separate
 * combine kernel (QMM_STAGE_SLOTS only; otherwise empty).  qmm_profile_read() waits for
 * the last profiled call's events and writes its QMM_PROFILE_PHASES phase times
 * in milliseconds; qmm_profile_read_call(i, ...) does the same for the i-th call
 * (0-based) since profiling was switched on, for the last QMM_PROFILE_RING such
 * calls, so that a caller can profile many calls without waiting between them.
 * Events belong to the current device and are created on first use; profiling
 * is off by default.  Other calls: QMM_ERR_INVALID_ARG.
 */
#define QMM_PROFILE_PHASES 5
#define QMM_PROFILE_RING 256
qmm_status qmm_profile_enable(int on);
qmm_status qmm_profile_read(float *ms_out);
qmm_status qmm_profile_read_call(long i, float *ms_out);

#ifdef __cplusplus
}
#endif
#endif /* QMM_H */
