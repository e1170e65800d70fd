// internal.cuh -- launch parameter blocks and launcher prototypes shared by the
// translation units of libhypic (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/hypic.h"

namespace hypic {

// Device status word bits (set by kernels, read by hypic_get_device_status).
enum : unsigned { kErrTimeout = 1u, kErrRange = 2u, kErrBounds = 4u };

// One segment of the launch table. The table is ordered longest first (LPT order:
// "Hypic: Position-Independent KV Caching ..." episode companion, "Segment parallelism:
// LPT scheduling across workers"); idx >= 0 is the segment's position in the caller's order,
// idx < 0 marks a piece of a split segment whose outputs go to piece slot -1 - idx.
struct SegEntry {
    int32_t start;
    int32_t len;
    int32_t idx;
    int32_t wsb;   // first workspace record of this segment (GDN / DeltaNet tensor-core build)
};

// Workspace record of the GDN / DeltaNet tensor-core build: one 64 x 64 bf16 matrix per
// (segment, value head, 64-token chunk).
constexpr int kGdnChunk = 64;
constexpr int64_t kGdnRecordBytes = kGdnChunk * kGdnChunk * 2;
constexpr int64_t kGdnWorkspaceTail = 256;   // after the records: the preparation's ticket counter
// The channel-gated delta rule (KDA) adds, per record, the chunk's gated keys Kt and Kh (bf16
// 64 x 128 each, row-major) and its per-channel log-decay c_C (128 fp32) plus their maximum m,
// in three arrays after the tail: [records][64][128], [records][64][128], [records][kKdaSide].
constexpr int64_t kKdaTileBytes = kGdnChunk * 128 * 2;
constexpr int kKdaSide = 132;
constexpr int64_t kKdaExtraBytes = 2 * kKdaTileBytes + kKdaSide * 4;

struct BuildParams {
    int32_t family;
    int32_t dtype;
    int32_t n_seg;
    int32_t H_k;
    int32_t H_v;
    int32_t D;          // d_k == d_v
    int32_t gqa;        // H_v / H_k
    int32_t max_len;    // longest segment
    int32_t n_tok;      // tokens in k / v (the last segment offset)
    int32_t pad0;
    int64_t seg_stride; // output units between segments
    const void *k;
    const void *v;
    const float *log_gate;
    const float *log_gamma;
    const float *beta;
    float *S;
    float *lam;
    float *P;
    void *workspace;
    unsigned *err;
    // outputs of segment pieces (SegEntry.idx < 0: slot -1 - idx, [slot][H_v] units) when a
    // long segment is built as several pieces and composed afterwards; else unused
    float *S_piece;
    float *P_piece;
    float *lam_piece;
    const void *q;        // segment outputs (exact path only): queries, outputs, start states
    void *O;
    const float *S_init;
    void *kda_kt;         // KDA tensor-core build: the gated-key and log-decay records above
    void *kda_kh;
    float *kda_side;
    SegEntry seg[HYPIC_MAX_SEGMENTS];
};

struct ComposeParams {
    int32_t family;
    int32_t n_seg;
    int64_t n_units;
    int32_t D;
    int32_t pad;
    const float *S;
    const float *lam;
    const float *P;
    const float *S0;
    float *prefix;
    float *lam_total;   // optional: sum_j lam_j per unit (per key row for DIAG)
    float *P_total;     // optional, dense families: P_{n-1} ... P_0 per unit
    float *prefix_last; // dense tensor-core compose, internal use: write only the last state,
                        // [n_units][d][d], instead of prefix
    // internal use (the convolution warm-up): with two segments, segment 1's S, lam and P in
    // arrays of their own ([n_units][d][d], [n_units] ([n_units][d] for DIAG)); NULL: segment
    // 1 follows segment 0 in S, lam and P
    const float *S1;
    const float *lam1;
    const float *P1;
    unsigned *err;
};

// Segment j of unit u in a [segment][unit][per] array, or in segment 1's own [unit][per] array
__host__ __device__ __forceinline__ const float *compose_seg(const float *a, const float *a1, int64_t j,
                                                             int64_t n_units, int64_t u, int64_t per) {
    return (j == 1 && a1) ? a1 + u * per : a + (j * n_units + u) * per;
}

// The convolution of the warm-up's head tokens (conv.cu): head row r is token
// seg_start[j] + r - head_off[j] of the prompt, for the segment j with head_off[j] <= r <
// head_off[j + 1].
struct ConvHeadParams {
    int32_t family;
    int32_t dtype;
    int32_t n_seg;
    int32_t H_k;
    int32_t H_v;
    int32_t D;          // d_k == d_v
    int32_t K;          // the convolution's width
    int32_t n_rows;     // head tokens of all segments
    const void *k_raw;
    const void *v_raw;
    const float *wk;
    const float *wv;
    const float *log_gate;   // gathered per head row into g_head when not NULL
    const float *beta;       // gathered into b_head when not NULL
    float *k_head;      // [n_rows][H_k][D]
    float *v_head;      // [n_rows][H_v][D]
    float *g_head;      // [n_rows][H_v] (DIAG, KDA: [n_rows][H_v][D])
    float *b_head;      // [n_rows][H_v]
    unsigned *err;
    int32_t seg_start[HYPIC_MAX_SEGMENTS];
    int32_t head_off[HYPIC_MAX_SEGMENTS + 1];
};

// Launchers (return the launch's cudaError_t).
cudaError_t launch_build_gated_simt(const BuildParams &p, cudaStream_t s);
cudaError_t launch_build_seq(const BuildParams &p, cudaStream_t s);
cudaError_t launch_compose_scaled(const ComposeParams &p, cudaStream_t s);
cudaError_t launch_compose_lam_total(const ComposeParams &p, cudaStream_t s);
cudaError_t launch_compose_dense_simt(const ComposeParams &p, cudaStream_t s);
cudaError_t launch_compose_dense_tc(const ComposeParams &p, cudaStream_t s);
bool compose_dense_tc_supported(const ComposeParams &p);
cudaError_t launch_compose_dense_cols(const ComposeParams &p, cudaStream_t s);
bool compose_dense_cols_supported(const ComposeParams &p);
cudaError_t launch_build_gated_tc(const BuildParams &p, cudaStream_t s);
bool build_gated_tc_supported(const BuildParams &p);
cudaError_t launch_build_gdn_tc(const BuildParams &p, cudaStream_t s);
cudaError_t launch_build_gdn_tc_outputs(const BuildParams &p, cudaStream_t s);
cudaError_t launch_build_gdn_prep(const BuildParams &p, cudaStream_t s);
cudaError_t launch_build_kda_tc(const BuildParams &p, cudaStream_t s);
cudaError_t launch_build_kda_prep(const BuildParams &p, cudaStream_t s);
cudaError_t launch_conv_heads(const ConvHeadParams &p, cudaStream_t s);
bool build_gdn_tc_supported(const BuildParams &p);

// fp32 view of one input element (bf16 or fp32 storage).
__device__ __forceinline__ float load_in(const void *base, int64_t idx, int dtype) {
    if (dtype == HYPIC_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
    return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void raise_error(unsigned *err, unsigned bit) {
    if (err) atomicOr(err, bit);
}

// Index checks of a debug-bounds build (compiled with -DHYPIC_DEBUG_BOUNDS, in place of a memory
// checker): a failing check sets kErrBounds in the status word and the caller skips the access
// (and the work after it). In a release build every check is the constant true.
#ifdef HYPIC_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, unsigned *err) {
    if (!ok) raise_error(err, kErrBounds);
    return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, unsigned *) { return true; }
#endif

}  // namespace hypic
