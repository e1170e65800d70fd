/*
 * hypic.h -- C ABI of the GB300 (sm_103a) library for HYPIC's linear-layer state path.
 *
 * Two operations, both from the linear-layer half of HYPIC:
 *
 *  hypic_build_segments  prefill every cached prompt segment C of one layer into the pair
 *                        (S(C|0), T_C): the zero-initial end state and the segment-cumulative
 *                        transition operator; optionally also the segment's outputs
 *                        o_t = S_t^T q_t for every token (the prefill's own outputs, from a
 *                        zero state or from a given prefix state).
 *                        Source: "Cut First-Token Latency by 3.25x: Introducing HYPIC for
 *                        Position-Independent Caching in Hybrid-Attention LLMs" (besthub.dev),
 *                        paragraph "For linear layers" (HYPIC stores the pair (T_C, S(C|0))
 *                        during the first prefill) and "HYPIC: Cache Acceleration for Hybrid
 *                        Attention Models" (agihunt.info), "Core Approach", Linear Layers.
 *
 *  hypic_compose_scan    chain cached segments algebraically: the inclusive prefix scan
 *                        prefix_j = T_j . prefix_{j-1} + S_j over n segments, for many
 *                        (layer, head) units at once.
 *                        Source: same besthub.dev paragraph (reuse composes
 *                        T_C2 . S(C1) + S(C2) in O(1) time), the agihunt.info "Core Approach"
 *                        (states combine in constant time for any prefix) and the besthub.dev
 *                        paragraph on segment parallelism (a combine worker assembles the
 *                        final state from the segments' results).
 *
 * State convention: per value head the state S is a d_k x d_v fp32 matrix (row = key
 * channel); T_C is d_k x d_k and acts on the left. Families and their step
 * (the pages name the families but print no equations; these are the standard forms):
 *
 *   HYPIC_FAM_LINEAR  S_t = S_{t-1} + k_t v_t^T                                T_C = I
 *   HYPIC_FAM_SCALAR  S_t = g_t S_{t-1} + k_t v_t^T   (RetNet, Mamba2)        T_C = (prod g_t) I
 *   HYPIC_FAM_DIAG    S_t = Diag(g_t) S_{t-1} + k_t v_t^T   (GLA)             T_C = Diag(prod g_t)
 *   HYPIC_FAM_DELTA   S_t = (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T       T_C = prod (I - b k k^T)
 *   HYPIC_FAM_GDN     S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T   T_C = prod a_t (I - b k k^T)
 *   HYPIC_FAM_KDA     S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T
 *                                                            T_C = prod (I - b k k^T) Diag(a_t)
 *                     (the channel-gated delta rule: a per-key-channel decay a_t)
 *
 * with products ordered latest step leftmost (GDN: "Gated Delta Networks: Improving Mamba2
 * with Delta Rule", reference 7 of the episode-companion page "Hypic: Position-Independent
 * KV Caching for Hybrid-Attention LLM Serving").
 *
 * Log-scaled transition storage. The gates of long segments drive T_C below the fp32
 * range (a 2048-token GDN segment with log a ~ -0.04 per token has |T_C| ~ 1e-36), so
 * T_C is stored as T_C = exp(lam) . P:
 *   LINEAR           lam = 0 (written), no P
 *   SCALAR           lam = sum_t log g_t                        [seg][head]
 *   DIAG             lam = sum_t log g_t (per key channel)      [seg][head][d_k]
 *   DELTA / GDN      lam = sum_t log a_t (0 for DELTA)          [seg][head]
 *                    P = prod_t (I - b_t k_t k_t^T), gate-free  [seg][head][d_k][d_k] fp32
 *   KDA              lam = a log-scale that keeps P in range   [seg][head]
 *                    P = exp(-lam) T_C                          [seg][head][d_k][d_k] fp32
 *                    (exact path: lam = sum_t max_i log a_t[i]; tensor-core path: the sum
 *                    over 64-token chunks of max_i sum_{t in chunk} log a_t[i])
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates and owns every buffer. The library allocates no
 *     memory on any call; it keeps per-device state of its own (a 4-byte status word per
 *     device that has run a kernel).
 *   - Memory: tensors are device pointers (cudaMalloc / torch CUDA tensors), row-major
 *     and contiguous; seg_offsets is a HOST array. Every tensor pointer must be 16-byte
 *     aligned (HYPIC_ERR_ALIGNMENT otherwise), except the fp32 gate / beta arrays
 *     (4-byte).
 *   - Asynchrony: calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and return without synchronising. Outputs may not alias inputs.
 *   - Errors: argument problems are detected on the host before anything is launched and
 *     returned as a status; nothing is written then. Faults the host cannot see (a wait
 *     that exceeded its iteration limit, a gate that leaves the supported range) are
 *     recorded in the device status word; hypic_get_device_status() reads and clears it.
 *   - Shapes: d_k == d_v, one of 32, 64, 128; H_v a multiple of H_k (grouped-query keys:
 *     value head h reads key head h / (H_v / H_k)); at most HYPIC_MAX_SEGMENTS segments.
 */
#ifndef HYPIC_H
#define HYPIC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HYPIC_MAX_SEGMENTS 1024

typedef enum {
    HYPIC_OK = 0,
    HYPIC_ERR_INVALID_ARG = 1,  /* NULL / missing tensor, bad count or offsets, host pointer */
    HYPIC_ERR_ALIGNMENT = 2,    /* a tensor pointer is not 16-byte (gates: 4-byte) aligned  */
    HYPIC_ERR_UNSUPPORTED = 3,  /* valid request outside what is built (head size, dtype)   */
    HYPIC_ERR_RANGE = 4,        /* a gate outside the supported range (device-detected)     */
    HYPIC_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, attribute query)     */
    HYPIC_ERR_TIMEOUT = 6,      /* a kernel wait ran out of its iteration limit             */
    HYPIC_ERR_BOUNDS = 7        /* an index check failed (debug-bounds builds only)         */
} hypic_status;

typedef enum {
    HYPIC_FAM_LINEAR = 0,
    HYPIC_FAM_SCALAR = 1,
    HYPIC_FAM_DIAG = 2,
    HYPIC_FAM_DELTA = 3,
    HYPIC_FAM_GDN = 4,
    HYPIC_FAM_KDA = 5
} hypic_family;

typedef enum { HYPIC_BF16 = 0, HYPIC_F32 = 1 } hypic_dtype;

/* Arguments of hypic_build_segments (one linear layer).
 *
 *   family, dtype     hypic_family, hypic_dtype of k and v (gates and beta are fp32)
 *   n_seg             number of segments, 0 <= n_seg <= HYPIC_MAX_SEGMENTS (0: no-op)
 *   H_k, H_v          key heads, value heads (H_v % H_k == 0)
 *   d_k, d_v          head sizes (equal; 32, 64 or 128)
 *   seg_offsets       HOST int64 [n_seg + 1]: 0 = o_0 <= o_1 <= ... <= o_n = N_tok; segment
 *                     j is tokens [o_j, o_{j+1}); empty segments give S = 0, T = I
 *   out_seg_stride    units between consecutive segments in S / lam / P, 0 = H_v (lets a
 *                     caller write layer l of a multi-layer cache at unit offset l * H_v)
 *   k                 [N_tok][H_k][d_k]  dtype
 *   v                 [N_tok][H_v][d_v]  dtype
 *   log_gate          SCALAR: [N_tok][H_v] log g_t (or NULL when log_gamma is given);
 *                     DIAG: [N_tok][H_v][d_k] log g_t; GDN: [N_tok][H_v] log a_t;
 *                     KDA: [N_tok][H_v][d_k] log a_t; LINEAR, DELTA: NULL
 *   log_gamma         SCALAR with a constant per-head decay: [H_v] log gamma_h; else NULL
 *   beta              DELTA, GDN, KDA: [N_tok][H_v] b_t; else NULL
 *   S                 out [n_seg][H_v][d_k][d_v] fp32 (segment stride out_seg_stride units)
 *   lam               out [n_seg][H_v] fp32, DIAG [n_seg][H_v][d_k]
 *   P                 out DELTA / GDN / KDA: [n_seg][H_v][d_k][d_k] fp32; else NULL
 *   workspace         device scratch, at least hypic_build_workspace_bytes() bytes, 16-byte
 *                     aligned (NULL when that is 0). What it holds:
 *                     - DELTA / GDN / KDA with bf16 k, v and d = 128: 8 KB per (segment,
 *                       value head, 64-token chunk), the chunk matrices (I + Diag(b) L)^-1
 *                       Diag(b) that the chain kernel reads back, and 256 bytes of
 *                       work-distribution counter set by the call itself; KDA adds 33,296
 *                       bytes per chunk (its gated keys e^{c} k and e^{-c} k in bf16, and the
 *                       chunk's per-channel log-decays).
 *                     - Any bf16, d = 128 build whose (segment, value head) units fill at most
 *                       half of the current device's SMs: each segment is built as up to 8
 *                       chunk-aligned pieces that are then composed back into its entry. A
 *                       DELTA / GDN build whose last round of units fills at most half of the
 *                       SMs builds its trailing equal-length segments as two halves each. The
 *                       pieces' S, (P,) lam follow.
 *                     No part needs to start at zero. The caller owns it; its contents are
 *                     undefined after the call and it may be reused by the next call on the
 *                     same stream, but not by a call still running on another stream. It must
 *                     not overlap any argument.
 *   q                 optional [N_tok][H_k][d_k] dtype, 16-byte aligned: the queries; given
 *                     exactly when O is
 *   O                 optional out [N_tok][H_v][d_v] dtype, 16-byte aligned: o_t = S_t^T q_t,
 *                     the state after token t read with its query, for every token of every
 *                     segment (besthub.dev, paragraph "For linear layers": the pair is stored
 *                     during the first prefill, whose outputs these are; paragraph "Segment
 *                     parallelism": cold segments are prefilled by scatter workers). It may
 *                     not overlap k, v, q, S, lam or P.
 *   S_init            optional [n_seg][H_v][d_k][d_v] fp32, 16-byte aligned: the state each
 *                     segment starts from (NULL = zero). With it, S is S(C|S_init) and O the
 *                     outputs of the segment reused after that prefix state; T_C does not
 *                     change. (S_init is indexed by segment and head, stride H_v, whatever
 *                     out_seg_stride is.)
 *   The DeltaNet / GDN tensor-core build (bf16, d = 128) computes O itself: a second CTA per
 *   (segment, value head) runs the S half again with the outputs, and no segment is split
 *   into pieces. Every other call with O, every call with S_init, and KDA with fp32 inputs,
 *   d < 128 or a log_gate pointer that is not 8-byte aligned runs the exact CUDA-core path
 *   (fp32 arithmetic). KDA on the tensor cores supports chunks whose log-decay
 *   sum_{t in chunk} log a_t[i] is at least -60 on every channel i (HYPIC_ERR_RANGE in the
 *   device status otherwise), as GDN does for its scalar gate.
 */
typedef struct {
    int32_t family;
    int32_t dtype;
    int32_t n_seg;
    int32_t H_k;
    int32_t H_v;
    int32_t d_k;
    int32_t d_v;
    int32_t reserved0;
    int64_t out_seg_stride;
    const int64_t *seg_offsets;
    const void *k;
    const void *v;
    const float *log_gate;
    const float *log_gamma;
    const float *beta;
    float *S;
    float *lam;
    float *P;
    void *workspace;
    size_t workspace_bytes;
    const void *q;          /* ABI 4 */
    void *O;
    const float *S_init;
} hypic_build_args;

/* Arguments of hypic_compose_scan.
 *
 *   family       hypic_family of the cached entries
 *   n_seg        segments to chain, in order (0: no-op)
 *   n_units      independent (layer, head) units scanned side by side
 *   d_k, d_v     head sizes (equal; 32, 64 or 128)
 *   S            [n_seg][n_units][d_k][d_v] fp32: S(C_j|0) of every segment
 *   lam          [n_seg][n_units] fp32 (DIAG: [n_seg][n_units][d_k]); NULL for LINEAR
 *   P            DELTA / GDN / KDA: [n_seg][n_units][d_k][d_k] fp32; else NULL
 *   S0           optional initial state [n_units][d_k][d_v] fp32; NULL = zero state
 *   prefix       out [n_seg][n_units][d_k][d_v] fp32: prefix[j] = state after segments
 *                0..j, i.e. exp(lam_j) P_j prefix[j-1] + S_j with prefix[-1] = S0
 *   lam_total    optional out (NULL = skip): the log-scale of the transition of all n_seg
 *                segments composed; [n_units] (DIAG: [n_units][d_k]); 4-byte aligned.
 *                sum_j lam_j (0 for LINEAR), minus E ln 2 when P_total carries a scale 2^E.
 *   P_total      optional out (NULL = skip), DELTA / GDN / KDA only (must be NULL otherwise, and
 *                needs lam_total): 2^E P_{n-1} ... P_0 [n_units][d_k][d_k] fp32, latest
 *                segment leftmost, 16-byte aligned. The product of many contractions leaves
 *                the fp32 range (64 segments of a few hundred tokens: about 1e-49), so the
 *                d = 128 kernel carries it scaled by powers of two and reports the exponent
 *                E >= 0 in lam_total; E = 0 while the product stays above 2^-24 in its
 *                largest entry, and always for d = 32, 64. exp(lam_total) P_total is the
 *                composed transition either way.
 *   With S0 = NULL, (prefix[n-1], exp(lam_total) P_total) is the cache entry
 *   (S(C|0), T_C) of the concatenation C = C_0 ... C_{n-1}: entries compose as
 *   T_C2 . S(C1) + S(C2) with transition T_C2 T_C1 (besthub.dev, paragraph "For linear
 *   layers"). Neither total may overlap an input or prefix.
 */
typedef struct {
    int32_t family;
    int32_t n_seg;
    int64_t n_units;
    int32_t d_k;
    int32_t d_v;
    const float *S;
    const float *lam;
    const float *P;
    const float *S0;
    float *prefix;
    float *lam_total;
    float *P_total;
} hypic_compose_args;

/* Build (S(C|0), T_C) for every segment and value head of one layer in one launch.
 * Segments run in parallel, longest first. Returns HYPIC_OK once the work is enqueued. */
hypic_status hypic_build_segments(const hypic_build_args *args, void *stream);

/* hypic_build_segments with library-owned scratch instead of args->workspace (which is
 * ignored): a file-scope device array of HYPIC_STATIC_WS_BYTES bytes, reserved when the
 * library's device code is loaded, so the call itself allocates nothing. The pages describe
 * no counterpart; it exists for callers that must not allocate device memory per call.
 *   - Requests whose hypic_build_workspace_bytes() exceeds HYPIC_STATIC_WS_BYTES return
 *     HYPIC_ERR_UNSUPPORTED before any device work (use hypic_build_segments then).
 *   - The scratch is one buffer per device: calls that overlap in time (two streams, or
 *     two host threads) race on it and give undefined results. Serialise them.
 *   - The first call on a device looks the buffer up (cudaGetSymbolAddress, once per
 *     device); make that first call before any stream capture.
 *   - No part of the scratch needs to start at zero.
 * Other arguments, results and errors are those of hypic_build_segments. */
#define HYPIC_STATIC_WS_BYTES (64u << 20)
hypic_status hypic_build_segments_static_ws(const hypic_build_args *args, void *stream);

/* Inclusive prefix scan of the composition over n_seg segments for n_units units, and
 * optionally the transition of all of them composed (lam_total, P_total). Units are scanned
 * side by side; the dense d = 128 scan without totals of at most (SMs / 4) units splits each
 * unit's state columns over four CTAs (columns compose independently), every other dense
 * d = 128 call takes one CTA per unit. */
hypic_status hypic_compose_scan(const hypic_compose_args *args, void *stream);

/* ---------------------------------------------------------------- convolution-state warm-up
 * "Cut First-Token Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For linear
 * layers": for convolutional variants HYPIC adds a "convolution state warm-up" patch. The pages
 * do not define the convolution; this library reads it as the short convolution of the Gated
 * DeltaNet layer ("Gated Delta Networks: Improving Mamba2 with Delta Rule", reference 7 of the
 * episode-companion page): per channel, a causal convolution of width K over the tokens,
 *     y_t[c] = silu(sum_{tau < K} w[c][tau] x_{t-K+1+tau}[c]),   silu(z) = z / (1 + e^-z),
 * on the raw keys and values (x taken as 0 before the prompt's first token), the keys then
 * L2-normalised per token and head for DELTA / GDN / KDA. A segment's tokens from min(K - 1,
 * length) on (its "rest") have their whole window inside the segment: their entry is
 * position-independent and is what a cache of a convolutional layer keeps (build it with
 * hypic_build_segments from the segment's own convolution, over the offsets shifted by the
 * head length). On reuse, the first min(K - 1, length) tokens (the "head") see the raw tokens
 * of the segment before in this prompt, so the call rebuilds them in context and composes the
 * head before the rest (T = T_rest T_head, S = T_rest S_head + S_rest), every segment at once:
 * a convolution kernel for the heads' tokens, the exact (fp32) build of the heads, and one
 * composition launch with totals.
 *
 *   family, dtype, n_seg, H_k, H_v, d_k, d_v   as in hypic_build_args (dtype of k_raw, v_raw)
 *   conv_k         K, the convolution's width, 1 <= K <= 8 (K = 1: empty heads)
 *   seg_offsets    HOST [n_seg + 1] int64: this prompt's segments, in order
 *   k_raw, v_raw   [N_tok][H_k][d_k], [N_tok][H_v][d_v] dtype, 16-byte aligned: the raw inputs
 *                  of the convolution for the whole prompt
 *   conv_wk, conv_wv  [H_k d_k][K], [H_v d_v][K] fp32, 4-byte aligned: the taps, tap K - 1 on
 *                  the token itself
 *   log_gate, log_gamma, beta   as in hypic_build_args, over the prompt's tokens
 *   S_rest, lam_rest, P_rest    the rests' cached entries, layouts of hypic_build_args' S,
 *                  lam, P with segment stride H_v (P_rest: DELTA / GDN / KDA only)
 *   S, lam, P      out: the segments' entries in this context, the same layouts; they may not
 *                  overlap any input
 *   workspace      at least hypic_warmup_workspace_bytes() bytes, 16-byte aligned
 * Errors: those of hypic_build_segments and hypic_compose_scan; K outside [1, 8] or a missing
 * rest entry is HYPIC_ERR_INVALID_ARG. Asynchronous on `stream`. */
typedef struct {
    int32_t family;
    int32_t dtype;
    int32_t n_seg;
    int32_t H_k;
    int32_t H_v;
    int32_t d_k;
    int32_t d_v;
    int32_t conv_k;
    const int64_t *seg_offsets;
    const void *k_raw;
    const void *v_raw;
    const float *conv_wk;
    const float *conv_wv;
    const float *log_gate;
    const float *log_gamma;
    const float *beta;
    const float *S_rest;
    const float *lam_rest;
    const float *P_rest;
    float *S;
    float *lam;
    float *P;
    void *workspace;
    size_t workspace_bytes;
} hypic_warmup_args;

size_t hypic_warmup_workspace_bytes(const hypic_warmup_args *args);
hypic_status hypic_conv_warmup(const hypic_warmup_args *args, void *stream);

/* Device scratch bytes hypic_build_segments needs for these arguments (host-only query;
 * reads the shapes, seg_offsets and, for KDA, the alignment of log_gate, never the tensors). 0 means no workspace; 0 also for
 * NULL or malformed arguments, which hypic_build_segments then rejects. */
size_t hypic_build_workspace_bytes(const hypic_build_args *args);

/* Name of the kernel hypic_build_segments / hypic_compose_scan would launch for these
 * arguments (host-only query: reads the shapes and, for a dense compose, the current
 * device's SM count; touches no tensor; "none" for an empty request, NULL for arguments the
 * call would reject on shape or family). Static strings. */
const char *hypic_build_kernel_name(const hypic_build_args *args);
const char *hypic_compose_kernel_name(const hypic_compose_args *args);

/* Synchronise `stream`, then read and clear the current device's status word: HYPIC_OK,
 * HYPIC_ERR_TIMEOUT or HYPIC_ERR_RANGE (HYPIC_ERR_BOUNDS, before both, in a library built with
 * HYPIC_DEBUG_BOUNDS: an index check in a kernel failed and that kernel skipped the access and
 * its remaining work); HYPIC_ERR_CUDA if the synchronisation failed. */
hypic_status hypic_get_device_status(void *stream);

/* Diagnostic for the kernels' failure path, so that it can be exercised on a GPU without
 * making any real kernel hang. The pages have no counterpart. Launches one CTA per SM of
 * the current device; each allocates tensor memory the way the build and compose kernels
 * do, waits on an mbarrier that nothing ever arrives at with the library's bounded wait
 * and a wall-clock limit of limit_us microseconds (1 .. 1,000,000), records
 * HYPIC_ERR_TIMEOUT in the device status word when the limit runs out (always, by
 * construction), passes the give-up on to a second wait through the CTA's abort flag as
 * the multi-role kernels do, frees its tensor memory and returns. Asynchronous on `stream`;
 * hypic_get_device_status() then reports HYPIC_ERR_TIMEOUT. Returns HYPIC_ERR_INVALID_ARG
 * for a limit outside the range, HYPIC_ERR_CUDA if the launch fails. */
hypic_status hypic_probe_wait_timeout(uint32_t limit_us, void *stream);

/* Static, NUL-terminated description of a status code. */
const char *hypic_status_string(hypic_status status);

/* Library ABI version (incremented on any change to the structs above or to the meaning of
 * their fields). 3: P_total needs lam_total and may carry a power-of-two scale. 4: KDA; the
 * build's q, O and S_init. 5: KDA on the tensor cores (its workspace, its lam);
 * HYPIC_ERR_BOUNDS; the convolution-state warm-up (hypic_warmup_args). */
int32_t hypic_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HYPIC_H */
