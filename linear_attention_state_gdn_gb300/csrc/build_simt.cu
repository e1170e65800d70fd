// build_simt.cu -- CUDA-core (FFMA) segment builds, one CTA per (segment, value head).
//
// These step the recurrence token by token with the state held in registers. They are
// the exact-fp32 path (fp32 inputs, where a 1e-4 relative error budget rules out bf16 or
// tf32 tensor-core operands) and the path for head sizes the tensor-core kernels do not
// take (d = 32, 64).
//
// What is computed: the pair (S(C|0), T_C) of every cached segment ("Cut First-Token
// Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For linear layers";
// "HYPIC: Cache Acceleration for Hybrid Attention Models", "Core Approach"), with T_C in
// the log-scaled form T_C = exp(lam) P.
#include "internal.cuh"

namespace hypic {
namespace {

constexpr int kGatedThreads = 256;
constexpr int kGatedChunk = 16;

// LINEAR / SCALAR / DIAG: S_t = Diag(g_t) S_{t-1} + k_t v_t^T (g = 1 for LINEAR, a scalar
// per token or per head for SCALAR, a vector for DIAG). Thread owns row i of S and NC
// consecutive columns.
template <int D>
__global__ void __launch_bounds__(kGatedThreads)
build_gated_simt_kernel(const __grid_constant__ BuildParams p) {
    constexpr int NC = D * D / kGatedThreads;     // columns per thread
    constexpr int GROUPS = D / NC;                // threads per row
    __shared__ __align__(16) float ks[kGatedChunk][D];
    __shared__ __align__(16) float vs[kGatedChunk][D];
    __shared__ __align__(16) float gs[kGatedChunk][D];

    if (!in_bounds((int)(blockIdx.x / p.H_v) < p.n_seg, p.err)) return;
    const SegEntry seg = p.seg[blockIdx.x / p.H_v];
    const int h = blockIdx.x % p.H_v;
    const int hk = h / p.gqa;
    const int tid = threadIdx.x;
    const int i = tid / GROUPS;
    const int c0 = (tid % GROUPS) * NC;
    const int fam = p.family;

    float s[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) s[c] = 0.f;
    float lam_acc = 0.f;
    const float const_lg = (fam == HYPIC_FAM_SCALAR && p.log_gamma) ? p.log_gamma[h] : 0.f;
    const float const_g = expf(const_lg);

    for (int t0 = 0; t0 < seg.len; t0 += kGatedChunk) {
        const int nt = min(kGatedChunk, seg.len - t0);
        __syncthreads();
        for (int e = tid; e < nt * D; e += kGatedThreads) {
            const int tt = e / D, d = e % D;
            const int64_t tok = (int64_t)seg.start + t0 + tt;
            ks[tt][d] = load_in(p.k, (tok * p.H_k + hk) * D + d, p.dtype);
            vs[tt][d] = load_in(p.v, (tok * p.H_v + h) * D + d, p.dtype);
            if (fam == HYPIC_FAM_DIAG)
                gs[tt][d] = p.log_gate[(tok * p.H_v + h) * D + d];
            else if (d == 0)
                gs[tt][0] = (fam == HYPIC_FAM_SCALAR && !p.log_gamma) ? p.log_gate[tok * p.H_v + h]
                                                                        : const_lg;
        }
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            const float lg = (fam == HYPIC_FAM_DIAG) ? gs[tt][i] : gs[tt][0];
            float g;
            if (fam == HYPIC_FAM_LINEAR) g = 1.f;
            else if (fam == HYPIC_FAM_SCALAR && p.log_gamma) g = const_g;
            else g = expf(lg);
            lam_acc += lg;
            const float ki = ks[tt][i];
#pragma unroll
            for (int c = 0; c < NC; c += 4) {
                const float4 vv = *reinterpret_cast<const float4 *>(&vs[tt][c0 + c]);
                s[c + 0] = fmaf(g, s[c + 0], ki * vv.x);
                s[c + 1] = fmaf(g, s[c + 1], ki * vv.y);
                s[c + 2] = fmaf(g, s[c + 2], ki * vv.z);
                s[c + 3] = fmaf(g, s[c + 3], ki * vv.w);
            }
        }
    }

    const int64_t unit = (int64_t)seg.idx * p.seg_stride + h;
    float *S = p.S + unit * D * D + (int64_t)i * D + c0;
#pragma unroll
    for (int c = 0; c < NC; c += 4)
        *reinterpret_cast<float4 *>(S + c) = make_float4(s[c], s[c + 1], s[c + 2], s[c + 3]);
    if (tid % GROUPS == 0) {
        if (fam == HYPIC_FAM_DIAG) {
            p.lam[unit * D + i] = lam_acc;
        } else if (i == 0) {
            float lam = 0.f;
            if (fam == HYPIC_FAM_SCALAR) lam = p.log_gamma ? (float)seg.len * const_lg : lam_acc;
            p.lam[unit] = lam;
        }
    }
}

constexpr int kSeqChunk = 16;

// Every family, stepped token by token in fp32. One CTA carries one half of a unit's
// augmented state Z = [S | P]: the S half, or the P half (only for the dense families DELTA /
// GDN / KDA, whose transition is not a scalar or a diagonal). Column n of the half is held in
// registers by TPC adjacent threads, RPT = D / TPC rows each; dot products over a column are
// partial sums over a thread's rows combined by shuffles inside the group. Per token t, with
// the family's gate A_t:
//   S <- A_t S                 A_t = g I (SCALAR), Diag(g) (DIAG), a I (GDN), Diag(a) (KDA)
//   S <- S + b k (v - k^T S)^T  (DELTA / GDN / KDA: the delta update)
//   S <- S + k v^T              (LINEAR / SCALAR / DIAG: the write)
//   P <- P~ then P <- P - b k (k^T P), P~ = P (DELTA, GDN: gate-free) or
//        Diag(a e^-m) P with m = max_i log a[i] (KDA), so lam = sum m and T = exp(lam) P
//   o_t = S^T q_t               (when the outputs are requested, read after the token)
// Each segment starts from S_init (when given) or zero. This is the exact path (fp32 inputs,
// where a 1e-4 relative error budget rules out bf16 or tf32 tensor-core operands), the path
// of the head sizes and families the tensor-core builds do not take (d = 32, 64; KDA), and
// the path of every build that asks for the segment outputs.
//
// Shared-memory vectors (k, q, per-channel gates) keep the rows of thread part r in 4-element
// chunks permuted by chunk ^ r, so that the TPC parts of a column group, which read the same
// chunk index of different row ranges at once, hit different banks.
template <int D, int TPC>
__device__ __forceinline__ int sidx(int i) {
    constexpr int RPT = D / TPC;
    return (i / RPT) * RPT + ((((i % RPT) >> 2) ^ (i / RPT)) << 2) + (i & 3);
}

// Partial x . z over this thread's RPT rows (x a swizzled shared vector, part r), as four
// independent sums, combined over the TPC threads of the column.
template <int D, int TPC>
__device__ __forceinline__ float col_dot(const float *x, const float (&z)[D / TPC], int r) {
    constexpr int RPT = D / TPC;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    const float *xr = x + r * RPT;
#pragma unroll
    for (int j = 0; j < RPT / 4; ++j) {
        const float4 v = *reinterpret_cast<const float4 *>(xr + ((j ^ r) << 2));
        a[0] = fmaf(v.x, z[4 * j], a[0]);
        a[1] = fmaf(v.y, z[4 * j + 1], a[1]);
        a[2] = fmaf(v.z, z[4 * j + 2], a[2]);
        a[3] = fmaf(v.w, z[4 * j + 3], a[3]);
    }
    float w = (a[0] + a[1]) + (a[2] + a[3]);
#pragma unroll
    for (int o = 1; o < TPC; o <<= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    return w;
}

template <int D, int TPC>
__global__ void __launch_bounds__(D * TPC)
build_seq_kernel(const __grid_constant__ BuildParams p) {
    constexpr int RPT = D / TPC;
    __shared__ __align__(16) float ks[kSeqChunk][D];
    __shared__ __align__(16) float vs[kSeqChunk][D];
    __shared__ __align__(16) float qs[kSeqChunk][D];
    __shared__ __align__(16) float gs[kSeqChunk][D];   // per-channel gates (log, then exp)
    __shared__ float lgs[kSeqChunk];                     // per-token log gate (SCALAR / GDN), KDA: m_t
    __shared__ float bs[kSeqChunk];

    const int fam = p.family;
    const bool delta = fam == HYPIC_FAM_DELTA || fam == HYPIC_FAM_GDN || fam == HYPIC_FAM_KDA;
    const int halves = delta ? 2 : 1;
    const int ux = blockIdx.x / halves;                       // (segment rank, value head)
    const bool is_S = blockIdx.x % halves == 0;               // the S half, else the P half
    if (!in_bounds(ux / p.H_v < p.n_seg, p.err)) return;      // uniform, before any set-up
    const SegEntry seg = p.seg[ux / p.H_v];
    const int h = ux % p.H_v;
    const int hk = h / p.gqa;
    const int n = threadIdx.x / TPC, r = threadIdx.x % TPC;   // column of the half, part of its rows
    const bool chan = fam == HYPIC_FAM_DIAG || fam == HYPIC_FAM_KDA;   // per-channel gates
    const bool tok_gate = fam == HYPIC_FAM_GDN || (fam == HYPIC_FAM_SCALAR && !p.log_gamma);
    const bool outs = p.O != nullptr;
    const int nthr = blockDim.x;
    const int tid = threadIdx.x;
    const float const_lg = (fam == HYPIC_FAM_SCALAR && p.log_gamma) ? p.log_gamma[h] : 0.f;
    const float const_g = expf(const_lg);
    const int64_t unit = (int64_t)seg.idx * p.seg_stride + h;

    float z[RPT];   // rows r RPT .. r RPT + RPT - 1 of column n
    if (is_S && p.S_init) {
        const float *s0 = p.S_init + ((int64_t)seg.idx * p.H_v + h) * D * D + (int64_t)r * RPT * D + n;
#pragma unroll
        for (int m = 0; m < RPT; ++m) z[m] = s0[(int64_t)m * D];
    } else {
#pragma unroll
        for (int m = 0; m < RPT; ++m) z[m] = (!is_S && r * RPT + m == n) ? 1.f : 0.f;
    }
    float lam_acc = 0.f;   // thread 0: sum of the scalar log-gates; DIAG: part 0 of column n

    for (int t0 = 0; t0 < seg.len; t0 += kSeqChunk) {
        const int nt = min(kSeqChunk, seg.len - t0);
        __syncthreads();
        for (int e = tid; e < nt * D; e += nthr) {
            const int tt = e / D, d = e % D;
            const int64_t tok = (int64_t)seg.start + t0 + tt;
            const int sd = sidx<D, TPC>(d);
            ks[tt][sd] = load_in(p.k, (tok * p.H_k + hk) * D + d, p.dtype);
            vs[tt][d] = load_in(p.v, (tok * p.H_v + h) * D + d, p.dtype);
            if (outs) qs[tt][sd] = load_in(p.q, (tok * p.H_k + hk) * D + d, p.dtype);
            if (chan) gs[tt][sd] = p.log_gate[(tok * p.H_v + h) * D + d];
        }
        if (tid < nt) {
            const int64_t tok = (int64_t)seg.start + t0 + tid;
            bs[tid] = delta ? p.beta[tok * p.H_v + h] : 0.f;
            lgs[tid] = tok_gate ? p.log_gate[tok * p.H_v + h] : const_lg;
        }
        __syncthreads();
        if (fam == HYPIC_FAM_DIAG && is_S && r == 0)   // lam of channel n: the chunk's log gates
            for (int tt = 0; tt < nt; ++tt) lam_acc += gs[tt][sidx<D, TPC>(n)];
        if (fam == HYPIC_FAM_KDA) {   // m_t = max_i log a_t[i], one warp per token
            for (int tt = tid >> 5; tt < nt; tt += nthr >> 5) {
                float m = -INFINITY;
                for (int d = tid & 31; d < D; d += 32) m = fmaxf(m, gs[tt][d]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if ((tid & 31) == 0) lgs[tt] = m;
            }
        }
        __syncthreads();
        if (chan) {
            for (int e = tid; e < nt * D; e += nthr) gs[e / D][e % D] = expf(gs[e / D][e % D]);
            __syncthreads();
        }
        for (int tt = 0; tt < nt; ++tt) {
            const int64_t tok = (int64_t)seg.start + t0 + tt;
            // the gate
            if (fam == HYPIC_FAM_SCALAR || (fam == HYPIC_FAM_GDN && is_S)) {
                const float g = (fam == HYPIC_FAM_SCALAR && p.log_gamma) ? const_g : expf(lgs[tt]);
#pragma unroll
                for (int m = 0; m < RPT; ++m) z[m] *= g;
            } else if (fam == HYPIC_FAM_DIAG || fam == HYPIC_FAM_KDA) {
                // S half: Diag(g); KDA's P half: Diag(a e^-m)
                const float em = (fam == HYPIC_FAM_KDA && !is_S) ? expf(-lgs[tt]) : 1.f;
                const float *gr = gs[tt] + r * RPT;
#pragma unroll
                for (int j = 0; j < RPT / 4; ++j) {
                    const float4 g = *reinterpret_cast<const float4 *>(gr + ((j ^ r) << 2));
                    z[4 * j] *= g.x * em, z[4 * j + 1] *= g.y * em, z[4 * j + 2] *= g.z * em,
                        z[4 * j + 3] *= g.w * em;
                }
            }
            const float *kr = ks[tt] + r * RPT;
            float coef;
            if (delta) {
                const float w = col_dot<D, TPC>(ks[tt], z, r);
                coef = bs[tt] * ((is_S ? vs[tt][n] : 0.f) - w);
            } else {
                coef = vs[tt][n];
            }
#pragma unroll
            for (int j = 0; j < RPT / 4; ++j) {   // z += coef k (the delta update or the write)
                const float4 kk = *reinterpret_cast<const float4 *>(kr + ((j ^ r) << 2));
                z[4 * j] = fmaf(coef, kk.x, z[4 * j]);
                z[4 * j + 1] = fmaf(coef, kk.y, z[4 * j + 1]);
                z[4 * j + 2] = fmaf(coef, kk.z, z[4 * j + 2]);
                z[4 * j + 3] = fmaf(coef, kk.w, z[4 * j + 3]);
            }
            if (outs && is_S) {   // uniform over the CTA: the shuffles stay inside it
                const float o = col_dot<D, TPC>(qs[tt], z, r);
                if (r == 0) {
                    const int64_t oi = (tok * p.H_v + h) * D + n;
                    if (p.dtype == HYPIC_BF16) reinterpret_cast<__nv_bfloat16 *>(p.O)[oi] = __float2bfloat16_rn(o);
                    else reinterpret_cast<float *>(p.O)[oi] = o;
                }
            }
            if (tid == 0 && fam != HYPIC_FAM_DIAG) lam_acc += lgs[tt];
        }
    }

    float *out = (is_S ? p.S : p.P) + unit * D * D + n + (int64_t)r * RPT * D;
#pragma unroll
    for (int m = 0; m < RPT; ++m) out[(int64_t)m * D] = z[m];
    if (fam == HYPIC_FAM_DIAG) {
        if (is_S && r == 0) p.lam[unit * D + n] = lam_acc;
    } else if (tid == 0 && is_S) {
        float lam = lam_acc;
        if (fam == HYPIC_FAM_LINEAR || fam == HYPIC_FAM_DELTA) lam = 0.f;
        else if (fam == HYPIC_FAM_SCALAR && p.log_gamma) lam = (float)seg.len * const_lg;
        p.lam[unit] = lam;
    }
}

template <typename K>
cudaError_t launch_1d(K kernel, int blocks, int threads, const BuildParams &p, cudaStream_t s) {
    if (blocks == 0) return cudaSuccess;
    kernel<<<blocks, threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_build_gated_simt(const BuildParams &p, cudaStream_t s) {
    const int blocks = p.n_seg * p.H_v;
    switch (p.D) {
    case 32: return launch_1d(build_gated_simt_kernel<32>, blocks, kGatedThreads, p, s);
    case 64: return launch_1d(build_gated_simt_kernel<64>, blocks, kGatedThreads, p, s);
    case 128: return launch_1d(build_gated_simt_kernel<128>, blocks, kGatedThreads, p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_build_seq(const BuildParams &p, cudaStream_t s) {
    const bool dense = p.family == HYPIC_FAM_DELTA || p.family == HYPIC_FAM_GDN || p.family == HYPIC_FAM_KDA;
    const int blocks = p.n_seg * p.H_v * (dense ? 2 : 1);   // the S and P halves of a unit apart
    switch (p.D) {   // 32 state rows per thread
    case 32: return launch_1d(build_seq_kernel<32, 1>, blocks, 32, p, s);
    case 64: return launch_1d(build_seq_kernel<64, 2>, blocks, 128, p, s);
    case 128: return launch_1d(build_seq_kernel<128, 4>, blocks, 512, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
