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

// x . z over D elements (x in shared memory, z in registers) as eight independent partial
// sums, so that the dependent chain is D / 8 fused multiply-adds long rather than D.
template <int D>
__device__ __forceinline__ float dot(const float *x, const float (&z)[D]) {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < D; i += 8) {
        const float4 x0 = *reinterpret_cast<const float4 *>(x + i);
        const float4 x1 = *reinterpret_cast<const float4 *>(x + i + 4);
        a[0] = fmaf(x0.x, z[i], a[0]);
        a[1] = fmaf(x0.y, z[i + 1], a[1]);
        a[2] = fmaf(x0.z, z[i + 2], a[2]);
        a[3] = fmaf(x0.w, z[i + 3], a[3]);
        a[4] = fmaf(x1.x, z[i + 4], a[4]);
        a[5] = fmaf(x1.y, z[i + 5], a[5]);
        a[6] = fmaf(x1.z, z[i + 6], a[6]);
        a[7] = fmaf(x1.w, z[i + 7], a[7]);
    }
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Every family, stepped token by token in fp32: thread n owns column n of the augmented state
// Z = [S | P] (d_k rows in registers; P only for the dense families DELTA / GDN / KDA, whose
// transition is not a scalar or a diagonal). Per token t, with the family's gate A_t:
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
template <int D>
__global__ void __launch_bounds__(2 * D)
build_seq_kernel(const __grid_constant__ BuildParams p) {
    __shared__ __align__(16) float ks[kSeqChunk][D];
    __shared__ __align__(16) float vs[kSeqChunk][D];
    __shared__ __align__(16) float qs[kSeqChunk][D];
    __shared__ __align__(16) float gs[kSeqChunk][D];   // exp of the gate: per channel, or [tt][0]
    __shared__ float lgs[kSeqChunk];                     // per-token log gate (SCALAR / GDN), KDA: m_t
    __shared__ float bs[kSeqChunk];

    const int fam = p.family;
    const SegEntry seg = p.seg[blockIdx.x / p.H_v];
    const int h = blockIdx.x % p.H_v;
    const int hk = h / p.gqa;
    const int n = threadIdx.x;
    const bool is_S = n < D;
    const bool delta = fam == HYPIC_FAM_DELTA || fam == HYPIC_FAM_GDN || fam == HYPIC_FAM_KDA;
    const bool chan = fam == HYPIC_FAM_DIAG || fam == HYPIC_FAM_KDA;   // per-channel gates
    const bool tok_gate = fam == HYPIC_FAM_GDN || (fam == HYPIC_FAM_SCALAR && !p.log_gamma);
    const bool outs = p.O != nullptr;
    const int nthr = blockDim.x;
    const int nwarp = nthr >> 5;
    const float const_lg = (fam == HYPIC_FAM_SCALAR && p.log_gamma) ? p.log_gamma[h] : 0.f;
    const float const_g = expf(const_lg);
    const int64_t unit = (int64_t)seg.idx * p.seg_stride + h;

    float z[D];
    if (is_S && p.S_init) {
        const float *s0 = p.S_init + ((int64_t)seg.idx * p.H_v + h) * D * D + n;
#pragma unroll
        for (int i = 0; i < D; ++i) z[i] = s0[(int64_t)i * D];
    } else {
#pragma unroll
        for (int i = 0; i < D; ++i) z[i] = (!is_S && i == n - D) ? 1.f : 0.f;
    }
    float lam_acc = 0.f;   // thread 0: sum of the scalar log-gates; DIAG: thread n, channel n

    for (int t0 = 0; t0 < seg.len; t0 += kSeqChunk) {
        const int nt = min(kSeqChunk, seg.len - t0);
        __syncthreads();
        for (int e = n; e < nt * D; e += nthr) {
            const int tt = e / D, d = e % D;
            const int64_t tok = (int64_t)seg.start + t0 + tt;
            ks[tt][d] = load_in(p.k, (tok * p.H_k + hk) * D + d, p.dtype);
            vs[tt][d] = load_in(p.v, (tok * p.H_v + h) * D + d, p.dtype);
            if (outs) qs[tt][d] = load_in(p.q, (tok * p.H_k + hk) * D + d, p.dtype);
            if (chan) gs[tt][d] = p.log_gate[(tok * p.H_v + h) * D + d];   // log, exponentiated below
        }
        if (n < nt) {
            const int64_t tok = (int64_t)seg.start + t0 + n;
            bs[n] = delta ? p.beta[tok * p.H_v + h] : 0.f;
            lgs[n] = tok_gate ? p.log_gate[tok * p.H_v + h] : const_lg;
        }
        __syncthreads();
        if (fam == HYPIC_FAM_KDA) {   // m_t = max_i log a_t[i], one warp per token
            for (int tt = n >> 5; tt < nt; tt += nwarp) {
                float m = -INFINITY;
                for (int d = n & 31; d < D; d += 32) m = fmaxf(m, gs[tt][d]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if ((n & 31) == 0) lgs[tt] = m;
            }
            __syncthreads();
        }
        if (chan) {
            for (int e = n; e < nt * D; e += nthr) {
                const int tt = e / D, d = e % D;
                const float lg = gs[tt][d];
                gs[tt][d] = expf(lg);
            }
            __syncthreads();
        }
        for (int tt = 0; tt < nt; ++tt) {
            const int64_t tok = (int64_t)seg.start + t0 + tt;
            // the gate
            if (fam == HYPIC_FAM_SCALAR || (fam == HYPIC_FAM_GDN && is_S)) {
                const float g = (fam == HYPIC_FAM_SCALAR && p.log_gamma) ? const_g : expf(lgs[tt]);
#pragma unroll
                for (int i = 0; i < D; ++i) z[i] *= g;
            } else if (fam == HYPIC_FAM_DIAG || (fam == HYPIC_FAM_KDA && is_S)) {
#pragma unroll
                for (int i = 0; i < D; i += 4) {
                    const float4 g = *reinterpret_cast<const float4 *>(&gs[tt][i]);
                    z[i] *= g.x, z[i + 1] *= g.y, z[i + 2] *= g.z, z[i + 3] *= g.w;
                }
            } else if (fam == HYPIC_FAM_KDA) {   // P half: Diag(a e^-m)
                const float em = expf(-lgs[tt]);
#pragma unroll
                for (int i = 0; i < D; i += 4) {
                    const float4 g = *reinterpret_cast<const float4 *>(&gs[tt][i]);
                    z[i] *= g.x * em, z[i + 1] *= g.y * em, z[i + 2] *= g.z * em, z[i + 3] *= g.w * em;
                }
            }
            if (delta) {
                const float w = dot<D>(ks[tt], z);
                const float coef = bs[tt] * ((is_S ? vs[tt][n] : 0.f) - w);
#pragma unroll
                for (int i = 0; i < D; i += 4) {
                    const float4 kk = *reinterpret_cast<const float4 *>(&ks[tt][i]);
                    z[i] = fmaf(coef, kk.x, z[i]);
                    z[i + 1] = fmaf(coef, kk.y, z[i + 1]);
                    z[i + 2] = fmaf(coef, kk.z, z[i + 2]);
                    z[i + 3] = fmaf(coef, kk.w, z[i + 3]);
                }
            } else {
                const float vn = vs[tt][n];
#pragma unroll
                for (int i = 0; i < D; i += 4) {
                    const float4 kk = *reinterpret_cast<const float4 *>(&ks[tt][i]);
                    z[i] = fmaf(kk.x, vn, z[i]);
                    z[i + 1] = fmaf(kk.y, vn, z[i + 1]);
                    z[i + 2] = fmaf(kk.z, vn, z[i + 2]);
                    z[i + 3] = fmaf(kk.w, vn, z[i + 3]);
                }
            }
            if (outs && is_S) {
                const float o = dot<D>(qs[tt], z);
                const int64_t oi = (tok * p.H_v + h) * D + n;
                if (p.dtype == HYPIC_BF16) reinterpret_cast<__nv_bfloat16 *>(p.O)[oi] = __float2bfloat16_rn(o);
                else reinterpret_cast<float *>(p.O)[oi] = o;
            }
            if (n == 0 && fam != HYPIC_FAM_DIAG) lam_acc += lgs[tt];
        }
        if (fam == HYPIC_FAM_DIAG && is_S)   // lam of channel n: the chunk's log gates
            for (int tt = 0; tt < nt; ++tt)
                lam_acc += p.log_gate[(((int64_t)seg.start + t0 + tt) * p.H_v + h) * D + n];
    }

    float *out = is_S ? p.S + unit * D * D + n : p.P + unit * D * D + (n - D);
#pragma unroll
    for (int i = 0; i < D; ++i) out[(int64_t)i * D] = z[i];
    if (fam == HYPIC_FAM_DIAG) {
        if (is_S) p.lam[unit * D + n] = lam_acc;
    } else if (n == 0) {
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
    const int blocks = p.n_seg * p.H_v;
    const bool dense = p.family == HYPIC_FAM_DELTA || p.family == HYPIC_FAM_GDN || p.family == HYPIC_FAM_KDA;
    switch (p.D) {
    case 32: return launch_1d(build_seq_kernel<32>, blocks, dense ? 64 : 32, p, s);
    case 64: return launch_1d(build_seq_kernel<64>, blocks, dense ? 128 : 64, p, s);
    case 128: return launch_1d(build_seq_kernel<128>, blocks, dense ? 256 : 128, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
