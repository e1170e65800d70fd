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

constexpr int kDeltaChunk = 32;

// DELTA / GDN: the augmented state Z = [S | P] (d_k x 2d) is stepped token by token;
// thread n owns column n of Z in registers. S columns follow
//   S <- a (I - b k k^T) S + b k v^T = a S + b k (v - a k^T S)^T,
// P columns follow the gate-free P <- (I - b k k^T) P from P = I, and lam = sum log a.
template <int D>
__global__ void __launch_bounds__(2 * D)
build_delta_seq_kernel(const __grid_constant__ BuildParams p) {
    __shared__ __align__(16) float ks[kDeltaChunk][D];
    __shared__ float vs[kDeltaChunk][D];
    __shared__ float bs[kDeltaChunk];
    __shared__ float as[kDeltaChunk];
    __shared__ float las[kDeltaChunk];

    const SegEntry seg = p.seg[blockIdx.x / p.H_v];
    const int h = blockIdx.x % p.H_v;
    const int hk = h / p.gqa;
    const int n = threadIdx.x;
    const bool is_S = n < D;
    const bool gdn = p.family == HYPIC_FAM_GDN;

    float z[D];
#pragma unroll
    for (int i = 0; i < D; ++i) z[i] = (!is_S && i == n - D) ? 1.f : 0.f;
    float lam_acc = 0.f;

    for (int t0 = 0; t0 < seg.len; t0 += kDeltaChunk) {
        const int nt = min(kDeltaChunk, seg.len - t0);
        __syncthreads();
        for (int e = n; e < nt * D; e += 2 * D) {
            const int tt = e / D, d = e % D;
            const int64_t tok = (int64_t)seg.start + t0 + tt;
            ks[tt][d] = load_in(p.k, (tok * p.H_k + hk) * D + d, p.dtype);
            vs[tt][d] = load_in(p.v, (tok * p.H_v + h) * D + d, p.dtype);
        }
        if (n < nt) {
            const int64_t tok = (int64_t)seg.start + t0 + n;
            bs[n] = p.beta[tok * p.H_v + h];
            const float la = gdn ? p.log_gate[tok * p.H_v + h] : 0.f;
            las[n] = la;
            as[n] = gdn ? expf(la) : 1.f;
        }
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float w = 0.f;
#pragma unroll
            for (int i = 0; i < D; i += 4) {
                const float4 kk = *reinterpret_cast<const float4 *>(&ks[tt][i]);
                w = fmaf(kk.x, z[i], w);
                w = fmaf(kk.y, z[i + 1], w);
                w = fmaf(kk.z, z[i + 2], w);
                w = fmaf(kk.w, z[i + 3], w);
            }
            const float b = bs[tt];
            if (is_S) {
                const float a = as[tt];
                const float coef = b * (vs[tt][n] - a * w);
#pragma unroll
                for (int i = 0; i < D; i += 4) {
                    const float4 kk = *reinterpret_cast<const float4 *>(&ks[tt][i]);
                    z[i] = fmaf(coef, kk.x, a * z[i]);
                    z[i + 1] = fmaf(coef, kk.y, a * z[i + 1]);
                    z[i + 2] = fmaf(coef, kk.z, a * z[i + 2]);
                    z[i + 3] = fmaf(coef, kk.w, a * z[i + 3]);
                }
            } else {
                const float coef = -b * w;
#pragma unroll
                for (int i = 0; i < D; i += 4) {
                    const float4 kk = *reinterpret_cast<const float4 *>(&ks[tt][i]);
                    z[i] = fmaf(coef, kk.x, z[i]);
                    z[i + 1] = fmaf(coef, kk.y, z[i + 1]);
                    z[i + 2] = fmaf(coef, kk.z, z[i + 2]);
                    z[i + 3] = fmaf(coef, kk.w, z[i + 3]);
                }
            }
            if (n == 0) lam_acc += las[tt];
        }
    }

    const int64_t unit = (int64_t)seg.idx * p.seg_stride + h;
    float *out = is_S ? p.S + unit * D * D + n : p.P + unit * D * D + (n - D);
#pragma unroll
    for (int i = 0; i < D; ++i) out[(int64_t)i * D] = z[i];
    if (n == 0) p.lam[unit] = lam_acc;
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

cudaError_t launch_build_delta_seq(const BuildParams &p, cudaStream_t s) {
    const int blocks = p.n_seg * p.H_v;
    switch (p.D) {
    case 32: return launch_1d(build_delta_seq_kernel<32>, blocks, 64, p, s);
    case 64: return launch_1d(build_delta_seq_kernel<64>, blocks, 128, p, s);
    case 128: return launch_1d(build_delta_seq_kernel<128>, blocks, 256, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
