// compose.cu -- prefix scan of the composition prefix_j = T_j prefix_{j-1} + S_j over the
// cached segments of many (layer, head) units ("Cut First-Token Latency by 3.25x:
// Introducing HYPIC ..." (besthub.dev), paragraph "For linear layers": reuse composes
// T_C2 . S(C1) + S(C2); paragraph on segment parallelism: the combine worker assembles the
// final state).
//
// compose_scaled: scalar and diagonal transitions, T_j = exp(lam_j) (per unit or per row).
//   A pure element-wise stream: each thread carries 4 consecutive state elements of one
//   unit through all segments, the S loads (and log-scales) of up to 16 segments in flight.
//   It also sums lam_total when asked (the first thread of each unit, or of each row for
//   diagonal gates) and, with prefix_last (a build composing the pieces of its segments),
//   writes only the last state. It is a programmatic dependent launch: it waits for the
//   kernel before it on the stream (the build of the pieces) before any global access.
// compose_dense_simt: dense transitions T_j = exp(lam_j) P_j on CUDA cores, used for head
//   sizes below 128 (the d = 128 case runs on the tensor cores, compose_tc.cu). With P_total
//   requested, units U .. 2U-1 of the grid carry the transition chain P_j ... P_0 instead.
// compose_lam_total: the log-scale of the composed transition, sum_j lam_j (the transition
//   of an entry composed from consecutive segments is T_{n-1} ... T_0).
#include "internal.cuh"

namespace hypic {
namespace {

constexpr int kScaledThreads = 256;
constexpr int kAhead = 16;   // segments whose S loads are in flight at once

__device__ __forceinline__ float4 ldg_stream(const float *p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void stg_stream(float *p, float4 v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

__global__ void __launch_bounds__(kScaledThreads)
compose_scaled_kernel(const __grid_constant__ ComposeParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int D = p.D;
    const int n4 = D * D / 4;
    const int bpu = (n4 + kScaledThreads - 1) / kScaledThreads;   // blocks per unit
    const int64_t u = blockIdx.x / bpu;
    const int e4 = (blockIdx.x % bpu) * kScaledThreads + threadIdx.x;
    if (e4 >= n4) return;
    const int row = (e4 * 4) / D;
    const int64_t DD = (int64_t)D * D;
    const bool diag = p.family == HYPIC_FAM_DIAG;
    const bool has_lam = p.family != HYPIC_FAM_LINEAR && p.lam != nullptr;

    float4 cur = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.S0) cur = ldg_stream(p.S0 + u * DD + e4 * 4);

    // a batch of up to kAhead segments: every S load of the batch is issued before the first is
    // used (the scan is short: one memory latency per batch instead of one per few segments)
    // (with the batch's log-scales: a load after a store of the loop below would wait for it)
    float4 ring[kAhead];
    float lv[kAhead];
    float lsum = 0.f;
    for (int j0 = 0; j0 < p.n_seg; j0 += kAhead) {
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            const int j = j0 + a;
            if (j < p.n_seg) {
                ring[a] = ldg_stream(compose_seg(p.S, p.S1, j, p.n_units, u, DD) + e4 * 4);
                lv[a] = !has_lam ? 0.f
                        : diag ? compose_seg(p.lam, p.lam1, j, p.n_units, u, D)[row]
                               : *compose_seg(p.lam, p.lam1, j, p.n_units, u, 1);
            }
        }
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            const int j = j0 + a;
            if (j < p.n_seg) {
                const float4 x = ring[a];
                const float sc = has_lam ? expf(lv[a]) : 1.f;
                lsum += lv[a];
                cur.x = fmaf(sc, cur.x, x.x);
                cur.y = fmaf(sc, cur.y, x.y);
                cur.z = fmaf(sc, cur.z, x.z);
                cur.w = fmaf(sc, cur.w, x.w);
                if (!p.prefix_last)
                    stg_stream(p.prefix + ((int64_t)j * p.n_units + u) * DD + e4 * 4, cur);
            }
        }
    }
    if (p.prefix_last) stg_stream(p.prefix_last + u * DD + e4 * 4, cur);
    if (p.lam_total) {   // the segments' lam in order, as compose_lam_total sums them
        if (diag && (e4 * 4) % D == 0) p.lam_total[u * D + row] = lsum;
        if (!diag && e4 == 0) p.lam_total[u] = lsum;
    }
}

constexpr int kDenseThreads = 256;
constexpr int kDenseCols = 32;

// One CTA per (unit, block of 32 state columns). The column block X of prefix_{j-1} stays
// in shared memory; P_j is staged whole; each thread forms RPT x 4 outputs.
template <int D>
__global__ void __launch_bounds__(kDenseThreads)
compose_dense_simt_kernel(const __grid_constant__ ComposeParams p) {
    constexpr int LDA = D + 4;
    constexpr int RPT = D * kDenseCols / kDenseThreads / 4;   // rows per thread
    extern __shared__ __align__(16) float smem[];
    float *A = smem;                   // [D][LDA]
    float *X = smem + D * LDA;         // [D][kDenseCols]

    // units 0 .. U-1: the prefix scan; U .. 2U-1 (with P_total): the transition chain
    // Q_j = P_j Q_{j-1}, Q_0 = P_0, of unit u - U, written once at the end
    const int64_t ublk = blockIdx.x / (D / kDenseCols);
    const bool trans = ublk >= p.n_units;
    const int64_t u = trans ? ublk - p.n_units : ublk;
    const int cb = (blockIdx.x % (D / kDenseCols)) * kDenseCols;
    const int tid = threadIdx.x;
    const int tx = tid % (kDenseCols / 4);   // 4-column group
    const int ty = tid / (kDenseCols / 4);   // row group
    const int64_t DD = (int64_t)D * D;

    bool have_state = trans || p.S0 != nullptr;
    if (have_state) {
        const float *X0 = trans ? p.P + u * DD : p.S0 + u * DD;
        for (int e = tid; e < D * kDenseCols; e += kDenseThreads)
            X[e] = X0[(int64_t)(e / kDenseCols) * D + cb + e % kDenseCols];
    }

    for (int j = trans ? 1 : 0; j < p.n_seg; ++j) {
        const int64_t base = ((int64_t)j * p.n_units + u) * DD;   // of prefix_j
        const float *Pj = compose_seg(p.P, p.P1, j, p.n_units, u, DD);
        const float *Sj = compose_seg(p.S, p.S1, j, p.n_units, u, DD);
        float acc[RPT][4];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
        if (have_state) {
            __syncthreads();
            for (int e = tid; e < D * D / 4; e += kDenseThreads) {
                const int r = (e * 4) / D, c = (e * 4) % D;
                const float4 a = *reinterpret_cast<const float4 *>(Pj + (int64_t)r * D + c);
                *reinterpret_cast<float4 *>(&A[r * LDA + c]) = a;
            }
            __syncthreads();
#pragma unroll 4
            for (int m = 0; m < D; ++m) {
                const float4 x = *reinterpret_cast<const float4 *>(&X[m * kDenseCols + tx * 4]);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const float a = A[(ty * RPT + r) * LDA + m];
                    acc[r][0] = fmaf(a, x.x, acc[r][0]);
                    acc[r][1] = fmaf(a, x.y, acc[r][1]);
                    acc[r][2] = fmaf(a, x.z, acc[r][2]);
                    acc[r][3] = fmaf(a, x.w, acc[r][3]);
                }
            }
        }
        const float sc = trans ? 1.f : have_state ? expf(*compose_seg(p.lam, p.lam1, j, p.n_units, u, 1)) : 0.f;
        __syncthreads();   // every thread is done reading X
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = ty * RPT + r;
            const int64_t off = base + (int64_t)row * D + cb + tx * 4;
            const int64_t in_off = (int64_t)row * D + cb + tx * 4;
            if (trans) {
                *reinterpret_cast<float4 *>(&X[row * kDenseCols + tx * 4]) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                continue;
            }
            const float4 s = *reinterpret_cast<const float4 *>(Sj + in_off);
            float4 o;
            o.x = fmaf(sc, acc[r][0], s.x);
            o.y = fmaf(sc, acc[r][1], s.y);
            o.z = fmaf(sc, acc[r][2], s.z);
            o.w = fmaf(sc, acc[r][3], s.w);
            *reinterpret_cast<float4 *>(p.prefix + off) = o;
            *reinterpret_cast<float4 *>(&X[row * kDenseCols + tx * 4]) = o;
        }
        have_state = true;
    }
    if (trans) {
        __syncthreads();
        for (int e = tid; e < D * kDenseCols; e += kDenseThreads)
            p.P_total[u * DD + (int64_t)(e / kDenseCols) * D + cb + e % kDenseCols] = X[e];
    }
}

__global__ void __launch_bounds__(256) compose_lam_total_kernel(const __grid_constant__ ComposeParams p) {
    const int nl = p.family == HYPIC_FAM_DIAG ? p.D : 1;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // unit * nl + row
    if (i >= p.n_units * nl) return;
    float acc = 0.f;
    if (p.family != HYPIC_FAM_LINEAR)
        for (int j = 0; j < p.n_seg; ++j)
            acc += (j == 1 && p.lam1) ? p.lam1[i] : p.lam[(int64_t)j * p.n_units * nl + i];
    p.lam_total[i] = acc;
}

template <int D>
cudaError_t launch_dense(const ComposeParams &p, cudaStream_t s) {
    const size_t smem = sizeof(float) * (D * (D + 4) + D * kDenseCols);
    cudaError_t e = cudaFuncSetAttribute(compose_dense_simt_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.n_units * (p.P_total ? 2 : 1) * (D / kDenseCols)));
    compose_dense_simt_kernel<D><<<grid, kDenseThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compose_scaled(const ComposeParams &p, cudaStream_t s) {
    if (p.n_seg == 0 || p.n_units == 0) return cudaSuccess;
    if (p.S1 && (p.n_seg != 2 || !p.lam1)) return cudaErrorInvalidValue;   // segment 1 of a two-segment scan
    const int n4 = p.D * p.D / 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_units * ((n4 + kScaledThreads - 1) / kScaledThreads)));
    cfg.blockDim = dim3(kScaledThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, compose_scaled_kernel, p);
}

cudaError_t launch_compose_lam_total(const ComposeParams &p, cudaStream_t s) {
    if (p.n_units == 0 || !p.lam_total) return cudaSuccess;
    if (p.lam1 && p.n_seg != 2) return cudaErrorInvalidValue;
    const int64_t n = p.n_units * (p.family == HYPIC_FAM_DIAG ? p.D : 1);
    compose_lam_total_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_compose_dense_simt(const ComposeParams &p, cudaStream_t s) {
    if (p.n_seg == 0 || p.n_units == 0) return cudaSuccess;
    if (p.S1 && (p.n_seg != 2 || !p.lam1 || !p.P1)) return cudaErrorInvalidValue;   // segment 1 of a two-segment scan
    switch (p.D) {
    case 32: return launch_dense<32>(p, s);
    case 64: return launch_dense<64>(p, s);
    case 128: return launch_dense<128>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
