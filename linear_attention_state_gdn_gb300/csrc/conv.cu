// conv.cu -- the convolution of the convolution-state warm-up's head tokens.
//
// "Cut First-Token Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For linear
// layers": for convolutional variants HYPIC adds a "convolution state warm-up" patch. The short
// convolution is read from the Gated DeltaNet layer ("Gated Delta Networks: Improving Mamba2
// with Delta Rule", reference 7 of the episode-companion page): per channel c of head h,
//     y_t[c] = silu(sum_{tau < K} w[h D + c][tau] x_{t-K+1+tau}[c]),   silu(z) = z / (1 + e^-z),
// with x taken as 0 before the prompt's first token, and for the delta-rule families the keys
// L2-normalised per token and head. A segment's first min(K - 1, length) tokens are its head:
// their windows reach into the segment before, so they are convolved here over the prompt's raw
// stream, in fp32, into compact arrays that the exact build then consumes. One CTA per (head
// row, key or value head), one thread per channel; the same CTAs gather the rows' gates and b.
#include "internal.cuh"

namespace hypic {
namespace {

__global__ void __launch_bounds__(128) conv_heads_kernel(const __grid_constant__ ConvHeadParams p) {
    const int r = blockIdx.x;
    const int c = threadIdx.x;
    const bool isk = (int)blockIdx.y < p.H_k;
    const int h = isk ? (int)blockIdx.y : (int)blockIdx.y - p.H_k;
    const int H = isk ? p.H_k : p.H_v;
    // the segment of row r: the last j with head_off[j] <= r (empty heads come and go)
    int lo = 0, hi = p.n_seg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.head_off[mid] <= r) lo = mid;
        else hi = mid - 1;
    }
    if (!in_bounds(r >= p.head_off[lo] && r < p.head_off[lo + 1], p.err)) return;   // uniform
    const int64_t t = (int64_t)p.seg_start[lo] + (r - p.head_off[lo]);
    const void *x = isk ? p.k_raw : p.v_raw;
    const float *w = (isk ? p.wk : p.wv) + ((int64_t)h * p.D + c) * p.K;
    float acc = 0.f;
    for (int tau = 0; tau < p.K; ++tau) {
        const int64_t s = t - (p.K - 1) + tau;
        if (s >= 0) acc = fmaf(w[tau], load_in(x, (s * H + h) * p.D + c, p.dtype), acc);
    }
    float y = acc / (1.f + expf(-acc));
    const bool delta = p.family == HYPIC_FAM_DELTA || p.family == HYPIC_FAM_GDN || p.family == HYPIC_FAM_KDA;
    if (isk && delta) {   // L2 norm over the head's D channels (one to four warps)
        __shared__ float part[4];
        float ss = y * y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((c & 31) == 0) part[c >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < p.D / 32; ++i) tot += part[i];
        const float n = sqrtf(tot);
        y = n > 0.f ? y / n : 0.f;
    }
    float *out = isk ? p.k_head : p.v_head;
    out[((int64_t)r * H + h) * p.D + c] = y;
    if (!isk) {   // the row's gates and b, in the build's layouts
        const bool chan = p.family == HYPIC_FAM_DIAG || p.family == HYPIC_FAM_KDA;
        if (p.g_head) {
            if (chan) p.g_head[((int64_t)r * p.H_v + h) * p.D + c] = p.log_gate[(t * p.H_v + h) * p.D + c];
            else if (c == 0) p.g_head[(int64_t)r * p.H_v + h] = p.log_gate[t * p.H_v + h];
        }
        if (p.b_head && c == 0) p.b_head[(int64_t)r * p.H_v + h] = p.beta[t * p.H_v + h];
    }
}

}  // namespace

cudaError_t launch_conv_heads(const ConvHeadParams &p, cudaStream_t s) {
    if (p.n_rows == 0) return cudaSuccess;
    if (p.D > 128 || p.D % 32 != 0) return cudaErrorInvalidValue;
    conv_heads_kernel<<<dim3((unsigned)p.n_rows, (unsigned)(p.H_k + p.H_v)), p.D, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hypic
