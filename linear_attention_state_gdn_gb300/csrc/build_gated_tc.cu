// build_gated_tc.cu -- segment build for plain linear attention, scalar decay (RetNet,
// Mamba2) and diagonal gates (GLA) on the 5th-generation tensor cores (bf16 k / v, d = 128).
//
// What is computed: for every cached segment C and value head, S(C|0) and lam with
// T_C = exp(lam) (scalar) or Diag(exp(lam)) (diagonal) ("Cut First-Token Latency by 3.25x:
// Introducing HYPIC ..." (besthub.dev), paragraph "For linear layers"; "Hypic:
// Position-Independent KV Caching for Hybrid-Attention LLM Serving", "Family comparison:
// scalar -> diagonal -> dense").
//
// Chunked form (exact algebra of S_t = Diag(g_t) S_{t-1} + k_t v_t^T): over a chunk of C
// tokens with channel log-gates l_t,
//     S <- Diag(exp(sum_t l_t)) S + Khat^T V,   Khat[t][i] = k_t[i] exp(sum_{s>t} l_s[i]),
// so every chunk is one C-deep bf16 contraction with fp32 accumulation, and no factor
// exceeds 1 (no overflow for any segment length).
//
// Data flow of one CTA (one (segment, value head) unit; two CTAs per SM):
//   * warp 8 streams k, v (and the per-channel log-gates) chunk by chunk by TMA into a
//     3-stage ring; k and v land 128B-swizzled with channels contiguous, which is directly
//     the MN-major operand layout of both MMA operands;
//   * warps 0-7 turn the chunk's gates into decay factors (one per token for linear /
//     scalar decay, one per token and channel for diagonal gates, written over the gate
//     tile; 0 past the segment end), then scale k in place into Khat with 16-byte vector
//     accesses and hand the stage to the MMA warp;
//   * warp 9 issues dS_c = Khat^T V into one of two TMEM accumulators (lane i, column n);
//   * warps 0-7 fold dS_c into the fp32 state they hold in registers (64 columns each):
//     S[i][:] = exp(sum_t l_t[i]) S[i][:] + dS_c[i][:].
// Every wait is bounded (HYPIC_ERR_TIMEOUT on expiry, after which the CTA winds down).
#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace hypic {
namespace {

using namespace ptx;

constexpr int D = 128;
constexpr int kThreads = 320;        // 8 state/decay warps, producer, MMA issuer
constexpr int kEpi = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// TMA ring depth: 3 stages at two CTAs per SM; 6 at one CTA per SM (calls with at most one
// unit per SM), whose single CTA needs more bytes in flight to keep HBM busy
// (RetNet, 128 units: 46.4 -> 41.3 us).
constexpr uint32_t kTmemCols = 256;   // two 128-column accumulators

enum { kLinear = 0, kScalar = 1, kDiag = 2 };

template <int KIND, int STAGES>
struct Geo {
    static constexpr int C = KIND == kDiag ? 32 : 64;          // tokens per chunk
    static constexpr uint32_t kHalf = C * 128;                  // 64 channels x C tokens, bf16
    static constexpr uint32_t kKV = 2 * kHalf;                  // one k (or v) chunk
    static constexpr uint32_t kG = KIND == kDiag ? C * D * 4 : 0;
    static constexpr uint32_t kStage = 2 * kKV + kG;
    static constexpr uint32_t kSmem = STAGES * kStage + 1024;
};

template <int STAGES>
struct Bars {
    uint64_t full[STAGES], kready[STAGES], empty[STAGES], dfull[2], dfree[2], fin;
};

// Named barrier of the 256 decay / state threads, plain and with an AND of a predicate (every
// thread leaves with the same outcome). Non-aligned forms: lanes may arrive at different times.
__device__ __forceinline__ void bar_state() {
    __syncwarp();
    asm volatile("barrier.sync 1, 256;" ::: "memory");
}
__device__ __forceinline__ bool bar_state_and(bool v) {
    uint32_t r;
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.red.and.pred po, 1, 256, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

template <int KIND, int STAGES>
__global__ void __launch_bounds__(kThreads, STAGES == 3 ? 2 : 1)
build_gated_tc_kernel(const __grid_constant__ BuildParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG) {
    constexpr int kStages = STAGES;
    using G = Geo<KIND, STAGES>;
    constexpr int C = G::C;
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived by offsetting the shared array itself so that the
    // compiler keeps the shared address space (plain ld/st.shared, not generic accesses)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars<STAGES> bars;
    __shared__ uint32_t tslot;
    __shared__ volatile int abort_flag;
    __shared__ __align__(16) float fac[kStages][64];   // per-token decay factors (linear / scalar)
    __shared__ float gtot[2][D];                        // chunk log-decay (per channel for diagonal)
    __shared__ float scan_tmp[2];

    const int warp = warp_id(), lane = lane_id();
    if (!in_bounds((int)(blockIdx.x / p.H_v) < p.n_seg, p.err)) return;   // uniform, before any set-up
    const SegEntry seg = p.seg[blockIdx.x / p.H_v];
    const int h = blockIdx.x % p.H_v;
    const int hk = h / p.gqa;
    const int nchunks = (seg.len + C - 1) / C;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.kready[s], kEpi);
            mbar_init(&bars.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.dfull[b], 1);
            mbar_init(&bars.dfree[b], kEpi);
        }
        mbar_init(&bars.fin, 1);
        abort_flag = 0;
        fence_mbar_init();
        // the kernel after this one (the merge of split segments) may launch and set up on SMs
        // this grid has left; it waits for this grid's completion before any access
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(&tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            if (KIND == kDiag) prefetch_tmap(&tmG);
            int c = 0;
            for (; c < nchunks; ++c) {
                const int s = c % kStages, use = c / kStages;
                if (use >= 1 && !mbar_wait_or_abort_compact(&bars.empty[s], (use - 1) & 1, p.err, kErrTimeout,
                                                    &abort_flag))
                    break;
                uint8_t *st = smem + s * G::kStage;
                const int32_t t0 = seg.start + c * C;
                mbar_arrive_expect_tx(&bars.full[s], G::kStage);
                tma_load_3d(st, &tmK, &bars.full[s], 0, hk, t0);
                tma_load_3d(st + G::kHalf, &tmK, &bars.full[s], 64, hk, t0);
                tma_load_3d(st + G::kKV, &tmV, &bars.full[s], 0, h, t0);
                tma_load_3d(st + G::kKV + G::kHalf, &tmV, &bars.full[s], 64, h, t0);
                if (KIND == kDiag) tma_load_3d(st + 2 * G::kKV, &tmG, &bars.full[s], 0, h, t0);
            }
            if (abort_flag)   // let the copies in flight land before leaving (bounded)
                for (int q = (c > kStages ? c - kStages : 0); q < c; ++q)
                    mbar_wait(&bars.full[q % kStages], (q / kStages) & 1, p.err, kErrTimeout);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t id = idesc(kFmtBF16, kFmtBF16, true, true, 128, 128);
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kStages, use = c / kStages, b = c & 1, buse = c >> 1;
                if (!mbar_wait_or_abort_compact(&bars.kready[s], use & 1, p.err, kErrTimeout, &abort_flag))
                    break;
                if (buse >= 1 && !mbar_wait_or_abort_compact(&bars.dfree[b], (buse - 1) & 1, p.err,
                                                     kErrTimeout, &abort_flag))
                    break;
                tc_fence_after();
                const uint32_t ka = smem_u32(smem + s * G::kStage);
                const uint32_t va = ka + G::kKV;
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16(tmem + b * 128, sdesc(ka + k * 2048, G::kHalf, 1024, kSwizzle128B),
                             sdesc(va + k * 2048, G::kHalf, 1024, kSwizzle128B), id, k > 0);
                mma_commit(&bars.empty[s]);
                mma_commit(&bars.dfull[b]);
            }
            if (abort_flag) {
                mma_commit(&bars.fin);
                mbar_wait(&bars.fin, 0, p.err, kErrTimeout);
            }
        }
    } else {
        // thread t: key channel i = t % 128 (= TMEM lane), state columns [64 hc, 64 hc + 64)
        // and, for the decay, the tokens of its half hc of each chunk
        const int t = threadIdx.x;
        const int i = t & 127, hc = t >> 7;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        float S[64];
#pragma unroll
        for (int n = 0; n < 64; ++n) S[n] = 0.f;
        float lam = 0.f;
        float gsum[2] = {0.f, 0.f};
        const float lgam = (KIND == kScalar && p.log_gamma) ? p.log_gamma[h] : 0.f;

        auto decay = [&](int c) -> bool {
            const int s = c % kStages;
            if (!bar_state_and(mbar_wait_or_abort_compact(&bars.full[s], (c / kStages) & 1, p.err, kErrTimeout,
                                                  &abort_flag)))
                return false;
            uint8_t *kt = smem + s * G::kStage;
            float *gt = reinterpret_cast<float *>(smem + s * G::kStage + 2 * G::kKV);
            const int valid = min(C, seg.len - c * C);
            // (1) decay factors: exp of the log-gates after each token inside the chunk. They
            //     only scale bf16 operands (relative rounding 2^-9), so the fast exponential
            //     (relative error near 2^-22 over this range) is exact enough; the fp32 state's
            //     per-chunk decay below keeps expf.
            if (KIND == kDiag) {
                // thread t < 128 walks channel t from the last token, writing the factor of each
                // token over its gate (same thread, same address: read before write)
                if (t < D) {
                    float suf = 0.f;
#pragma unroll 8
                    for (int tt = C - 1; tt >= 0; --tt) {
                        const float l = tt < valid ? gt[tt * D + t] : 0.f;
                        gt[tt * D + t] = tt < valid ? __expf(suf) : 0.f;
                        suf += l;
                    }
                    gtot[c & 1][t] = suf;
                }
            } else if (KIND == kScalar && p.log_gamma) {
                if (t < C) fac[s][t] = t < valid ? expf(lgam * (float)(valid - 1 - t)) : 0.f;
                if (t == 0) gtot[c & 1][0] = lgam * (float)valid;
            } else if (KIND == kScalar) {
                // threads 0-63: inclusive scan of the per-token log-gates, suffix = total - scan
                float l = 0.f, x = 0.f;
                if (t < C) {
                    l = t < valid ? p.log_gate[((int64_t)seg.start + c * C + t) * p.H_v + h] : 0.f;
                    x = l;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    if (lane == 31) scan_tmp[t >> 5] = x;
                }
                bar_state();
                if (t < C) {
                    const float total = scan_tmp[0] + scan_tmp[1];
                    const float incl = t >= 32 ? x + scan_tmp[0] : x;
                    fac[s][t] = t < valid ? __expf(total - incl) : 0.f;
                    if (t == 0) gtot[c & 1][0] = total;
                }
            } else {
                if (t < C) fac[s][t] = t < valid ? 1.f : 0.f;
                if (t == 0) gtot[c & 1][0] = 0.f;
            }
            bar_state();
            gsum[c & 1] = KIND == kDiag ? gtot[c & 1][i] : gtot[c & 1][0];
            lam += gsum[c & 1];
            // (2) Khat = factors * k, 16 bytes (8 channels of one token) per access. Row tok of
            //     a 64-channel half holds physical 16-byte chunk pc = logical chunk ^ (tok % 8).
            if (KIND != kLinear || valid < C) {
#pragma unroll 1
                for (int m = 0; m < C * 16 / kEpi; ++m) {
                    const int e = t + kEpi * m;
                    const int tok = e >> 4, hf = (e >> 3) & 1, pc = e & 7;
                    uint4 *ptr = reinterpret_cast<uint4 *>(kt + hf * G::kHalf + tok * 128 + pc * 16);
                    const uint4 w = *ptr;
                    auto scale2 = [](uint32_t wj, float f0, float f1) {
                        return pack_bf16x2(__uint_as_float(wj << 16) * f0, __uint_as_float(wj & 0xffff0000u) * f1);
                    };
                    uint4 o;
                    if (KIND == kDiag) {
                        const int ch = 64 * hf + 8 * (pc ^ (tok & 7));
                        const float4 f0 = *reinterpret_cast<const float4 *>(gt + tok * D + ch);
                        const float4 f1 = *reinterpret_cast<const float4 *>(gt + tok * D + ch + 4);
                        o = make_uint4(scale2(w.x, f0.x, f0.y), scale2(w.y, f0.z, f0.w), scale2(w.z, f1.x, f1.y),
                                       scale2(w.w, f1.z, f1.w));
                    } else {
                        const float ft = fac[s][tok];
                        o = make_uint4(scale2(w.x, ft, ft), scale2(w.y, ft, ft), scale2(w.z, ft, ft),
                                       scale2(w.w, ft, ft));
                    }
                    *ptr = o;
                }
            }
            fence_async_shared();
            mbar_arrive(&bars.kready[s]);
            return true;
        };
        auto fold = [&](int c) -> bool {
            const int b = c & 1;
            if (!bar_state_and(mbar_wait_or_abort_compact(&bars.dfull[b], (c >> 1) & 1, p.err, kErrTimeout,
                                                  &abort_flag)))
                return false;
            tc_fence_after();
            const float e = (KIND == kLinear) ? 1.f : expf(gsum[b]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t r[16];
                tmem_ld16(tmem + lane_off + b * 128 + 64 * hc + 16 * q, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) S[16 * q + j] = fmaf(e, S[16 * q + j], __uint_as_float(r[j]));
            }
            tc_fence_before();
            mbar_arrive(&bars.dfree[b]);
            return true;
        };

        bool ok = true;
        if (nchunks > 0) ok = decay(0);
        for (int c = 1; ok && c < nchunks; ++c) ok = decay(c) && fold(c - 1);
        if (ok && nchunks > 0) ok = fold(nchunks - 1);

        // a piece of a split segment writes its own slot; a whole segment the caller's output
        const bool piece = seg.idx < 0;
        const int64_t unit = piece ? (int64_t)(-1 - seg.idx) * p.H_v + h : (int64_t)seg.idx * p.seg_stride + h;
        float *lam_out = piece ? p.lam_piece : p.lam;
        float4 *out = reinterpret_cast<float4 *>((piece ? p.S_piece : p.S) + unit * D * D + (int64_t)i * D + 64 * hc);
#pragma unroll
        for (int n = 0; n < 64; n += 4) out[n / 4] = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
        if (hc == 0) {
            if (KIND == kDiag) {
                lam_out[unit * D + i] = lam;
            } else if (i == 0) {
                float l = 0.f;
                if (KIND == kScalar) l = p.log_gamma ? (float)seg.len * lgam : lam;
                lam_out[unit] = l;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int KIND, int STAGES>
cudaError_t launch_kind(const BuildParams &p, cudaStream_t s) {
    using G = Geo<KIND, STAGES>;
    const int64_t N = p.n_tok > 0 ? p.n_tok : 1;
    CUtensorMap tmK, tmV, tmG;
    if (!make_tmap_3d(&tmK, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_k, N, (uint64_t)D * 2,
                      (uint64_t)p.H_k * D * 2, 64, 1, G::C, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tmV, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_v, N, (uint64_t)D * 2,
                      (uint64_t)p.H_v * D * 2, 64, 1, G::C, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (KIND == kDiag) {
        if (!make_tmap_3d(&tmG, p.log_gate, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, p.H_v, N,
                          (uint64_t)D * 4, (uint64_t)p.H_v * D * 4, D, 1, G::C,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        tmG = tmV;   // unused
    }
    cudaError_t e = cudaFuncSetAttribute(build_gated_tc_kernel<KIND, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem);
    if (e != cudaSuccess) return e;
    const int blocks = p.n_seg * p.H_v;
    if (blocks == 0) return cudaSuccess;
    build_gated_tc_kernel<KIND, STAGES><<<blocks, kThreads, G::kSmem, s>>>(p, tmK, tmV, tmG);
    return cudaGetLastError();
}

}  // namespace

bool build_gated_tc_supported(const BuildParams &p) {
    return p.D == D && p.dtype == HYPIC_BF16 &&
           (p.family == HYPIC_FAM_LINEAR || p.family == HYPIC_FAM_SCALAR ||
            p.family == HYPIC_FAM_DIAG);
}

cudaError_t launch_build_gated_tc(const BuildParams &p, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const bool deep = (int64_t)p.n_seg * p.H_v <= sms;   // at most one unit per SM
    switch (p.family) {
    case HYPIC_FAM_LINEAR: return deep ? launch_kind<kLinear, 6>(p, s) : launch_kind<kLinear, 3>(p, s);
    case HYPIC_FAM_SCALAR: return deep ? launch_kind<kScalar, 6>(p, s) : launch_kind<kScalar, 3>(p, s);
    case HYPIC_FAM_DIAG: return deep ? launch_kind<kDiag, 6>(p, s) : launch_kind<kDiag, 3>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hypic
