// compose_tc.cu -- dense compose prefix scan on the 5th-generation tensor cores (d = 128).
//
// For every (layer, head) unit: prefix_j = exp(lam_j) P_j prefix_{j-1} + S_j over the
// cached segments j ("Cut First-Token Latency by 3.25x: Introducing HYPIC ..."
// (besthub.dev), paragraph "For linear layers": reuse composes T_C2 . S(C1) + S(C2), with
// T_C stored as exp(lam) P; paragraph on segment parallelism: a combine worker assembles
// the final state from the segments' results).
//
// Precision. fp32-accurate products from three tf32 MMAs (hi/lo split of both operands:
// A_hi B_hi + A_lo B_hi + A_hi B_lo, error ~2^-21 relative), fp32 accumulation. The hi parts
// are rounded to tf32 explicitly (to nearest), so that the lo parts carry no bias.
//
// Data flow of one CTA (persistent over units, one unit at a time):
//   * the transposed running state prefix_{j-1}^T, scaled by exp(lam_j) and split into
//     (hi, lo), lives in TMEM as the A operand (lane = state column n, column = row k);
//   * P_j streams in by TMA (128B-swizzled, K-major: rows m, k contiguous) into one of two
//     64 KB stages; the epilogue warps truncate it to tf32 in place and write its low part
//     into a two-slot ring of 16 KB k-blocks, so the MMAs of block b overlap the split of
//     block b+1;
//   * D^T = A P_j^T accumulates in TMEM (lane n, column m) = (P_j prefix_{j-1})[:, n], in one
//     of two accumulators that alternate by step;
//   * S_j arrives by TMA into shared memory; the epilogue thread of state column n forms
//     prefix_j[:, n] = D^T[n, :] + S_j[:, n], stores it (coalesced across the warp) and
//     writes the next A operand, in two halves of A's K range: after the first half the next
//     step's products on it start (into the other accumulator) while the second is written.
// Transition units: with P_total requested, units U .. 2U-1 of the persistent loop carry
// the chain Q_j = P_j Q_{j-1} from Q_0 = P_0 (loaded like an S tile) through the same
// products, without S, and write only Q_{n-1} = P_total of unit u - U: the transition of the
// entry composed from all n segments is exp(sum_j lam_j) Q_{n-1}. Each P_j is a product of
// contractions, so a long chain drives Q below the fp32 range (64 cached segments of a few
// hundred tokens: about 1e-49). The chain is therefore carried scaled by powers of two: once
// the largest entry of the carried matrix falls below 2^-24 (found by a max-reduction of the
// previous step's values over the epilogue threads, on an mbarrier), the next operand is
// multiplied by the power of two that brings it back into [1, 2); the exponents are summed
// and P_total = 2^E Q_{n-1} is written with lam_total = sum_j lam_j - E ln 2 (the scaling is
// exact, and E = 0 whenever the chain stays in range). The transition unit writes lam_total;
// without P_total it is summed by the normal unit's epilogue (thread 0, segment order). With
// prefix_last (a build composing the pieces of its segments), only the last state is written.
// Roles: warps 0-7 epilogue (warps w and w + 4 share TMEM lanes 32 (w % 4) .. + 31, one state
// column per lane, and each take half of the column's rows and of every P split), warp 8 TMA
// producer, warp 9 MMA issuer.
// Every wait is bounded; on expiry the CTA records HYPIC_ERR_TIMEOUT, lets its in-flight
// copies and MMAs finish (bounded), frees its TMEM and returns.
#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace hypic {
namespace {

using namespace ptx;

constexpr int D = 128;
constexpr int kEpiWarps = 8;
constexpr int kEpi = kEpiWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTile = D * D * 4;          // one fp32 128x128 matrix: 64 KB
constexpr uint32_t kBlock = D * 32 * 4;        // one 32-column k-block of P: 16 KB
constexpr uint32_t kOffP = 0;                  // two P stages
constexpr uint32_t kOffLo = 2 * kTile;         // two low-part k-block slots
constexpr uint32_t kOffS = 2 * kTile + 2 * kBlock;
constexpr uint32_t kSmemBytes = kOffS + kTile + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 512;            // A_hi [0,128) A_lo [128,256) D 2 x [256,384)

struct Bars {
    uint64_t p_full[2], p_empty[2], lo_full[2], lo_empty[2];
    uint64_t s_full, s_empty, a_full[2], d_full, fin;
    uint64_t red;   // the epilogue threads' max-reduction of a transition unit's step
};

// The power-of-two exponent e with 2^e <= x < 2^(e+1), for a normal positive float x.
__device__ __forceinline__ int exponent_of(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127; }

// x rounded to the nearest tf32 value, ties away from zero (sign-magnitude: adding half a tf32
// unit to the magnitude bits, then clearing the 13 low mantissa bits). The hi part of every
// split is rounded this way, so that the lo part x - hi (exact in fp32) takes either sign and
// the tensor core's reading of it (it keeps tf32 bits only) errs both ways: a truncated hi
// made every lo part the same sign as x, and that bias accumulated over long chains of
// products.
__device__ __forceinline__ float tf32_rna(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void st_stream(float *p, float v) {
    asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// FUSED: lam_total summed here and prefix_last honoured (compiled separately, so that the
// plain scan's code is unchanged)
template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
compose_dense_tc_kernel(const __grid_constant__ ComposeParams p,
                        const __grid_constant__ CUtensorMap tmP,
                        const __grid_constant__ CUtensorMap tmS,
                        const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmP1,
                        const __grid_constant__ CUtensorMap tmS1) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived by offsetting the shared array itself so that the
    // compiler keeps the shared address space (plain ld/st.shared, not generic accesses)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars bars;
    __shared__ uint32_t tslot;
    __shared__ volatile int abort_flag;
    __shared__ unsigned red_max[3];   // largest |value| of a transition step (float bits), three slots

    const int warp = warp_id(), lane = lane_id();
    const int U = (int)p.n_units, NS = p.n_seg;
    const int UT = p.P_total ? 2 * U : U;   // units, then transition units
    const bool has_s0 = p.S0 != nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.p_full[i], 1);
            mbar_init(&bars.p_empty[i], 1);
            mbar_init(&bars.lo_full[i], kEpiWarps * 32);
            mbar_init(&bars.lo_empty[i], 1);
        }
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.s_empty, kEpiWarps * 32);
        mbar_init(&bars.a_full[0], kEpiWarps * 32);
        mbar_init(&bars.a_full[1], kEpiWarps * 32);
        mbar_init(&bars.d_full, 1);
        mbar_init(&bars.fin, 1);
        mbar_init(&bars.red, kEpiWarps * 32);
        red_max[0] = red_max[1] = red_max[2] = 0u;
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    const uint32_t tA_hi = tmem, tA_lo = tmem + 128, tD = tmem + 256;
    // launched as a programmatic dependent of the previous kernel on the stream: the set-up
    // above may overlap its tail; every global access comes after its completion
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == kProducerWarp) {
        if (lane == 0) {
            prefetch_tmap(&tmP);
            prefetch_tmap(&tmS);
            prefetch_tmap(&tmQ);
            if (FUSED && p.S1) {
                prefetch_tmap(&tmP1);
                prefetch_tmap(&tmS1);
            }
            uint32_t pc = 0, sc = 0;
            for (int ux = blockIdx.x; ux < UT && !abort_flag; ux += gridDim.x) {
                const bool tr = ux >= U;
                const int u = tr ? ux - U : ux;
                for (int j = 0; j < NS; ++j) {
                    // segment 1 in arrays of its own (fused instance only)
                    const bool sep = FUSED && j == 1 && p.S1 != nullptr;
                    const int32_t row = sep ? (int32_t)((int64_t)u * D) : (int32_t)(((int64_t)j * U + u) * D);
                    if (j > 0 || (has_s0 && !tr)) {
                        const uint32_t st = pc & 1, use = pc >> 1;
                        if (use >= 1 && !mbar_wait_or_abort(&bars.p_empty[st], (use - 1) & 1, p.err,
                                                            kErrTimeout, &abort_flag))
                            goto producer_done;
                        mbar_arrive_expect_tx(&bars.p_full[st], kTile);
                        for (int b = 0; b < 4; ++b)
                            tma_load_2d(smem + kOffP + st * kTile + b * kBlock, sep ? &tmP1 : &tmP,
                                        &bars.p_full[st], 32 * b, row);
                        ++pc;
                    }
                    if (tr && j > 0) continue;   // the transition chain adds no S
                    if (sc >= 1 && !mbar_wait_or_abort(&bars.s_empty, (sc - 1) & 1, p.err,
                                                       kErrTimeout, &abort_flag))
                        goto producer_done;
                    mbar_arrive_expect_tx(&bars.s_full, kTile);
                    tma_load_2d(smem + kOffS, tr ? &tmQ : sep ? &tmS1 : &tmS, &bars.s_full, 0, row);   // Q_0 = P_0
                    ++sc;
                }
            }
        producer_done:
            if (abort_flag) {
                // let the loads still in flight land before the CTA leaves (bounded)
                for (uint32_t q = pc > 2 ? pc - 2 : 0; q < pc; ++q)
                    mbar_wait(&bars.p_full[q & 1], (q >> 1) & 1, p.err, kErrTimeout);
                if (sc) mbar_wait(&bars.s_full, (sc - 1) & 1, p.err, kErrTimeout);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t id = idesc(kFmtTF32, kFmtTF32, false, false, 128, 128);
            uint32_t pc = 0, lb = 0, ac = 0;
            for (int ux = blockIdx.x; ux < UT && !abort_flag; ux += gridDim.x) {
                const bool tr = ux >= U;
                for (int j = 0; j < NS; ++j) {
                    if (!(j > 0 || (has_s0 && !tr))) continue;
                    const uint32_t st = pc & 1;
                    const uint32_t dacc = tD + 128 * (pc & 1);   // the two D buffers alternate by step
                    for (int b = 0; b < 4; ++b) {
                        if ((b & 1) == 0) {   // A's k-blocks 0-1, then 2-3, as the epilogue writes them
                            if (!mbar_wait_or_abort(&bars.a_full[b >> 1], ac & 1, p.err, kErrTimeout,
                                                    &abort_flag))
                                goto mma_done;
                            tc_fence_after();
                        }
                        const uint32_t slot = lb & 1, use = lb >> 1;
                        if (!mbar_wait_or_abort(&bars.lo_full[slot], use & 1, p.err, kErrTimeout,
                                                &abort_flag))
                            goto mma_done;
                        tc_fence_after();
                        const uint64_t dhi =
                            sdesc(smem_u32(smem + kOffP + st * kTile + b * kBlock), 16, 1024, kSwizzle128B);
                        const uint64_t dlo =
                            sdesc(smem_u32(smem + kOffLo + slot * kBlock), 16, 1024, kSwizzle128B);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint32_t kc = (uint32_t)(32 * b + 8 * s);   // A column of this k-step
                            mma_tf32_ta(dacc, tA_hi + kc, dhi + 2 * s, id, (b | s) != 0);
                            mma_tf32_ta(dacc, tA_lo + kc, dhi + 2 * s, id, 1);
                            mma_tf32_ta(dacc, tA_hi + kc, dlo + 2 * s, id, 1);
                        }
                        mma_commit(&bars.lo_empty[slot]);
                        ++lb;
                    }
                    ++ac;
                    mma_commit(&bars.p_empty[st]);
                    mma_commit(&bars.d_full);
                    ++pc;
                }
            }
        mma_done:
            if (abort_flag) {
                // every MMA issued so far completes before TMEM is released (bounded)
                mma_commit(&bars.fin);
                mbar_wait(&bars.fin, 0, p.err, kErrTimeout);
            }
        }
    } else {
        // epilogue: thread t owns state column n = t % 128 = TMEM lane n. A step's rows are
        // written in two parts, A's k-blocks 0-1 (rows 0-63) and then 2-3 (rows 64-127); in each
        // part half eh = t / 128 of the threads takes 32 rows. After each part the threads split
        // the matching k-blocks of the next step's P, so that the next step's products on those
        // k-blocks (into the other D buffer) run while the second part is still being written.
        const int t = threadIdx.x, n = t & 127, eh = t >> 7;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t pc = 0, sc = 0, lb = 0, dc = 0, rc = 0;
        const float *Ssm = reinterpret_cast<const float *>(smem + kOffS);
        // hi / lo split of k-blocks [b0, b1) of the next P stage to be consumed (pc), in place
        // and into the low-part ring; block 0 waits for the stage, block 3 retires it
        auto split = [&](int b0, int b1) -> bool {
            const uint32_t st = pc & 1, use = pc >> 1;
            if (b0 == 0 && !mbar_wait_or_abort(&bars.p_full[st], use & 1, p.err, kErrTimeout, &abort_flag))
                return false;
            for (int b = b0; b < b1; ++b) {
                const uint32_t slot = lb & 1, luse = lb >> 1;
                if (luse >= 1 && !mbar_wait_or_abort(&bars.lo_empty[slot], (luse - 1) & 1,
                                                     p.err, kErrTimeout, &abort_flag))
                    return false;
                float4 *src = reinterpret_cast<float4 *>(smem + kOffP + st * kTile + b * kBlock);
                float4 *dst = reinterpret_cast<float4 *>(smem + kOffLo + slot * kBlock);
#pragma unroll
                for (int q = 0; q < 1024 / kEpi; ++q) {
                    const int idx = t + kEpi * q;
                    const float4 x = src[idx];
                    float4 h, l;
                    h.x = tf32_rna(x.x); l.x = x.x - h.x;
                    h.y = tf32_rna(x.y); l.y = x.y - h.y;
                    h.z = tf32_rna(x.z); l.z = x.z - h.z;
                    h.w = tf32_rna(x.w); l.w = x.w - h.w;
                    src[idx] = h;
                    dst[idx] = l;
                }
                fence_async_shared();
                mbar_arrive(&bars.lo_full[slot]);
                ++lb;
            }
            if (b1 == 4) ++pc;
            return true;
        };
        for (int ux = blockIdx.x; ux < UT && !abort_flag; ux += gridDim.x) {
            const bool tr = ux >= U;
            const int u = tr ? ux - U : ux;
            float lsum = 0.f;   // thread 0: sum of lam over the segments (lam_total)
            // transition units: the power of two the next operand is multiplied by, the sum of
            // the exponents applied so far, and this thread's largest |value| of the step
            float s_pow = 1.f, vmax = 0.f;
            int e_sum = 0;
            if (has_s0 && !tr) {
                // A = split(exp(lam_0) S0^T) for the first step
                const float sc0 = expf(p.lam[u]);
                const float *s0 = p.S0 + (int64_t)u * D * D + n;
                for (int c = 4 * eh; c < 4 * eh + 4; ++c) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float x = s0[(16 * c + i) * D] * sc0;
                        const float h = tf32_rna(x);
                        hi[i] = __float_as_uint(h);
                        lo[i] = __float_as_uint(x - h);
                    }
                    tmem_st16(tA_hi + lane_off + 16 * c, hi);
                    tmem_st16(tA_lo + lane_off + 16 * c, lo);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars.a_full[0]);
                mbar_arrive(&bars.a_full[1]);
            }
            bool split_ahead = false;   // this step's P was split during the previous step
            for (int j = 0; j < NS; ++j) {
                const bool mma = j > 0 || (has_s0 && !tr);
                uint32_t dacc = tD;
                if (mma) {
                    if (!split_ahead && !split(0, 4)) goto epi_done;
                    dacc = tD + 128 * (dc & 1);
                    if (!mbar_wait_or_abort(&bars.d_full, dc & 1, p.err, kErrTimeout, &abort_flag))
                        goto epi_done;
                    ++dc;
                    tc_fence_after();
                    if (FUSED && tr) {
                        // the largest |entry| of the previous step's values over all epilogue
                        // threads (non-negative floats order like their bit patterns), in slot
                        // rc % 3. Thread 0 then clears slot (rc + 2) % 3: every thread read it
                        // (reduction rc - 1) before arriving here, and none writes it before
                        // reduction rc + 2, which needs thread 0's next arrival
                        atomicMax(&red_max[rc % 3], __float_as_uint(vmax));
                        mbar_arrive(&bars.red);
                        if (!mbar_wait_or_abort(&bars.red, rc & 1, p.err, kErrTimeout, &abort_flag))
                            goto epi_done;
                        const float m = __uint_as_float(red_max[rc % 3]) * s_pow;   // largest |entry| of A_j
                        if (t == 0) red_max[(rc + 2) % 3] = 0u;
                        ++rc;
                        s_pow = 1.f;
                        // (the last step writes no next operand: no scale, no exponent)
                        if (j + 1 < NS && m > 0.f && m < 0x1p-24f) {
                            const int e = -exponent_of(m);   // m 2^e in [1, 2)
                            s_pow = __uint_as_float((uint32_t)(127 + e) << 23);
                            e_sum += e;
                        }
                        vmax = 0.f;
                    }
                }
                const bool has_s = !(tr && j > 0);   // S_j (Q_0 = P_0 for the transition chain)
                if (has_s) {
                    if (!mbar_wait_or_abort(&bars.s_full, sc & 1, p.err, kErrTimeout, &abort_flag))
                        goto epi_done;
                    ++sc;
                }
                const bool next = j + 1 < NS;
                const float scale_next =
                    !next ? 0.f
                    : tr  ? s_pow
                          : expf(FUSED && j == 0 && p.lam1 ? p.lam1[u] : p.lam[(int64_t)(j + 1) * U + u]);
                if (FUSED && t == 0 && p.lam_total) lsum += j == 1 && p.lam1 ? p.lam1[u] : p.lam[(int64_t)j * U + u];
                // prefix_j (only the last one with prefix_last), or for the transition chain
                // only its last state, P_total
                float *out = tr ? (next ? nullptr : p.P_total + (int64_t)u * D * D + n)
                           : (FUSED && p.prefix_last) ? (next ? nullptr : p.prefix_last + (int64_t)u * D * D + n)
                                           : p.prefix + ((int64_t)j * U + u) * D * D + n;
                for (int part = 0; part < 2; ++part) {
                    for (int c = 4 * part + 2 * eh; c < 4 * part + 2 * eh + 2; ++c) {
                        uint32_t r[16];
                        if (mma) {
                            tmem_ld16(dacc + lane_off + 16 * c, r);
                            tmem_ld_wait();
                        }
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = 16 * c + i;
                            const float v = (mma ? __uint_as_float(r[i]) : 0.f) + (has_s ? Ssm[m * D + n] : 0.f);
                            if (out) st_stream(out + (int64_t)m * D, v);
                            if (FUSED && tr) vmax = fmaxf(vmax, fabsf(v));
                            const float x = v * scale_next;
                            const float h = tf32_rna(x);
                            hi[i] = __float_as_uint(h);
                            lo[i] = __float_as_uint(x - h);
                        }
                        if (next) {
                            tmem_st16(tA_hi + lane_off + 16 * c, hi);
                            tmem_st16(tA_lo + lane_off + 16 * c, lo);
                        }
                    }
                    if (part == 1 && has_s) mbar_arrive(&bars.s_empty);
                    if (next) {
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(&bars.a_full[part]);
                        if (!split(2 * part, 2 * part + 2)) goto epi_done;
                    }
                }
                split_ahead = next;
            }
            // lam_total: by the transition unit when there is one (with the exponents of its
            // scaling), else by the normal unit
            if (FUSED && t == 0 && p.lam_total && tr == (p.P_total != nullptr))
                p.lam_total[u] = lsum - (float)e_sum * 0.69314718055994531f;
        }
    epi_done:;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

bool compose_dense_tc_supported(const ComposeParams &p) {
    return p.D == D && (int64_t)p.n_seg * p.n_units * D <= INT32_MAX;
}

cudaError_t launch_compose_dense_tc(const ComposeParams &p, cudaStream_t s) {
    if (p.n_seg == 0 || p.n_units == 0) return cudaSuccess;
    const uint64_t rows = (uint64_t)p.n_seg * p.n_units * D;
    CUtensorMap tmP, tmS, tmQ;
    // P is only read for steps with a carried state; any valid base serves otherwise
    const float *pbase = p.P ? p.P : p.S;
    if (!make_tmap_2d(&tmP, pbase, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows, D * 4, 32, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tmS, p.S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows, D * 4, 128, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tmQ, pbase, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows, D * 4, 128, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE))   // P_0 read whole, like an S tile
        return cudaErrorInvalidValue;
    // segment 1 in arrays of its own ([n_units] rows of d x d): its own maps, else unused copies
    CUtensorMap tmP1 = tmP, tmS1 = tmS;
    if (p.S1) {
        if (p.n_seg != 2 || !p.P1 || !p.lam1) return cudaErrorInvalidValue;
        const uint64_t rows1 = (uint64_t)p.n_units * D;
        if (!make_tmap_2d(&tmP1, p.P1, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows1, D * 4, 32, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap_2d(&tmS1, p.S1, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows1, D * 4, 128, 128,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    const bool fused = p.lam_total != nullptr || p.prefix_last != nullptr || p.S1 != nullptr;
    auto kern = fused ? compose_dense_tc_kernel<true> : compose_dense_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t units = p.n_units * (p.P_total ? 2 : 1);
    const int grid = (int)std::min<int64_t>(units, sm_count());
    // a programmatic dependent launch: CTAs may set up while the previous kernel finishes
    // (the chain of a build call, whose pieces this merges) and wait for it before any access
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, tmP, tmS, tmQ, tmP1, tmS1);
}

}  // namespace hypic
