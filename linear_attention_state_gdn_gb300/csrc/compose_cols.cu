// compose_cols.cu -- dense compose prefix scan on the tensor cores for calls with few units
// (d = 128): one CTA per (unit, block of 32 state columns).
//
// Computes the same scan as compose_tc.cu, prefix_j = exp(lam_j) P_j prefix_{j-1} + S_j over
// the cached segments j ("Cut First-Token Latency by 3.25x: Introducing HYPIC ..."
// (besthub.dev), paragraph "For linear layers": reuse composes T_C2 . S(C1) + S(C2), with T_C
// stored as exp(lam) P), with the same fp32-accurate products (three tf32 MMAs on hi/lo splits
// of both operands, hi rounded to nearest). The scan is sequential in j, so with one CTA per
// unit a call of a few dozen units leaves most SMs idle and its time is n steps of a whole
// 128 x 128 x 128 product each. Columns of the state are independent (prefix_j[:, c] depends
// only on prefix_{j-1}[:, c]), so here four CTAs share a unit, each carrying 32 columns, and a
// step's products shrink to 128 x 32 x 128.
//
// Data flow of one CTA, block of columns [n0, n0 + 32):
//   * D = P_j X_{j-1} accumulates in TMEM (lane = row m, column = state column n - n0), with
//     X_{j-1} = exp(lam_j) prefix_{j-1}[:, block] the B operand, stored transposed (rows n,
//     k contiguous, 128B-swizzled) as tf32 hi and lo parts in shared memory;
//   * P_j streams in by TMA into a ring of two 64 KB stages and is split into tf32 hi and lo
//     parts written into TMEM as the A operand (lane = row m, column = k), k-block by k-block,
//     each as soon as the previous step's products on that k-block have completed. A stays out
//     of shared memory: with four CTAs reading every P_j, shared-memory bandwidth (TMA writes,
//     split, operand reads) bounded the step;
//   * S_j's column block streams in by TMA into a ring of four 16 KB slots, steps ahead of its
//     use (read from global memory by the epilogue itself, its latency sat on every step);
//   * the epilogue reads D, adds S_j, writes the next X and releases it to the MMA issuers;
//     then it writes prefix_j over S_j in the slot, and one TMA store writes the block out.
//     (Each thread's contiguous bytes stored directly made every warp store touch 32 lines;
//     the stores queued ahead of the shared-memory operations of the other roles and cost
//     about a third of every step.) The slot returns to the producer once the store has read
//     it.
// Roles. Warps 0-3 epilogue and warps 4-7 split (warp w = rows m and TMEM lanes 32 (w % 4)
// .. + 31); warps 8-11 MMA issuers, issuer i taking k-step i of every k-block (its three
// products) into its own accumulator D_i (D = the sum of the four, formed by the epilogue).
// One issuing thread starts about one product per 50 cycles on GB300, whatever its size
// (measured: 48 tf32 128 x 32 x 8 products take 2500 cycles from one thread, 1500 from two,
// 1040 from four); going through the k-blocks in order, the issuers release A's k-blocks one
// after another, so the split of the next step's A follows the products closely. There is no
// producer warp (a thirteenth warp would leave four on one SM sub-partition, and 128 registers
// a thread): the first split thread refills a P stage once all split threads have read it,
// and the first epilogue thread refills an S slot once the prefix store has read it.
// Plain scan only (optionally from S0); the totals and the merge of a build's pieces run on
// compose_tc.cu.
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
constexpr int NB = 32;                          // state columns per CTA
constexpr int kCols = D / NB;                   // CTAs per unit
constexpr int kEpi = 128, kSplit = 128;         // warps 0-3, warps 4-7
constexpr int kMmaWarp0 = 8;                    // warps 8 .. 11: issuer warp - 8
constexpr int kThreads = 12 * 32;
constexpr int kStages = 2;
constexpr int kSSlots = 4;
constexpr uint32_t kTile = D * D * 4;           // one fp32 128 x 128 matrix: 64 KB
constexpr uint32_t kBlock = D * 32 * 4;         // one 32-column k-block of P: 16 KB
constexpr uint32_t kSBlock = D * NB * 4;        // one column block of S: 16 KB
constexpr uint32_t kXBlock = NB * 128;          // one k-block of X^T: NB rows of 128 B
constexpr uint32_t kOffP = 0;                   // the P stages
constexpr uint32_t kOffS = kStages * kTile;     // the S slots
constexpr uint32_t kOffXhi = kOffS + kSSlots * kSBlock;
constexpr uint32_t kOffXlo = kOffXhi + 4 * kXBlock;
// + alignment slack; the size also keeps a second CTA (and its TMEM allocation) off the SM
constexpr uint32_t kSmemBytes = kOffXlo + 4 * kXBlock + 1024;
constexpr uint32_t kTmemCols = 512;             // A_hi [0,128) A_lo [128,256) D_b [256+32b, +32)

struct Bars {
    uint64_t p_full[kStages], p_empty[kStages], s_full[kSSlots], a_full[4], a_empty[4];
    uint64_t x_full, d_full, fin[4];
    uint64_t st_ready;   // the epilogue threads have written their rows of the prefix block
};

// x rounded to the nearest tf32 value, ties away from zero (adding half a tf32 unit to the
// magnitude bits, then clearing the 13 low mantissa bits), so that the low part x - hi takes
// either sign and the tensor core's truncating reading of it errs both ways.
__device__ __forceinline__ float tf32_rna(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__global__ void __launch_bounds__(kThreads, 1)
compose_dense_cols_kernel(const __grid_constant__ ComposeParams p,
                          const __grid_constant__ CUtensorMap tmP,
                          const __grid_constant__ CUtensorMap tmS,
                          const __grid_constant__ CUtensorMap tmO) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars bars;
    __shared__ uint32_t tslot;
    __shared__ volatile int abort_flag;

    const int warp = warp_id(), lane = lane_id();
    const int U = (int)p.n_units, NS = p.n_seg;
    const int tiles = U * kCols;
    const bool has_s0 = p.S0 != nullptr;
    // this CTA's tiles blockIdx.x + t gridDim.x, their steps (t, j) in order, and the steps
    // with a carried state (MMA steps): j >= 1, or all with S0
    const int my_tiles = (tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int mma_per_tile = has_s0 ? NS : NS - 1;
    const uint32_t nS = (uint32_t)(my_tiles * NS), nP = (uint32_t)(my_tiles * mma_per_tile);
    // the [row][column] box origin of step t NS + j (unit u, column block n0)
    auto origin = [&](uint32_t t, int j, int32_t &col, int32_t &row) {
        const int tile = (int)blockIdx.x + (int)t * (int)gridDim.x;
        const int u = tile / kCols;
        col = NB * (tile % kCols);
        row = (int32_t)(((int64_t)j * U + u) * D);
    };
    // P_j of MMA step q into its stage; S_j of step q into its slot
    auto load_p = [&](uint32_t q) {
        const uint32_t st = q % kStages;
        int32_t col, row;
        origin(q / (uint32_t)mma_per_tile, (int)(q % (uint32_t)mma_per_tile) + (has_s0 ? 0 : 1), col, row);
        mbar_arrive_expect_tx(&bars.p_full[st], kTile);
        for (int b = 0; b < 4; ++b)
            tma_load_2d(smem + kOffP + st * kTile + b * kBlock, &tmP, &bars.p_full[st], 32 * b, row);
    };
    auto load_s = [&](uint32_t q) {
        const uint32_t sl = q % kSSlots;
        int32_t col, row;
        origin(q / (uint32_t)NS, (int)(q % (uint32_t)NS), col, row);
        mbar_arrive_expect_tx(&bars.s_full[sl], kSBlock);
        tma_load_2d(smem + kOffS + sl * kSBlock, &tmS, &bars.s_full[sl], col, row);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars.p_full[i], 1);
            mbar_init(&bars.p_empty[i], kSplit);
        }
        for (int i = 0; i < kSSlots; ++i) mbar_init(&bars.s_full[i], 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bars.a_full[i], kSplit);
            mbar_init(&bars.a_empty[i], 4);   // one commit per issuer
            mbar_init(&bars.fin[i], 1);
        }
        mbar_init(&bars.x_full, kEpi);
        mbar_init(&bars.d_full, 4);
        mbar_init(&bars.st_ready, kEpi);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tA_hi = tslot, tA_lo = tslot + 128, tD = tslot + 256;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp >= kMmaWarp0) {
        if (lane == 0) {
            constexpr uint32_t id = idesc(kFmtTF32, kFmtTF32, false, false, 128, NB);
            const int i = warp - kMmaWarp0;
            const uint32_t tDi = tD + NB * i;
            for (uint32_t pc = 0; pc < nP && !abort_flag; ++pc) {
                // X_{j-1} (the previous products' D has been read), then A k-block by k-block
                if (!mbar_wait_or_abort(&bars.x_full, pc & 1, p.err, kErrTimeout, &abort_flag, true))
                    goto mma_done;
                for (int b = 0; b < 4; ++b) {
                    if (!mbar_wait_or_abort(&bars.a_full[b], pc & 1, p.err, kErrTimeout, &abort_flag, true))
                        goto mma_done;
                    tc_fence_after();
                    // k-step i of k-block b: 8 tf32 = 32 bytes into each B row
                    const uint32_t kc = (uint32_t)(32 * b + 8 * i);
                    const uint64_t bhi = sdesc(smem_u32(smem + kOffXhi + b * kXBlock), 16, 1024, kSwizzle128B) + 2 * i;
                    const uint64_t blo = sdesc(smem_u32(smem + kOffXlo + b * kXBlock), 16, 1024, kSwizzle128B) + 2 * i;
                    mma_tf32_ta(tDi, tA_hi + kc, bhi, id, b != 0);
                    mma_tf32_ta(tDi, tA_lo + kc, bhi, id, 1);
                    mma_tf32_ta(tDi, tA_hi + kc, blo, id, 1);
                    mma_commit(&bars.a_empty[b]);
                }
                mma_commit(&bars.d_full);
            }
        mma_done:
            if (abort_flag) {   // every MMA this thread issued completes before TMEM is released
                mma_commit(&bars.fin[i]);
                mbar_wait(&bars.fin[i], 0, p.err, kErrTimeout);
            }
        }
    } else if (warp >= 4) {
        // split: thread = row m of every P stage; k-block b to tf32 hi and lo parts in A's TMEM
        // columns, once the previous step's products on it completed. Every wait is left by
        // the whole warp together (__all_sync): its tcgen05 stores are warp-collective.
        const int m = threadIdx.x - kEpi;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t issued = 0, landed = 0;   // P loads issued (by thread m = 0) and waited for
        if (m == 0)
            for (; issued < nP && issued < (uint32_t)kStages; ++issued) load_p(issued);
        for (uint32_t pc = 0; pc < nP && !abort_flag; ++pc) {
            const uint32_t st = pc % kStages;
            if (!__all_sync(~0u, mbar_wait_or_abort(&bars.p_full[st], (pc / kStages) & 1, p.err, kErrTimeout,
                                                    &abort_flag)))
                goto split_done;
            landed = pc + 1;
            for (int b = 0; b < 4; ++b) {
                // row m of the k-block: eight 16-byte chunks, 128B-swizzled (conflict-free:
                // the warp's 32 rows spread each chunk over all banks)
                const uint8_t *src = smem + kOffP + st * kTile + b * kBlock;
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 x = *reinterpret_cast<const float4 *>(src + sw128((uint32_t)m, 16u * c));
                    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float hv = tf32_rna(xs[e]);
                        hi[4 * c + e] = __float_as_uint(hv);
                        lo[4 * c + e] = __float_as_uint(xs[e] - hv);
                    }
                }
                if (b == 3) mbar_arrive(&bars.p_empty[st]);   // this thread's reads of the stage are done
                if (pc >= 1 && !__all_sync(~0u, mbar_wait_or_abort(&bars.a_empty[b], (pc - 1) & 1, p.err,
                                                                   kErrTimeout, &abort_flag)))
                    goto split_done;
                const uint32_t ta = lane_off + 32 * b;
                tmem_st16(tA_hi + ta, *reinterpret_cast<const uint32_t(*)[16]>(hi));
                tmem_st16(tA_hi + ta + 16, *reinterpret_cast<const uint32_t(*)[16]>(hi + 16));
                tmem_st16(tA_lo + ta, *reinterpret_cast<const uint32_t(*)[16]>(lo));
                tmem_st16(tA_lo + ta + 16, *reinterpret_cast<const uint32_t(*)[16]>(lo + 16));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars.a_full[b]);
            }
            // the first split thread refills the stage, once every split thread has read it
            bool ok = true;
            if (m == 0 && pc + kStages < nP) {
                ok = mbar_wait_or_abort(&bars.p_empty[st], (pc / kStages) & 1, p.err, kErrTimeout, &abort_flag);
                if (ok) load_p(issued++);
            }
            if (!__shfl_sync(~0u, ok, 0)) goto split_done;   // warp 4 stays converged
        }
    split_done:
        if (m == 0 && abort_flag)   // the loads still in flight land before the CTA leaves
            for (uint32_t q = landed; q < issued; ++q)
                mbar_wait(&bars.p_full[q % kStages], (q / kStages) & 1, p.err, kErrTimeout);
    } else {
        // epilogue: thread t owns row m = t (TMEM lane t) of the column block; in X^T it is
        // column k = m, in k-block m / 32 = warp. Every wait is left by the whole warp together.
        const int m = threadIdx.x;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        uint8_t *xhi = smem + kOffXhi + warp * kXBlock, *xlo = smem + kOffXlo + warp * kXBlock;
        const uint32_t kbyte = 4u * (uint32_t)lane;
        uint32_t dc = 0, sc = 0, issued = 0;   // S loads issued by thread m = 0
        if (m == 0)
            for (; issued < nS && issued < (uint32_t)kSSlots; ++issued) load_s(issued);
        // X rows n = 0 .. NB-1 of column k = m from v[] (scaled): hi and lo parts, then released
        // to the MMA issuers
        auto put_x = [&](const float (&v)[NB], float scale) {
#pragma unroll
            for (int n = 0; n < NB; ++n) {
                const float x = v[n] * scale;
                const float hv = tf32_rna(x);
                const uint32_t off = sw128((uint32_t)n, kbyte);
                *reinterpret_cast<float *>(xhi + off) = hv;
                *reinterpret_cast<float *>(xlo + off) = x - hv;
            }
            fence_async_shared();
            tc_fence_before();
            mbar_arrive(&bars.x_full);
        };
        for (uint32_t t = 0; t < (uint32_t)my_tiles && !abort_flag; ++t) {
            const int tile = (int)blockIdx.x + (int)t * (int)gridDim.x;
            const int u = tile / kCols, n0 = NB * (tile % kCols);
            float v[NB];
            if (has_s0) {
                const float4 *s0 = reinterpret_cast<const float4 *>(p.S0 + ((int64_t)u * D + m) * D + n0);
#pragma unroll
                for (int i = 0; i < NB / 4; ++i) {
                    const float4 x = __ldcs(s0 + i);
                    v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
                }
                put_x(v, expf(p.lam[u]));
            }
            // lam_{j+1} scales the operand written at step j; its load is issued a step ahead
            float lam_next = NS > 1 ? p.lam[(int64_t)U + u] : 0.f;
            for (int j = 0; j < NS; ++j) {
                const bool next = j + 1 < NS;
                const float lam_after = j + 2 < NS ? p.lam[(int64_t)(j + 2) * U + u] : 0.f;
                const float scale_next = next ? expf(lam_next) : 0.f;
                lam_next = lam_after;
                const uint32_t sl = sc % kSSlots;
                if (!__all_sync(~0u, mbar_wait_or_abort(&bars.s_full[sl], (sc / kSSlots) & 1, p.err, kErrTimeout,
                                                        &abort_flag)))
                    goto epi_done;
                ++sc;
                uint8_t *ssm = smem + kOffS + sl * kSBlock;
                // v = (D_0 + D_1) + (D_2 + D_3) + S_j's row segment (S_j alone at a first step
                // without S0)
                if (j > 0 || has_s0) {
                    if (!__all_sync(~0u, mbar_wait_or_abort(&bars.d_full, dc & 1, p.err, kErrTimeout, &abort_flag)))
                        goto epi_done;
                    ++dc;
                    tc_fence_after();
                    uint32_t r0[NB], r1[NB];
                    tmem_ld32(tD + lane_off, r0);
                    tmem_ld32(tD + NB + lane_off, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < NB; ++i) v[i] = __uint_as_float(r0[i]) + __uint_as_float(r1[i]);
                    tmem_ld32(tD + 2 * NB + lane_off, r0);
                    tmem_ld32(tD + 3 * NB + lane_off, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < NB; ++i) v[i] += __uint_as_float(r0[i]) + __uint_as_float(r1[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < NB; ++i) v[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < NB / 4; ++i) {
                    const float4 x = *reinterpret_cast<const float4 *>(ssm + sw128((uint32_t)m, 16u * i));
                    v[4 * i] += x.x; v[4 * i + 1] += x.y; v[4 * i + 2] += x.z; v[4 * i + 3] += x.w;
                }
                if (next) put_x(v, scale_next);
                // prefix_j's row over S_j's in the slot; thread 0 stores the block once every
                // row is in, then refills the previous step's slot (its store has read it)
#pragma unroll
                for (int i = 0; i < NB / 4; ++i)
                    *reinterpret_cast<float4 *>(ssm + sw128((uint32_t)m, 16u * i)) =
                        make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                fence_async_shared();
                mbar_arrive(&bars.st_ready);
                bool stored = true;
                if (m == 0) {
                    stored = mbar_wait_or_abort(&bars.st_ready, (sc - 1) & 1, p.err, kErrTimeout, &abort_flag);
                    if (stored) {
                        tma_store_2d(&tmO, ssm, n0, (int32_t)(((int64_t)j * U + u) * D));
                        bulk_commit();
                        bulk_wait_read<1>();
                        if (sc >= 2 && issued < nS) load_s(issued++);   // = step sc - 2 + kSSlots
                    }
                }
                if (!__shfl_sync(~0u, stored, 0)) goto epi_done;   // warp 0 stays converged
            }
        }
    epi_done:
        if (m == 0) {
            bulk_wait<0>();   // the prefix stores complete before the CTA exits
            if (abort_flag)   // and the loads still in flight land
                for (uint32_t q = sc; q < issued; ++q)
                    mbar_wait(&bars.s_full[q % kSSlots], (q / kSSlots) & 1, p.err, kErrTimeout);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tA_hi, kTmemCols);   // the allocation's base
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

// Plain scans (no totals, no merge) of d = 128 whose (unit, column block) tiles all fit on the
// SMs at once.
bool compose_dense_cols_supported(const ComposeParams &p) {
    if (p.D != D || p.lam_total || p.P_total || p.prefix_last || p.S1) return false;
    if ((int64_t)p.n_seg * p.n_units * D > INT32_MAX) return false;
    const int sms = sm_count();
    return sms > 0 && p.n_units * kCols <= sms;
}

cudaError_t launch_compose_dense_cols(const ComposeParams &p, cudaStream_t s) {
    if (p.n_seg == 0 || p.n_units == 0) return cudaSuccess;
    const uint64_t rows = (uint64_t)p.n_seg * p.n_units * D;
    CUtensorMap tmP, tmS, tmO;
    const float *pbase = p.P ? p.P : p.S;   // P is only read for steps with a carried state
    if (!make_tmap_2d(&tmP, pbase, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows, D * 4, 32, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tmS, p.S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows, D * 4, NB, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tmO, p.prefix, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, rows, D * 4, NB, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(compose_dense_cols_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int sms = std::max(1, sm_count());
    const int grid = (int)std::min<int64_t>(p.n_units * kCols, sms);
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
    return cudaLaunchKernelEx(&cfg, compose_dense_cols_kernel, p, tmP, tmS, tmO);
}

}  // namespace hypic
