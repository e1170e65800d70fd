// build_gdn_tc.cu -- DeltaNet / Gated DeltaNet segment build on the 5th-generation tensor
// cores (bf16 k / v, d_k = d_v = 128, fp32 state): the serial chunk chain. It runs after
// build_gdn_prep.cu, which leaves one bf16 matrix M2 = N Diag(b) per 64-token chunk in the
// workspace (N = (I + Diag(b) L)^-1, L the strictly lower part of the chunk's gram K K^T).
//
// What is computed: for every cached segment C and value head the pair (S(C|0), T_C) with
// T_C = exp(lam) P, P = prod_t (I - b_t k_t k_t^T) (latest factor leftmost), lam = sum log a_t
// ("Cut First-Token Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For
// linear layers": HYPIC stores (T_C, S(C|0)) for DeltaNet / GDN layers; GDN recurrence from
// "Gated Delta Networks: Improving Mamba2 with Delta Rule", reference 7 of the episode
// companion page "Hypic: Position-Independent KV Caching for Hybrid-Attention LLM Serving").
//
// Chunked form (exact algebra; c_t = sum_{s<=t} log a_s inside the chunk, c_C = c_63):
//     W = M2 K,   U = M2 Diag(e^-c) V,
//     S <- e^{c_C} (S + K^T (U - W S)),     P <- P + K^T (-W P).
// W and U do not depend on the state. The state is carried as Z = [S~ | P] with
// S = exp(Lam) S~, Lam a running log-scale reset to 0 whenever Lam + c_C < -30 (S~ is then
// multiplied by exp(Lam) first), so every chunk is
//     D_S = exp(-Lam) U - W S~,   D_P = -W P,   Z <- Z + K^T [D_S | D_P],   Lam += c_C,
// two dependent MMA groups per half with a bf16 rounding of Z and of D in between.
//
// The chain is bound by shared-memory bandwidth when its operands go through shared memory,
// so both dependent products take their A operand from TMEM: the state and the D
// accumulators are rounded to bf16 in place in TMEM (tcgen05.ld / st, two values per
// column), and only the B operands (-W^T and the k chunk) are read from shared memory.
//
// Layout (one CTA = one (segment, value head) unit, 480 threads, one CTA per SM):
//   TMEM  [0,128) Z_S^T, [128,256) Z_P^T   fp32 state, lane n = state column, column = key row
//         [256,320) D_S^T, [320,384) D_P^T fp32 accumulators (lane n, column t); the bf16 D^T
//                                         (A of the update) is written over their first half
//         [384,448) bf16 Z_S^T (A of d_S); between d_S(c) and the next Z pass it holds the
//                   fp32 W^T(c+1) accumulator (lane i, column t')
//         [448,512) bf16 Z_P^T (A of d_P)
//   SMEM  a ring of three k chunks and a ring of three {v chunk, M2 record} (TMA,
//         128B-swizzled); -W^T bf16 (MN-major B of d, two slots); M1 = M2 Diag(exp(-Lam - c))
//         bf16 (K-major B of U, two slots).
// Roles: warps 0-3 carry the S~ half and warps 4-7 the P half (thread = TMEM lane = state
// column: Z^T -> bf16, D^T -> bf16), warps 8-11 prepare the state-independent operands
// (gates, M1, -W^T -> bf16), warp 12 issues TMA, warp 13 the S~ half's MMAs and the state-
// independent ones, warp 14 the P half's MMAs:
//     warp 13, per chunk c:  d_S(c): D_S += Z_S^T (-W^T);  W(c+1): W^T = K^T M2^T;
//                            f_S(c): Z_S^T += D_S^T K;     U(c+1): D_S = V^T M1^T
//     warp 14, per chunk c:  d_P(c): D_P = Z_P^T (-W^T);   f_P(c): Z_P^T += D_P^T K
// Two issuers keep the tensor pipe fed: it queues only a few instructions, so while one half
// waits for its operands the other half's products run.
//
// Outputs instance. When the call asks for the segment outputs o_t = S_t^T q_t, a second set of
// CTAs (blockIdx >= units) runs the S~ half again without the P half and computes, per chunk,
//     O^T = S~^T Q^T + D_S^T A^T,   A = the masked Q K^T (A_ts = q_t . k_s for s <= t),
//     o_t = exp(Lam + c_t) O^T[:, t]
// (with Delta = exp(Lam) D_S the chunk's delta values, o_t = e^{c_t} (S_before^T q_t +
// sum_{s<=t} (q_t . k_s) Delta_s)): the S~ issuer adds Q S~ (A = the bf16 Z_S^T already in TMEM,
// B = the q chunk) before d_S and the intra-chunk product (A = the bf16 D_S^T, B = A) after f_S,
// into the Z_P columns (two 64-column buffers by chunk parity, so that a chunk's products do
// not wait for the previous chunk's read-out); the P issuer computes Q K^T (M = 64) into the
// D_P columns;
// the P-half warps turn it into the bf16 operand A (masked) and read the outputs out, scaled
// with the chunk's gate slot (four slots, so that the slot outlives the read-out).
// KDA instance (the channel-gated delta rule, one decay per key channel; build_gdn_prep.cu
// derives its chunk form). The preparation leaves per chunk M2 (of the gated gram), the gated
// keys Kt = e^{c} k and Kh = e^{-c} k, and the per-channel log-decay c_C with its maximum m.
// The chunk maps the state to Diag(e^{c_C}) (Z + Kh^T D), so the chain is the same with
// W = M2 Kt, U = M2 V (no M1), the update Z += Kh^T D, and instead of the running log-scale the
// chunk's row scaling applied in the next Z pass: the conversion warps scale Z by Diag(e^{c_C})
// (S half) or Diag(e^{c_C - m}) (P half) of the previous chunk, write it back and take the bf16
// copy of the scaled state; the outputs get the last chunk's scaling. The transition is stored as
// exp(sum m) P with P in range. Kt and Kh share the k ring's slot; the scales of a chunk sit in
// one of four slots in the M1 area, each with its own barrier.
// Every wait is bounded; a wait that runs out sets the status word and the CTA drains.
#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace hypic {
namespace {

using namespace ptx;

constexpr int D = 128;
constexpr int C = kGdnChunk;
constexpr int kThreads = 480;
constexpr int kAuxWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarpS = 13;   // issues the S~ half's products and W, U
constexpr int kMmaWarpP = 14;   // issues the P half's products
constexpr float kRenormBelow = -30.f;       // reset Lam when Lam + c_C would drop below this
constexpr float kMinChunkLogDecay = -60.f;  // supported range of c_C

// shared-memory map (offsets from the 1024-aligned base)
constexpr uint32_t kHalf = 64 * 128;          // 64 rows x 128 B: one 64-channel half of a chunk
constexpr uint32_t kKV = 2 * kHalf;           // k (or v) chunk, 16 KB
constexpr uint32_t kRec = 64 * 128;           // M2 record, 8 KB
constexpr uint32_t kVR = kKV + kRec;          // v chunk + M2 record, 24 KB
constexpr int kKSlots = 3;                    // k is read until the lagging half's update
constexpr int kVSlots = 3;                    // {v, M2} slots: loads requested two chunks ahead
constexpr uint32_t kOffK = 0;                 // k ring: 3 x 16 KB
constexpr uint32_t kOffVR = kKSlots * kKV;    // {v, M2} ring: 3 x 24 KB
constexpr uint32_t kOffWop = kOffVR + kVSlots * kVR;  // -W^T bf16: 2 slots x [128 rows i][128 B]
constexpr uint32_t kOffM1 = kOffWop + 2 * kKV;  // M1: 2 slots x 8 KB
constexpr uint32_t kSmemBytes = kOffM1 + 2 * kRec + 1024;
// outputs instance only: a ring of two q chunks and two slots of the masked Q K^T (bf16)
constexpr uint32_t kOffQ = kOffM1 + 2 * kRec;
constexpr uint32_t kOffAq = kOffQ + 2 * kKV;
constexpr uint32_t kSmemBytesOut = kOffAq + 2 * kRec + 1024;
// KDA instance: k-ring slots of two tiles (Kt, Kh); the gate slots take the M1 area
constexpr uint32_t kSmemBytesKda = kKSlots * 2 * kKV + kVSlots * kVR + 2 * kKV + 2 * kRec + 1024;

constexpr uint32_t kTZ = 0, kTD = 256, kTZK = 384;
constexpr uint32_t kTO = 128, kTAq = 320;   // outputs instance: O^T (two buffers) and Q K^T (the P half's columns)

struct Slot {   // per-chunk values from the operand warps (two slots)
    float ex[C];      // exp(-Lam_start - c_t)
    float rscale;     // exp(Lam) before the reset (used when renorm)
    int renorm;       // S~ is multiplied by rscale before this chunk
    float lam_after;  // Lam after this chunk
    float lam_sum;    // sum of c_C up to and including this chunk
};

// KDA: the chunk's per-channel scales of the S and P halves and the running sum of m
struct KdaSlot {
    float gs[D], gp[D];
    float lam_sum, pad[3];
};
constexpr int kKdaSlots = 4;
static_assert(kKdaSlots * sizeof(KdaSlot) <= 2 * kRec, "KDA gate slots exceed the M1 area");

struct Bars {
    uint64_t kfull[kKSlots], kempty[kKSlots];   // k ring
    uint64_t vfull[kVSlots], vempty[kVSlots];   // {v, M2} ring
    uint64_t wfull;               // W^T accumulated
    // -W^T operand of a chunk written (and the W^T TMEM columns free), one per operand slot:
    // the P half's issuer may lag, so one barrier could be two phases ahead of its wait
    uint64_t wready[2];
    uint64_t wfree[2];            // d_P has read a -W^T slot (d_S is ordered by wfull)
    uint64_t m1ready[2];          // M1 (and the slot) of a chunk, one barrier per slot
    uint64_t zready[2], dfull[2], dready[2], zfull[2];   // per half
    uint64_t fin[2];
    // outputs instance: the q ring (emptied by Q S~ and Q K^T), Q K^T in TMEM (written by the
    // P issuer, read by the output warps), its bf16 slots, and the output accumulator
    uint64_t qfull[2], qempty[2], aqfull, aqfree, aqready[2], ofull[2], ofree[2];   // O: two buffers
    uint64_t gready[kKdaSlots];   // KDA: a chunk's gate slot written (operand warps)
};

// Named barrier of the 128 operand-warp threads, and the same with an AND of a predicate
// (every thread leaves with the same outcome). Non-aligned forms: the lanes of a warp may
// arrive at different times.
__device__ __forceinline__ void bar_aux() {
    __syncwarp();
    asm volatile("barrier.sync 2, 128;" ::: "memory");
}
__device__ __forceinline__ bool bar_aux_and(bool v) {
    uint32_t r;
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.red.and.pred po, 2, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t bf2(float lo, float hi) { return pack_bf16x2(lo, hi); }

__device__ __forceinline__ void ld64(uint32_t taddr, uint32_t (&z)[64]) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&z[0]));
    tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&z[32]));
}

// 64 fp32 values of this lane -> 32 TMEM columns of bf16 pairs (even element in the low
// half), the A-operand form of a kind::f16 MMA with A in TMEM.
__device__ __forceinline__ void st_bf16x64(uint32_t taddr, const uint32_t (&z)[64]) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            pk[j] = bf2(__uint_as_float(z[32 * g + 2 * j]), __uint_as_float(z[32 * g + 2 * j + 1]));
        tmem_st16(taddr + 16 * g, pk);
    }
}

// OUT: the instance launched when the call asks for the segment outputs (both kinds of CTA);
// the plain build compiles without any of the outputs code. KDA: the channel-gated instance.
template <bool OUT, bool KDA>
__global__ void __launch_bounds__(kThreads, 1)
build_gdn_tc_kernel(const __grid_constant__ BuildParams p, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmR,
                    const __grid_constant__ CUtensorMap tmQ) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived by offsetting the shared array itself so that the
    // compiler keeps the shared address space (plain ld/st.shared, not generic accesses)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars bars;
    // per-chunk gate slots: the outputs instance reads a chunk's slot after its last product
    // while its S~ issuer runs up to two chunks ahead (two output buffers), so it keeps four
    constexpr int kSlots = OUT ? 4 : 2;
    __shared__ __align__(16) Slot slots[kSlots];
    __shared__ uint32_t tslot;
    __shared__ volatile int abort_flag;
    __shared__ float scan_tmp[2];
    // outputs instance: exp(Lam_start + c_t), the outputs' scale, per gate slot
    __shared__ __align__(16) float s_oscale[OUT ? kSlots : 1][C];

    const int warp = warp_id(), lane = lane_id();
    const int units = p.n_seg * p.H_v;
    const bool outm = OUT && (int)blockIdx.x >= units;   // the outputs instance of unit blockIdx - units
    const int ux = outm ? (int)blockIdx.x - units : (int)blockIdx.x;
    const SegEntry seg = p.seg[ux / p.H_v];
    const int h = ux % p.H_v;
    const int hk = h / p.gqa;
    const int nch = (seg.len + C - 1) / C;
    const bool gdn = p.family == HYPIC_FAM_GDN;
    // shared-memory map of this instance (KDA: two tiles per k-ring slot, gate slots over M1)
    constexpr uint32_t kKSl = KDA ? 2 * kKV : kKV;
    constexpr uint32_t oVR = kKSlots * kKSl;
    constexpr uint32_t oWop = oVR + kVSlots * kVR;
    constexpr uint32_t oM1 = oWop + 2 * kKV;
    KdaSlot *kslots = reinterpret_cast<KdaSlot *>(smem + oM1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kKSlots; ++s) {
            mbar_init(&bars.kfull[s], 1);
            mbar_init(&bars.kempty[s], 2);   // both halves' updates read the k chunk
        }
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(&bars.vfull[s], 1);
            mbar_init(&bars.vempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.m1ready[s], 128);
            mbar_init(&bars.zready[s], 128);
            mbar_init(&bars.dfull[s], 1);
            mbar_init(&bars.dready[s], 128);
            mbar_init(&bars.zfull[s], 1);
            mbar_init(&bars.wfree[s], 1);
            mbar_init(&bars.wready[s], 128);
        }
        mbar_init(&bars.wfull, 1);
        mbar_init(&bars.fin[0], 1);
        mbar_init(&bars.fin[1], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.qfull[s], 1);
            mbar_init(&bars.qempty[s], 2);   // Q S~ (S~ issuer) and Q K^T (P issuer)
            mbar_init(&bars.aqready[s], 128);
        }
        mbar_init(&bars.aqfull, 1);
        mbar_init(&bars.aqfree, 128);
        for (int s = 0; s < kKdaSlots; ++s) mbar_init(&bars.gready[s], 128);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.ofull[s], 1);
            mbar_init(&bars.ofree[s], 128);
        }
        abort_flag = 0;
        fence_mbar_init();
        // the kernel after this one (the merge of split segments) may launch and set up on SMs
        // this grid has left; it waits for this grid's completion before any access
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(&tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    auto wait = [&](uint64_t *b, uint32_t par) {
        return mbar_wait_or_abort_compact(b, par, p.err, kErrTimeout, &abort_flag);
    };
    // every lane waits; the warp leaves with one outcome (tcgen05.ld / st are warp-wide)
    auto wwait = [&](uint64_t *b, uint32_t par) { return __all_sync(0xffffffffu, wait(b, par)) != 0; };

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmR);
            if (outm) prefetch_tmap(&tmQ);
            int c = 0, kc = 0, qc = 0;   // chunks whose {v, M2} / k / q loads were issued
            const SegEntry &last = p.seg[p.n_seg - 1];
            const int64_t records = (int64_t)last.wsb + (int64_t)p.H_v * ((last.len + C - 1) / C);
            for (; c < nch; ++c) {
                const int32_t t0 = seg.start + c * C;
                if (!in_bounds((int64_t)seg.wsb + (int64_t)h * nch + c < records &&
                                   seg.start + (int64_t)c * C < (int64_t)p.n_tok, p.err)) {
                    abort_flag = 1;   // the other roles give up their waits; the loads drain below
                    break;
                }
                const int ks = c % kKSlots, kuse = c / kKSlots;
                if (kuse >= 1 && !wait(&bars.kempty[ks], (kuse - 1) & 1)) break;
                uint8_t *kt = smem + kOffK + ks * kKSl;
                const int32_t rrow = (seg.wsb + h * nch + c) * 64;
                if constexpr (KDA) {   // Kt and Kh: records of the preparation (see below)
                    if (c == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                    mbar_arrive_expect_tx(&bars.kfull[ks], 2 * kKV);
                    tma_load_2d(kt, &tmK, &bars.kfull[ks], 0, rrow);
                    tma_load_2d(kt + kHalf, &tmK, &bars.kfull[ks], 64, rrow);
                    tma_load_2d(kt + kKV, &tmQ, &bars.kfull[ks], 0, rrow);
                    tma_load_2d(kt + kKV + kHalf, &tmQ, &bars.kfull[ks], 64, rrow);
                } else {
                    mbar_arrive_expect_tx(&bars.kfull[ks], kKV);
                    tma_load_3d(kt, &tmK, &bars.kfull[ks], 0, hk, t0);
                    tma_load_3d(kt + kHalf, &tmK, &bars.kfull[ks], 64, hk, t0);
                }
                kc = c + 1;
                // the records are written by the preparation kernel, which may still be
                // running (this grid is a programmatic dependent launch): wait for it to
                // complete before the first record load (k and v above are inputs)
                if (!KDA && c == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                const int vs = c % kVSlots, vuse = c / kVSlots;
                if (vuse >= 1 && !wait(&bars.vempty[vs], (vuse - 1) & 1)) break;
                uint8_t *vt = smem + oVR + vs * kVR;
                mbar_arrive_expect_tx(&bars.vfull[vs], kVR);
                tma_load_3d(vt, &tmV, &bars.vfull[vs], 0, h, t0);
                tma_load_3d(vt + kHalf, &tmV, &bars.vfull[vs], 64, h, t0);
                tma_load_2d(vt + kKV, &tmR, &bars.vfull[vs], 0, rrow);
                if (outm) {
                    const int qs = c & 1, quse = c >> 1;
                    if (quse >= 1 && !wait(&bars.qempty[qs], (quse - 1) & 1)) break;
                    uint8_t *qt = smem + kOffQ + qs * kKV;
                    mbar_arrive_expect_tx(&bars.qfull[qs], kKV);
                    tma_load_3d(qt, &tmQ, &bars.qfull[qs], 0, hk, t0);
                    tma_load_3d(qt + kHalf, &tmQ, &bars.qfull[qs], 64, hk, t0);
                    qc = c + 1;
                }
            }
            if (abort_flag) {   // let the loads in flight land before the CTA exits
                for (int q = (kc > kKSlots ? kc - kKSlots : 0); q < kc; ++q)
                    mbar_wait(&bars.kfull[q % kKSlots], (q / kKSlots) & 1, p.err, kErrTimeout);
                for (int q = (c > kVSlots ? c - kVSlots : 0); q < c; ++q)
                    mbar_wait(&bars.vfull[q % kVSlots], (q / kVSlots) & 1, p.err, kErrTimeout);
                for (int q = (qc > 2 ? qc - 2 : 0); q < qc; ++q)
                    mbar_wait(&bars.qfull[q & 1], (q >> 1) & 1, p.err, kErrTimeout);
            }
        }
    } else if (warp == kMmaWarpS || warp == kMmaWarpP) {
        // ---------------------------------------------------------------- MMA issuers
        // Two issuing threads, one per state half: the tensor pipe queues only a few
        // instructions, so a thread that waits between its groups leaves it idle unless the
        // other half has work queued. Every descriptor is built once; an MMA then costs a
        // 64-bit add and the issue itself.
        if (lane == 0 && nch > 0) {
            auto wait = [&](uint64_t *b, uint32_t par) {
                return mbar_wait_or_abort(b, par, p.err, kErrTimeout, &abort_flag, true);
            };
            constexpr uint32_t idA = idesc(kFmtBF16, kFmtBF16, true, false, 128, 64);
            constexpr uint32_t idD = idesc(kFmtBF16, kFmtBF16, false, true, 128, 64);
            constexpr uint32_t idF = idesc(kFmtBF16, kFmtBF16, false, true, 128, 128);
            const uint32_t sb = smem_u32(smem);
            const uint64_t dK = sdesc(sb + kOffK, kHalf, 1024, kSwizzle128B);         // MN-major
            const uint64_t dV = sdesc(sb + oVR, kHalf, 1024, kSwizzle128B);           // MN-major
            const uint64_t dR = sdesc(sb + oVR + kKV, 16, 1024, kSwizzle128B);        // K-major
            const uint64_t dW = sdesc(sb + oWop, kHalf, 1024, kSwizzle128B);          // MN-major
            const uint64_t dM = sdesc(sb + oM1, 16, 1024, kSwizzle128B);              // K-major
            const uint64_t dQ = sdesc(sb + kOffQ, 16, 1024, kSwizzle128B);            // K-major
            const uint64_t dKk = sdesc(sb + kOffK, 16, 1024, kSwizzle128B);           // K-major
            const uint64_t dAq = sdesc(sb + kOffAq, 16, 1024, kSwizzle128B);          // K-major
            constexpr uint32_t idO = idesc(kFmtBF16, kFmtBF16, false, false, 128, 64);
            constexpr uint32_t idQK = idesc(kFmtBF16, kFmtBF16, false, false, 64, 64);
            constexpr uint64_t kRow16 = 2048 >> 4;   // 16 rows of 128 B (MN-major K step)
            constexpr uint64_t kCol16 = 32 >> 4;     // 16 bf16 columns (K-major K step)
            const int hf = warp == kMmaWarpS ? 0 : 1;
            // D^T(hf) += Z^T(hf) (-W^T) with A = bf16 Z^T in TMEM (the P half starts from zero)
            auto issue_d = [&](int c) {
                const uint64_t b = dW + (((c & 1) * kKV) >> 4);
                const uint32_t d = tmem + kTD + 64 * hf, a = tmem + kTZK + 64 * hf;
                mma_bf16_ta(d, a, b, idD, hf == 0 ? 1u : 0u);
#pragma unroll
                for (int s = 1; s < 8; ++s) mma_bf16_ta(d, a + 8 * s, b + s * kRow16, idD, 1u);
                mma_commit(&bars.dfull[hf]);
            };
            // Z^T(hf) += D^T(hf) K(c) with A = bf16 D^T in TMEM; with the other half's update
            // it frees the k slot
            auto issue_f = [&](int c) {   // KDA: B = Kh, the slot's second tile
                const uint64_t b = dK + (((c % kKSlots) * kKSl + (KDA ? kKV : 0)) >> 4);
                const uint32_t d = tmem + kTZ + 128 * hf, a = tmem + kTD + 64 * hf;
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16_ta(d, a + 8 * s, b + s * kRow16, idF, 1u);
                if (!outm) {
                    mma_commit(&bars.zfull[hf]);
                    mma_commit(&bars.kempty[c % kKSlots]);
                }
            };
            // outputs instance: O^T = S~^T Q^T (A = the bf16 Z_S^T of d_S, B = the q chunk,
            // K-major, 64-channel halves), and O^T += D_S^T A^T (A = the bf16 D_S^T of f_S,
            // B = the masked Q K^T of the chunk, K-major)
            auto issue_qs = [&](int c) {
                const uint64_t b = dQ + (((c & 1) * kKV) >> 4);
                const uint32_t d = tmem + kTO + 64 * (c & 1);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16_ta(d, tmem + kTZK + 8 * s, b + (((s >> 2) * kHalf) >> 4) + (s & 3) * kCol16,
                                idO, s > 0 ? 1u : 0u);
            };
            auto issue_intra = [&](int c) {
                const uint64_t b = dAq + (((c & 1) * kRec) >> 4);
                const uint32_t d = tmem + kTO + 64 * (c & 1);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16_ta(d, tmem + kTD + 8 * s, b + s * kCol16, idO, 1u);
            };
            bool ok = true;
            if (hf == 0) {
                // W^T(c) = K^T M2^T into the S~ half's bf16-Z^T columns (A: the k chunk read
                // MN-major, B: the M2 record K-major)
                auto issue_w = [&](int c) {   // KDA: A = Kt
                    const uint64_t a = dK + (((c % kKSlots) * kKSl) >> 4), b = dR + (((c % kVSlots) * kVR) >> 4);
                    mma_bf16(tmem + kTZK, a, b, idA, 0u);
#pragma unroll
                    for (int s = 1; s < 4; ++s) mma_bf16(tmem + kTZK, a + s * kRow16, b + s * kCol16, idA, 1u);
                    mma_commit(&bars.wfull);
                };
                // D_S^T(c) = V^T M1^T (A: the v chunk read MN-major, B: M1 K-major); frees the
                // {v, M2} slot of chunk c
                auto issue_u = [&](int c) {   // KDA: B = the M2 record itself
                    const uint64_t a = dV + (((c % kVSlots) * kVR) >> 4);
                    const uint64_t b = KDA ? dR + (((c % kVSlots) * kVR) >> 4) : dM + (((c & 1) * kRec) >> 4);
                    mma_bf16(tmem + kTD, a, b, idA, 0u);
#pragma unroll
                    for (int s = 1; s < 4; ++s) mma_bf16(tmem + kTD, a + s * kRow16, b + s * kCol16, idA, 1u);
                    mma_commit(&bars.vempty[c % kVSlots]);
                };
                // per chunk: d_S(c), W(c+1), f_S(c), U(c+1). W(c+1) overwrites the columns
                // d_S(c) reads as A and U(c+1) the D_S columns f_S(c) reads as A, so each is
                // issued only once that product's completion has been observed.
                ok = wait(&bars.kfull[0], 0) && wait(&bars.vfull[0], 0);
                if (ok) {
                    tc_fence_after();
                    issue_w(0);
                    if ((ok = wait(&bars.m1ready[0], 0))) {
                        tc_fence_after();
                        issue_u(0);
                    }
                }
                for (int c = 0; ok && c < nch; ++c) {
                    const bool more = c + 1 < nch;
                    if (!(ok = wait(&bars.wready[c & 1], (c >> 1) & 1) && wait(&bars.zready[0], c & 1))) break;
                    if (outm && !(ok = wait(&bars.qfull[c & 1], (c >> 1) & 1) &&
                                       (c < 2 || wait(&bars.ofree[c & 1], ((c - 2) >> 1) & 1))))
                        break;
                    tc_fence_after();
                    if (outm) issue_qs(c);
                    issue_d(c);
                    if (outm) mma_commit(&bars.qempty[c & 1]);
                    if (more) {
                        if (!(ok = wait(&bars.dfull[0], c & 1) && wait(&bars.kfull[(c + 1) % kKSlots], ((c + 1) / kKSlots) & 1) &&
                                   wait(&bars.vfull[(c + 1) % kVSlots], ((c + 1) / kVSlots) & 1)))
                            break;
                        tc_fence_after();
                        issue_w(c + 1);
                    }
                    if (!(ok = wait(&bars.dready[0], c & 1))) break;
                    tc_fence_after();
                    issue_f(c);
                    if (outm) {
                        if (!(ok = wait(&bars.aqready[c & 1], (c >> 1) & 1))) break;
                        tc_fence_after();
                        issue_intra(c);
                        mma_commit(&bars.zfull[0]);
                        mma_commit(&bars.kempty[c % kKSlots]);
                        mma_commit(&bars.ofull[c & 1]);
                    }
                    if (more) {
                        if (!(ok = wait(&bars.zfull[0], c & 1) && wait(&bars.m1ready[(c + 1) & 1], ((c + 1) >> 1) & 1)))
                            break;
                        tc_fence_after();
                        issue_u(c + 1);
                    }
                }
            } else if (outm) {
                // outputs instance: Q K^T of every chunk (M = 64: A the q chunk, B the k chunk,
                // both K-major) into the D_P columns, once the output warps have read the last
                for (int c = 0; ok && c < nch; ++c) {
                    if (!(ok = wait(&bars.qfull[c & 1], (c >> 1) & 1) &&
                               wait(&bars.kfull[c % kKSlots], (c / kKSlots) & 1) &&
                               (c < 1 || wait(&bars.aqfree, (c - 1) & 1))))
                        break;
                    tc_fence_after();
                    const uint64_t a = dQ + (((c & 1) * kKV) >> 4), b = dKk + (((c % kKSlots) * kKV) >> 4);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint64_t o = (((s >> 2) * kHalf) >> 4) + (s & 3) * kCol16;
                        mma_bf16(tmem + kTAq, a + o, b + o, idQK, s > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars.aqfull);
                    mma_commit(&bars.qempty[c & 1]);
                    mma_commit(&bars.kempty[c % kKSlots]);
                }
            } else {
                // per chunk: d_P(c) (frees the -W^T slot for the operand warps), f_P(c).
                // zready_P(c) implies f_P(c-1) is complete (the P half waited for it).
                for (int c = 0; ok && c < nch; ++c) {
                    if (!(ok = wait(&bars.wready[c & 1], (c >> 1) & 1) && wait(&bars.zready[1], c & 1))) break;
                    tc_fence_after();
                    issue_d(c);
                    mma_commit(&bars.wfree[c & 1]);
                    if (!(ok = wait(&bars.dready[1], c & 1))) break;
                    tc_fence_after();
                    issue_f(c);
                }
            }
            if (!ok) {   // let this thread's MMAs in flight finish before the CTA exits
                mma_commit(&bars.fin[hf]);
                mbar_wait(&bars.fin[hf], 0, p.err, kErrTimeout);
            }
        }
    } else if (warp >= kAuxWarp0 && warp < kProducerWarp) {
        // ---------------------------------------------------------------- operand warps 8-11
        const int q = threadIdx.x - 32 * kAuxWarp0;    // 0..127 = TMEM lane of W^T
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        float Lam = 0.f, lam_sum = 0.f;
        float la_next = 0.f;   // log-gate of the next chunk (thread q < 64: token q)
        if (q < C && nch > 0 && gdn) {
            const int64_t tok = (int64_t)seg.start + q;
            la_next = q < min(C, seg.len) ? p.log_gate[tok * p.H_v + h] : 0.f;
        }
        for (int c = 0; c < nch; ++c) {
            if constexpr (KDA) {
                // (1) the chunk's scales from the preparation's record: S half e^{c_C}, P half
                //     e^{c_C - m}. Slot c % 4 was last read (for chunk c - 4) in the Z passes of
                //     chunk c - 3: the waits of chunk c - 1 below (W(c - 1) complete, hence
                //     d_S(c - 2); d_P(c - 3) complete) imply that both halves are done with them.
                if (c == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                const float *side = p.kda_side + ((int64_t)seg.wsb + (int64_t)h * nch + c) * kKdaSide;
                const float cq = side[q], mC = side[128];
                KdaSlot &ks = kslots[c % kKdaSlots];
                ks.gs[q] = expf(cq);
                ks.gp[q] = expf(cq - mC);
                lam_sum += mC;
                if (q == 0) ks.lam_sum = lam_sum;
                mbar_arrive(&bars.gready[c % kKdaSlots]);
                // (2) no M1: U reads the record itself
                mbar_arrive(&bars.m1ready[c & 1]);
            } else {
            Slot &sl = slots[c % kSlots];
            // (1) gates: prefix sums c_t, chunk total c_C, the log-scale bookkeeping.
            //     Slot c % 2 was last read for chunk c - 2, whose W product has been issued.
            float x = la_next;
            if (q < C && gdn && c + 1 < nch) {
                const int64_t tok = (int64_t)seg.start + (c + 1) * C + q;
                la_next = q < min(C, seg.len - (c + 1) * C) ? p.log_gate[tok * p.H_v + h] : 0.f;
            }
            if (q < C) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane == 31) scan_tmp[q >> 5] = x;
            }
            bar_aux();
            const float cC = scan_tmp[0] + scan_tmp[1];
            const bool renorm = Lam + cC < kRenormBelow;
            const float lam0 = renorm ? 0.f : Lam;
            if (q < C) sl.ex[q] = expf(-lam0 - (q >= 32 ? x + scan_tmp[0] : x));
            if (OUT && q < C) s_oscale[c % kSlots][q] = expf(lam0 + (q >= 32 ? x + scan_tmp[0] : x));
            if (q == 0) {
                sl.renorm = renorm ? 1 : 0;
                sl.rscale = expf(Lam);
                sl.lam_after = lam0 + cC;
                sl.lam_sum = lam_sum + cC;
                if (cC < kMinChunkLogDecay) atomicOr(p.err, kErrRange);
            }
            Lam = lam0 + cC;
            lam_sum += cC;
            bar_aux();   // ex visible; every read of scan_tmp done before the next writes
            // (2) M1[t'][t] = M2[t'][t] exp(-Lam_start - c_t), same swizzled layout
            if (!bar_aux_and(wait(&bars.vfull[c % kVSlots], (c / kVSlots) & 1))) break;
            {
                const uint8_t *rec = smem + oVR + (c % kVSlots) * kVR + kKV;
                uint8_t *m1 = smem + oM1 + (c & 1) * kRec;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int e = q + 128 * m;   // 16-byte piece: row t', columns 8 t8 .. 8 t8 + 7
                    const int tp = e >> 3, t8 = e & 7;
                    const uint32_t off = sw128(tp, 16 * t8);
                    const uint4 r = *reinterpret_cast<const uint4 *>(rec + off);
                    const float4 e0 = reinterpret_cast<const float4 *>(sl.ex + 8 * t8)[0];
                    const float4 e1 = reinterpret_cast<const float4 *>(sl.ex + 8 * t8)[1];
                    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
                    float f[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        f[2 * j] = __uint_as_float(w[j] << 16);
                        f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                    }
                    *reinterpret_cast<uint4 *>(m1 + off) =
                        make_uint4(bf2(f[0] * e0.x, f[1] * e0.y), bf2(f[2] * e0.z, f[3] * e0.w),
                                   bf2(f[4] * e1.x, f[5] * e1.y), bf2(f[6] * e1.z, f[7] * e1.w));
                }
            }
            fence_async_shared();
            mbar_arrive(&bars.m1ready[c & 1]);
            }
            // (3) W^T(c) -> -W^T bf16, MN-major B operand (row i = this thread's lane). The
            //     slot was last read by d_S(c-2) (ordered before W(c) by its issuer) and by
            //     d_P(c-2), whose completion is signalled on wfree.
            if (!bar_aux_and(wait(&bars.wfull, c & 1) &&
                             (outm || c < 2 || wait(&bars.wfree[c & 1], ((c - 2) >> 1) & 1))))
                break;
            tc_fence_after();
            {
                uint32_t z[64];
                ld64(tmem + lane_off + kTZK, z);
                tmem_ld_wait();
                uint8_t *wop = smem + oWop + (c & 1) * kKV;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 pk;
                    pk.x = bf2(-__uint_as_float(z[8 * j + 0]), -__uint_as_float(z[8 * j + 1]));
                    pk.y = bf2(-__uint_as_float(z[8 * j + 2]), -__uint_as_float(z[8 * j + 3]));
                    pk.z = bf2(-__uint_as_float(z[8 * j + 4]), -__uint_as_float(z[8 * j + 5]));
                    pk.w = bf2(-__uint_as_float(z[8 * j + 6]), -__uint_as_float(z[8 * j + 7]));
                    *reinterpret_cast<uint4 *>(wop + sw128((uint32_t)q, 16 * j)) = pk;
                }
            }
            fence_async_shared();
            tc_fence_before();
            mbar_arrive(&bars.wready[c & 1]);
        }
    } else if (outm && warp >= 4) {   // warps 4-7 (warps 8 and up took the branches above)
        // ---------------------------------------------------------------- output warps 4-7
        // Per chunk c: (a) the masked Q K^T (M = 64 accumulator: rows 16 (warp % 4) + lane in
        // lanes 0-15) -> bf16 rows t of the K-major B operand, columns s <= t; (b) the outputs,
        // o_t[n] = O^T[n][t] exp(Lam + c_t), the scale written with the chunk's gate slot.
        // The masked Q K^T of chunk c + 1 is prepared before the outputs of chunk c are read
        // out and stored, so that the S~ issuer's intra-chunk product of c + 1 does not wait
        // for chunk c's stores.
        const int n = threadIdx.x & 127;   // state column = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        __nv_bfloat16 *Ob = static_cast<__nv_bfloat16 *>(p.O);
        auto prep_aq = [&](int c) -> bool {
            if (!wwait(&bars.aqfull, c & 1)) return false;
            tc_fence_after();
            uint32_t z[64];
            ld64(tmem + lane_off + kTAq, z);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bars.aqfree);
            if (lane < 16) {
                const int t = 16 * (warp & 3) + lane;
                uint8_t *aq = smem + kOffAq + (c & 1) * kRec;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = (8 * j + e <= t) ? __uint_as_float(z[8 * j + e]) : 0.f;
                    *reinterpret_cast<uint4 *>(aq + sw128((uint32_t)t, 16u * j)) =
                        make_uint4(bf2(f[0], f[1]), bf2(f[2], f[3]), bf2(f[4], f[5]), bf2(f[6], f[7]));
                }
            }
            fence_async_shared();
            mbar_arrive(&bars.aqready[c & 1]);
            return true;
        };
        bool ok = nch == 0 || prep_aq(0);
        for (int c = 0; ok && c < nch; ++c) {
            if (c + 1 < nch && !(ok = prep_aq(c + 1))) break;
            if (!(ok = wwait(&bars.ofull[c & 1], (c >> 1) & 1))) break;
            tc_fence_after();
            uint32_t z[64];
            ld64(tmem + lane_off + kTO + 64 * (c & 1), z);
            tmem_ld_wait();
            // scaled with the chunk's gate slot before the accumulator is freed: freeing it
            // lets the next chunks run on, and the slot is rewritten four chunks later
            {
                const float4 *os4 = reinterpret_cast<const float4 *>(s_oscale[c % kSlots]);
#pragma unroll
                for (int t4 = 0; t4 < C / 4; ++t4) {
                    const float4 e = os4[t4];
                    z[4 * t4] = __float_as_uint(__uint_as_float(z[4 * t4]) * e.x);
                    z[4 * t4 + 1] = __float_as_uint(__uint_as_float(z[4 * t4 + 1]) * e.y);
                    z[4 * t4 + 2] = __float_as_uint(__uint_as_float(z[4 * t4 + 2]) * e.z);
                    z[4 * t4 + 3] = __float_as_uint(__uint_as_float(z[4 * t4 + 3]) * e.w);
                }
            }
            tc_fence_before();
            mbar_arrive(&bars.ofree[c & 1]);
            const int nv = min(C, seg.len - c * C);
            const int64_t tok0 = (int64_t)seg.start + (int64_t)c * C;
            {
                __nv_bfloat16 *op = Ob + ((tok0 * p.H_v + h) * D + n);
                const int64_t st = (int64_t)p.H_v * D;
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    if (t < nv) *op = __float2bfloat16_rn(__uint_as_float(z[t]));
                    op += st;
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- chain warps 0-7
        const int hf = warp >> 2;                  // 0: S~ half, 1: P half
        const int n = threadIdx.x & 127;           // state column = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t zcol = kTZ + 128 * hf, dcol = kTD + 64 * hf, zkcol = kTZK + 64 * hf;
        {   // Z^T = 0 (S~ half) or I (P half); the TMEM address of a warp-wide store must be
            // the same in all lanes, so every lane stores every column group
            uint32_t z[16];
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) z[j] = (hf == 1 && c0 + j == n) ? __float_as_uint(1.f) : 0u;
                tmem_st16(tmem + lane_off + zcol + c0, z);
            }
            tmem_st_wait();
        }
        bool ok = true;
        for (int c = 0; ok && c < nch; ++c) {
            // (1) Z^T -> bf16 A operand in TMEM (S~ half: multiplied by exp(Lam) first on a
            //     reset). The S~ half's bf16 columns hold W^T(c) until its pass has read it.
            if (c >= 1 && !(ok = wwait(&bars.zfull[hf], (c - 1) & 1))) break;
            bool renorm = false;
            float rs = 1.f;
            if constexpr (KDA) {   // both halves read the previous chunk's gate slot
                if (!(ok = (c == 0 || wwait(&bars.gready[(c - 1) % kKdaSlots], ((c - 1) / kKdaSlots) & 1)) &&
                           (hf == 1 || wwait(&bars.wready[c & 1], (c >> 1) & 1))))
                    break;
            } else if (hf == 0) {
                if (!(ok = wwait(&bars.m1ready[c & 1], (c >> 1) & 1) && wwait(&bars.wready[c & 1], (c >> 1) & 1)))
                    break;
                renorm = slots[c % kSlots].renorm != 0;
                rs = slots[c % kSlots].rscale;
            }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t z[64];
                ld64(tmem + lane_off + zcol + 64 * cb, z);
                tmem_ld_wait();
                if (KDA && c > 0) {
                    // the previous chunk's row scaling, written back, then the bf16 copy for d
                    const KdaSlot &ks = kslots[(c - 1) % kKdaSlots];
                    const float4 *g4 = reinterpret_cast<const float4 *>((hf == 0 ? ks.gs : ks.gp) + 64 * cb);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float4 gg = g4[j];
                        z[4 * j] = __float_as_uint(__uint_as_float(z[4 * j]) * gg.x);
                        z[4 * j + 1] = __float_as_uint(__uint_as_float(z[4 * j + 1]) * gg.y);
                        z[4 * j + 2] = __float_as_uint(__uint_as_float(z[4 * j + 2]) * gg.z);
                        z[4 * j + 3] = __float_as_uint(__uint_as_float(z[4 * j + 3]) * gg.w);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tmem_st16(tmem + lane_off + zcol + 64 * cb + 16 * j, *reinterpret_cast<uint32_t(*)[16]>(&z[16 * j]));
                }
                if (renorm) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) z[j] = __float_as_uint(__uint_as_float(z[j]) * rs);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tmem_st16(tmem + lane_off + zcol + 64 * cb + 16 * j,
                                  *reinterpret_cast<uint32_t(*)[16]>(&z[16 * j]));
                }
                st_bf16x64(tmem + lane_off + zkcol + 32 * cb, z);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars.zready[hf]);
            // (2) D^T -> bf16 A operand of the update, over the accumulator's first columns
            if (!(ok = wwait(&bars.dfull[hf], c & 1))) break;
            tc_fence_after();
            {
                uint32_t z[64];
                ld64(tmem + lane_off + dcol, z);
                tmem_ld_wait();
                st_bf16x64(tmem + lane_off + dcol, z);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars.dready[hf]);
        }
        // outputs: S = exp(Lam) S~ (column n) or P (column n), and lam (the outputs instance
        // writes only O)
        if (ok && nch > 0) ok = wwait(&bars.zfull[hf], (nch - 1) & 1);
        // KDA: the last chunk's row scaling is applied here
        if (KDA && ok && nch > 0) ok = wwait(&bars.gready[(nch - 1) % kKdaSlots], ((nch - 1) / kKdaSlots) & 1);
        tc_fence_after();

        if (!outm) {
            // a piece of a split segment writes its own slot; a whole segment the caller's output
            const bool piece = seg.idx < 0;
            const int64_t unit = piece ? (int64_t)(-1 - seg.idx) * p.H_v + h : (int64_t)seg.idx * p.seg_stride + h;
            float *O = (hf == 0 ? (piece ? p.S_piece : p.S) : (piece ? p.P_piece : p.P)) + unit * D * D + n;
            const float sc = (!KDA && hf == 0 && nch > 0) ? expf(slots[(nch - 1) % kSlots].lam_after) : 1.f;
            const float *gl = nullptr;
            if (KDA && nch > 0) gl = hf == 0 ? kslots[(nch - 1) % kKdaSlots].gs : kslots[(nch - 1) % kKdaSlots].gp;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t z[32];
                tmem_ld32(tmem + lane_off + zcol + c0, z);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    O[(int64_t)(c0 + j) * D] = __uint_as_float(z[j]) * (KDA && gl ? gl[c0 + j] : sc);
            }
            if (hf == 0 && n == 0)
                (piece ? p.lam_piece : p.lam)[unit] =
                    nch == 0 ? 0.f : KDA ? kslots[(nch - 1) % kKdaSlots].lam_sum : slots[(nch - 1) % kSlots].lam_sum;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

#if !defined(HYPIC_GDN_TC_OUTPUTS) && !defined(HYPIC_GDN_TC_KDA)
bool build_gdn_tc_supported(const BuildParams &p) {
    return p.D == D && p.dtype == HYPIC_BF16 &&
           (p.family == HYPIC_FAM_GDN || p.family == HYPIC_FAM_DELTA || p.family == HYPIC_FAM_KDA);
}
#endif

namespace {

template <bool OUT, bool KDA>
cudaError_t launch_chain(const BuildParams &p, cudaStream_t s) {
    // with the segment outputs, a second CTA per unit runs the outputs instance
    const int blocks = p.n_seg * p.H_v * (p.O ? 2 : 1);
    if (blocks == 0) return cudaSuccess;
    int64_t records = 0;
    for (int r = 0; r < p.n_seg; ++r) records += (int64_t)p.H_v * ((p.seg[r].len + C - 1) / C);
    const int64_t N = p.n_tok > 0 ? p.n_tok : 1;
    CUtensorMap tmK, tmV, tmR, tmQ;
    if (!make_tmap_3d(&tmK, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_k, N, (uint64_t)D * 2,
                      (uint64_t)p.H_k * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tmV, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_v, N, (uint64_t)D * 2,
                      (uint64_t)p.H_v * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (KDA) {   // the gated keys Kt (in tmK's place) and Kh (in tmQ's), [records x 64 rows][128]
        if (records > 0 &&
            (!make_tmap_2d(&tmK, p.kda_kt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)records * 64, D * 2, 64,
                           64, CU_TENSOR_MAP_SWIZZLE_128B) ||
             !make_tmap_2d(&tmQ, p.kda_kh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)records * 64, D * 2, 64,
                           64, CU_TENSOR_MAP_SWIZZLE_128B)))
            return cudaErrorInvalidValue;
        if (records == 0) tmQ = tmK;
    } else if (p.O) {
        if (!make_tmap_3d(&tmQ, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_k, N, (uint64_t)D * 2,
                          (uint64_t)p.H_k * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else {
        tmQ = tmK;   // no outputs instance: never read
    }
    if (records > 0) {
        if (!p.workspace ||
            !make_tmap_2d(&tmR, p.workspace, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, (uint64_t)records * 64,
                          128, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else {
        tmR = tmK;   // no chunk anywhere: the kernel issues no load
    }
    cudaError_t e = KDA ? launch_build_kda_prep(p, s) : launch_build_gdn_prep(p, s);
    if (e != cudaSuccess) return e;
    const uint32_t smem = KDA ? kSmemBytesKda : OUT ? kSmemBytesOut : kSmemBytes;
    auto kern = build_gdn_tc_kernel<OUT, KDA>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (records == 0) {
        kern<<<blocks, kThreads, smem, s>>>(p, tmK, tmV, tmR, tmQ);
        return cudaGetLastError();
    }
    // launched as a programmatic dependent of the preparation kernel: CTAs may start (set-up,
    // k / v loads) on SMs the preparation has left, and wait for its completion before
    // reading its records
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, tmK, tmV, tmR, tmQ);
}

}  // namespace

// The instances are compiled in separate translation units (this file; build_gdn_tc_out.cu and
// build_gdn_tc_kda.cu, which include it with HYPIC_GDN_TC_OUTPUTS or HYPIC_GDN_TC_KDA defined):
// with two in one unit the plain chain measured 6.5% slower on GB300 (0.311 against 0.292 ms
// per build call).
#if defined(HYPIC_GDN_TC_KDA)
cudaError_t launch_build_kda_tc(const BuildParams &p, cudaStream_t s) { return launch_chain<false, true>(p, s); }
#elif defined(HYPIC_GDN_TC_OUTPUTS)
cudaError_t launch_build_gdn_tc_outputs(const BuildParams &p, cudaStream_t s) { return launch_chain<true, false>(p, s); }
#else
cudaError_t launch_build_gdn_tc(const BuildParams &p, cudaStream_t s) {
    if (p.family == HYPIC_FAM_KDA) return launch_build_kda_tc(p, s);
    return p.O ? launch_build_gdn_tc_outputs(p, s) : launch_chain<false, false>(p, s);
}
#endif

}  // namespace hypic
