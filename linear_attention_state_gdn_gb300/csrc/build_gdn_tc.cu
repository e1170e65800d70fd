// build_gdn_tc.cu -- DeltaNet / Gated DeltaNet segment build on the 5th-generation tensor
// cores (bf16 k / v, d_k = d_v = 128, fp32 state).
//
// What is computed: for every cached segment C and value head the pair (S(C|0), T_C) with
// T_C = exp(lam) P, P = prod_t (I - b_t k_t k_t^T) (latest factor leftmost), lam = sum log a_t
// ("Cut First-Token Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For
// linear layers": HYPIC stores (T_C, S(C|0)) for DeltaNet / GDN layers; GDN recurrence from
// "Gated Delta Networks: Improving Mamba2 with Delta Rule", reference 7 of the episode
// companion page "Hypic: Position-Independent KV Caching for Hybrid-Attention LLM Serving").
//
// Chunked form (exact algebra, chunks of C = 64 tokens, c_t = sum_{s<=t} log a_s inside
// the chunk, A_ts = b_t (k_t . k_s) exp(c_t - c_s) for s < t, M = (I + A)^-1):
//     S <- e^{c_C} (S + K^T Diag(e^-c) M Diag(b) (V - Diag(e^c) K S)),
//     P <- P - K^T Diag(e^-c) M Diag(b e^c) K P,
// i.e. with Y = K [S | P] and R = Diag(b) [V - Diag(e^c) Y_S | -Diag(e^c) Y_P] every chunk
// adds K^T Diag(e^-c) M R to the state. The state is carried as Z = [S~ | P] with
// S = exp(Lam) S~ (Lam a running log-scale, folded into S~ when it drops below -20):
//     Y = K Z,  R = Diag(b) [exp(-Lam) V - Diag(e^c) Y_S | -Diag(e^c) Y_P],
//     Z <- Z + K^T D',  D' = Diag(e^-c) M R.
// Only M depends on the chunk's gram; everything that touches the state is three MMAs
// (Y, M R, K^T D') plus two per-lane transforms.
//
// Layout (one CTA = one (segment, value head) unit, 320 threads):
//   TMEM  Z^T      [0,256)   lane = state column n (S~ half, then P half), column = key row i
//         Y^T/D^T  [256,384) lane n, column t: Y^T = Z^T K^T, then (M R)^T in the same place
//         G        [384,512) two gram slots (M = 64 layout), one per chunk parity
//   SMEM  two TMA stages of (k, v) chunks (128B-swizzled, channels contiguous); the bf16
//         K-major operands Z^T (A of Y), R^T then D'^T (A of M R, then of the update) and M
//         (B of M R); the fp32 A and M of the inversion; per-chunk gate vectors (3 slots).
// Roles: warps 0-3 carry the chain (Z^T -> bf16, R, D'; thread n = TMEM lane n), warps 4-7
// prepare M for the next chunk (gates, A from the gram, 16 x 16-blocked inverse in fp32),
// warp 8 issues TMA, warp 9 issues the MMAs. Every wait is bounded.
#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace hypic {
namespace {

using namespace ptx;

constexpr int D = 128;
constexpr int C = 64;
constexpr int kThreads = 320;
constexpr int kPrepWarp0 = 4;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRenorm = -20.f;     // fold exp(Lam) into S~ below this log-scale
constexpr float kMinChunkLogDecay = -60.f;

// shared-memory map (offsets from the 1024-aligned base)
constexpr uint32_t kKTile = C * 256;                  // k chunk: two 64-channel halves, 16 KB
constexpr uint32_t kStage = 2 * kKTile;               // k + v
constexpr uint32_t kOffStage = 0;                     // 2 stages: 64 KB
constexpr uint32_t kOffAZ = 2 * kStage;               // Z^T bf16, 2 K-blocks x 256 rows x 128 B
constexpr uint32_t kOffAR = kOffAZ + 65536;           // R^T / D'^T bf16, 256 rows x 128 B
constexpr uint32_t kOffBM = kOffAR + 32768;           // M bf16, 64 rows t x 128 B
constexpr uint32_t kLDA = 68;                         // padded row stride of the fp32 A (16-B rows)
constexpr uint32_t kOffA32 = kOffBM + 8192;           // fp32 A, 64 x 68
constexpr uint32_t kOffM32 = kOffA32 + 64 * kLDA * 4; // fp32 M, 64 x 64
constexpr uint32_t kOffT = kOffM32 + 64 * 64 * 4;     // fp32 block products, 3 x 16 x 16
constexpr uint32_t kOffVec = kOffT + 3 * 256 * 4;     // per-chunk vectors (3 slots)

constexpr uint32_t kTZ = 0, kTY = 256, kTG = 384;

struct Vec {   // one slot of per-chunk vectors
    float beta[C], c[C], ecp[C], ecm[C], bec[C];
    float cC;  // chunk total log decay
    float pad[3];
};
constexpr uint32_t kSmemBytes = kOffVec + 3 * sizeof(Vec) + 1024;

struct Bars {
    uint64_t kv_full[2], kv_empty[2];
    uint64_t gfull[2];   // one per gram slot, so a wait can never alias a later phase
    // one per gate-vector slot: the prep may run two chunks ahead of the chain's wait on
    // these (its progress past chunk c + 1 only needs the chain's step 2 of chunk c), so
    // a single barrier could be two phases ahead and alias the awaited parity
    uint64_t vready[3];
    uint64_t mready, zbf_ready, yfull, rready, dfull, dready, zfull, fin;
};

// Named barrier of the 128 prep threads. The non-aligned form counts threads, not warps,
// so it stays correct when the lanes of a warp reach it at different times (for example
// lane 0 returning later from an mbarrier wait than its warp-mates); __syncwarp first
// reconverges the warp anyway.
__device__ __forceinline__ void bar_prep() {
    __syncwarp();
    asm volatile("barrier.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ uint32_t bf2(float lo, float hi) { return pack_bf16x2(lo, hi); }

// One level of the blocked inverse M = (I + A)^-1 (64 x 64, 16 x 16 blocks): the NB = 4 - L
// blocks (a, b) with a - b = L, from M_ab = -M_aa sum_{k=b}^{a-1} A_ak M_kb. Prep thread q
// owns entries (row r0 + 8h, column j) of every block, r0 = q / 16, j = q % 16, h = 0, 1;
// all loops are compile-time so the independent dot products interleave.
template <int L>
__device__ __forceinline__ void inverse_level(const float *A32, float *M32, float *T32, int q) {
    constexpr int NB = 4 - L;
    const int j = q & 15, r0 = q >> 4;
    float t[2 * NB];
#pragma unroll
    for (int m = 0; m < 2 * NB; ++m) t[m] = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int k = b; k < b + L; ++k) {
            float mc[16];
#pragma unroll
            for (int s = 0; s < 16; ++s) mc[s] = M32[(16 * k + s) * C + 16 * b + j];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float4 *ar = reinterpret_cast<const float4 *>(A32 + (16 * (b + L) + r0 + 8 * hh) * kLDA + 16 * k);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const float4 x = ar[s4];
                    float &acc = t[2 * b + hh];
                    acc = fmaf(x.x, mc[4 * s4 + 0], acc);
                    acc = fmaf(x.y, mc[4 * s4 + 1], acc);
                    acc = fmaf(x.z, mc[4 * s4 + 2], acc);
                    acc = fmaf(x.w, mc[4 * s4 + 3], acc);
                }
            }
        }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) T32[b * 256 + (r0 + 8 * hh) * 16 + j] = t[2 * b + hh];
    bar_prep();
    float res[2 * NB];   // all loads first, then the stores (no load/store interleaving)
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int a = b + L;
        float tc[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) tc[s] = T32[b * 256 + s * 16 + j];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = r0 + 8 * hh;
            const float4 *mr = reinterpret_cast<const float4 *>(M32 + (16 * a + r) * C + 16 * a);
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const float4 x = mr[s4];
                acc0 = fmaf(x.x, tc[4 * s4 + 0], acc0);
                acc1 = fmaf(x.y, tc[4 * s4 + 1], acc1);
                acc0 = fmaf(x.z, tc[4 * s4 + 2], acc0);
                acc1 = fmaf(x.w, tc[4 * s4 + 3], acc1);
            }
            res[2 * b + hh] = -(acc0 + acc1);
        }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) M32[(16 * (b + L) + r0 + 8 * hh) * C + 16 * b + j] = res[2 * b + hh];
    bar_prep();
}

__global__ void __launch_bounds__(kThreads, 1)
build_gdn_tc_kernel(const __grid_constant__ BuildParams p, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived by offsetting the shared array itself so that the
    // compiler keeps the shared address space (plain ld/st.shared, not generic accesses)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars bars;
    __shared__ uint32_t tslot;
    __shared__ volatile int abort_flag;
    __shared__ float scan_tmp[2];
    __shared__ int prep_flag[2];

    const int warp = warp_id(), lane = lane_id();
    const SegEntry seg = p.seg[blockIdx.x / p.H_v];
    const int h = blockIdx.x % p.H_v;
    const int hk = h / p.gqa;
    const int nch = (seg.len + C - 1) / C;
    const bool gdn = p.family == HYPIC_FAM_GDN;
    Vec *vec = reinterpret_cast<Vec *>(smem + kOffVec);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        mbar_init(&bars.gfull[0], 1);
        mbar_init(&bars.gfull[1], 1);
        for (int s = 0; s < 3; ++s) mbar_init(&bars.vready[s], 128);
        mbar_init(&bars.mready, 128);
        mbar_init(&bars.zbf_ready, 128);
        mbar_init(&bars.yfull, 1);
        mbar_init(&bars.rready, 128);
        mbar_init(&bars.dfull, 1);
        mbar_init(&bars.dready, 128);
        mbar_init(&bars.zfull, 1);
        mbar_init(&bars.fin, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    auto wait = [&](uint64_t *b, uint32_t par) {
        return mbar_wait_or_abort(b, par, p.err, kErrTimeout, &abort_flag);
    };

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            int c = 0;
            for (; c < nch; ++c) {
                const int s = c & 1, use = c >> 1;
                if (use >= 1 && !wait(&bars.kv_empty[s], (use - 1) & 1)) break;
                uint8_t *st = smem + kOffStage + s * kStage;
                const int32_t t0 = seg.start + c * C;
                mbar_arrive_expect_tx(&bars.kv_full[s], kStage);
                tma_load_3d(st, &tmK, &bars.kv_full[s], 0, hk, t0);
                tma_load_3d(st + kKTile / 2, &tmK, &bars.kv_full[s], 64, hk, t0);
                tma_load_3d(st + kKTile, &tmV, &bars.kv_full[s], 0, h, t0);
                tma_load_3d(st + kKTile + kKTile / 2, &tmV, &bars.kv_full[s], 64, h, t0);
            }
            if (abort_flag)
                for (int q = (c > 2 ? c - 2 : 0); q < c; ++q)
                    mbar_wait(&bars.kv_full[q & 1], (q >> 1) & 1, p.err, kErrTimeout);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idG = idesc(kFmtBF16, kFmtBF16, false, false, 64, 64);
            constexpr uint32_t idKK = idesc(kFmtBF16, kFmtBF16, false, false, 128, 64);
            constexpr uint32_t idZ = idesc(kFmtBF16, kFmtBF16, false, true, 128, 128);
            const uint32_t sb = smem_u32(smem);
            auto issue_gram = [&](int c) -> bool {
                if (!wait(&bars.kv_full[c & 1], (c >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t k = sb + kOffStage + (c & 1) * kStage;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t a = k + (s >> 2) * (kKTile / 2) + (s & 3) * 32;
                    mma_bf16(tmem + kTG + 64 * (c & 1), sdesc(a, 16, 1024, kSwizzle128B),
                             sdesc(a, 16, 1024, kSwizzle128B), idG, s > 0);
                }
                mma_commit(&bars.gfull[c & 1]);
                return true;
            };
            bool ok = issue_gram(0);
            for (int c = 0; ok && c < nch; ++c) {
                const uint32_t k = sb + kOffStage + (c & 1) * kStage;
                // Y^T = Z^T K^T (S~ and P halves)
                if (!(ok = wait(&bars.zbf_ready, c & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t a = sb + kOffAZ + (s >> 2) * 32768 + hf * 16384 + (s & 3) * 32;
                        const uint32_t b = k + (s >> 2) * (kKTile / 2) + (s & 3) * 32;
                        mma_bf16(tmem + kTY + 64 * hf, sdesc(a, 16, 1024, kSwizzle128B),
                                 sdesc(b, 16, 1024, kSwizzle128B), idKK, s > 0);
                    }
                mma_commit(&bars.yfull);
                // the next chunk's gram, into the other slot
                if (c + 1 < nch && !(ok = issue_gram(c + 1))) break;
                // (M R)^T = R^T M^T
                if (!(ok = wait(&bars.rready, c & 1) && wait(&bars.mready, c & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16(tmem + kTY + 64 * hf,
                                 sdesc(sb + kOffAR + hf * 16384 + s * 32, 16, 1024, kSwizzle128B),
                                 sdesc(sb + kOffBM + s * 32, 16, 1024, kSwizzle128B), idKK, s > 0);
                mma_commit(&bars.dfull);
                // Z^T += D'^T K
                if (!(ok = wait(&bars.dready, c & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16(tmem + kTZ + 128 * hf,
                                 sdesc(sb + kOffAR + hf * 16384 + s * 32, 16, 1024, kSwizzle128B),
                                 sdesc(k + s * 2048, kKTile / 2, 1024, kSwizzle128B), idZ, 1);
                mma_commit(&bars.zfull);
                mma_commit(&bars.kv_empty[c & 1]);
            }
            if (abort_flag) {
                mma_commit(&bars.fin);
                mbar_wait(&bars.fin, 0, p.err, kErrTimeout);
            }
        }
    } else if (warp >= kPrepWarp0) {
        // ---------------------------------------------------------------- prep warps 4-7
        const int q = threadIdx.x - 128;          // 0..127
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        float *A32 = reinterpret_cast<float *>(smem + kOffA32);
        float *M32 = reinterpret_cast<float *>(smem + kOffM32);
        float *T32 = reinterpret_cast<float *>(smem + kOffT);
        float b_next = 0.f, la_next = 0.f;   // gates of the next chunk (thread q < 64: token q)
        if (q < C && nch > 0) {
            const int64_t tok = (int64_t)seg.start + q;
            const bool in = q < min(C, seg.len);
            b_next = in ? p.beta[tok * p.H_v + h] : 0.f;
            la_next = (in && gdn) ? p.log_gate[tok * p.H_v + h] : 0.f;
        }
        // one elected thread waits; the outcome reaches the other 127 through the named
        // barrier, so every prep thread takes the same branch (no thread is left behind
        // at a barrier when a wait gives up)
        uint32_t nw = 0;
        auto pwait = [&](uint64_t *b, uint32_t par) -> bool {
            volatile int *f = &prep_flag[nw & 1];
            if (q == 0) *f = wait(b, par) ? 1 : 0;
            bar_prep();
            const bool r = *f != 0;
            ++nw;
            return r;
        };
        for (int c = 0; c < nch; ++c) {   // leaves only through a broadcast pwait outcome
            // (a) gates of chunk c (loaded one chunk ahead into registers), prefix sums.
            //     Slot c % 3 was last read by the chain for chunk c - 3, long finished.
            Vec &v = vec[c % 3];
            const int valid = min(C, seg.len - c * C);
            float b_cur = b_next, la_cur = la_next;
            if (q < C && c + 1 < nch) {
                const int64_t tok = (int64_t)seg.start + (c + 1) * C + q;
                const bool in = q < min(C, seg.len - (c + 1) * C);
                b_next = in ? p.beta[tok * p.H_v + h] : 0.f;
                la_next = (in && gdn) ? p.log_gate[tok * p.H_v + h] : 0.f;
            }
            if (q < C) {
                if (q >= valid) b_cur = la_cur = 0.f;
                float x = la_cur;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane == 31) scan_tmp[q >> 5] = x;
                v.beta[q] = b_cur;
                v.c[q] = x;
            }
            bar_prep();
            if (q < C) {
                const float cc = q >= 32 ? v.c[q] + scan_tmp[0] : v.c[q];
                const float e = expf(cc);
                v.c[q] = cc;
                v.ecp[q] = e;
                v.ecm[q] = expf(-cc);
                v.bec[q] = v.beta[q] * e;
                if (q == C - 1) {
                    v.cC = cc;
                    if (cc < kMinChunkLogDecay) atomicOr(p.err, kErrRange);
                }
            }
            mbar_arrive(&bars.vready[c % 3]);
            // (b) gram -> A (rows t = 16 (warp - 4) + lane for lanes < 16), padded rows
            if (!pwait(&bars.gfull[c & 1], (c >> 1) & 1)) break;
            tc_fence_after();
            {
                const int t = 16 * (warp - kPrepWarp0) + lane;
                uint32_t g[64];
                const uint32_t gcol = kTG + 64 * (c & 1);
                tmem_ld32(tmem + lane_off + gcol, *reinterpret_cast<uint32_t(*)[32]>(&g[0]));
                tmem_ld32(tmem + lane_off + gcol + 32, *reinterpret_cast<uint32_t(*)[32]>(&g[32]));
                tmem_ld_wait();
                if (lane < 16) {
                    // all loads before any store (stores to A may not pass loads from the
                    // same shared memory, so interleaving them would serialise the loop)
                    const float bt = v.beta[t] * v.ecp[t];
                    float em[C];
#pragma unroll
                    for (int s4 = 0; s4 < C / 4; ++s4) {
                        const float4 e4 = reinterpret_cast<const float4 *>(v.ecm)[s4];
                        em[4 * s4] = e4.x, em[4 * s4 + 1] = e4.y, em[4 * s4 + 2] = e4.z, em[4 * s4 + 3] = e4.w;
                    }
                    float4 *row = reinterpret_cast<float4 *>(A32 + t * kLDA);
#pragma unroll
                    for (int s4 = 0; s4 < C / 4; ++s4) {
                        float4 a4;
                        const int s2 = 4 * s4;
                        a4.x = s2 + 0 < t ? bt * __uint_as_float(g[s2 + 0]) * em[s2 + 0] : 0.f;
                        a4.y = s2 + 1 < t ? bt * __uint_as_float(g[s2 + 1]) * em[s2 + 1] : 0.f;
                        a4.z = s2 + 2 < t ? bt * __uint_as_float(g[s2 + 2]) * em[s2 + 2] : 0.f;
                        a4.w = s2 + 3 < t ? bt * __uint_as_float(g[s2 + 3]) * em[s2 + 3] : 0.f;
                        row[s4] = a4;
                    }
                }
            }
            tc_fence_before();
            bar_prep();
            // (c) M = (I + A)^-1 by 16 x 16 blocks: diagonal blocks by forward substitution
            //     (thread = one column of one block, each row's A entries loaded ahead),
            //     then the blocks below the diagonal level by level.
            if (q < C) {
                const int a = q >> 4, j = q & 15;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float4 *Ar = reinterpret_cast<const float4 *>(A32 + (16 * a + r) * kLDA + 16 * a);
                    float ar[16];
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const float4 t4 = Ar[s4];
                        ar[4 * s4] = t4.x, ar[4 * s4 + 1] = t4.y, ar[4 * s4 + 2] = t4.z, ar[4 * s4 + 3] = t4.w;
                    }
                    float acc[4] = {(r == j) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int s2 = 0; s2 < r; ++s2) acc[s2 & 3] = fmaf(-ar[s2], x[s2], acc[s2 & 3]);
                    x[r] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) M32[(16 * a + r) * C + 16 * a + j] = x[r];
            } else {
                // zero the six blocks above the diagonal
                for (int e = q - C; e < 6 * 256; e += C) {
                    const int blk = e >> 8, r = (e >> 4) & 15, j = e & 15;
                    const int a = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                    const int b = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                    M32[(16 * a + r) * C + 16 * b + j] = 0.f;
                }
            }
            bar_prep();
            inverse_level<1>(A32, M32, T32, q);
            inverse_level<2>(A32, M32, T32, q);
            inverse_level<3>(A32, M32, T32, q);
            // (d) M as bf16 K-major rows t, once the M R product of chunk c - 1 has read it
            if (c >= 1 && !pwait(&bars.dfull, (c - 1) & 1)) break;
            {
                uint8_t *bm = smem + kOffBM;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int e8 = q + 128 * m;            // 8 consecutive entries of row t
                    const int t = e8 >> 3, s8 = (e8 & 7) * 8;
                    const float4 lo = reinterpret_cast<const float4 *>(M32 + t * C + s8)[0];
                    const float4 hi = reinterpret_cast<const float4 *>(M32 + t * C + s8)[1];
                    *reinterpret_cast<uint4 *>(bm + sw128(t, 2 * s8)) =
                        make_uint4(bf2(lo.x, lo.y), bf2(lo.z, lo.w), bf2(hi.x, hi.y), bf2(hi.z, hi.w));
                }
            }
            fence_async_shared();
            mbar_arrive(&bars.mready);
        }
    } else {
        // ---------------------------------------------------------------- chain warps 0-3
        const int n = threadIdx.x;   // state column (and TMEM lane)
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        float Lam = 0.f, lam_total = 0.f;
        // Z^T = [0 | I]
        {
            uint32_t z[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) z[j] = 0u;
#pragma unroll
            for (int c0 = 0; c0 < 256; c0 += 16) tmem_st16(tmem + lane_off + kTZ + c0, z);
            tmem_st_wait();
            // identity in the P half: every lane stores every column group (the TMEM
            // address of a warp-wide store must be the same in all lanes)
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) z[j] = (c0 + j == n) ? __float_as_uint(1.f) : 0u;
                tmem_st16(tmem + lane_off + kTZ + 128 + c0, z);
            }
            tmem_st_wait();
        }
        uint8_t *az = smem + kOffAZ, *ar = smem + kOffAR;
        const uint32_t vhalf = (uint32_t)(n >> 6) * (kKTile / 2), vbyte = (uint32_t)(n & 63) * 2;
        bool ok = true;
        for (int c = 0; ok && c < nch; ++c) {
            // (1) Z^T -> bf16 A operand (renormalising S~ when the log-scale got small)
            if (c >= 1 && !(ok = wait(&bars.zfull, (c - 1) & 1))) break;
            tc_fence_after();
            const bool renorm = Lam < kRenorm;
            const float sc = renorm ? expf(Lam) : 1.f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {   // 64 key rows per batch: K-block cb
                    uint32_t z[64];
                    const uint32_t col = kTZ + 128 * hf + 64 * cb;
                    tmem_ld32(tmem + lane_off + col, *reinterpret_cast<uint32_t(*)[32]>(&z[0]));
                    tmem_ld32(tmem + lane_off + col + 32, *reinterpret_cast<uint32_t(*)[32]>(&z[32]));
                    tmem_ld_wait();
                    if (hf == 0 && renorm) {
#pragma unroll
                        for (int j = 0; j < 64; ++j) z[j] = __float_as_uint(__uint_as_float(z[j]) * sc);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tmem_st16(tmem + lane_off + col + 16 * j, *reinterpret_cast<uint32_t(*)[16]>(&z[16 * j]));
                    }
                    uint8_t *rowb = az + cb * 32768;
                    const uint32_t r = 128 * hf + n;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 pk;
                        pk.x = bf2(__uint_as_float(z[8 * j + 0]), __uint_as_float(z[8 * j + 1]));
                        pk.y = bf2(__uint_as_float(z[8 * j + 2]), __uint_as_float(z[8 * j + 3]));
                        pk.z = bf2(__uint_as_float(z[8 * j + 4]), __uint_as_float(z[8 * j + 5]));
                        pk.w = bf2(__uint_as_float(z[8 * j + 6]), __uint_as_float(z[8 * j + 7]));
                        *reinterpret_cast<uint4 *>(rowb + sw128(r, 16 * j)) = pk;
                    }
                }
            }
            if (renorm) {
                tmem_st_wait();
                Lam = 0.f;
            }
            fence_async_shared();
            tc_fence_before();
            mbar_arrive(&bars.zbf_ready);
            // (2) R^T[n][t] = b_t (exp(-Lam) V[t][n] - e^{c_t} Y_S^T[n][t]), -b_t e^{c_t} Y_P^T[n][t]
            if (!(ok = wait(&bars.vready[c % 3], (c / 3) & 1) && wait(&bars.yfull, c & 1))) break;
            tc_fence_after();
            const Vec &v = vec[c % 3];
            const float eL = expf(-Lam);
            const uint8_t *vt = smem + kOffStage + (c & 1) * kStage + kKTile + vhalf;
#pragma unroll
            for (int c0 = 0; c0 < C; c0 += 32) {
                uint32_t ys[32], yp[32];
                tmem_ld32(tmem + lane_off + kTY + c0, ys);
                tmem_ld32(tmem + lane_off + kTY + 64 + c0, yp);
                // every shared-memory load of the batch before its stores
                float vv[32], bb[32], be[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    vv[j] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(vt + sw128(c0 + j, vbyte)));
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 b4 = reinterpret_cast<const float4 *>(v.beta + c0)[j4];
                    const float4 e4 = reinterpret_cast<const float4 *>(v.bec + c0)[j4];
                    bb[4 * j4] = b4.x, bb[4 * j4 + 1] = b4.y, bb[4 * j4 + 2] = b4.z, bb[4 * j4 + 3] = b4.w;
                    be[4 * j4] = e4.x, be[4 * j4 + 1] = e4.y, be[4 * j4 + 2] = e4.z, be[4 * j4 + 3] = e4.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float rs[8], rp[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int jj = 8 * j8 + j;
                        rs[j] = fmaf(bb[jj] * eL, vv[jj], -be[jj] * __uint_as_float(ys[jj]));
                        rp[j] = -be[jj] * __uint_as_float(yp[jj]);
                    }
                    const uint32_t bo = (c0 + 8 * j8) * 2;
                    *reinterpret_cast<uint4 *>(ar + sw128(n, bo)) =
                        make_uint4(bf2(rs[0], rs[1]), bf2(rs[2], rs[3]), bf2(rs[4], rs[5]), bf2(rs[6], rs[7]));
                    *reinterpret_cast<uint4 *>(ar + sw128(128 + n, bo)) =
                        make_uint4(bf2(rp[0], rp[1]), bf2(rp[2], rp[3]), bf2(rp[4], rp[5]), bf2(rp[6], rp[7]));
                }
            }
            fence_async_shared();
            tc_fence_before();
            mbar_arrive(&bars.rready);
            // (3) D'^T[n][t] = e^{-c_t} (M R)^T[n][t], into the same operand tile
            if (!(ok = wait(&bars.dfull, c & 1))) break;
            tc_fence_after();
            const float cC = v.cC;
#pragma unroll
            for (int c0 = 0; c0 < C; c0 += 32) {
                uint32_t ds[32], dp[32];
                tmem_ld32(tmem + lane_off + kTY + c0, ds);
                tmem_ld32(tmem + lane_off + kTY + 64 + c0, dp);
                float em[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 e4 = reinterpret_cast<const float4 *>(v.ecm + c0)[j4];
                    em[4 * j4] = e4.x, em[4 * j4 + 1] = e4.y, em[4 * j4 + 2] = e4.z, em[4 * j4 + 3] = e4.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float a8[8], b8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int jj = 8 * j8 + j;
                        const float e = em[jj];
                        a8[j] = e * __uint_as_float(ds[jj]);
                        b8[j] = e * __uint_as_float(dp[jj]);
                    }
                    const uint32_t bo = (c0 + 8 * j8) * 2;
                    *reinterpret_cast<uint4 *>(ar + sw128(n, bo)) =
                        make_uint4(bf2(a8[0], a8[1]), bf2(a8[2], a8[3]), bf2(a8[4], a8[5]), bf2(a8[6], a8[7]));
                    *reinterpret_cast<uint4 *>(ar + sw128(128 + n, bo)) =
                        make_uint4(bf2(b8[0], b8[1]), bf2(b8[2], b8[3]), bf2(b8[4], b8[5]), bf2(b8[6], b8[7]));
                }
            }
            fence_async_shared();
            tc_fence_before();
            mbar_arrive(&bars.dready);
            Lam += cC;
            lam_total += cC;
        }
        // outputs: S = exp(Lam) S~ (column n), P (column n), lam
        if (ok && nch > 0) ok = wait(&bars.zfull, (nch - 1) & 1);
        tc_fence_after();
        const int64_t unit = (int64_t)seg.idx * p.seg_stride + h;
        float *So = p.S + unit * D * D + n;
        float *Po = p.P + unit * D * D + n;
        const float sc = expf(Lam);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t z[32];
                tmem_ld32(tmem + lane_off + kTZ + 128 * hf + c0, z);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float val = __uint_as_float(z[j]);
                    if (hf == 0) So[(int64_t)(c0 + j) * D] = val * sc;
                    else Po[(int64_t)(c0 + j) * D] = val;
                }
            }
        if (n == 0) p.lam[unit] = lam_total;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool build_gdn_tc_supported(const BuildParams &p) {
    return p.D == D && p.dtype == HYPIC_BF16 &&
           (p.family == HYPIC_FAM_GDN || p.family == HYPIC_FAM_DELTA);
}

cudaError_t launch_build_gdn_tc(const BuildParams &p, cudaStream_t s) {
    const int64_t N = p.n_tok > 0 ? p.n_tok : 1;
    CUtensorMap tmK, tmV;
    if (!make_tmap_3d(&tmK, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_k, N, (uint64_t)D * 2,
                      (uint64_t)p.H_k * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tmV, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_v, N, (uint64_t)D * 2,
                      (uint64_t)p.H_v * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(build_gdn_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int blocks = p.n_seg * p.H_v;
    if (blocks == 0) return cudaSuccess;
    build_gdn_tc_kernel<<<blocks, kThreads, kSmemBytes, s>>>(p, tmK, tmV);
    return cudaGetLastError();
}

}  // namespace hypic
