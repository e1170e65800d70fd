// build_gdn_prep.cu -- chunk preparation of the DeltaNet / GDN segment build (bf16 k,
// d_k = d_v = 128, chunks of 64 tokens): for every (segment, value head, chunk) the matrix
//     M2 = N Diag(b),   N = (I + Diag(b) L)^-1,   L_ts = k_t . k_s for s < t (0 otherwise),
// rounded to bf16 and written as one 8 KB record (64 rows t' x 64 columns t, row-major) into
// the caller's workspace. The chain kernel (build_gdn_tc.cu) reads the records back.
//
// Why N carries everything the chain needs: with c_t = sum_{s<=t} log a_s inside the chunk,
// the chunked recurrence of "Gated Delta Networks: Improving Mamba2 with Delta Rule"
// (reference 7 of the episode-companion page "Hypic: Position-Independent KV Caching for
// Hybrid-Attention LLM Serving") needs M = (I + A)^-1 with A_ts = b_t (k_t . k_s) e^{c_t - c_s}
// (s < t). A = Diag(b e^c) L Diag(e^-c), so I + A = Diag(e^c) (I + Diag(b) L) Diag(e^-c) and
// M = Diag(e^c) N Diag(e^-c): the inverse itself never sees the gates a_t. The chain applies
// them as diagonal scalings of M2. The product of the chunk's transitions
// prod_t (I - b_t k_t k_t^T) (latest leftmost) equals I - K^T M2 K, the transition part of
// the pair (S(C|0), T_C) that "Cut First-Token Latency by 3.25x: Introducing HYPIC ..."
// (besthub.dev), paragraph "For linear layers", stores for DeltaNet / GDN layers.
//
// Persistent CTAs of 128 threads. A unit of work is R records of one (segment, chunk): with
// an even grouped-query factor R = 2, the two value heads of one key head, which share the k
// tile, the gram and its shared-memory copy, and whose two inverses run side by side;
// otherwise R = 1. Four CTAs per SM (all 512 TMEM columns, about 52 KB of shared memory and at
// most 128 registers each). Units are handed out as tickets: a CTA
// starts with two fixed units and takes each further one from a counter in the workspace
// (zeroed before the launch), so CTAs that run faster take more units and all CTAs finish
// within about one unit of each other. The k tile of the next unit is requested as soon as
// the current gram has read the single k buffer, its gram is issued while the current
// inverses finish (two TMEM buffers), and b is loaded a unit ahead, so loads and grams
// overlap the inversions. A CTA that has drawn its last ticket lets the chain
// kernel launch (programmatic dependent launch); the chain waits for this grid's completion
// before it reads any record.
//   1. TMA the chunk's k (two 128B-swizzled 64-channel halves); b masked past the segment end.
//   2. One thread issues the gram K K^T (M = 64 tcgen05 MMA, fp32 accumulator in TMEM).
//   3. The raw gram G = K K^T in shared memory, 16 x 16 blocks: the blocks left of the
//      diagonal rounded to tf32 once (they are only ever MMA operands), the diagonal blocks
//      exact (forward substitution); the blocks right of the diagonal are not stored.
//      A = Diag(b) L is never formed: b scales rows inside the consumers, and the strictly
//      lower mask is the consumers' index range.
//   4. N by 16 x 16 blocks: the four diagonal blocks by forward substitution (one warp each;
//      lanes 0-15 solve the first record's columns, lanes 16-31 the second's),
//      then the blocks below level by level, N_ab = -N_aa Diag(b_a) sum_{k=b}^{a-1} G_ak N_kb,
//      as 16 x 8 half-blocks spread over the four warps. The 16 x 16 x 16 products run on
//      the warp-level tensor-core MMA (m16n8k8, tf32 inputs, fp32 accumulation): tcgen05's
//      smallest tile (M = 64) would waste most of its work on products this small and each
//      would need a round trip through TMEM. Every MMA operand in shared memory is stored
//      already rounded to tf32, so the fragments are loaded without conversions.
//   5. Columns scaled by b_t, rounded to bf16, stored (16-byte coalesced stores).
// Tokens past the segment end have b = 0, so their rows and columns of M2 are zero.
#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace hypic {
namespace {

using namespace ptx;

constexpr int D = 128;
constexpr int C = kGdnChunk;
constexpr int kThreads = 128;
// Shared-memory layout of G and N: only the ten 16 x 16 blocks on and below the diagonal are
// stored, block (a, b) at word kBlk (a (a + 1) / 2 + b), and element (r, c) of a block at
// 16 r + (c ^ sw(r)). The swizzle makes the warp-level MMA's A fragments (8 rows x 4 columns),
// its B fragments (4 rows x 8 columns), the 16 x 8 result stores and the row-wise accesses
// each touch 32 distinct banks. The 8 words after each block put the blocks of one row in
// different banks (record stage) and start N's second record 16 banks after the first (the two
// records' diagonal solves store side by side). The per-warp 16 x 8 scratch (a B operand) has
// unpadded rows of 8.
constexpr int kBlk = 264;
constexpr int kTri = 10 * kBlk;   // one matrix
constexpr int kLDT = 8;
__device__ __forceinline__ int sw(int r) { return ((r << 2) & 8) | (r & 4); }
__device__ __forceinline__ int blk(int a, int b) { return kBlk * (a * (a + 1) / 2 + b); }
// b of a record: entry e at vbi(e), 16 words of padding after the first 32 entries, so that the
// record stage's loads of b touch distinct banks
constexpr int kVb = 80;
__device__ __forceinline__ int vbi(int e) { return e + ((e >> 5) << 4); }
// R records per iteration: the value heads h, h + 1 that share a key head (R = 2, when the
// grouped-query factor is even) share the k tile, the gram and its shared-memory copy, and
// their two inverses run side by side; R = 1 otherwise.
template <int R>
struct PrepGeo {
    static constexpr uint32_t kOffK = 0;                              // k tile, 16 KB
    static constexpr uint32_t kOffG32 = 16384;                        // the gram K K^T, 10 blocks
    static constexpr uint32_t kOffN32 = kOffG32 + kTri * 4;           // R x N (tf32-rounded), 10 blocks each
    static constexpr uint32_t kOffT = kOffN32 + R * kTri * 4;         // 4 warps x 16 x 8 fp32
    static constexpr uint32_t kSmemBytes = kOffT + 4 * 16 * kLDT * 4 + 1024;
    static constexpr int kCtasPerSm = 4;                              // 4 x 128 TMEM columns
};
constexpr int kCtl = 96;   // warp 3 lane 0 issues loads and grams (warp 3 has the least level work)

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// x rounded to tf32 (round to nearest), kept as a float with the low 13 mantissa bits zero
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(to_tf32(x)); }

// c (16 x 8, m16n8 accumulator layout) += X (16 x 16) * Y[:, yc .. yc + 7] (16 x 8), holding
// tf32-rounded values: X a swizzled block; Y a swizzled block (YS) or the unswizzled 16 x 8
// scratch (row stride kLDT, yc = 0).
template <bool YS>
__device__ __forceinline__ void mma16x8x16(float (&c)[4], const float *X, const float *Y, int yc, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int sx = sw(g);   // rows g and g + 8 share it
    constexpr int ldy = YS ? 16 : kLDT;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const int c0 = (8 * ks + t) ^ sx, c1 = (8 * ks + t + 4) ^ sx;
        const int r0 = 8 * ks + t, r1 = r0 + 4;
        const uint32_t a0 = __float_as_uint(X[g * 16 + c0]);
        const uint32_t a1 = __float_as_uint(X[(g + 8) * 16 + c0]);
        const uint32_t a2 = __float_as_uint(X[g * 16 + c1]);
        const uint32_t a3 = __float_as_uint(X[(g + 8) * 16 + c1]);
        const uint32_t b0 = __float_as_uint(Y[r0 * ldy + ((yc + g) ^ (YS ? sw(r0) : 0))]);
        const uint32_t b1 = __float_as_uint(Y[r1 * ldy + ((yc + g) ^ (YS ? sw(r1) : 0))]);
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Half-block (a, b, hh) of N: columns 16 b + 8 hh .. + 7 of block row a, from the blocks of
// N already computed: T = Diag(b_a) sum_{k=b}^{a-1} G_ak N_kb[:, half], N_ab[:, half] =
// -N_aa T (bv: the chunk's b).
__device__ __forceinline__ void half_block(const float *G32, float *N32, float *Tw, const float *bv, int a,
                                           int b, int hh, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = b; k < a; ++k) mma16x8x16<true>(c, G32 + blk(a, k), N32 + blk(k, b), 8 * hh, lane);
    const float b0 = bv[vbi(16 * a + g)], b1 = bv[vbi(16 * a + g + 8)];
    *reinterpret_cast<float2 *>(Tw + g * kLDT + 2 * t) = make_float2(tf32r(c[0] * b0), tf32r(c[1] * b0));
    *reinterpret_cast<float2 *>(Tw + (g + 8) * kLDT + 2 * t) = make_float2(tf32r(c[2] * b1), tf32r(c[3] * b1));
    __syncwarp();
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16<false>(d, N32 + blk(a, a), Tw, 0, lane);
    float *o = N32 + blk(a, b) + ((8 * hh + 2 * t) ^ sw(g));   // rows g and g + 8 share the swizzle
    *reinterpret_cast<float2 *>(o + g * 16) = make_float2(tf32r(-d[0]), tf32r(-d[1]));
    *reinterpret_cast<float2 *>(o + (g + 8) * 16) = make_float2(tf32r(-d[2]), tf32r(-d[3]));
    __syncwarp();   // Tw is reused by this warp's next half-block
}

// Work units (R records each) are numbered in the order (segment rank, chunk, value heads
// h .. h + R - 1), so the units that share a key head read the same k tile back to back
// (from L2); segment rank r owns numbers [wsb_r / R, (wsb_r + H_v nch_r) / R). A number is
// turned back into its unit by a binary search over the segment table.
struct Walk {
    int r, c, h;   // segment rank, chunk, first value head; r == n_seg: no unit
};

template <int R>
__device__ __forceinline__ Walk decode(const BuildParams &p, int64_t t, int64_t units) {
    Walk w{p.n_seg, 0, 0};
    if (t >= units) return w;
    int lo = 0, hi = p.n_seg - 1;   // the last rank with wsb / R <= t (empty segments come last)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].wsb / R <= t) lo = mid;
        else hi = mid - 1;
    }
    const int local = (int)(t - p.seg[lo].wsb / R), per_chunk = p.H_v / R;
    w.r = lo;
    w.c = local / per_chunk;
    w.h = R * (local - w.c * per_chunk);
    return w;
}

__device__ __forceinline__ int64_t total_records(const BuildParams &p) {
    const SegEntry &l = p.seg[p.n_seg - 1];
    return (int64_t)l.wsb + (int64_t)p.H_v * ((l.len + C - 1) / C);
}

template <int R>
__global__ void __launch_bounds__(kThreads, PrepGeo<R>::kCtasPerSm)
build_gdn_prep_kernel(const __grid_constant__ BuildParams p, const __grid_constant__ CUtensorMap tmK) {
    using G = PrepGeo<R>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t kfull, gfull[2];
    __shared__ uint32_t tslot;
    __shared__ int s_ok;
    __shared__ Walk s_n2[2];   // the unit after `nxt`, drawn by thread kCtl (two slots)
    __shared__ __align__(16) float vb[2][R][kVb];   // the records' b at vbi(token)

    const int64_t total = total_records(p), units = total / R;
    unsigned *tickets = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(p.workspace) + total * kGdnRecordBytes);
    auto nch_of = [&](int r) { return (p.seg[r].len + C - 1) / C; };
    Walk cur = decode<R>(p, blockIdx.x, units);
    if (cur.r >= p.n_seg) return;   // uniform: the whole CTA leaves before any set-up
    const int q = threadIdx.x, warp = q >> 5, lane = q & 31;
    float *G32 = reinterpret_cast<float *>(smem + G::kOffG32);
    float *N32 = reinterpret_cast<float *>(smem + G::kOffN32);   // record rr at N32 + rr * kTri
    float *Tw = reinterpret_cast<float *>(smem + G::kOffT) + warp * 16 * kLDT;

    if (q == 0) {
        mbar_init(&kfull, 1);
        mbar_init(&gfull[0], 1);
        mbar_init(&gfull[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tslot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    constexpr uint32_t idG = idesc(kFmtBF16, kFmtBF16, false, false, 64, 64);
    int kiss = 0, kwait = 0, giss[2] = {0, 0}, gwait[2] = {0, 0};   // thread kCtl
    auto load_k = [&](const Walk &w) {   // thread kCtl
        ++kiss;
        const int32_t t0 = p.seg[w.r].start + w.c * C;
        mbar_arrive_expect_tx(&kfull, 16384);
        tma_load_3d(smem + G::kOffK, &tmK, &kfull, 0, w.h / p.gqa, t0);
        tma_load_3d(smem + G::kOffK + 8192, &tmK, &kfull, 64, w.h / p.gqa, t0);
    };
    auto gram = [&](int b) -> bool {   // thread kCtl: the k tile -> TMEM buffer b
        if (!mbar_wait(&kfull, kwait & 1, p.err, kErrTimeout)) return false;
        ++kwait;
        ++giss[b];
        tc_fence_after();
        const uint32_t k = smem_u32(smem + G::kOffK);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint32_t a = k + (s >> 2) * 8192 + (s & 3) * 32;
            mma_bf16(tmem + 64 * b, sdesc(a, 16, 1024, kSwizzle128B), sdesc(a, 16, 1024, kSwizzle128B), idG,
                     s > 0);
        }
        mma_commit(&gfull[b]);
        return true;
    };
    // b of a unit's records (thread q < 64 R: token q % 64 of record q / 64), a unit ahead
    auto load_beta = [&](const Walk &w) -> float {
        const int tq = q & (C - 1), rr = q / C;
        if (rr >= R || w.r >= p.n_seg) return 0.f;
        const SegEntry sg = p.seg[w.r];
        return tq < min(C, sg.len - w.c * C) ? p.beta[((int64_t)sg.start + w.c * C + tq) * p.H_v + w.h + rr] : 0.f;
    };
    bool ok = true;
    int64_t ticket = 0;   // thread kCtl
    Walk nxt = decode<R>(p, (int64_t)gridDim.x + blockIdx.x, units);
    float beta_cur = load_beta(cur);
    if (q == kCtl) {
        prefetch_tmap(&tmK);
        load_k(cur);
        ok = gram(0);
    }
    for (int i = 0; cur.r < p.n_seg; ++i) {
        const int b = i & 1;
        const SegEntry seg = p.seg[cur.r];
        const int nch = nch_of(cur.r);
        // every thread decodes the same unit: a failing check leaves the loop uniformly
        if (!in_bounds(cur.c < nch && cur.h + R <= p.H_v &&
                           (int64_t)seg.wsb + (int64_t)(cur.h + R - 1) * nch + cur.c < total, p.err))
            break;
        if (q < R * C) vb[b][q / C][vbi(q & (C - 1))] = beta_cur;
        const float beta_next = load_beta(nxt);
        // gram(i) done: the k tile is free for the next record
        if (q == kCtl) {
            ok = ok && mbar_wait(&gfull[b], gwait[b] & 1, p.err, kErrTimeout);
            if (ok) {
                ++gwait[b];
                if (nxt.r < p.n_seg) load_k(nxt);
            }
            s_ok = ok ? 1 : 0;
            // the ticket of the record after `nxt` (the counter's answer is used only at
            // level 3 below, so its latency overlaps this record's inverse)
            if (nxt.r < p.n_seg) ticket = 2 * (int64_t)gridDim.x + atomicAdd(tickets, 1u);
        }
        __syncthreads();
        if (!s_ok) break;   // uniform
        tc_fence_after();
        {   // gram rows 16 warp + lane (lanes < 16, M = 64 accumulator layout): row `lane` of
            // block row `warp`; its blocks left of the diagonal are stored tf32-rounded, its
            // diagonal block exact, the blocks right of it not at all. Columns in two halves of
            // 32 (warps 0-1 need only the first).
            const uint32_t taddr = tmem + 64 * b + ((uint32_t)(32 * warp) << 16);
            const int r = lane & 15;
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                if (hc == 1 && warp < 2) break;   // uniform
                uint32_t gr[32];
                tmem_ld32(taddr + 32 * hc, gr);
                tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int s4 = 0; s4 < 8; ++s4) {
                        const int k = 2 * hc + (s4 >> 2), cb = 4 * (s4 & 3);
                        if (k > warp) break;   // uniform
                        float4 g4 = make_float4(__uint_as_float(gr[4 * s4]), __uint_as_float(gr[4 * s4 + 1]),
                                                __uint_as_float(gr[4 * s4 + 2]), __uint_as_float(gr[4 * s4 + 3]));
                        if (k < warp) g4 = make_float4(tf32r(g4.x), tf32r(g4.y), tf32r(g4.z), tf32r(g4.w));
                        *reinterpret_cast<float4 *>(G32 + blk(warp, k) + 16 * r + (cb ^ sw(r))) = g4;
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        // diagonal block `warp`: lane j < 16 solves column j of record 0 (lanes 16-31 that of
        // record 1 when R = 2) by forward substitution,
        // x_r = [r == j] - b_r sum_{s<r} G_rs x_s (A = Diag(b) L restricted to the block)
        if (R == 2 || lane < 16) {
            const int a = warp, j = lane & 15, rr_ = lane >> 4;
            const float *bv = vb[b][rr_];
            const float *Gd = G32 + blk(a, a);
            float *Nd = N32 + rr_ * kTri + blk(a, a);
            float x[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                float gr[16];
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(Gd + 16 * rr + ((4 * s4) ^ sw(rr)));
                    gr[4 * s4] = t4.x, gr[4 * s4 + 1] = t4.y, gr[4 * s4 + 2] = t4.z, gr[4 * s4 + 3] = t4.w;
                }
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < rr; ++s) acc[s & 3] = fmaf(gr[s], x[s], acc[s & 3]);
                x[rr] = fmaf(-bv[vbi(16 * a + rr)], (acc[0] + acc[1]) + (acc[2] + acc[3]), (rr == j) ? 1.f : 0.f);
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) Nd[16 * rr + (j ^ sw(rr))] = tf32r(x[rr]);
        }
        __syncthreads();
        // level 1: (1,0), (2,1), (3,2) as six half-blocks; level 2: (2,0), (3,1); level 3: (3,0).
        // Warps 0-1 take one half-block per level, warps 2-3 two in level 1 and none in level 3.
        // Each half-block is done for every record of the unit.
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            half_block(G32, N32 + rr * kTri, Tw, vb[b][rr], 1 + (warp >> 1), warp >> 1, warp & 1, lane);
            if (warp >= 2) half_block(G32, N32 + rr * kTri, Tw, vb[b][rr], 3, 2, warp & 1, lane);
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
            half_block(G32, N32 + rr * kTri, Tw, vb[b][rr], 2 + (warp >> 1), warp >> 1, warp & 1, lane);
        __syncthreads();
        if (warp < 2) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) half_block(G32, N32 + rr * kTri, Tw, vb[b][rr], 3, 0, warp, lane);
        }
        // warps 2-3 have no level-3 work: the next record's gram (its k tile was requested at
        // the top of this iteration) into the other TMEM buffer, last read a record ago
        // and the ticket of the record after it
        if (q == kCtl) {
            if (ok && nxt.r < p.n_seg) ok = gram(b ^ 1);
            s_n2[b] = nxt.r < p.n_seg ? decode<R>(p, ticket, units) : nxt;
        }
        __syncthreads();
        const Walk n2 = s_n2[b];   // slot b is written again two records later
        if (n2.r >= p.n_seg) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // records: N Diag(b) as bf16 rows t' (blocks above the diagonal are zero)
#pragma unroll
        for (int m = 0; m < 4 * R; ++m) {
            const int rr = m / 4;
            uint8_t *dst = static_cast<uint8_t *>(p.workspace) +
                           ((int64_t)seg.wsb + (int64_t)(cur.h + rr) * nch + cur.c) * (int64_t)kGdnRecordBytes;
            const float *Nr = N32 + rr * kTri;
            const int e8 = q + 128 * (m & 3);   // 8 consecutive entries of row t'
            const int tp = e8 >> 3, s8 = (e8 & 7) * 8;
            const int ba = tp >> 4, bb = s8 >> 4, r = tp & 15;   // block (ba, bb), row r in it
            uint4 pk = make_uint4(0u, 0u, 0u, 0u);
            if (bb <= ba) {
                // the eight lanes of a row read the two halves of their 8 entries in an order
                // chosen per lane, so that each load of N and of b touches distinct banks
                const int h0 = 4 * ((bb & 1) ^ ((sw(r) >> 2) & 1)), h1 = h0 ^ 4;
                const float *src = Nr + blk(ba, bb) + 16 * r;
                const float4 x0 = *reinterpret_cast<const float4 *>(src + (((s8 & 15) + h0) ^ sw(r)));
                const float4 x1 = *reinterpret_cast<const float4 *>(src + (((s8 & 15) + h1) ^ sw(r)));
                const float4 b0 = *reinterpret_cast<const float4 *>(vb[b][rr] + vbi(s8 + h0));
                const float4 b1 = *reinterpret_cast<const float4 *>(vb[b][rr] + vbi(s8 + h1));
                const uint32_t p0 = pack_bf16x2(x0.x * b0.x, x0.y * b0.y), p1 = pack_bf16x2(x0.z * b0.z, x0.w * b0.w);
                const uint32_t p2 = pack_bf16x2(x1.x * b1.x, x1.y * b1.y), p3 = pack_bf16x2(x1.z * b1.z, x1.w * b1.w);
                pk = h0 == 0 ? make_uint4(p0, p1, p2, p3) : make_uint4(p2, p3, p0, p1);
            }
            *reinterpret_cast<uint4 *>(dst + tp * 128 + s8 * 2) = pk;
        }
        cur = nxt;
        nxt = n2;
        beta_cur = beta_next;
    }
    if (q == kCtl) {   // after a wait gave up: let every copy and MMA in flight land first
        for (; kwait < kiss; ++kwait) mbar_wait(&kfull, kwait & 1, nullptr, 0);
        for (int b = 0; b < 2; ++b)
            for (; gwait[b] < giss[b]; ++gwait[b]) mbar_wait(&gfull[b], gwait[b] & 1, nullptr, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

template <int R>
cudaError_t launch_prep(const BuildParams &p, int64_t total, const CUtensorMap &tmK, int sms, cudaStream_t s) {
    using G = PrepGeo<R>;
    cudaError_t e = cudaFuncSetAttribute(build_gdn_prep_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         G::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(total / R, (int64_t)sms * G::kCtasPerSm);
    build_gdn_prep_kernel<R><<<grid, kThreads, G::kSmemBytes, s>>>(p, tmK);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------ KDA
// The channel-gated delta rule: S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T with
// one decay per key channel, a_t in (0, 1]^{d_k} (KDA is among the linear layers "Cut First-Token
// Latency by 3.25x ..." (besthub.dev), paragraph "For linear layers", names). Inside a chunk let
// c_t = sum_{s<=t} log a_s per channel (valid tokens only) and, elementwise,
//     kt_t = e^{c_t} k_t,   kh_s = e^{-c_s} k_s.
// The chunk's delta values Delta (S_t = Diag(e^{c_t})(S0 + sum_{s<=t} kh_s Delta_s^T)) solve
// (I + A) Delta = Diag(b)(V - Kt S0) with A_ts = b_t (kt_t . kh_s) for s < t, and the state after
// the chunk is Diag(e^{c_C}) (S0 + Kh^T Delta). The gates do not factor out of A here (they
// differ per channel), so the inverse is taken of the gated gram: M2 = (I + Diag(b) L)^-1 Diag(b)
// with L the strictly lower part of Kt Kh^T, by the same blocked algorithm as above. One record
// per (segment, value head, chunk): M2 (bf16 8 KB), Kt and Kh (bf16 64 x 128, written by bulk
// tensor stores from the gram's operand tiles), c_C (128 fp32) and m = max_i c_C[i].
// c_C <= c_t <= 0 and c_C >= -60 keep e^{-c_t} within the range of bf16; a chunk below that
// sets the range status.
constexpr float kKdaMinChunkLogDecay = -60.f;

// 2^x by the hardware's approximate base-2 exponential (relative error about 2^-22 on the
// arguments used here, |x| <= 87: far below the bf16 rounding of every value it scales)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Four CTAs per SM: the two operand tiles, G and N (the level products' 16 x 8 scratch sits in
// the Kh tile once its store has read it; the token halves' gate sums at the start of G).
struct KdaGeo {
    static constexpr uint32_t kOffK = 0;                  // k tile, then Kt in place, 16 KB
    static constexpr uint32_t kOffH = 16384;              // Kh, then the scratch
    static constexpr uint32_t kOffG32 = 32768;            // the gram, 10 blocks
    static constexpr uint32_t kOffN32 = kOffG32 + kTri * 4;
    static constexpr uint32_t kSmemBytes = kOffN32 + kTri * 4 + 1024;
    static constexpr int kCtasPerSm = 4;
};

__global__ void __launch_bounds__(kThreads, KdaGeo::kCtasPerSm)
build_kda_prep_kernel(const __grid_constant__ BuildParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmKh) {
    using G = KdaGeo;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t kfull, gfull;
    __shared__ uint32_t tslot;
    __shared__ Walk s_n2[2];
    __shared__ float s_max[4];
    __shared__ __align__(16) float vb[kVb];

    const int64_t total = total_records(p);
    unsigned *tickets = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(p.workspace) + total * kGdnRecordBytes);
    Walk cur = decode<1>(p, blockIdx.x, total);
    if (cur.r >= p.n_seg) return;   // uniform: the whole CTA leaves before any set-up
    const int q = threadIdx.x, warp = q >> 5, lane = q & 31;
    uint8_t *tK = smem + G::kOffK, *tH = smem + G::kOffH;
    float *G32 = reinterpret_cast<float *>(smem + G::kOffG32);
    float *N32 = reinterpret_cast<float *>(smem + G::kOffN32);
    float *Tw = reinterpret_cast<float *>(tH) + warp * 16 * kLDT;
    float2 (*s_part)[64] = reinterpret_cast<float2 (*)[64]>(G32);   // [token half][channel pair]

    if (q == 0) {
        mbar_init(&kfull, 1);
        mbar_init(&gfull, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tslot, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    constexpr uint32_t idG = idesc(kFmtBF16, kFmtBF16, false, false, 64, 64);
    int kiss = 0, giss = 0, kwait = 0, gwait = 0;   // issued by thread kCtl; waited by every thread
    bool stored = false;                             // thread kCtl: a group of record stores issued
    auto load_k = [&](const Walk &w) {   // thread kCtl
        ++kiss;
        const int32_t t0 = p.seg[w.r].start + w.c * C;
        mbar_arrive_expect_tx(&kfull, 16384);
        tma_load_3d(tK, &tmK, &kfull, 0, w.h / p.gqa, t0);
        tma_load_3d(tK + 8192, &tmK, &kfull, 64, w.h / p.gqa, t0);
    };
    bool ok = true;
    int64_t ticket = 0;   // thread kCtl
    Walk nxt = decode<1>(p, (int64_t)gridDim.x + blockIdx.x, total);
    if (q == kCtl) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmKt);
        prefetch_tmap(&tmKh);
        load_k(cur);
    }
    // Thread q takes the key channels 2 pc, 2 pc + 1 (pc = q % 64) over the tokens of one half
    // of the chunk, th = q / 64: the pair's bf16 elements of a token are one word of a 64 x 128
    // bf16 tile held as two 128B-swizzled 64-channel halves.
    const int pc = q & 63, th = q >> 6;
    const uint32_t hoff = (uint32_t)(pc >> 5) * 8192u, qb = 4u * (uint32_t)(pc & 31);
    // the pair's log-gates over the half's valid tokens (0 past the segment end) and b of token
    // q < 64, loaded a unit ahead so that their latency overlaps the previous inverse
    constexpr int CH = C / 2;
    float2 g[CH];
    float beta_cur = 0.f;
    auto load_gates = [&](const Walk &w) {
        const SegEntry sg = p.seg[w.r];
        const int nvw = min(C, sg.len - w.c * C);
        const int64_t t0 = (int64_t)sg.start + (int64_t)w.c * C;
        const float2 *gp = reinterpret_cast<const float2 *>(p.log_gate + ((t0 + CH * th) * p.H_v + w.h) * D) + pc;
        const int64_t gs = (int64_t)p.H_v * (D / 2);
#pragma unroll
        for (int t = 0; t < CH; ++t) g[t] = CH * th + t < nvw ? __ldg(gp + t * gs) : make_float2(0.f, 0.f);
        beta_cur = q < nvw ? p.beta[(t0 + q) * p.H_v + w.h] : 0.f;
    };
    load_gates(cur);
    for (int i = 0; cur.r < p.n_seg; ++i) {
        const SegEntry seg = p.seg[cur.r];
        const int nch = (seg.len + C - 1) / C;
        const int64_t rec = (int64_t)seg.wsb + (int64_t)cur.h * nch + cur.c;
        if (!in_bounds(cur.c < nch && cur.h < p.H_v && rec < total, p.err)) break;   // uniform
        // (1) b of the unit; the pair's log-decay over this token half
        if (q < C) vb[vbi(q)] = beta_cur;
        {
            float2 sh = make_float2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < CH; ++t) sh.x += g[t].x, sh.y += g[t].y;
            s_part[th][pc] = sh;
        }
        if (q == kCtl && nxt.r < p.n_seg) ticket = 2 * (int64_t)gridDim.x + atomicAdd(tickets, 1u);
        ok = ok && mbar_wait(&kfull, kwait & 1, p.err, kErrTimeout);
        ++kwait;
        if (!__syncthreads_and(ok)) break;   // uniform
        // (2) the pair's elements of Kt (over k) and Kh, token by token
        const float2 p0 = s_part[0][pc], p1 = s_part[1][pc];
        const float2 cC = make_float2(p0.x + p1.x, p0.y + p1.y);
        {
            constexpr float kLog2e = 1.4426950408889634f;
            float cx = th ? p0.x : 0.f, cy = th ? p0.y : 0.f;
#pragma unroll
            for (int t = 0; t < CH; ++t) {
                cx += g[t].x;
                cy += g[t].y;
                const uint32_t off = hoff + sw128((uint32_t)(CH * th + t), qb);
                const uint32_t kw = *reinterpret_cast<const uint32_t *>(tK + off);
                const float kx = __uint_as_float(kw << 16), ky = __uint_as_float(kw & 0xffff0000u);
                *reinterpret_cast<uint32_t *>(tK + off) =
                    pack_bf16x2(kx * ex2_approx(cx * kLog2e), ky * ex2_approx(cy * kLog2e));
                *reinterpret_cast<uint32_t *>(tH + off) =
                    pack_bf16x2(kx * ex2_approx(-cx * kLog2e), ky * ex2_approx(-cy * kLog2e));
            }
        }
        if (fminf(cC.x, cC.y) < kKdaMinChunkLogDecay) atomicOr(p.err, kErrRange);
        float mx = fmaxf(cC.x, cC.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_max[warp] = mx;
        fence_async_shared();   // Kt and Kh are read by the tensor core and the bulk stores
        __syncthreads();
        if (q == kCtl) {
            tc_fence_after();
            // the gram Kt Kh^T (M = 64) into TMEM; the read-out below waits for it
            const uint32_t a0 = smem_u32(tK), b0 = smem_u32(tH);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t o = (s >> 2) * 8192 + (s & 3) * 32;
                mma_bf16(tmem, sdesc(a0 + o, 16, 1024, kSwizzle128B), sdesc(b0 + o, 16, 1024, kSwizzle128B), idG,
                         s > 0);
            }
            mma_commit(&gfull);
            ++giss;
            // Kt and Kh to their records (64 rows each, two 64-channel boxes)
            const int32_t row = (int32_t)(rec * C);
            tma_store_2d(&tmKt, tK, 0, row);
            tma_store_2d(&tmKt, tK + 8192, 64, row);
            tma_store_2d(&tmKh, tH, 0, row);
            tma_store_2d(&tmKh, tH + 8192, 64, row);
            bulk_commit();
            stored = true;
        }
        {
            const float m = fmaxf(fmaxf(s_max[0], s_max[1]), fmaxf(s_max[2], s_max[3]));
            float *side = p.kda_side + rec * kKdaSide;
            if (th == 0) reinterpret_cast<float2 *>(side)[pc] = cC;
            if (q == 0) side[128] = m;
        }
        ok = ok && mbar_wait(&gfull, gwait & 1, p.err, kErrTimeout);
        ++gwait;
        if (!__syncthreads_and(ok)) break;   // uniform
        tc_fence_after();
        {   // gram rows into G32 (as in the GDN preparation, one TMEM buffer)
            const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
            const int r = lane & 15;
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                if (hc == 1 && warp < 2) break;   // uniform
                uint32_t gr[32];
                tmem_ld32(taddr + 32 * hc, gr);
                tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int s4 = 0; s4 < 8; ++s4) {
                        const int k = 2 * hc + (s4 >> 2), cb = 4 * (s4 & 3);
                        if (k > warp) break;   // uniform
                        float4 g4 = make_float4(__uint_as_float(gr[4 * s4]), __uint_as_float(gr[4 * s4 + 1]),
                                                __uint_as_float(gr[4 * s4 + 2]), __uint_as_float(gr[4 * s4 + 3]));
                        if (k < warp) g4 = make_float4(tf32r(g4.x), tf32r(g4.y), tf32r(g4.z), tf32r(g4.w));
                        *reinterpret_cast<float4 *>(G32 + blk(warp, k) + 16 * r + (cb ^ sw(r))) = g4;
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        // the stores must have read Kt and Kh before the next k tile lands over Kt and the
        // level products' scratch is written over Kh (after the barrier below); the next unit's
        // gates
        if (q == kCtl) {
            bulk_wait_read<0>();
            if (nxt.r < p.n_seg) load_k(nxt);
        }
        if (nxt.r < p.n_seg) load_gates(nxt);
        // diagonal blocks by forward substitution, lane j < 16 of warp a: column j of block a
        if (lane < 16) {
            const int a = warp, j = lane;
            const float *Gd = G32 + blk(a, a);
            float *Nd = N32 + blk(a, a);
            float x[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                float gr[16];
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(Gd + 16 * rr + ((4 * s4) ^ sw(rr)));
                    gr[4 * s4] = t4.x, gr[4 * s4 + 1] = t4.y, gr[4 * s4 + 2] = t4.z, gr[4 * s4 + 3] = t4.w;
                }
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < rr; ++s) acc[s & 3] = fmaf(gr[s], x[s], acc[s & 3]);
                x[rr] = fmaf(-vb[vbi(16 * a + rr)], (acc[0] + acc[1]) + (acc[2] + acc[3]), (rr == j) ? 1.f : 0.f);
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) Nd[16 * rr + (j ^ sw(rr))] = tf32r(x[rr]);
        }
        __syncthreads();
        half_block(G32, N32, Tw, vb, 1 + (warp >> 1), warp >> 1, warp & 1, lane);
        if (warp >= 2) half_block(G32, N32, Tw, vb, 3, 2, warp & 1, lane);
        __syncthreads();
        half_block(G32, N32, Tw, vb, 2 + (warp >> 1), warp >> 1, warp & 1, lane);
        __syncthreads();
        if (warp < 2) half_block(G32, N32, Tw, vb, 3, 0, warp, lane);
        if (q == kCtl) s_n2[i & 1] = nxt.r < p.n_seg ? decode<1>(p, ticket, total) : nxt;
        __syncthreads();
        const Walk n2 = s_n2[i & 1];
        if (n2.r >= p.n_seg) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // the record: N Diag(b) as bf16 rows t' (blocks above the diagonal are zero)
        uint8_t *dst = static_cast<uint8_t *>(p.workspace) + rec * kGdnRecordBytes;
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const int e8 = q + 128 * mm;
            const int tp = e8 >> 3, s8 = (e8 & 7) * 8;
            const int ba = tp >> 4, bb = s8 >> 4, r = tp & 15;
            uint4 pk = make_uint4(0u, 0u, 0u, 0u);
            if (bb <= ba) {
                const int h0 = 4 * ((bb & 1) ^ ((sw(r) >> 2) & 1)), h1 = h0 ^ 4;
                const float *src = N32 + blk(ba, bb) + 16 * r;
                const float4 x0 = *reinterpret_cast<const float4 *>(src + (((s8 & 15) + h0) ^ sw(r)));
                const float4 x1 = *reinterpret_cast<const float4 *>(src + (((s8 & 15) + h1) ^ sw(r)));
                const float4 b0 = *reinterpret_cast<const float4 *>(vb + vbi(s8 + h0));
                const float4 b1 = *reinterpret_cast<const float4 *>(vb + vbi(s8 + h1));
                const uint32_t p0 = pack_bf16x2(x0.x * b0.x, x0.y * b0.y), p1 = pack_bf16x2(x0.z * b0.z, x0.w * b0.w);
                const uint32_t p2 = pack_bf16x2(x1.x * b1.x, x1.y * b1.y), p3 = pack_bf16x2(x1.z * b1.z, x1.w * b1.w);
                pk = h0 == 0 ? make_uint4(p0, p1, p2, p3) : make_uint4(p2, p3, p0, p1);
            }
            *reinterpret_cast<uint4 *>(dst + tp * 128 + s8 * 2) = pk;
        }
        __syncthreads();   // every read of vb, G32, N32 and the scratch done before the next unit
        cur = nxt;
        nxt = n2;
    }
    if (q == kCtl) {   // the record stores complete; after a wait gave up, every copy and MMA lands
        if (stored) bulk_wait<0>();
        for (; kwait < kiss; ++kwait) mbar_wait(&kfull, kwait & 1, nullptr, 0);
        for (; gwait < giss; ++gwait) mbar_wait(&gfull, gwait & 1, nullptr, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

}  // namespace

cudaError_t launch_build_gdn_prep(const BuildParams &p, cudaStream_t s) {
    if (p.n_seg == 0) return cudaSuccess;
    const SegEntry &l = p.seg[p.n_seg - 1];
    const int64_t total = (int64_t)l.wsb + (int64_t)p.H_v * ((l.len + C - 1) / C);
    if (total == 0) return cudaSuccess;
    if (total > INT32_MAX / 2) return cudaErrorInvalidValue;
    const int64_t N = p.n_tok > 0 ? p.n_tok : 1;
    CUtensorMap tmK;
    if (!make_tmap_3d(&tmK, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_k, N, (uint64_t)D * 2,
                      (uint64_t)p.H_k * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // the ticket counter after the records (the workspace tail), zeroed for this launch
    e = cudaMemsetAsync(static_cast<uint8_t *>(p.workspace) + total * kGdnRecordBytes, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    // pairs of value heads share a key head when the grouped-query factor is even
    return p.gqa % 2 == 0 ? launch_prep<2>(p, total, tmK, sms, s) : launch_prep<1>(p, total, tmK, sms, s);
}

cudaError_t launch_build_kda_prep(const BuildParams &p, cudaStream_t s) {
    if (p.n_seg == 0) return cudaSuccess;
    const SegEntry &l = p.seg[p.n_seg - 1];
    const int64_t total = (int64_t)l.wsb + (int64_t)p.H_v * ((l.len + C - 1) / C);
    if (total == 0) return cudaSuccess;
    if (total > INT32_MAX / C) return cudaErrorInvalidValue;
    const int64_t N = p.n_tok > 0 ? p.n_tok : 1;
    CUtensorMap tmK, tmKt, tmKh;
    if (!make_tmap_3d(&tmK, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H_k, N, (uint64_t)D * 2,
                      (uint64_t)p.H_k * D * 2, 64, 1, C, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tmKt, p.kda_kt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)total * C, D * 2, 64, C,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tmKh, p.kda_kh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)total * C, D * 2, 64, C,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = cudaMemsetAsync(static_cast<uint8_t *>(p.workspace) + total * kGdnRecordBytes, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(build_kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KdaGeo::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(total, (int64_t)sms * KdaGeo::kCtasPerSm);
    build_kda_prep_kernel<<<grid, kThreads, KdaGeo::kSmemBytes, s>>>(p, tmK, tmKt, tmKh);
    return cudaGetLastError();
}

}  // namespace hypic
