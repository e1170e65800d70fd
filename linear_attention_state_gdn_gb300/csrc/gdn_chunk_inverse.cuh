// gdn_chunk_inverse.cuh -- the per-chunk matrix of the DeltaNet / GDN segment build
//     M2 = N Diag(b),   N = (I + Diag(b) L)^-1,   L_ts = k_t . k_s for s < t (0 otherwise),
// for one 64-token chunk, computed by four warps of the chain kernel (build_gdn_tc.cu) from the
// chunk's k tile in shared memory, a chunk or two ahead of the chain that consumes it.
//
// Why N carries everything the chain needs: with c_t = sum_{s<=t} log a_s inside the chunk,
// the chunked recurrence of "Gated Delta Networks: Improving Mamba2 with Delta Rule"
// (reference 7 of the episode-companion page "Hypic: Position-Independent KV Caching for
// Hybrid-Attention LLM Serving") needs M = (I + A)^-1 with A_ts = b_t (k_t . k_s) e^{c_t - c_s}
// (s < t). A = Diag(b e^c) L Diag(e^-c), so I + A = Diag(e^c) (I + Diag(b) L) Diag(e^-c) and
// M = Diag(e^c) N Diag(e^-c): the inverse itself never sees the gates a_t. The chain applies
// them as diagonal scalings of M2.
//
// Steps (the four warps 0-3 here are the kernel's four chunk-inverse warps):
//   1. The gram G = K K^T, only its ten 16 x 16 blocks on and below the diagonal, on the
//      warp-level tensor-core MMA (m16n8k16, bf16 inputs from the swizzled k tile, fp32
//      accumulation), three or two blocks per warp. Blocks left of the diagonal are rounded
//      to tf32 once (they are only ever MMA operands); the diagonal blocks stay exact.
//      A = Diag(b) L is never formed: b scales rows inside the consumers, and the strictly
//      lower mask is the consumers' index range.
//   2. N by 16 x 16 blocks: the four diagonal blocks by forward substitution (one warp each,
//      lane j < 16 solves column j), then the blocks below level by level,
//      N_ab = -N_aa Diag(b_a) sum_{k=b}^{a-1} G_ak N_kb, as 16 x 8 half-blocks spread over
//      the four warps, on the warp-level MMA (m16n8k8, tf32 inputs, fp32 accumulation).
//   3. Columns scaled by b_t, rounded to bf16, stored as the chain's 128B-swizzled K-major
//      operand (64 rows t' of 128 bytes).
// Tokens past the segment end have b = 0, so their rows and columns of M2 are zero.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace hypic {
namespace gdninv {

// Shared-memory layout of G and N: only the ten 16 x 16 blocks on and below the diagonal are
// stored, block (a, b) at word kBlk (a (a + 1) / 2 + b), and element (r, c) of a block at
// 16 r + (c ^ sw(r)). The swizzle makes the warp-level MMA's A fragments (8 rows x 4 columns),
// its B fragments (4 rows x 8 columns), the 16 x 8 result stores and the row-wise accesses
// each touch 32 distinct banks. The 8 words after each block put the blocks of one row in
// different banks (record stage). The per-warp 16 x 8 scratch (a B operand) has unpadded
// rows of 8.
constexpr int kBlk = 264;
constexpr int kTri = 10 * kBlk;   // one matrix, in words
constexpr int kLDT = 8;
__device__ __forceinline__ int sw(int r) { return ((r << 2) & 8) | (r & 4); }
__device__ __forceinline__ int blk(int a, int b) { return kBlk * (a * (a + 1) / 2 + b); }
// b of a chunk: entry e at vbi(e), 16 words of padding after the first 32 entries, so that
// the record stage's loads of b touch distinct banks
constexpr int kVb = 80;
__device__ __forceinline__ int vbi(int e) { return e + ((e >> 5) << 4); }

// shared-memory bytes of the four warps' working set: G, N and four 16 x 8 scratch tiles
constexpr uint32_t kSmemBytes = 2 * kTri * 4 + 4 * 16 * kLDT * 4;

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

// Shared-memory byte offset of the 16 bytes holding channels i .. i + 7 (i a multiple of 8) of
// token row t in a k tile stored as two 64-channel halves of 64 rows x 128 bytes with the
// 128-byte swizzle (the TMA box layout the chain loads).
__device__ __forceinline__ uint32_t ktile_off(int t, int i) {
    return (uint32_t)(i >> 6) * 8192u + ptx::sw128((uint32_t)t, (uint32_t)(i & 63) * 2u);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Step 1 for warp w (0-3): the gram blocks (a, b), b <= a, of this warp, from the k tile at
// shared address ktile, into G32. Warp 0: (0,0), (1,0), (1,1); warp 1: (2,0), (2,1), (2,2);
// warp 2: (3,0), (3,1); warp 3: (3,2), (3,3).
__device__ __forceinline__ void gram_blocks(uint32_t ktile, float *G32, int w, int lane) {
    const int nb = w < 2 ? 3 : 2;
    int ba[3], bb[3];
    if (w == 0) { ba[0] = 0; bb[0] = 0; ba[1] = 1; bb[1] = 0; ba[2] = 1; bb[2] = 1; }
    else if (w == 1) { ba[0] = 2; bb[0] = 0; ba[1] = 2; bb[1] = 1; ba[2] = 2; bb[2] = 2; }
    else if (w == 2) { ba[0] = 3; bb[0] = 0; ba[1] = 3; bb[1] = 1; ba[2] = 3; bb[2] = 1; }
    else { ba[0] = 3; bb[0] = 2; ba[1] = 3; bb[1] = 3; ba[2] = 3; bb[2] = 3; }
    float acc[3][2][4];
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][n][j] = 0.f;
    // ldmatrix row addresses: A (16 tokens x 16 channels) row (l & 7) + 8 ((l >> 3) & 1),
    // channel half (l >> 4); B (two 8-token column tiles x 16 channels) row (l & 7) + 8 (l >> 4),
    // channel half ((l >> 3) & 1)
    const int ar = (lane & 7) + 8 * ((lane >> 3) & 1), ac = 8 * (lane >> 4);
    const int br = (lane & 7) + 8 * (lane >> 4), bc = 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            if (i < nb) {   // uniform
                uint32_t af[4], bf[4];
                ldsm_x4(ktile + ktile_off(16 * ba[i] + ar, 16 * ks + ac), af);
                ldsm_x4(ktile + ktile_off(16 * bb[i] + br, 16 * ks + bc), bf);
                mma_bf16_16816(acc[i][0], af, bf[0], bf[1]);
                mma_bf16_16816(acc[i][1], af, bf[2], bf[3]);
            }
        }
    }
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        if (i < nb) {
            const bool diag = ba[i] == bb[i];
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                float *o = G32 + blk(ba[i], bb[i]) + ((8 * n + 2 * t) ^ sw(g));   // rows g, g + 8 share it
                float2 lo = make_float2(acc[i][n][0], acc[i][n][1]), hi = make_float2(acc[i][n][2], acc[i][n][3]);
                if (!diag) {
                    lo = make_float2(tf32r(lo.x), tf32r(lo.y));
                    hi = make_float2(tf32r(hi.x), tf32r(hi.y));
                }
                *reinterpret_cast<float2 *>(o + g * 16) = lo;
                *reinterpret_cast<float2 *>(o + (g + 8) * 16) = hi;
            }
        }
    }
}

// Step 2, diagonal block w: lane j < 16 solves column j by forward substitution,
// x_r = [r == j] - b_r sum_{s<r} G_rs x_s (A = Diag(b) L restricted to the block).
__device__ __forceinline__ void diag_solve(const float *G32, float *N32, const float *bv, int w, int lane) {
    if (lane >= 16) return;
    const int a = w, j = lane;
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
        x[rr] = fmaf(-bv[vbi(16 * a + rr)], (acc[0] + acc[1]) + (acc[2] + acc[3]), (rr == j) ? 1.f : 0.f);
    }
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) Nd[16 * rr + (j ^ sw(rr))] = tf32r(x[rr]);
}

// Step 3 for thread q (0-127): N Diag(b) as bf16, rows t' of 128 bytes in the 128B-swizzled
// layout at `m2` (blocks above the diagonal are zero). The eight lanes of a row read the two
// halves of their 8 entries in an order chosen per lane, so that each load of N and of b
// touches distinct banks.
__device__ __forceinline__ void store_m2(const float *N32, const float *bv, uint8_t *m2, int q) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int e8 = q + 128 * m;   // 8 consecutive entries of row t'
        const int tp = e8 >> 3, s8 = (e8 & 7) * 8;
        const int ba = tp >> 4, bb = s8 >> 4, r = tp & 15;   // block (ba, bb), row r in it
        uint4 pk = make_uint4(0u, 0u, 0u, 0u);
        if (bb <= ba) {
            const int h0 = 4 * ((bb & 1) ^ ((sw(r) >> 2) & 1)), h1 = h0 ^ 4;
            const float *src = N32 + blk(ba, bb) + 16 * r;
            const float4 x0 = *reinterpret_cast<const float4 *>(src + (((s8 & 15) + h0) ^ sw(r)));
            const float4 x1 = *reinterpret_cast<const float4 *>(src + (((s8 & 15) + h1) ^ sw(r)));
            const float4 b0 = *reinterpret_cast<const float4 *>(bv + vbi(s8 + h0));
            const float4 b1 = *reinterpret_cast<const float4 *>(bv + vbi(s8 + h1));
            const uint32_t p0 = ptx::pack_bf16x2(x0.x * b0.x, x0.y * b0.y), p1 = ptx::pack_bf16x2(x0.z * b0.z, x0.w * b0.w);
            const uint32_t p2 = ptx::pack_bf16x2(x1.x * b1.x, x1.y * b1.y), p3 = ptx::pack_bf16x2(x1.z * b1.z, x1.w * b1.w);
            pk = h0 == 0 ? make_uint4(p0, p1, p2, p3) : make_uint4(p2, p3, p0, p1);
        }
        *reinterpret_cast<uint4 *>(m2 + ptx::sw128((uint32_t)tp, (uint32_t)s8 * 2u)) = pk;
    }
}

}  // namespace gdninv
}  // namespace hypic
