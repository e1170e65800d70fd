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
// otherwise R = 1. Four CTAs per SM (all 512 TMEM columns, about 50 KB of shared memory and at
// most 128 registers each). Units are handed out as tickets: a CTA
// starts with two fixed units and takes each further one from a counter in the workspace
// (zeroed before the launch), so CTAs that run faster take more units and all CTAs finish
// within about one unit of each other. The k tile of the next unit is requested as soon as
// the current gram has read the single k buffer, its gram is issued once the current diagonal
// blocks are solved (two TMEM buffers), and b is loaded a unit ahead, so loads and grams
// overlap the inversions. A CTA that is on its last unit lets the chain kernel launch
// (programmatic dependent launch); the chain waits for this grid's completion before it reads
// any record. Three CTA barriers per unit: at its top, after the diagonal solves, and between
// steps 4 (ii) and (iii). Per unit:
//   1. TMA the chunk's k (two 128B-swizzled 64-channel halves); b masked past the segment end.
//   2. One thread issues the gram K K^T (M = 64 tcgen05 MMA, fp32 accumulator in TMEM).
//   3. Warp w reads block row w of the raw gram G = K K^T into shared memory as 16 x 16 blocks:
//      the blocks left of the diagonal rounded to tf32 once (they are only ever MMA operands),
//      the diagonal block exact (forward substitution); the blocks right of it are not stored.
//      A = Diag(b) L is never formed: b scales rows inside the consumers, and the strictly
//      lower mask is the consumers' index range.
//   4. N by 16 x 16 blocks. (i) Warp a solves diagonal block a by forward substitution (lanes
//      0-15 the first record's columns, lanes 16-31 the second's); it needs only its own gram
//      rows, so no CTA barrier precedes it. (ii) The blocks (1,0) and (3,2), which complete the
//      inverses N11 and N22 of the two 32 x 32 diagonal halves: N_ab = -N_aa Diag(b_a) G_ab N_bb.
//      (iii) The lower-left 32 x 32 quarter, N21 = -N22 Diag(b) G21 N11, by columns: a warp
//      takes 8 columns of one record and forms both T = Diag(b) G21 N11 rows and both N21 rows
//      for them with nothing but its own scratch, so no barrier separates the two products.
//      All products are 16 x 8 x 16 pieces on the warp-level tensor-core MMA (m16n8k8, tf32
//      inputs, fp32 accumulation): tcgen05's smallest tile (M = 64) would waste most of its
//      work on products this small and each would need a round trip through TMEM. Operands
//      come by ldmatrix: A operands from row-major blocks, B operands from transposed copies
//      (a block is stored in the orientations its consumers need), all already rounded to
//      tf32.
//   5. Every block of N is scaled by b over its columns, rounded to bf16 and stored into the
//      record straight from the registers that computed it; warps 0-1 write the blocks above the
//      diagonal as zeros after their diagonal solves.
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
// Shared-memory layout. G keeps its ten 16 x 16 blocks on and below the diagonal, block (a, b)
// at word 256 (a (a + 1) / 2 + b), row-major with element (r, c) at 16 r + (c ^ sw(r)). N keeps,
// per record, the blocks its products read: row-major N11, N22, N32, N33 (A operands) and
// transposed N00, N10, N11, N22 (B operands: element (r, c) at 16 c + (r ^ sw(c))). The swizzle
// makes every ldmatrix phase (8 rows of 16 bytes), the gram's and the diagonal solves' stores
// and the step (ii) stores of N32 touch 32 distinct banks (those of N10 touch 16). A record's N
// takes kNRec words, 16 more than its blocks, so that the second record's row-major blocks sit
// 16 banks after the first's (the two records' diagonal solves store side by side). Each warp
// has 2 R scratch tiles T (16 x 8), held transposed as 8 rows of stride kLdT = 20 words, which
// keeps both their stores from the accumulators and their ldmatrix reads conflict-free.
constexpr int kLdT = 20;
constexpr int kN11 = 0, kN22 = 256, kN32 = 512, kN33 = 768;                 // row-major
constexpr int kT00 = 1024, kT10 = 1280, kT11 = 1536, kT22 = 1792;           // transposed
constexpr int kNRec = 2048 + 16;
constexpr int kGWords = 10 * 256;
constexpr int kTile = 8 * kLdT;   // one transposed 16 x 8 T tile
__device__ __forceinline__ int sw(int r) { return ((r << 2) & 8) | (r & 4); }
__host__ __device__ constexpr int gblk(int a, int b) { return 256 * (a * (a + 1) / 2 + b); }
// b of a record: entry e at vbi(e), 16 words of padding after the first 32 entries, so that the
// diagonal solves' loads of b touch distinct banks
constexpr int kVb = 80;
__device__ __forceinline__ int vbi(int e) { return e + ((e >> 5) << 4); }
// R records per iteration: the value heads h, h + 1 that share a key head (R = 2, when the
// grouped-query factor is even) share the k tile, the gram and its shared-memory copy, and
// their two inverses run side by side; R = 1 otherwise.
template <int R>
struct PrepGeo {
    static constexpr uint32_t kOffK = 0;                              // k tile, 16 KB
    static constexpr uint32_t kOffG32 = 16384;                        // the gram K K^T, 10 blocks
    static constexpr uint32_t kOffN32 = kOffG32 + kGWords * 4;        // R x N (tf32-rounded)
    static constexpr uint32_t kOffT = kOffN32 + R * kNRec * 4;        // 4 warps x 2 R tiles
    static constexpr uint32_t kSmemBytes = kOffT + 4 * 2 * R * kTile * 4 + 1024;
    static constexpr int kCtasPerSm = 4;                              // 4 x 128 TMEM columns
};
constexpr int kCtl = 0;   // warp 0 lane 0 issues loads and grams (warp 0 reads the fewest gram rows)

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// x rounded to tf32 (round to nearest), kept as a float with the low 13 mantissa bits zero
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(to_tf32(x)); }

// four 8 x 8 b16 matrices; read as 32-bit words, lane l receives word (l / 4, l % 4) of each
// matrix's 8 rows of 16 bytes, which is how a tf32 MMA fragment is laid out
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void mma_m16n8k8(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A lane's byte offsets of the ldmatrix row addresses, and its place (g, t) in the m16n8
// accumulator: rows g, g + 8, columns 2 t, 2 t + 1.
struct Lanes {
    uint32_t a0, a1;   // A fragments, k-steps 0 and 1, of a row-major 16 x 16 block
    uint32_t bn;       // B fragments, both k-steps, of rows 0-7 of a transposed block of N
    uint32_t b;        // B fragments, both k-steps, of a T tile
    int g, t;
};

__device__ __forceinline__ Lanes lanes_of(int lane) {
    Lanes L;
    // matrices 0-3 of an A fragment: rows 0-7 and 8-15 of k-columns 8 ks .. + 3, then + 4 .. + 7
    const int r = (lane & 7) | (lane & 8), c = 4 * (lane >> 4);
    L.a0 = 4u * (uint32_t)(16 * r + (c ^ sw(r)));
    L.a1 = 4u * (uint32_t)(16 * r + ((8 + c) ^ sw(r)));
    // matrices 0-3 of a B fragment: columns 0-7 of k-rows 0-3, 4-7, 8-11, 12-15 (rows 8-15 of a
    // transposed block share the swizzle of rows 0-7)
    L.bn = 4u * (uint32_t)(16 * (lane & 7) + ((4 * (lane >> 3)) ^ sw(lane & 7)));
    L.b = 4u * (uint32_t)(kLdT * (lane & 7) + 4 * (lane >> 3));
    L.g = lane >> 2;
    L.t = lane & 3;
    return L;
}

// c += X Y for a row-major 16 x 16 block X (shared address) and the B fragments of a 16 x 8 Y
__device__ __forceinline__ void mma16(float (&c)[4], uint32_t X, const uint32_t (&y)[4], const Lanes &L) {
    uint32_t a[4], a2[4];
    ldsm4(a, X + L.a0);
    ldsm4(a2, X + L.a1);
    mma_m16n8k8(c, a, y[0], y[1]);
    mma_m16n8k8(c, a2, y[2], y[3]);
}

// T = Diag(b_lo rows, b_hi rows) c, rounded to tf32, into a transposed tile (element (m, n) at
// kLdT n + m)
__device__ __forceinline__ void put_t(float *Tt, const float (&c)[4], float b_lo, float b_hi, const Lanes &L) {
    float *o = Tt + kLdT * (2 * L.t) + L.g;
    o[0] = tf32r(c[0] * b_lo);
    o[kLdT] = tf32r(c[1] * b_lo);
    o[8] = tf32r(c[2] * b_hi);
    o[kLdT + 8] = tf32r(c[3] * b_hi);
}

// the record's entries (row0 + g, col0 + 2 t, + 1) and (row0 + g + 8, ...) from N values -d:
// M2 = N Diag(b), bf16, rows of 128 bytes
__device__ __forceinline__ void put_rec(uint8_t *rec, int row0, int col0, const float (&d)[4], const float *bv,
                                        const Lanes &L) {
    const int r = row0 + L.g, c = col0 + 2 * L.t;
    const float2 bc = *reinterpret_cast<const float2 *>(bv + vbi(c));
    *reinterpret_cast<uint32_t *>(rec + r * 128 + c * 2) = pack_bf16x2(-d[0] * bc.x, -d[1] * bc.y);
    *reinterpret_cast<uint32_t *>(rec + (r + 8) * 128 + c * 2) = pack_bf16x2(-d[2] * bc.x, -d[3] * bc.y);
}

// Step 4 (i): diagonal block `warp` of each record. Lane j < 16 solves column j of record 0
// (lanes 16-31 that of record 1 when R = 2) by forward substitution,
// x_r = [r == j] - b_r sum_{s<r} G_rs x_s (A = Diag(b) L restricted to the block), then stores
// the column into the copies the products read and into the record.
template <int R>
__device__ __forceinline__ void diag_blocks(const float *G32, float *N32, const float (*vb)[kVb],
                                            uint8_t *const (&rec)[R], int warp, int lane) {
    if (R == 2 || lane < 16) {
        const int a = warp, j = lane & 15, rr_ = R == 2 ? lane >> 4 : 0;
        const float *bv = vb[rr_];
        const float *Gd = G32 + gblk(a, a);
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
        float *Nr = N32 + rr_ * kNRec;
        if (a >= 1) {   // row-major copy: N11, N22, N33
            float *Nd = Nr + (a == 1 ? kN11 : a == 2 ? kN22 : kN33);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) Nd[16 * rr + (j ^ sw(rr))] = tf32r(x[rr]);
        }
        if (a <= 2) {   // transposed copy: N00, N11, N22 (column j is row j)
            float *Td = Nr + (a == 0 ? kT00 : a == 1 ? kT11 : kT22) + 16 * j;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4)
                *reinterpret_cast<float4 *>(Td + ((4 * s4) ^ sw(j))) = make_float4(
                    tf32r(x[4 * s4]), tf32r(x[4 * s4 + 1]), tf32r(x[4 * s4 + 2]), tf32r(x[4 * s4 + 3]));
        }
        const float bj = bv[vbi(16 * a + j)];
        uint8_t *dst = (rr_ ? rec[R - 1] : rec[0]) + (16 * a) * 128 + (16 * a + j) * 2;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr)
            *reinterpret_cast<uint16_t *>(dst + rr * 128) = (uint16_t)pack_bf16x2(x[rr] * bj, 0.f);
    }
}

// Step 4 (ii): columns 8 h .. 8 h + 7 of block (1,0) (B32 = false) or (3,2) (true) of each of the
// unit's R records, N_ab = -N_aa Diag(b_a) G_ab N_bb; the records share the G fragments and run
// side by side (record rr in scratch tile rr). N10 is stored transposed (a B operand of step
// (iii)), N32 row-major (an A operand).
template <bool B32, int R>
__device__ __forceinline__ void level_one(uint32_t sG, float *N32, float *Tw, const float (*vb)[kVb],
                                          uint8_t *const (&rec)[R], int h, const Lanes &L) {
    constexpr int a = B32 ? 3 : 1, b = B32 ? 2 : 0;
    const uint32_t sN = smem_u32(N32), sT = smem_u32(Tw);
    uint32_t ga[4], ga2[4], y[R][4];
    ldsm4(ga, sG + 4u * gblk(a, b) + L.a0);
    ldsm4(ga2, sG + 4u * gblk(a, b) + L.a1);
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
        ldsm4(y[rr], sN + 4u * (uint32_t)(rr * kNRec + (B32 ? kT22 : kT00) + 128 * h) + L.bn);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_m16n8k8(c, ga, y[rr][0], y[rr][1]);
        mma_m16n8k8(c, ga2, y[rr][2], y[rr][3]);
        put_t(Tw + rr * kTile, c, vb[rr][vbi(16 * a + L.g)], vb[rr][vbi(16 * a + L.g + 8)], L);
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < R; ++rr) ldsm4(y[rr], sT + 4u * (uint32_t)(rr * kTile) + L.b);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        float *Nr = N32 + rr * kNRec;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma16(d, sN + 4u * (uint32_t)(rr * kNRec + (B32 ? kN33 : kN11)), y[rr], L);
        if (B32) {
            float *o = Nr + kN32 + ((8 * h + 2 * L.t) ^ sw(L.g));   // rows g and g + 8 share the swizzle
            *reinterpret_cast<float2 *>(o + 16 * L.g) = make_float2(tf32r(-d[0]), tf32r(-d[1]));
            *reinterpret_cast<float2 *>(o + 16 * (L.g + 8)) = make_float2(tf32r(-d[2]), tf32r(-d[3]));
        } else {   // N10 transposed: rows n = 8 h + 2 t, + 1 (the same swizzle), columns g, g + 8
            const int n = 8 * h + 2 * L.t;
            float *o = Nr + kT10 + 16 * n;
            o[L.g ^ sw(n)] = tf32r(-d[0]);
            o[16 + (L.g ^ sw(n + 1))] = tf32r(-d[1]);
            o[(L.g + 8) ^ sw(n)] = tf32r(-d[2]);
            o[16 + ((L.g + 8) ^ sw(n + 1))] = tf32r(-d[3]);
        }
        put_rec(rec[rr], 16 * a, 16 * b + 8 * h, d, vb[rr], L);
    }
    __syncwarp();   // the scratch tiles are rewritten by this warp's next piece
}

// Step 4 (iii): columns 16 X + 8 h .. + 7 of the lower-left quarter of R records (record rr takes
// block column X ^ rr, in scratch tiles 2 rr and 2 rr + 1; the records' products run side by
// side): T2, T3 = Diag(b) (G21 N11) rows 32-47, 48-63 (N11's block column: blocks 0-1 for column
// 0, block 1 for column 1), then N(2,.) = -N22 T2 and N(3,.) = -(N32 T2 + N33 T3), straight into
// the record.
template <int X, int R>
__device__ __forceinline__ void level_two(uint32_t sG, const float *N32, float *Tw, const float (*vb)[kVb],
                                          uint8_t *const (&rec)[R], int h, const Lanes &L) {
    const uint32_t sN = smem_u32(N32), sT = smem_u32(Tw), hoff = 4u * (uint32_t)(128 * h);
    float c2[R][4], c3[R][4];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int x = X ^ rr;
        const uint32_t nb = sN + 4u * (uint32_t)(rr * kNRec) + hoff + L.bn;
        uint32_t y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c2[rr][i] = c3[rr][i] = 0.f;
        if (x == 0) {
            ldsm4(y, nb + 4u * kT00);
            mma16(c2[rr], sG + 4u * gblk(2, 0), y, L);
            mma16(c3[rr], sG + 4u * gblk(3, 0), y, L);
            ldsm4(y, nb + 4u * kT10);
        } else {
            ldsm4(y, nb + 4u * kT11);
        }
        mma16(c2[rr], sG + 4u * gblk(2, 1), y, L);
        mma16(c3[rr], sG + 4u * gblk(3, 1), y, L);
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        put_t(Tw + 2 * rr * kTile, c2[rr], vb[rr][vbi(32 + L.g)], vb[rr][vbi(40 + L.g)], L);
        put_t(Tw + (2 * rr + 1) * kTile, c3[rr], vb[rr][vbi(48 + L.g)], vb[rr][vbi(56 + L.g)], L);
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const uint32_t na = sN + 4u * (uint32_t)(rr * kNRec);
        float d2[4] = {0.f, 0.f, 0.f, 0.f}, d3[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t y[4];
        ldsm4(y, sT + 4u * (uint32_t)(2 * rr * kTile) + L.b);
        mma16(d2, na + 4u * kN22, y, L);
        mma16(d3, na + 4u * kN32, y, L);
        ldsm4(y, sT + 4u * (uint32_t)((2 * rr + 1) * kTile) + L.b);
        mma16(d3, na + 4u * kN33, y, L);
        put_rec(rec[rr], 32, 16 * (X ^ rr) + 8 * h, d2, vb[rr], L);
        put_rec(rec[rr], 48, 16 * (X ^ rr) + 8 * h, d3, vb[rr], L);
    }
    __syncwarp();   // the scratch tiles are rewritten by this warp's next piece
}

// The record's blocks above the diagonal, as zeros: 192 pieces of 16 bytes per record (block
// row 0 from column 16, row 1 from 32, row 2 from 48), by threads q < NT.
template <int R, int NT>
__device__ __forceinline__ void zero_upper(uint8_t *const (&rec)[R], int q) {
#pragma unroll
    for (int id = q; id < 192 * R; id += NT) {
        const int rr = R == 2 ? (id >= 192) : 0, z = id - 192 * rr;
        int row, piece;
        if (z < 96) row = z / 6, piece = 2 + z % 6;
        else if (z < 160) row = 16 + (z - 96) / 4, piece = 4 + (z - 96) % 4;
        else row = 32 + (z - 160) / 2, piece = 6 + (z - 160) % 2;
        *reinterpret_cast<uint4 *>((rr ? rec[R - 1] : rec[0]) + row * 128 + piece * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Steps 4 (ii) and (iii) for the unit's R records, with one CTA barrier between them. Step
// (ii): warps 0-1 take the halves of (1,0), warps 2-3 those of (3,2), for every record. Step
// (iii): warp w takes
// column half h = w % 2 of block column w / 2 of record 0 and, when R = 2, of the other block
// column of record 1, so that every warp has the same work; the two records' pieces interleave.
template <int R>
__device__ __forceinline__ void off_diagonal(uint32_t sG, float *N32, float *Tw, const float (*vb)[kVb],
                                             uint8_t *const (&rec)[R], int warp, const Lanes &L) {
    const int h = warp & 1;
    if (warp < 2) level_one<false, R>(sG, N32, Tw, vb, rec, h, L);
    else level_one<true, R>(sG, N32, Tw, vb, rec, h, L);
    __syncthreads();
    if (warp < 2) level_two<0, R>(sG, N32, Tw, vb, rec, h, L);
    else level_two<1, R>(sG, N32, Tw, vb, rec, h, L);
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
    __shared__ Walk s_walk[2];   // the unit after the next, drawn by thread kCtl (two slots)
    __shared__ __align__(16) float vb[2][R][kVb];   // the records' b at vbi(token)

    const int64_t total = total_records(p), units = total / R;
    unsigned *tickets = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(p.workspace) + total * kGdnRecordBytes);
    auto nch_of = [&](int r) { return (p.seg[r].len + C - 1) / C; };
    Walk cur = decode<R>(p, blockIdx.x, units);
    if (cur.r >= p.n_seg) return;   // uniform: the whole CTA leaves before any set-up
    const int q = threadIdx.x, warp = q >> 5, lane = q & 31;
    float *G32 = reinterpret_cast<float *>(smem + G::kOffG32);
    float *N32 = reinterpret_cast<float *>(smem + G::kOffN32);   // record rr at N32 + rr * kNRec
    float *Tw = reinterpret_cast<float *>(smem + G::kOffT) + warp * 2 * R * kTile;
    const uint32_t sG = smem_u32(G32);
    const Lanes L = lanes_of(lane);

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
    // every thread decodes unit 1; later units come through s_walk. Thread kCtl keeps its own
    // copy `kn`: the unit after the current one at the top of an iteration (its k tile is
    // requested there), the unit after that once its ticket is decoded.
    Walk nxt = decode<R>(p, (int64_t)gridDim.x + blockIdx.x, units);
    Walk kn = nxt;
    float beta_cur = load_beta(cur);
    if (q == kCtl) {
        prefetch_tmap(&tmK);
        load_k(cur);
        ok = gram(0);
        s_walk[1] = nxt;
    }
    for (int i = 0; cur.r < p.n_seg; ++i) {
        const int b = i & 1;
        const SegEntry seg = p.seg[cur.r];
        const int nch = nch_of(cur.r);
        // every thread decodes the same unit: a failing check leaves the loop uniformly
        if (!in_bounds(cur.c < nch && cur.h + R <= p.H_v &&
                           (int64_t)seg.wsb + (int64_t)(cur.h + R - 1) * nch + cur.c < total, p.err))
            break;
        uint8_t *rec[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
            rec[rr] = static_cast<uint8_t *>(p.workspace) +
                      ((int64_t)seg.wsb + (int64_t)(cur.h + rr) * nch + cur.c) * (int64_t)kGdnRecordBytes;
        if (q < R * C) vb[b][q / C][vbi(q & (C - 1))] = beta_cur;
        // gram(i) done: the k tile is free for the next unit
        if (q == kCtl) {
            ok = ok && mbar_wait(&gfull[b], gwait[b] & 1, p.err, kErrTimeout);
            if (ok) {
                ++gwait[b];
                if (kn.r < p.n_seg) load_k(kn);
            }
            s_ok = ok ? 1 : 0;
            // the ticket of the unit after the next (the counter's answer is used only once
            // this unit's diagonal blocks are solved, so its latency overlaps them)
            if (kn.r < p.n_seg) ticket = 2 * (int64_t)gridDim.x + atomicAdd(tickets, 1u);
        }
        __syncthreads();
        if (!s_ok) break;   // uniform
        nxt = s_walk[(i + 1) & 1];
        if (nxt.r >= p.n_seg) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        const float beta_next = load_beta(nxt);
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
                        *reinterpret_cast<float4 *>(G32 + gblk(warp, k) + 16 * r + (cb ^ sw(r))) = g4;
                    }
                }
            }
        }
        __syncwarp();   // the diagonal block's rows were stored by this warp
        diag_blocks<R>(G32, N32, vb[b], rec, warp, lane);
        if (warp < 2) zero_upper<R, 64>(rec, q);   // warps 0-1 read the fewest gram rows
        // the next unit's gram (its k tile was requested at the top of this unit) into the other
        // TMEM buffer, last read a unit ago, and the walk of the unit after it
        if (q == kCtl) {
            if (ok && kn.r < p.n_seg) ok = gram(b ^ 1);
            const Walk w2 = kn.r < p.n_seg ? decode<R>(p, ticket, units) : kn;
            s_walk[b] = w2;
            kn = w2;
        }
        tc_fence_before();
        __syncthreads();
        off_diagonal<R>(sG, N32, Tw, vb[b], rec, warp, L);
        cur = nxt;
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

// Four CTAs per SM: the two operand tiles, G and N (the level products' scratch tiles sit in the
// Kh tile once its store has read it).
struct KdaGeo {
    static constexpr uint32_t kOffK = 0;                  // k tile, then Kt in place, 16 KB
    static constexpr uint32_t kOffH = 16384;              // Kh, then the scratch
    static constexpr uint32_t kOffG32 = 32768;            // the gram, 10 blocks
    static constexpr uint32_t kOffN32 = kOffG32 + kGWords * 4;
    static constexpr uint32_t kSmemBytes = kOffN32 + kNRec * 4 + 1024;
    static constexpr int kCtasPerSm = 4;
};
static_assert(4 * 2 * kTile * 4 <= 16384, "the scratch tiles fit in the Kh tile");
// warp 3 lane 0 issues loads, grams and the operand stores: its wait for the stores' reads comes
// after its diagonal solve, which its larger share of gram rows delays anyway
constexpr int kKdaCtl = 96;

__global__ void __launch_bounds__(kThreads, KdaGeo::kCtasPerSm)
build_kda_prep_kernel(const __grid_constant__ BuildParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmKh) {
    using G = KdaGeo;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t kfull, gfull;
    __shared__ uint32_t tslot;
    __shared__ Walk s_walk[2];
    __shared__ float s_max[4];
    __shared__ float2 s_part[2][64];                  // [token half][channel pair]
    __shared__ __align__(16) float vb[2][1][kVb];     // two units' b

    const int64_t total = total_records(p);
    unsigned *tickets = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(p.workspace) + total * kGdnRecordBytes);
    Walk cur = decode<1>(p, blockIdx.x, total);
    if (cur.r >= p.n_seg) return;   // uniform: the whole CTA leaves before any set-up
    const int q = threadIdx.x, warp = q >> 5, lane = q & 31;
    uint8_t *tK = smem + G::kOffK, *tH = smem + G::kOffH;
    float *G32 = reinterpret_cast<float *>(smem + G::kOffG32);
    float *N32 = reinterpret_cast<float *>(smem + G::kOffN32);
    float *Tw = reinterpret_cast<float *>(tH) + warp * 2 * kTile;
    const uint32_t sG = smem_u32(G32);
    const Lanes L = lanes_of(lane);

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
    int kiss = 0, giss = 0, kwait = 0, gwait = 0;   // issued by thread kKdaCtl; waited by every thread
    bool stored = false;                             // thread kKdaCtl: a group of record stores issued
    auto load_k = [&](const Walk &w) {   // thread kKdaCtl
        ++kiss;
        const int32_t t0 = p.seg[w.r].start + w.c * C;
        mbar_arrive_expect_tx(&kfull, 16384);
        tma_load_3d(tK, &tmK, &kfull, 0, w.h / p.gqa, t0);
        tma_load_3d(tK + 8192, &tmK, &kfull, 64, w.h / p.gqa, t0);
    };
    bool ok = true;
    int64_t ticket = 0;   // thread kKdaCtl
    Walk nxt = decode<1>(p, (int64_t)gridDim.x + blockIdx.x, total);
    if (q == kKdaCtl) {
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
        const int b = i & 1;
        const SegEntry seg = p.seg[cur.r];
        const int nch = (seg.len + C - 1) / C;
        const int64_t rec_i = (int64_t)seg.wsb + (int64_t)cur.h * nch + cur.c;
        if (!in_bounds(cur.c < nch && cur.h < p.H_v && rec_i < total, p.err)) break;   // uniform
        uint8_t *const rec[1] = {static_cast<uint8_t *>(p.workspace) + rec_i * kGdnRecordBytes};
        // (1) b of the unit; the pair's log-decay over this token half
        if (q < C) vb[b][0][vbi(q)] = beta_cur;
        {
            float2 sh = make_float2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < CH; ++t) sh.x += g[t].x, sh.y += g[t].y;
            s_part[th][pc] = sh;
        }
        if (q == kKdaCtl && nxt.r < p.n_seg) ticket = 2 * (int64_t)gridDim.x + atomicAdd(tickets, 1u);
        zero_upper<1, kThreads>(rec, q);
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
        if (q == kKdaCtl) {
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
            const int32_t row = (int32_t)(rec_i * C);
            tma_store_2d(&tmKt, tK, 0, row);
            tma_store_2d(&tmKt, tK + 8192, 64, row);
            tma_store_2d(&tmKh, tH, 0, row);
            tma_store_2d(&tmKh, tH + 8192, 64, row);
            bulk_commit();
            stored = true;
        }
        {
            const float m = fmaxf(fmaxf(s_max[0], s_max[1]), fmaxf(s_max[2], s_max[3]));
            float *side = p.kda_side + rec_i * kKdaSide;
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
                        *reinterpret_cast<float4 *>(G32 + gblk(warp, k) + 16 * r + (cb ^ sw(r))) = g4;
                    }
                }
            }
        }
        __syncwarp();   // the diagonal block's rows were stored by this warp
        diag_blocks<1>(G32, N32, vb[b], rec, warp, lane);
        // the stores must have read Kt and Kh before the next k tile lands over Kt and the
        // level products' scratch is written over Kh (after the barrier below); the next unit's
        // gates and walk
        if (q == kKdaCtl) {
            bulk_wait_read<0>();
            if (nxt.r < p.n_seg) load_k(nxt);
            s_walk[b] = nxt.r < p.n_seg ? decode<1>(p, ticket, total) : nxt;
        }
        if (nxt.r < p.n_seg) load_gates(nxt);
        tc_fence_before();
        __syncthreads();
        const Walk n2 = s_walk[b];   // slot b is written again two units later
        if (n2.r >= p.n_seg) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        off_diagonal<1>(sG, N32, Tw, vb[b], rec, warp, L);
        cur = nxt;
        nxt = n2;
    }
    if (q == kKdaCtl) {   // the record stores complete; after a wait gave up, every copy and MMA lands
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
