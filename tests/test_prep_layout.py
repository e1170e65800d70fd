"""Host model of the chunk preparation's shared-memory layout, fragment loads and record writes
(csrc/build_gdn_prep.cu).

G (the chunk's gram) keeps its ten 16 x 16 blocks on and below the diagonal, block (a, b) at word
256 (a (a + 1) / 2 + b), row-major with element (r, c) at 16 r + (c ^ sw(r)), sw(r) = 8 bit1(r) +
4 bit2(r). N keeps, per record, the row-major blocks N11, N22, N32, N33 (A operands, the same
swizzle) and the transposed blocks N00, N10, N11, N22 (B operands: element (r, c) at
16 c + (r ^ sw(c))). The products' scratch tiles T (16 x 8) are transposed, element (m, n) at
20 n + m. The b values of a record sit at e + 16 (e >> 5). The tests restate those index functions and every access of the kernel, and
check that

- the ldmatrix row addresses deliver each lane exactly the elements of the m16n8k8 tf32 A and B
  fragments (a0..a3 = (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4); b0, b1 = (t, g), (t + 4, g));
- each warp-wide access needs no more shared-memory wavefronts than its width requires (ldmatrix
  x4: one per 8 x 16-byte matrix; 4-, 8-, 16-byte accesses by a full warp: 1, 2, 4);
- every element of a record (64 x 64 bf16) is written exactly once: the diagonal solves, the
  pieces of steps (ii) and (iii), and the zeros above the diagonal; every piece of a unit's
  inverse is computed by exactly one warp;
- the blocked algebra of steps (i)-(iii), replayed in numpy in the kernel's block order, is the
  inverse (I + Diag(b) L)^-1.

A planted layout without the swizzle fails the fragment-conflict check, and a planted transposed
operand fails the fragment-content check.
"""
import numpy as np
import pytest

LDT = 20
N11, N22, N32, N33 = 0, 256, 512, 768
T00, T10, T11, T22 = 1024, 1280, 1536, 1792
NREC = 2048 + 16
GW = 10 * 256
TILE = 8 * LDT
KDA_SCRATCH = 16384   # the Kh tile the KDA preparation's scratch tiles sit in


def sw(r):
    return ((r << 2) & 8) | (r & 4)


def gblk(a, b):
    return 256 * (a * (a + 1) // 2 + b)


def el_rm(base, r, c, swizzle=sw):
    return base + 16 * r + (c ^ swizzle(r))


def el_t(base, r, c):
    """Element (r, c) of a block of N stored transposed."""
    return base + 16 * c + (r ^ sw(c))


def el_tile(base, m, n):
    """Element (m, n) of a 16 x 8 scratch tile (stored transposed)."""
    return base + LDT * n + m


def vbi(e):
    return e + ((e >> 5) << 4)


def wavefronts(addrs, width):
    """Shared-memory wavefronts of one warp-wide access of `width` words per lane: lanes are
    served in phases of 32 / width lanes, and a phase takes as many wavefronts as the most
    distinct words that fall in one bank."""
    per = 32 // width
    total = 0
    for ph in range(0, 32, per):
        banks = {}
        for lane in range(ph, ph + per):
            if addrs[lane] is None:
                continue
            for w in range(width):
                banks.setdefault((addrs[lane] + w) % 32, set()).add(addrs[lane] + w)
        total += max((len(v) for v in banks.values()), default=0)
    return total


def ldsm_wavefronts(addrs):
    """ldmatrix .x4: lanes 8 m .. 8 m + 7 give the row addresses (16 bytes) of matrix m; each
    matrix is one phase."""
    total = 0
    for m in range(4):
        banks = {}
        for lane in range(8 * m, 8 * m + 8):
            for w in range(4):
                banks.setdefault((addrs[lane] + w) % 32, set()).add(addrs[lane] + w)
        total += max(len(v) for v in banks.values())
    return total


def ldsm_words(addrs):
    """The word each lane receives in registers 0-3 of an ldmatrix .x4 read as 32-bit words:
    lane l gets word l % 4 of row l / 4 of matrix m."""
    return [[addrs[8 * m + (l >> 2)] + (l & 3) for m in range(4)] for l in range(32)]


def a_addrs(base, ks, swizzle=sw):
    out = []
    for l in range(32):
        r, c = (l & 7) | (l & 8), 4 * (l >> 4)
        out.append(base + 16 * r + ((8 * ks + c) ^ swizzle(r)))
    return out


def b_addrs(base, h):
    """B fragments of columns 8 h .. 8 h + 7 of a transposed block of N."""
    return [base + 16 * (8 * h + (l & 7)) + ((4 * (l >> 3)) ^ sw(l & 7)) for l in range(32)]


def tile_addrs(base):
    """B fragments of a scratch tile."""
    return [base + LDT * (l & 7) + 4 * (l >> 3) for l in range(32)]


def test_a_fragments_hold_the_mma_layout():
    for ks in range(2):
        got = ldsm_words(a_addrs(0, ks))
        for l in range(32):
            g, t = l >> 2, l & 3
            want = [el_rm(0, g, 8 * ks + t), el_rm(0, g + 8, 8 * ks + t),
                    el_rm(0, g, 8 * ks + t + 4), el_rm(0, g + 8, 8 * ks + t + 4)]
            assert got[l] == want, (ks, l)


def test_b_fragments_hold_the_mma_layout():
    """B (16 x 8) = columns 8 h .. 8 h + 7 of a transposed block, or a T tile: lane (g, t) needs
    k-rows t, t + 4 (k-step 0) and 8 + t, 12 + t (k-step 1) of column g."""
    for h in range(2):
        got = ldsm_words(b_addrs(0, h))
        for l in range(32):
            g, t = l >> 2, l & 3
            want = [el_t(0, k, 8 * h + g) for k in (t, t + 4, 8 + t, 12 + t)]
            assert got[l] == want, (h, l)
    got = ldsm_words(tile_addrs(0))
    for l in range(32):
        g, t = l >> 2, l & 3
        assert got[l] == [el_tile(0, k, g) for k in (t, t + 4, 8 + t, 12 + t)], l


def test_planted_transposed_operand_is_caught():
    """A B operand read from a row-major block (the transposed copy forgotten) delivers N[g][k]
    instead of N[k][g]: every lane off the diagonal gets other elements."""
    got = ldsm_words(b_addrs(0, 0))
    wrong = 0
    for l in range(32):
        g, t = l >> 2, l & 3
        for i, k in enumerate((t, t + 4, 8 + t, 12 + t)):
            if k != g:
                wrong += got[l][i] != el_rm(0, k, g)
    assert wrong == sum(1 for l in range(32) for k in ((l & 3), (l & 3) + 4, 8 + (l & 3), 12 + (l & 3))
                        if k != (l >> 2))


def test_ldmatrix_reads_are_conflict_free():
    bases_a = [gblk(a, b) for a in range(4) for b in range(a + 1)] + [N11, N22, N32, N33]
    for base in bases_a:
        for ks in range(2):
            assert ldsm_wavefronts(a_addrs(base, ks)) == 4, (base, ks)
    for base in (T00, T10, T11, T22):
        for h in range(2):
            assert ldsm_wavefronts(b_addrs(base, h)) == 4, (base, h)
    for tile in range(4):
        assert ldsm_wavefronts(tile_addrs(tile * TILE)) == 4


def test_planted_unswizzled_layout_conflicts():
    assert max(ldsm_wavefronts(a_addrs(gblk(2, 0), ks, swizzle=lambda r: 0)) for ks in range(2)) > 4


def result_store_addrs(kind, base, h):
    """The four 4-byte stores of a 16 x 8 result piece (put_t into a tile, or N10 transposed),
    or the two 8-byte stores of N32 (row-major)."""
    out = []
    if kind in ("tile", "transposed"):
        el = el_tile if kind == "tile" else el_t
        for dm, dn in ((0, 0), (0, 1), (8, 0), (8, 1)):
            out.append(([el(base, (l >> 2) + dm, 8 * h + 2 * (l & 3) + dn) for l in range(32)], 1))
    else:
        for dm in (0, 8):
            out.append(([el_rm(base, (l >> 2) + dm, 8 * h + 2 * (l & 3)) for l in range(32)], 2))
    return out


def test_result_stores_are_conflict_free():
    """The scratch tiles' and N32's stores take the minimum wavefronts; N10's (four stores of a
    step (ii) piece) take two."""
    for tile in range(4):
        for addrs, width in result_store_addrs("tile", tile * TILE, 0):
            assert wavefronts(addrs, width) == width
    for h in range(2):
        for addrs, width in result_store_addrs("transposed", T10, h):
            assert wavefronts(addrs, width) <= 2
        for addrs, width in result_store_addrs("row-major", N32, h):
            assert wavefronts(addrs, width) == width
            assert all(el_rm(N32, r, c) + 1 == el_rm(N32, r, c + 1) for r in range(16) for c in range(0, 16, 2))


def test_gram_row_stores_are_conflict_free():
    for w in range(4):   # lanes < 16 of warp w store row `lane` of block row w, 16 bytes a lane
        for k in range(w + 1):
            for cb in range(0, 16, 4):
                addrs = [el_rm(gblk(w, k), l, cb) if l < 16 else None for l in range(32)]
                assert wavefronts(addrs, 4) == 2
                assert all((cb ^ sw(l)) % 4 == 0 for l in range(16))


def test_diagonal_solve_stores_are_conflict_free():
    """Lanes 0-15 store record 0's columns, lanes 16-31 record 1's."""
    for base in (N11, N22, N33):
        for rr in range(16):
            addrs = [(l >> 4) * NREC + el_rm(base, rr, l & 15) for l in range(32)]
            assert wavefronts(addrs, 1) == 1
    for base in (T00, T11, T22):
        for s4 in range(4):
            addrs = [(l >> 4) * NREC + base + 16 * (l & 15) + ((4 * s4) ^ sw(l & 15)) for l in range(32)]
            assert wavefronts(addrs, 4) == 4
            for l in range(16):   # the 16-byte piece is elements 4 s4 .. 4 s4 + 3 of row l, in order
                assert [el_t(base, 4 * s4 + e, l) for e in range(4)] == list(
                    range(base + 16 * l + ((4 * s4) ^ sw(l)), base + 16 * l + ((4 * s4) ^ sw(l)) + 4))
    for a in range(4):
        for rr in range(16):
            assert wavefronts([(l >> 4) * 80 + vbi(16 * a + rr) for l in range(32)], 1) == 1


def test_every_word_is_its_own_and_inside_the_allocation():
    words = set()
    for base in (N11, N22, N32, N33):
        for r in range(16):
            for c in range(16):
                words.add(el_rm(base, r, c))
    for base in (T00, T10, T11, T22):
        for r in range(16):
            for c in range(16):
                words.add(el_t(base, r, c))
    assert len(words) == 8 * 256 and max(words) < NREC
    assert NREC % 32 == 16 and NREC % 4 == 0   # record 1's row-major blocks 16 banks over
    g = {el_rm(gblk(a, b), r, c) for a in range(4) for b in range(a + 1) for r in range(16) for c in range(16)}
    assert len(g) == 10 * 256 and max(g) < GW
    t = {tile * TILE + el_tile(0, m, n) for tile in range(4) for m in range(16) for n in range(8)}
    assert len(t) == 4 * 128 and max(t) < 4 * TILE
    assert 4 * 2 * TILE * 4 <= KDA_SCRATCH   # the KDA preparation (one record): two tiles a warp
    assert len({vbi(e) for e in range(64)}) == 64 and vbi(63) < 80
    # the GDN preparation's shared memory at R = 2, four CTAs per SM (the static part measured
    # by the compiler: 1344 bytes)
    dyn = 16384 + GW * 4 + 2 * NREC * 4 + 4 * 4 * TILE * 4 + 1024
    assert 4 * (dyn + 1344 + 1024) <= 228 * 1024


def zero_pieces(R, q, nt):
    """The zero pieces thread q < nt writes (the GDN preparation: warps 0-1, nt = 64; the KDA
    preparation: all 128 threads)."""
    out = []
    for idx in range(q, 192 * R, nt):
        rr = 1 if (R == 2 and idx >= 192) else 0
        z = idx - 192 * rr
        if z < 96:
            row, piece = z // 6, 2 + z % 6
        elif z < 160:
            row, piece = 16 + (z - 96) // 4, 4 + (z - 96) % 4
        else:
            row, piece = 32 + (z - 160) // 2, 6 + (z - 160) % 2
        out.append((rr, row, piece))
    return out


def pieces_of_warp(R, warp):
    """The (record, step, block column X, half h) pieces warp `warp` computes (off_diagonal)."""
    h = warp & 1
    out = [(rr, "one", 1 if warp < 2 else 3, h) for rr in range(R)]
    for rr in range(R):
        x = 0 if (warp >> 1) == rr else 1
        out.append((rr, "two", x, h))
    return out


@pytest.mark.parametrize("R, nt", [(1, 64), (2, 64), (1, 128)])
def test_every_record_entry_is_written_once(R, nt):
    count = np.zeros((R, 64, 64), dtype=int)
    for warp in range(4):   # diagonal solves: lane j < 16 (record lane >> 4 when R = 2)
        for lane in range(32):
            if R == 1 and lane >= 16:
                continue
            rr, j = (lane >> 4) if R == 2 else 0, lane & 15
            for row in range(16):
                count[rr, 16 * warp + row, 16 * warp + j] += 1
    for warp in range(4):
        for rr, step, x, h in pieces_of_warp(R, warp):
            if step == "one":
                blocks = [(x, x - 1)]   # (1,0) or (3,2)
            else:
                blocks = [(2, x), (3, x)]
            for a, b in blocks:
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    for dr in (0, 8):
                        for dc in (0, 1):
                            count[rr, 16 * a + g + dr, 16 * b + 8 * h + 2 * t + dc] += 1
    for q in range(nt):
        for rr, row, piece in zero_pieces(R, q, nt):
            assert row < 64 and piece < 8
            count[rr, row, 8 * piece:8 * piece + 8] += 1
    assert (count == 1).all()


def test_step_two_work_is_balanced_at_r2():
    """Each warp takes one piece of block column 0 (7 products of 16 x 8 x 16) and one of
    column 1 (5), so the four warps have equal work."""
    for warp in range(4):
        xs = sorted(x for rr, step, x, h in pieces_of_warp(2, warp) if step == "two")
        assert xs == [0, 1]


def blocked_inverse(Gm, b):
    """Steps (i)-(iii) in the kernel's block order, in float64: diagonal blocks by forward
    substitution, then (1,0) and (3,2), then the lower-left quarter by block columns."""
    n = np.zeros((64, 64))
    B = lambda i: slice(16 * i, 16 * i + 16)   # noqa: E731
    for a in range(4):
        for j in range(16):
            x = np.zeros(16)
            for r in range(16):
                acc = sum(Gm[16 * a + r, 16 * a + s] * x[s] for s in range(r))
                x[r] = (1.0 if r == j else 0.0) - b[16 * a + r] * acc
            n[B(a), 16 * a + j] = x
    for a, c in ((1, 0), (3, 2)):
        t = np.diag(b[B(a)]) @ Gm[B(a), B(c)] @ n[B(c), B(c)]
        n[B(a), B(c)] = -n[B(a), B(a)] @ t
    for x in range(2):
        if x == 0:
            t2 = Gm[B(2), B(0)] @ n[B(0), B(0)] + Gm[B(2), B(1)] @ n[B(1), B(0)]
            t3 = Gm[B(3), B(0)] @ n[B(0), B(0)] + Gm[B(3), B(1)] @ n[B(1), B(0)]
        else:
            t2 = Gm[B(2), B(1)] @ n[B(1), B(1)]
            t3 = Gm[B(3), B(1)] @ n[B(1), B(1)]
        t2 = np.diag(b[B(2)]) @ t2
        t3 = np.diag(b[B(3)]) @ t3
        n[B(2), B(x)] = -n[B(2), B(2)] @ t2
        n[B(3), B(x)] = -(n[B(3), B(2)] @ t2 + n[B(3), B(3)] @ t3)
    return n


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_blocked_algebra_is_the_inverse(seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((64, 128))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    Gm = k @ k.T
    b = rng.uniform(0.0, 1.0, 64)
    b[50:] = 0.0 if seed == 2 else b[50:]   # a ragged chunk: tokens past the end have b = 0
    ref = np.linalg.inv(np.eye(64) + np.diag(b) @ np.tril(Gm, -1))
    got = blocked_inverse(Gm, b)
    assert np.allclose(got, ref, atol=1e-10, rtol=1e-10)


def sw128(row, byte):
    return row * 128 + (byte ^ ((row & 7) << 4))


def test_kda_tile_pass_is_conflict_free():
    """The KDA preparation's pass over a chunk: thread q takes the key channels 2 pc, 2 pc + 1
    (pc = q % 64) over the token half q / 64 and reads, then writes, their bf16 pair (one word)
    of the k tile and the gated tiles, all 64 x 128 bf16 as two 128B-swizzled 64-channel
    halves of 8 KB, token by token: each warp-wide access is one wavefront."""
    for w in range(4):
        for t in range(32):
            addrs = []
            for l in range(32):
                q = 32 * w + l
                pc, th = q & 63, q >> 6
                addrs.append(((pc >> 5) * 8192 + sw128(32 * th + t, 4 * (pc & 31))) // 4)
            assert len(set(addrs)) == 32
            assert wavefronts(addrs, 1) == 1


# The kernel source this model was last checked against (code only; comments do not count).
MODELLED_SOURCE = ("build_gdn_prep.cu", "87c7e3551c14")


def test_model_is_checked_against_the_current_kernel_source():
    from tests.helpers import kernel_code_hash
    name, recorded = MODELLED_SOURCE
    assert kernel_code_hash(name) == recorded, (
        f"{name} changed since this model was checked against it: re-check the model "
        f"against the new code, then record the new hash {kernel_code_hash(name)}")
