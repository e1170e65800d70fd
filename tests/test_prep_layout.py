"""Host model of the shared-memory layout of the chunk preparation (csrc/build_gdn_prep.cu).

G (the chunk's gram) and N (the inverse, one per record of a unit) keep only their ten 16 x 16
blocks on and below the diagonal: block (a, b) starts at word 264 (a (a + 1) / 2 + b), and
element (r, c) of a block sits at 16 r + (c ^ sw(r)) with sw(r) = 8 bit1(r) + 4 bit2(r). The b
values of a record sit at e + 16 (e >> 5). The tests restate those index functions and every
access pattern of the kernel, and check that

- every element has its own word, inside the allocation;
- each warp-wide access needs no more shared-memory wavefronts than its width requires
  (1 for 4-byte, 2 for 8-byte, 4 for 16-byte accesses by a full warp): the warp-level MMA's A
  and B fragments, the 16 x 8 result stores, the gram's row stores, the diagonal solves' stores
  and reads of b, and the record stage's loads of N and b.

A planted layout without the swizzle fails the fragment check.
"""
import pytest

BLK = 264            # words per block, including 8 words of padding
TRI = 10 * BLK       # one matrix (G, or one record of N)


def sw(r):
    return ((r << 2) & 8) | (r & 4)


def blk(a, b):
    return BLK * (a * (a + 1) // 2 + b)


def el(a, b, r, c, swizzle=sw):
    return blk(a, b) + 16 * r + (c ^ swizzle(r))


def vbi(e):
    return e + ((e >> 5) << 4)


def wavefronts(addrs, width):
    """Shared-memory wavefronts of one warp-wide access: lanes are served in phases of
    32 / width lanes, and a phase takes as many wavefronts as the most distinct words that
    fall in one bank."""
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


def fragment_accesses(swizzle=sw):
    """(name, addresses, width) of every A / B fragment load and result store of the level
    products N_ab = -N_aa Diag(b_a) sum_k G_ak N_kb (16 x 8 halves)."""
    out = []
    for a in range(4):
        for b in range(a):
            for k in range(b, a + 1):
                for hh in range(2):
                    for ks in range(2):
                        for j in range(2):
                            for rh in range(2):
                                out.append(("A of G", [el(a, k, (l >> 2) + 8 * rh, 8 * ks + (l & 3) + 4 * j, swizzle)
                                                       for l in range(32)], 1))
                                out.append(("A of N_aa", [el(a, a, (l >> 2) + 8 * rh, 8 * ks + (l & 3) + 4 * j, swizzle)
                                                          for l in range(32)], 1))
                            out.append(("B of N", [el(k, b, 8 * ks + (l & 3) + 4 * j, 8 * hh + (l >> 2), swizzle)
                                                   for l in range(32)], 1))
            for hh in range(2):
                for rh in range(2):
                    out.append(("result store", [el(a, b, (l >> 2) + 8 * rh, 8 * hh + 2 * (l & 3), swizzle)
                                                 for l in range(32)], 2))
    return out


def test_every_element_has_its_own_word():
    words = set()
    for rec in range(2):
        for a in range(4):
            for b in range(a + 1):
                for r in range(16):
                    for c in range(16):
                        words.add(rec * TRI + el(a, b, r, c))
    assert len(words) == 2 * 10 * 256
    assert max(words) < 2 * TRI
    assert len({vbi(e) for e in range(64)}) == 64 and vbi(63) < 80


def test_vector_pieces_stay_contiguous_and_aligned():
    for r in range(16):
        for c in range(0, 16, 4):   # 16-byte pieces: gram row stores, solve reads, record loads
            phys = [x ^ sw(r) for x in range(c, c + 4)]
            assert phys == list(range(phys[0], phys[0] + 4)) and phys[0] % 4 == 0
        for c in range(0, 16, 2):   # 8-byte result stores
            assert (c ^ sw(r)) + 1 == ((c + 1) ^ sw(r))


def test_fragments_and_result_stores_are_conflict_free():
    for name, addrs, width in fragment_accesses():
        assert wavefronts(addrs, width) == {1: 1, 2: 2}[width], name


def test_row_accesses_are_conflict_free():
    for w in range(4):   # gram row stores: lanes < 16 of warp w store row `lane` of block row w
        for s4 in range(4 * (w + 1)):
            k, c = s4 >> 2, 4 * (s4 & 3)
            assert wavefronts([el(w, k, l, c) if l < 16 else None for l in range(32)], 4) == 2
    for a in range(4):   # diagonal solves: lanes 0-15 record 0, 16-31 record 1
        for rr in range(16):
            assert wavefronts([(l >> 4) * TRI + el(a, a, rr, l & 15) for l in range(32)], 1) == 1
            assert wavefronts([(l >> 4) * 80 + vbi(16 * a + rr) for l in range(32)], 1) == 1


def test_record_stage_is_conflict_free():
    for m in range(4):
        for w in range(4):
            for first in (True, False):
                an, ab = [], []
                for l in range(32):
                    e8 = 32 * w + l + 128 * m
                    tp, j = e8 >> 3, e8 & 7
                    a, r, b, c0 = tp >> 4, tp & 15, j >> 1, 8 * (j & 1)
                    h0 = 4 * ((b & 1) ^ ((sw(r) >> 2) & 1))
                    h = h0 if first else h0 ^ 4
                    an.append(TRI + el(a, b, r, c0 + h) if b <= a else None)
                    ab.append(80 + vbi(8 * j + h) if b <= a else None)
                assert wavefronts(an, 4) == 4
                assert wavefronts(ab, 4) <= 4


def sw128(row, byte):
    return row * 128 + (byte ^ ((row & 7) << 4))


def test_kda_tile_pass_is_conflict_free():
    """The KDA preparation's pass over a chunk: thread q takes the key channels 2 pc, 2 pc + 1
    (pc = q % 64) over the token half q / 64 and reads, then writes, their bf16 pair (one word)
    of the k tile and the three gated tiles, all 64 x 128 bf16 as two 128B-swizzled 64-channel
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


def test_planted_unswizzled_layout_conflicts():
    worst = max(wavefronts(addrs, width) - {1: 1, 2: 2}[width]
                for _, addrs, width in fragment_accesses(swizzle=lambda r: 0))
    assert worst > 0


# The kernel source this model was last checked against (code only; comments do not count).
MODELLED_SOURCE = ("build_gdn_prep.cu", "19a64ce16b42")


def test_model_is_checked_against_the_current_kernel_source():
    from tests.helpers import kernel_code_hash
    name, recorded = MODELLED_SOURCE
    assert kernel_code_hash(name) == recorded, (
        f"{name} changed since this model was checked against it: re-check the model "
        f"against the new code, then record the new hash {kernel_code_hash(name)}")
