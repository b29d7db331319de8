"""The shifted vector loads of the chunked draw, checked on a model.

On a row that is not 16-byte aligned the chunked draw reads each 32-byte
group through the aligned 16-byte vectors that overlap it (three vectors, or
two when the group happens to be aligned) and moves the wanted words into
place: ws = mis >> 2 whole words, then a 16-bit funnel shift when the offset
is 2 mod 4 (bf16 rows).  The model repeats that word arithmetic on a random
byte buffer, little-endian as on the GPU, and checks that

* every group at every 2-byte aligned address comes out as the bytes there;
* every vector the kernel reads overlaps the group, so no read reaches past
  the aligned 16-byte granules that hold the group's bytes (an aligned
  16-byte vector never straddles a page);
* the select never indexes past the words loaded.

A planted error (a funnel shift of 8 bits instead of 16) must fail the model.
"""
import numpy as np

MASK = 0xFFFFFFFF


def funnel_r(lo, hi, sh):
    return ((hi << 32 | lo) >> (sh & 31)) & MASK


def shifted_group(buf, addr, half_shift=16):
    """The model of the kernel's load of the 32 bytes at ``addr``: returns the
    8 words and the byte ranges of the vectors it read."""
    mis = addr & 15
    base = addr - mis
    nvec = 3 if mis else 2
    reads = [(base + 16 * k, base + 16 * k + 16) for k in range(nvec)]
    w = [int.from_bytes(bytes(buf[base + 4 * j: base + 4 * j + 4]), "little")
         for j in range(4 * nvec)] + [0] * (12 - 4 * nvec)
    ws, hs = mis >> 2, (half_shift if mis & 2 else 0)
    assert ws + 8 <= 11, "select past the loaded words"
    d = [w[j + ws] for j in range(9)]
    return [funnel_r(d[j], d[j + 1], hs) for j in range(8)], reads


def _check(half_shift):
    rng = np.random.default_rng(7)
    buf = rng.integers(0, 256, size=2048, dtype=np.uint8)
    wrong = 0
    for addr in range(0, 2048 - 48, 2):
        got, reads = shifted_group(buf, addr, half_shift)
        want = [int.from_bytes(bytes(buf[addr + 4 * j: addr + 4 * j + 4]), "little")
                for j in range(8)]
        wrong += got != want
        for lo, hi in reads:
            assert lo < addr + 32 and hi > addr, (addr, lo, hi)
    return wrong


def test_shifted_groups_are_the_bytes_at_every_offset():
    assert _check(16) == 0


def test_the_model_detects_a_wrong_half_word_shift():
    assert _check(8) > 0


# --- the top-k draw's single-vector form --------------------------------------
# On a row that is not 16-byte aligned the top-k draw reads vector vi (16
# bytes at row + 16 vi, element vi * kN < V) through the aligned vector that
# holds its first byte and, only when it still holds a byte of the row, the
# next one; the words are moved into place the same way, and the elements at
# or past V are cleared.


def shifted_vec(buf, row, vi, V, es, half_shift=16):
    kN = 16 // es
    a = row + 16 * vi
    end = row + V * es
    mis = a & 15
    base = a - mis
    reads = [(base, base + 16)]
    w = [int.from_bytes(bytes(buf[base + 4 * j: base + 4 * j + 4]), "little") for j in range(4)]
    if base + 16 < end:
        reads.append((base + 16, base + 32))
        w += [int.from_bytes(bytes(buf[base + 16 + 4 * j: base + 20 + 4 * j]), "little")
              for j in range(4)]
    else:
        w += [0] * 4
    ws, hs = mis >> 2, (half_shift if mis & 2 else 0)
    d = [w[j + ws] for j in range(5)]
    o = [funnel_r(d[j], d[j + 1], hs) for j in range(4)]
    n = V - vi * kN
    for e in range(n, kN):
        if es == 4:
            o[e] = 0
        else:
            o[e >> 1] &= 0x0000FFFF if e & 1 else 0xFFFF0000
    return o, reads


def _check_vec(half_shift):
    rng = np.random.default_rng(11)
    buf = rng.integers(0, 256, size=4096, dtype=np.uint8)
    wrong = 0
    for es in (2, 4):
        kN = 16 // es
        for mis in range(es, 16, es):              # every unaligned row start
            for V in (1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 40):
                row = 1024 + mis
                end = row + V * es
                for vi in range(-(-V // kN)):
                    got, reads = shifted_vec(buf, row, vi, V, es, half_shift)
                    a = row + 16 * vi
                    want = bytearray(buf[a: a + 16])
                    for e in range(V - vi * kN, kN):    # elements past V read as zero
                        want[e * es: e * es + es] = bytes(es)
                    want = [int.from_bytes(bytes(want[4 * j: 4 * j + 4]), "little") for j in range(4)]
                    wrong += got != want
                    for lo, hi in reads:                 # every read holds a byte of the row
                        assert lo < end and hi > row, (es, mis, V, vi, lo, hi)
    return wrong


def test_topk_shifted_vectors_are_the_row_bytes():
    assert _check_vec(16) == 0


def test_topk_vector_model_detects_a_wrong_half_word_shift():
    assert _check_vec(8) > 0
