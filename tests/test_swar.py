"""The digest byte match used by the kernels (common.cuh byte_match4) must
flag every byte equal to the digest: it may flag a few extra bytes (a key
compare rejects those), never miss one.  Checked exhaustively over byte
pairs below a matching byte and on random words (host mirror of the
arithmetic: zero-byte flags of w ^ pattern, gathered by one multiply)."""
import random

M = 0xFFFFFFFF


def zero_byte_flags(x):
    return ((x - 0x01010101) & M) & (~x & M) & 0x80808080


def byte_match4(w, pat):
    return ((zero_byte_flags(w ^ pat) * 0x00204081) & M) >> 28


def exact(w, pat):
    return sum(1 << i for i in range(4) if ((w >> (8 * i)) & 255) == ((pat >> (8 * i)) & 255))


def test_never_misses_an_equal_byte_exhaustive_pairs():
    for d in range(256):
        pat = d * 0x01010101
        for lo in range(256):
            for hi in (d, d ^ 1, (d + 1) & 255, lo):
                w = lo | (hi << 8) | (d << 16) | (lo << 24)
                assert exact(w, pat) & ~byte_match4(w, pat) == 0


def test_never_misses_random_words():
    rng = random.Random(7)
    for _ in range(50000):
        d = rng.randrange(256)
        pat = d * 0x01010101
        w = sum(rng.choice([d, d ^ 1, rng.randrange(256)]) << (8 * i) for i in range(4))
        assert exact(w, pat) & ~byte_match4(w, pat) == 0
