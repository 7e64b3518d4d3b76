"""The decode kernel reads E4M3 codes by integer operations alone: the code moved to the top byte,
shifted right arithmetically by 4 and masked with 0x87F00000 is an f32 whose value is the code's
times 2^-120 (the kernel multiplies 2^120 back per partial sum).  This host model of that rule,
for every byte position of a 32-bit word, must give the oracle's value for every finite code."""
import struct

import numpy as np

from oracle import moe_ffn as O


def _kernel_rule(word: int, k: int) -> float:
    x = (word << (24 - 8 * k)) & 0xFFFFFFFF
    xi = x - (1 << 32) if x & 0x80000000 else x          # the int view
    bits = (xi >> 4) & 0x87F00000                          # arithmetic shift, then the mask
    return struct.unpack("<f", struct.pack("<I", bits & 0xFFFFFFFF))[0] * 2.0 ** 120


def test_integer_decode_matches_the_format_for_every_finite_code():
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    ref = O.e4m3_to_float(np.array(codes, np.uint8))
    for k in range(4):
        for c, r in zip(codes, ref):
            neighbours = 0x5A5A5A5A & ~(0xFF << (8 * k))   # other bytes of the word must not leak in
            got = _kernel_rule(neighbours | (c << (8 * k)), k)
            assert got == r or (got == 0.0 and r == 0.0), (hex(c), k, got, r)
