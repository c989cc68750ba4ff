"""Test-side packer: codes -> MLX-affine words, written independently of the
oracle's bit reader (whole-integer shifts over one Python int per row)."""
import numpy as np


def pack_row(codes, bits):
    """Pack one row of codes low code first into little-endian uint32 words."""
    acc = 0
    for i, c in enumerate(codes):
        c = int(c)
        assert 0 <= c < (1 << bits)
        acc |= c << (i * bits)
    nbits = len(codes) * bits
    assert nbits % 32 == 0, "a row must end on a word"
    return np.array([(acc >> (32 * w)) & 0xFFFFFFFF for w in range(nbits // 32)], dtype=np.uint32)


def pack(codes2d, bits):
    return np.stack([pack_row(r, bits) for r in codes2d]).astype(np.uint32)


def row_bytes(words):
    return np.asarray(words, dtype=np.uint32).view(np.uint8)
