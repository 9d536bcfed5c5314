"""Bit-position reader for k-quant blocks, used to pin the oracle's decoder.

Written independently of oracle/kq_oracle.c from the same layout description,
but as positions in one little-endian bit string per field rather than byte
loops, and vectorised over many blocks with numpy.  Returns integer fields only
(no floating point), so a wrong byte index, shift or mask in either decoder
shows up as a mismatch.
"""
import numpy as np


def _bits(field: np.ndarray, start: int, width: int) -> np.ndarray:
    """Bits [start, start+width) of each row of ``field`` read as a little-endian bit string."""
    bits = np.unpackbits(field, axis=1, bitorder="little")
    w = 1 << np.arange(width, dtype=np.int64)
    return (bits[:, start:start + width].astype(np.int64) * w).sum(axis=1)


def q4k_like(blocks: np.ndarray, five_bit: bool):
    """Fields of Q4_K (five_bit False) or Q5_K blocks: d, dmin bits, sc[8], m[8], q[256]."""
    blocks = np.atleast_2d(blocks)
    d = _bits(blocks[:, 0:2], 0, 16)
    dmin = _bits(blocks[:, 2:4], 0, 16)
    s = blocks[:, 4:16]
    sc = np.zeros((len(blocks), 8), np.int64)
    m = np.zeros((len(blocks), 8), np.int64)
    for j in range(8):
        if j < 4:
            sc[:, j] = _bits(s, 8 * j, 6)
            m[:, j] = _bits(s, 8 * (j + 4), 6)
        else:
            sc[:, j] = _bits(s, 8 * (j + 4), 4) | (_bits(s, 8 * (j - 4) + 6, 2) << 4)
            m[:, j] = _bits(s, 8 * (j + 4) + 4, 4) | (_bits(s, 8 * j + 6, 2) << 4)
    qs = blocks[:, 48:176] if five_bit else blocks[:, 16:144]
    qh = blocks[:, 16:48]
    q = np.zeros((len(blocks), 256), np.int64)
    for i in range(256):
        g, r = divmod(i, 64)
        half, l = divmod(r, 32)
        q[:, i] = _bits(qs, (32 * g + l) * 8 + 4 * half, 4)
        if five_bit:
            q[:, i] |= _bits(qh, 8 * l + 2 * g + half, 1) << 4
    return d, dmin, sc, m, q


def q6k(blocks: np.ndarray):
    """Fields of Q6_K blocks: d bits, sc[16] (signed), q[256] (0..63, unbiased)."""
    blocks = np.atleast_2d(blocks)
    ql, qh = blocks[:, 0:128], blocks[:, 128:192]
    sc = blocks[:, 192:208].view(np.int8).astype(np.int64)
    d = _bits(blocks[:, 208:210], 0, 16)
    q = np.zeros((len(blocks), 256), np.int64)
    for i in range(256):
        h, r = divmod(i, 128)
        t, l = divmod(r, 32)
        low = _bits(ql, (64 * h + 32 * (t % 2) + l) * 8 + 4 * (t // 2), 4)
        high = _bits(qh, (32 * h + l) * 8 + 2 * t, 2)
        q[:, i] = low | (high << 4)
    return d, sc, q


def dequant_f64(qtype: int, blocks: np.ndarray) -> np.ndarray:
    """Dequantized weights (n_blocks, 256) in float64 from the bit reader's fields,
    with d/dmin decoded by numpy's float16."""
    def h(bits):
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if qtype == 3:
        d, sc, q = q6k(blocks)
        return h(d)[:, None] * np.repeat(sc, 16, axis=1) * (q - 32)
    d, dmin, sc, m, q = q4k_like(blocks, five_bit=(qtype == 2))
    return (h(d)[:, None] * np.repeat(sc, 32, axis=1) * q
            - h(dmin)[:, None] * np.repeat(m, 32, axis=1))
