"""Independent Q4_K superblock packer for tests, written from the format text in
include/spec_verify.h (canonical layout).  It shares nothing with the oracle's
decoder: it builds bytes from explicit fields so the decoder can be checked.

  bytes 0..1 d, 2..3 dmin (binary16 little endian)
  bytes 4..15 96-bit little-endian field: sc_j at bits 6j.., m_j at bits 48+6j..
  bytes 16..143: element e of sub-block j=e//32, r=e%32 in byte 16+16j+(r%16),
                 low nibble when r < 16, high nibble otherwise.
"""
import numpy as np


def half_bits(x: float) -> int:
    return int(np.array([x], dtype=np.float16).view(np.uint16)[0])


def pack_superblock(d: float, dmin: float, sc, m, codes) -> np.ndarray:
    assert len(sc) == 8 and len(m) == 8 and len(codes) == 256
    out = np.zeros(144, dtype=np.uint8)
    hd, hm = half_bits(d), half_bits(dmin)
    out[0], out[1] = hd & 0xFF, hd >> 8
    out[2], out[3] = hm & 0xFF, hm >> 8
    field = 0
    for j in range(8):
        assert 0 <= sc[j] < 64 and 0 <= m[j] < 64
        field |= int(sc[j]) << (6 * j)
        field |= int(m[j]) << (48 + 6 * j)
    for i in range(12):
        out[4 + i] = (field >> (8 * i)) & 0xFF
    for e in range(256):
        q = int(codes[e])
        assert 0 <= q < 16
        j, r = divmod(e, 32)
        byte = 16 + 16 * j + (r % 16)
        if r < 16:
            out[byte] |= q
        else:
            out[byte] |= q << 4
    return out


def dequant_fields(d: float, dmin: float, sc, m, codes) -> np.ndarray:
    """w_e = d*sc_j*q_e - dmin*m_j in fp64 from the fields (d, dmin as stored fp16)."""
    d = float(np.float16(d))
    dmin = float(np.float16(dmin))
    return np.array([d * sc[e // 32] * codes[e] - dmin * m[e // 32] for e in range(256)])
