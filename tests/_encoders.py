"""Independent encoders for the tests: known fields -> GGUF Q4_K / Q6_K block bytes (the inverse
of the public GGUF layouts), plus f16 bit helpers. They share nothing with the oracle's decoders
or the CUDA library; tests use them to build blocks whose decoded values are known by hand."""
import numpy as np


def f16_bits(x: float) -> int:
    return int(np.array([x], np.float16).view(np.uint16)[0])


def f16_val(bits: int) -> float:
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def encode_q4k(d_bits, dmin_bits, sc, mn, q):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([d_bits], np.uint16).view(np.uint8)
    blk[2:4] = np.array([dmin_bits], np.uint16).view(np.uint8)
    s = np.zeros(12, np.int64)
    for j in range(8):
        if j < 4:
            s[j] |= sc[j] & 63
            s[j + 4] |= mn[j] & 63
        else:
            s[j + 4] |= (sc[j] & 15) | ((mn[j] & 15) << 4)
            s[j - 4] |= (sc[j] >> 4) << 6
            s[j] |= (mn[j] >> 4) << 6
    blk[4:16] = s.astype(np.uint8)
    for c in range(4):
        for l in range(32):
            blk[16 + 32 * c + l] = (q[64 * c + l] & 15) | ((q[64 * c + 32 + l] & 15) << 4)
    return blk


def encode_q6k(d_bits, sc, q):
    blk = np.zeros(210, np.uint8)
    for i in range(256):
        h, t, l = i // 128, (i % 128) // 32, i % 32
        lo, hi = q[i] & 15, (q[i] >> 4) & 3
        idx = 64 * h + l + 32 * (t & 1)
        blk[idx] |= lo if t < 2 else (lo << 4)
        blk[128 + 32 * h + l] |= hi << (2 * t)
    blk[192:208] = np.array(sc, np.int8).view(np.uint8)
    blk[208:210] = np.array([d_bits], np.uint16).view(np.uint8)
    return blk


