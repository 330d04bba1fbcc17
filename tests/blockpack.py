"""Test-side block encoders, written from the GGUF layout description.

They turn explicit fields (f16 scales, integer sub-block scales/mins, codes)
into canonical block bytes so the pins can build blocks with known contents.
Independent of the oracle (no shared code) and of the CUDA library.
"""
import numpy as np


def f16(v):
    return np.array([v], dtype=np.float16).view(np.uint8)


def pack_q4_k(d, dmin, sc, mn, codes):
    """sc, mn: 8 ints in 0..63; codes: 256 ints in 0..15 -> 144 bytes."""
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = f16(d)
    b[2:4] = f16(dmin)
    s = np.zeros(12, dtype=np.int64)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    b[4:16] = s.astype(np.uint8)
    for c in range(4):
        for l in range(32):
            lo = codes[64 * c + l]
            hi = codes[64 * c + 32 + l]
            b[16 + 32 * c + l] = lo | (hi << 4)
    return b


def pack_q5_k(d, dmin, sc, mn, codes):
    """sc, mn: 8 ints in 0..63; codes: 256 ints in 0..31 -> 176 bytes (header as Q4_K, then 32 high-bit
    bytes -- element 64c + l takes bit 2c of byte l, element 64c + 32 + l bit 2c + 1 -- then the low
    nibbles in the Q4_K arrangement)."""
    q4 = pack_q4_k(d, dmin, sc, mn, [c & 15 for c in codes])
    b = np.zeros(176, dtype=np.uint8)
    b[0:16] = q4[0:16]
    for c in range(4):
        for l in range(32):
            b[16 + l] |= ((codes[64 * c + l] >> 4) & 1) << (2 * c)
            b[16 + l] |= ((codes[64 * c + 32 + l] >> 4) & 1) << (2 * c + 1)
    b[48:176] = q4[16:144]
    return b


def pack_q6_k(d, sc, codes):
    """sc: 16 ints in -128..127; codes: 256 ints in 0..63 -> 210 bytes."""
    b = np.zeros(210, dtype=np.uint8)
    for h in range(2):
        for l in range(32):
            c = [codes[128 * h + l + 32 * q] for q in range(4)]
            b[64 * h + l] = (c[0] & 15) | ((c[2] & 15) << 4)
            b[64 * h + l + 32] = (c[1] & 15) | ((c[3] & 15) << 4)
            b[128 + 32 * h + l] = (c[0] >> 4) | ((c[1] >> 4) << 2) | ((c[2] >> 4) << 4) | ((c[3] >> 4) << 6)
    b[192:208] = np.array(sc, dtype=np.int64).astype(np.int8).view(np.uint8)
    b[208:210] = f16(d)
    return b


def pack_q8_0(d, w):
    b = np.zeros(34, dtype=np.uint8)
    b[0:2] = f16(d)
    b[2:34] = np.array(w, dtype=np.int64).astype(np.int8).view(np.uint8)
    return b


def parse_fixture(path, block_bytes):
    """Yield (name, block bytes, {index: value}, rest) from a hand-derived fixture."""
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, sets, expect = [p.strip() for p in line.split("|")]
            blk = np.zeros(block_bytes, dtype=np.uint8)
            for tok in sets.split():
                off, val = tok.split("=")
                blk[int(off)] = int(val, 16)
            exp = {}
            for tok in expect.split():
                idx, val = tok.split("=")
                if ".." in idx:
                    lo, hi = idx.split("..")
                    for i in range(int(lo), int(hi) + 1):
                        exp[i] = float(val)
                else:
                    exp[int(idx)] = float(val)
            yield name, blk, exp
