"""Hand-built GGUF blocks with values known in closed form.

The bloomery pages name the block types the card experts use (Q4_K..Q6_K,
Q8_0, MXFP4, and the Q3_K_M files of the large model: "bloomery README
0.3.1", Status table, "Quant types" row) but print no
block bytes and no worked example.  These blocks are built by hand from the
public GGUF layout, byte by byte, with a packer written here on its own (it
shares nothing with the synthetic-input encoder or the oracle), so that the
dequantized value of every weight is an exact small number.

Run as a script to (re)write the <type>_blocks.txt fixtures; the tests
read those text fixtures and also rebuild the bytes here to check them.
"""
from __future__ import annotations

import os
import struct

HERE = os.path.dirname(os.path.abspath(__file__))


def fp16_bytes(bits: int) -> bytes:
    return struct.pack("<H", bits)


# ---------------------------------------------------------------- Q8_0 (34 B / 32)

def q8_0_block(d_bits: int, q: list[int]) -> bytes:
    assert len(q) == 32 and all(-128 <= v <= 127 for v in q)
    return fp16_bytes(d_bits) + bytes((v + 256) % 256 for v in q)


def q8_0_cases():
    """name -> (bytes, expected weights as exact fractions given by a lambda)."""
    return {
        # d = 0.25 (0x3400), q_i = i - 16  ->  w_i = (i - 16) / 4
        "ramp": (q8_0_block(0x3400, [i - 16 for i in range(32)]),
                 [(i - 16) * 0.25 for i in range(32)]),
        # the int8 extremes with d = 1: -128 and 127 alternate
        "extremes": (q8_0_block(0x3C00, [-128 if i % 2 else 127 for i in range(32)]),
                     [-128.0 if i % 2 else 127.0 for i in range(32)]),
        # d = 0 gives zeros whatever q is
        "zero_scale": (q8_0_block(0x0000, [i - 7 for i in range(32)]), [0.0] * 32),
        # smallest fp16 subnormal d = 2^-24
        "subnormal_scale": (q8_0_block(0x0001, [i - 16 for i in range(32)]),
                            [(i - 16) * 2.0 ** -24 for i in range(32)]),
        # negative scale d = -2 (0xC000)
        "negative_scale": (q8_0_block(0xC000, [3] * 16 + [-5] * 16), [-6.0] * 16 + [10.0] * 16),
    }


# ---------------------------------------------------------------- Q4_K (144 B / 256)

def q4_k_block(d_bits: int, dmin_bits: int, sc: list[int], m: list[int], q: list[int]) -> bytes:
    """One super-block: fp16 d, fp16 dmin, 12 scale bytes, 128 quant bytes.

    Scale bytes, written out one by one:
      bytes 0..3  : sc[0..3] in bits 0-5, bits 4-5 of sc[4..7] in bits 6-7
      bytes 4..7  : m[0..3]  in bits 0-5, bits 4-5 of m[4..7]  in bits 6-7
      bytes 8..11 : bits 0-3 of sc[4..7] in the low nibble, of m[4..7] in the high
    Quant bytes: 32*c + i holds q[64c + i] low and q[64c + 32 + i] high.
    """
    assert len(sc) == 8 and len(m) == 8 and len(q) == 256
    S = bytearray(12)
    for j in range(4):
        S[j] = (sc[j] & 0x3F) | (((sc[j + 4] >> 4) & 0x3) << 6)
        S[j + 4] = (m[j] & 0x3F) | (((m[j + 4] >> 4) & 0x3) << 6)
        S[j + 8] = (sc[j + 4] & 0xF) | ((m[j + 4] & 0xF) << 4)
    Q = bytearray(128)
    for c in range(4):
        for i in range(32):
            Q[32 * c + i] = (q[64 * c + i] & 0xF) | ((q[64 * c + 32 + i] & 0xF) << 4)
    return fp16_bytes(d_bits) + fp16_bytes(dmin_bits) + bytes(S) + bytes(Q)


def q4_k_cases():
    cases = {}
    # d = 1, dmin = 0.5, sc_j = j+1, m_j = 2j, q = i mod 16 (i = index in the block)
    #   -> w = (j+1) * (i mod 16) - j   (exact small integers)
    sc = [j + 1 for j in range(8)]
    m = [2 * j for j in range(8)]
    q = [i % 16 for i in range(256)]
    exp = [(i // 32 + 1) * (i % 16) - (i // 32) for i in range(256)]
    cases["ladder"] = (q4_k_block(0x3C00, 0x3800, sc, m, q), [float(v) for v in exp])
    # every field at its maximum: sc = m = 63, q = 15, d = 1, dmin = 1 -> w = 63*15 - 63 = 882
    cases["all_max"] = (q4_k_block(0x3C00, 0x3C00, [63] * 8, [63] * 8, [15] * 256), [882.0] * 256)
    # high bits only: sc = m = 48 (0b110000) for j >= 4, 0 elsewhere; q = 1
    #   -> w = 48 - 48 = 0 for j >= 4 would hide them, so use dmin = 0.5: 48 - 24 = 24
    scs = [0, 0, 0, 0, 48, 48, 48, 48]
    ms = [0, 0, 0, 0, 48, 48, 48, 48]
    cases["high_bits"] = (q4_k_block(0x3C00, 0x3800, scs, ms, [1] * 256),
                          [0.0] * 128 + [24.0] * 128)
    # distinct high bits in every scale and min: w = 2*sc_j - m_j/4
    scm = [1, 2, 3, 4, 17, 33, 49, 63]
    mm = [5, 6, 7, 8, 60, 44, 28, 12]
    cases["mixed_fields"] = (q4_k_block(0x3C00, 0x3400, scm, mm, [2] * 256),
                             [2.0 * scm[i // 32] - 0.25 * mm[i // 32] for i in range(256)])
    # one sub-block at a time: only sub-block j has sc = 1 and q = 7 (others sc = 0, q = 15)
    for j in range(8):
        scj = [1 if jj == j else 0 for jj in range(8)]
        qj = [7 if i // 32 == j else 15 for i in range(256)]
        expj = [7.0 if i // 32 == j else 0.0 for i in range(256)]
        cases[f"only_sub{j}"] = (q4_k_block(0x3C00, 0x0000, scj, [0] * 8, qj), expj)
    # low vs high nibble: q = 3 in even sub-blocks, 12 in odd ones, sc = 1, d = 0.5
    qn = [3 if (i // 32) % 2 == 0 else 12 for i in range(256)]
    cases["nibbles"] = (q4_k_block(0x3800, 0x0000, [1] * 8, [0] * 8, qn),
                        [1.5 if (i // 32) % 2 == 0 else 6.0 for i in range(256)])
    return cases


# ---------------------------------------------------------------- Q5_K (176 B / 256)

def q5_k_block(d_bits: int, dmin_bits: int, sc: list[int], m: list[int], q: list[int]) -> bytes:
    """One super-block: the 16 header bytes of Q4_K (d, dmin, packed scales and mins), then
    32 bytes whose bit j of byte i is bit 4 of q[32j + i], then the low nibbles of q laid
    out as the Q4_K quant bytes."""
    assert len(q) == 256 and all(0 <= v < 32 for v in q)
    head = q4_k_block(d_bits, dmin_bits, sc, m, [v & 0xF for v in q])
    QH = bytearray(32)
    for j in range(8):
        for i in range(32):
            if q[32 * j + i] & 0x10:
                QH[i] |= 1 << j
    return head[:16] + bytes(QH) + head[16:]


def q5_k_cases():
    cases = {}
    # d = 1, dmin = 0.5, sc_j = j+1, m_j = 2j, q = i mod 32  ->  w = (j+1)(i mod 32) - j
    sc = [j + 1 for j in range(8)]
    m = [2 * j for j in range(8)]
    cases["ladder"] = (q5_k_block(0x3C00, 0x3800, sc, m, [i % 32 for i in range(256)]),
                       [float((i // 32 + 1) * (i % 32) - (i // 32)) for i in range(256)])
    # every field at its maximum: 63 * 31 - 63
    cases["all_max"] = (q5_k_block(0x3C00, 0x3C00, [63] * 8, [63] * 8, [31] * 256), [1890.0] * 256)
    # the fifth bit alone, in a pattern that shifts from sub-block to sub-block: q = 16 or 0
    qf = [16 if (i % 32 + i // 32) % 3 == 0 else 0 for i in range(256)]
    cases["fifth_bit"] = (q5_k_block(0x3C00, 0x0000, [1] * 8, [0] * 8, qf), [float(v) for v in qf])
    # one sub-block at a time: sc = 1 and q = 23 (fifth bit set) there; sc = 0 and q = 15
    # (fifth bit clear) elsewhere
    for j in range(8):
        scj = [1 if jj == j else 0 for jj in range(8)]
        qj = [23 if i // 32 == j else 15 for i in range(256)]
        cases[f"only_sub{j}"] = (q5_k_block(0x3C00, 0x0000, scj, [0] * 8, qj),
                                 [23.0 if i // 32 == j else 0.0 for i in range(256)])
    # distinct high bits in every scale and min, q = 17: w = 17/2 sc_j - m_j/4
    scm = [1, 2, 3, 4, 17, 33, 49, 63]
    mm = [5, 6, 7, 8, 60, 44, 28, 12]
    cases["mixed_fields"] = (q5_k_block(0x3800, 0x3400, scm, mm, [17] * 256),
                             [8.5 * scm[i // 32] - 0.25 * mm[i // 32] for i in range(256)])
    return cases


# ---------------------------------------------------------------- Q6_K (210 B / 256)

def q6_k_block(d_bits: int, scales: list[int], q: list[int]) -> bytes:
    """One super-block from signed quants q[256] in [-32, 31] and int8 scales[16].

    Written byte by byte: for half h (weights 128h..128h+127) and quarter r, weight
    128h + 32r + l stores u = q + 32 (6 bits) as
      low 4 bits  -> byte 64h + 32(r % 2) + l of the first 128 bytes,
                     low nibble when r < 2, high nibble when r >= 2;
      high 2 bits -> bits 2r..2r+1 of byte 128 + 32h + l;
    then 16 scale bytes (two's complement), then fp16 d."""
    assert len(q) == 256 and all(-32 <= v < 32 for v in q)
    assert len(scales) == 16 and all(-128 <= v < 128 for v in scales)
    QL = bytearray(128)
    QH = bytearray(64)
    for h in range(2):
        for r in range(4):
            for l in range(32):
                u = q[128 * h + 32 * r + l] + 32
                at = 64 * h + 32 * (r % 2) + l
                QL[at] |= (u & 0xF) << (0 if r < 2 else 4)
                QH[32 * h + l] |= (u >> 4) << (2 * r)
    return bytes(QL) + bytes(QH) + bytes((v + 256) % 256 for v in scales) + fp16_bytes(d_bits)


def q6_k_cases():
    cases = {}
    # d = 0.5, scale of group g = 2g - 15 (odd, never 0), q a permutation of [-32, 31] per 64
    sg = [2 * g - 15 for g in range(16)]
    qp = [(37 * i) % 64 - 32 for i in range(256)]
    cases["ladder"] = (q6_k_block(0x3800, sg, qp), [0.5 * sg[i // 16] * qp[i] for i in range(256)])
    # extremes of q and of the int8 scale
    se = [127 if g % 2 == 0 else -128 for g in range(16)]
    qe = [31 if i % 2 == 0 else -32 for i in range(256)]
    cases["extremes"] = (q6_k_block(0x3C00, se, qe), [float(se[i // 16] * qe[i]) for i in range(256)])
    # one quarter of one half at a time: q = 5 there, 0 (stored 32) elsewhere, scale 1
    for h in range(2):
        for r in range(4):
            sel = [(i // 128 == h and (i % 128) // 32 == r) for i in range(256)]
            cases[f"only_h{h}_r{r}"] = (q6_k_block(0x3C00, [1] * 16, [5 if t else 0 for t in sel]),
                                        [5.0 if t else 0.0 for t in sel])
    # the high pairs alone: q = 16a - 32 with a = (i // 32) % 4 cycling per quarter
    qh = [16 * ((i // 32 + i // 128) % 4) - 32 for i in range(256)]
    cases["high_pairs"] = (q6_k_block(0x3C00, [1] * 16, qh), [float(v) for v in qh])
    return cases


# ---------------------------------------------------------------- Q3_K (110 B / 256)

def q3_k_block(d_bits: int, scales: list[int], q: list[int]) -> bytes:
    """One super-block from signed quants q[256] in [-4, 3] and scales[16] in [-32, 31].

    Written byte by byte: weight 128h + 32r + l stores v = q + 4 as
      bit 2 of v (the "high" bit) -> bit 4h + r of byte l (the first 32 bytes),
      bits 0-1 of v               -> bits 2r..2r+1 of byte 32 + 32h + l;
    scale j is stored as s = scales[j] + 32 (6 bits):
      bits 0-3 -> low nibble of byte 96 + j (j < 8), high nibble of byte 96 + j - 8 (j >= 8),
      bits 4-5 -> bits 2(j // 4)..2(j // 4)+1 of byte 104 + j % 4;
    then fp16 d."""
    assert len(q) == 256 and all(-4 <= v < 4 for v in q)
    assert len(scales) == 16 and all(-32 <= v < 32 for v in scales)
    HM = bytearray(32)
    QS = bytearray(64)
    for h in range(2):
        for r in range(4):
            for l in range(32):
                v = q[128 * h + 32 * r + l] + 4
                if v & 4:
                    HM[l] |= 1 << (4 * h + r)
                QS[32 * h + l] |= (v & 3) << (2 * r)
    S = bytearray(12)
    for j in range(16):
        s = scales[j] + 32
        if j < 8:
            S[j] |= s & 0xF
        else:
            S[j - 8] |= (s & 0xF) << 4
        S[8 + j % 4] |= ((s >> 4) & 3) << (2 * (j // 4))
    return bytes(HM) + bytes(QS) + bytes(S) + fp16_bytes(d_bits)


def q3_k_cases():
    cases = {}
    # d = 0.25, scale of group g = 2g - 15, q = i mod 8 - 4
    sg = [2 * g - 15 for g in range(16)]
    cases["ladder"] = (q3_k_block(0x3400, sg, [i % 8 - 4 for i in range(256)]),
                       [0.25 * sg[i // 16] * (i % 8 - 4) for i in range(256)])
    # extremes: scales -32 / 31, q -4 / 3
    se = [-32 if g % 2 == 0 else 31 for g in range(16)]
    qe = [-4 if i % 3 == 0 else 3 for i in range(256)]
    cases["extremes"] = (q3_k_block(0x3C00, se, qe), [float(se[i // 16] * qe[i]) for i in range(256)])
    # every bit of every stored scale: s + 32 takes these 6-bit values, q = 1
    raw = [1, 2, 4, 8, 16, 32, 48, 63, 0, 17, 34, 51, 5, 10, 20, 40]
    cases["scale_bits"] = (q3_k_block(0x3C00, [v - 32 for v in raw], [1] * 256),
                           [float(raw[i // 16] - 32) for i in range(256)])
    # one quarter of one half at a time: q = -4 (high bit clear) there, 0 (high bit set) elsewhere
    for h in range(2):
        for r in range(4):
            sel = [(i // 128 == h and (i % 128) // 32 == r) for i in range(256)]
            cases[f"only_h{h}_r{r}"] = (q3_k_block(0x3C00, [1] * 16, [-4 if t else 0 for t in sel]),
                                        [-4.0 if t else 0.0 for t in sel])
    # the low parts alone with every high bit set: q = (i // 32 + i) % 4
    ql = [(i // 32 + i) % 4 for i in range(256)]
    cases["low_parts"] = (q3_k_block(0x3C00, [1] * 16, ql), [float(v) for v in ql])
    return cases


# ---------------------------------------------------------------- MXFP4 (17 B / 32)

# FP4 E2M1 magnitudes of codes 0..7, as listed by the OCP Microscaling formats specification;
# codes 8..15 are the same magnitudes negated.
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1_value(code: int) -> float:
    v = E2M1[code & 7]
    return -v if code & 8 else v


def mxfp4_block(e: int, codes: list[int]) -> bytes:
    """One block: the E8M0 scale byte e, then byte j = codes[j] | codes[j + 16] << 4."""
    assert 0 <= e < 256 and len(codes) == 32 and all(0 <= c < 16 for c in codes)
    return bytes([e]) + bytes(codes[j] | (codes[j + 16] << 4) for j in range(16))


def mxfp4_cases():
    cases = {}
    # every code once in each half, the second half reversed: element order is visible
    codes = [i for i in range(16)] + [15 - i for i in range(16)]
    vals = [e2m1_value(c) for c in codes]
    cases["codes_scale1"] = (mxfp4_block(127, codes), vals)
    cases["codes_scale8"] = (mxfp4_block(130, codes), [8.0 * v for v in vals])
    cases["codes_scale_2^-27"] = (mxfp4_block(100, codes), [v * 2.0 ** -27 for v in vals])
    cases["codes_min_scale"] = (mxfp4_block(0, codes), [v * 2.0 ** -127 for v in vals])
    cases["codes_max_scale"] = (mxfp4_block(254, codes), [v * 2.0 ** 127 for v in vals])
    # low and high nibbles of each byte differ: 0.5 in the first half, -6 in the second
    cases["halves"] = (mxfp4_block(127, [1] * 16 + [15] * 16), [0.5] * 16 + [-6.0] * 16)
    # e = 255 is not a number; every element decodes to NaN
    cases["nan_scale"] = (mxfp4_block(255, codes), [float("nan")] * 32)
    return cases


BLOCK_TYPES = {
    # name -> (weights per block, bytes per block, cases)
    "Q8_0": (32, 34, q8_0_cases),
    "Q4_K": (256, 144, q4_k_cases),
    "Q5_K": (256, 176, q5_k_cases),
    "Q6_K": (256, 210, q6_k_cases),
    "Q3_K": (256, 110, q3_k_cases),
    "MXFP4": (32, 17, mxfp4_cases),
}


def write_fixtures():
    hdr = ("# Hand-built {kind} blocks (GGUF layout); the bloomery pages print no block bytes,\n"
           "# so every expected value is the closed form stated in tests/golden/blocks.py.\n"
           "# format: <name> <hex bytes>\n")
    for kind, (_, _, make) in BLOCK_TYPES.items():
        cases = make()
        path = os.path.join(HERE, f"{kind.lower()}_blocks.txt")
        with open(path, "w") as f:
            f.write(hdr.format(kind=kind))
            for name, (blk, _) in cases.items():
                f.write(f"{name} {blk.hex()}\n")


def read_fixture(kind: str) -> dict[str, bytes]:
    path = os.path.join(HERE, f"{kind.lower()}_blocks.txt")
    out = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, hx = line.split()
            out[name] = bytes.fromhex(hx)
    return out


if __name__ == "__main__":
    write_fixtures()
