"""Hand-built GGUF blocks with values known in closed form.

The bloomery pages name the block types the card experts use (Q4_K..Q6_K,
Q8_0: "bloomery README 0.3.1", Status table, "Quant types" row) but print no
block bytes and no worked example.  These blocks are built by hand from the
public GGUF layout, byte by byte, with a packer written here on its own (it
shares nothing with the synthetic-input encoder or the oracle), so that the
dequantized value of every weight is an exact small number.

Run as a script to (re)write q8_0_blocks.txt and q4_k_blocks.txt; the tests
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


def write_fixtures():
    hdr = ("# Hand-built {kind} blocks (GGUF layout); the bloomery pages print no block bytes,\n"
           "# so every expected value is the closed form stated in tests/golden/blocks.py.\n"
           "# format: <name> <hex bytes>\n")
    for kind, cases in (("Q8_0", q8_0_cases()), ("Q4_K", q4_k_cases())):
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
