"""Hand-assembles the payload fixtures in ``decode_fixtures.txt``.

This script calls nothing from the oracle or the library.  It places each field of a block at the
bit position the format layout gives (bit p of a block is bit p % 8 of byte p // 8, so multi-byte
words are little-endian) using a generic bit writer, from a per-format table of
(field, index, bit offset, width).  The fixture stores the field values next to the bytes; the tests
recompute the expected decoded values from the fields and compare them with both decoders.

Field values are seeded draws.  The layout follows the format descriptions of PR #2513
("IQ2_XXS packs a 4-bit sub-block scale into the same 32-bit word as four 7-bit sign indices";
IQ2_S "a full eight-bit sign mask per group"; IQ1_M "the FP16 super-block scale is reassembled from
the top nibble of each of four scale words", a local scale per two groups and a delta per group),
with the remaining bit order fixed by this library's header.

Run:  python tests/golden/make_decode_fixtures.py  (rewrites decode_fixtures.txt)
"""
import os

import numpy as np

BLOCK_BYTES = {"IQ2_XXS": 66, "IQ2_XS": 74, "IQ2_S": 82, "IQ1_S": 50, "IQ1_M": 56}


def layout(fmt):
    """(field, index, bit offset, width) for every field of one block."""
    L = []
    if fmt != "IQ1_M":
        L.append(("d16", 0, 0, 16))
    if fmt == "IQ2_XXS":
        for s in range(8):
            base = (2 + 8 * s) * 8
            for k in range(4):
                L.append(("idx", 4 * s + k, base + 8 * k, 8))
                L.append(("sign7", 4 * s + k, base + 32 + 7 * k, 7))
            L.append(("scale", s, base + 32 + 28, 4))
    elif fmt == "IQ2_XS":
        for g in range(32):
            L.append(("idx", g, (2 + 2 * g) * 8, 9))
            L.append(("sign7", g, (2 + 2 * g) * 8 + 9, 7))
        for cg in range(16):
            L.append(("scale", cg, (66 + cg // 2) * 8 + 4 * (cg % 2), 4))
    elif fmt == "IQ2_S":
        for g in range(32):
            L.append(("idx_lo", g, (2 + g) * 8, 8))
            L.append(("sign8", g, (34 + g) * 8, 8))
            L.append(("idx_hi", g, (66 + g // 4) * 8 + 2 * (g % 4), 2))
        for cg in range(16):
            L.append(("scale", cg, (74 + cg // 2) * 8 + 4 * (cg % 2), 4))
    elif fmt == "IQ1_S":
        for g in range(32):
            L.append(("idx_lo", g, (2 + g) * 8, 8))
            L.append(("idx_hi", g, (34 + 2 * (g // 4)) * 8 + 3 * (g % 4), 3))
        for s in range(8):
            L.append(("scale", s, (34 + 2 * s) * 8 + 12, 3))
            L.append(("dbit", s, (34 + 2 * s) * 8 + 15, 1))
    elif fmt == "IQ1_M":
        for g in range(32):
            L.append(("idx_lo", g, g * 8, 8))
            L.append(("idx_hi", g, (32 + g // 2) * 8 + 4 * (g % 2), 3))
            L.append(("dbit", g, (32 + g // 2) * 8 + 4 * (g % 2) + 3, 1))
        for cg in range(16):
            L.append(("scale", cg, (48 + 2 * (cg // 4)) * 8 + 3 * (cg % 4), 3))
        for k in range(4):
            L.append(("d16_nib", k, (48 + 2 * k) * 8 + 12, 4))
    return L


def write_bits(buf, pos, width, value):
    for b in range(width):
        if (value >> b) & 1:
            p = pos + b
            buf[p // 8] |= 1 << (p % 8)


def draw_fields(fmt, rng):
    entries = {"IQ2_XXS": 256, "IQ2_XS": 512, "IQ2_S": 1024, "IQ1_S": 2048, "IQ1_M": 2048}[fmt]
    f = {}
    # a positive normal fp16 scale with a varied mantissa
    f["d16"] = int(rng.integers(0x1400, 0x2c00))
    idx = rng.integers(0, entries, 32)
    f["idx"] = [int(v) for v in idx]
    if fmt in ("IQ2_XXS", "IQ2_XS"):
        f["sign7"] = [int(v) for v in rng.integers(0, 128, 32)]
    if fmt == "IQ2_S":
        f["sign8"] = [int(v) for v in rng.integers(0, 256, 32)]
    n_scale = {"IQ2_XXS": 8, "IQ2_XS": 16, "IQ2_S": 16, "IQ1_S": 8, "IQ1_M": 16}[fmt]
    top = 16 if fmt.startswith("IQ2") else 8
    f["scale"] = [int(v) for v in rng.integers(0, top, n_scale)]
    if fmt == "IQ1_S":
        f["dbit"] = [int(v) for v in rng.integers(0, 2, 8)]
    if fmt == "IQ1_M":
        f["dbit"] = [int(v) for v in rng.integers(0, 2, 32)]
    return f


def assemble(fmt, f):
    buf = bytearray(BLOCK_BYTES[fmt])
    for name, i, pos, width in layout(fmt):
        if name == "d16":
            v = f["d16"]
        elif name == "idx":
            v = f["idx"][i]
        elif name == "idx_lo":
            v = f["idx"][i] & 0xFF
        elif name == "idx_hi":
            v = f["idx"][i] >> 8
        elif name == "d16_nib":
            v = (f["d16"] >> (4 * i)) & 0xF
        else:
            v = f[name][i]
        write_bits(buf, pos, width, v)
    return bytes(buf)


def main():
    rng = np.random.default_rng(20261202)
    lines = ["# fmt | fields (name=comma list) | payload hex — hand-assembled by make_decode_fixtures.py"]
    for fmt in ("IQ2_XXS", "IQ2_XS", "IQ2_S", "IQ1_S", "IQ1_M"):
        for _ in range(3):
            f = draw_fields(fmt, rng)
            fields = ";".join(f"{k}=" + (",".join(map(str, v)) if isinstance(v, list) else str(v))
                              for k, v in f.items())
            lines.append(f"{fmt}|{fields}|{assemble(fmt, f).hex()}")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_fixtures.txt")
    with open(path, "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
