"""Writes q8_0_blocks.txt: hand-made Q8_0 blocks and their values.

Each value is d * q with d an exactly representable fp16 chosen by hand, following the
block format of the Q8_0 re-quantiser on the gemma4/model.rs page (fp16 scale, little
endian, then 32 int8).  Nothing here calls the oracle or the CUDA library.
Run from the repository root: python tests/golden/write_q8_0_blocks.py
"""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def block(dbits, qs):
    b = [dbits & 0xFF, dbits >> 8] + [(q + 256) % 256 for q in qs]
    return " ".join(f"{x:02x}" for x in b)


def main():
    lines = ["# Hand-made Q8_0 blocks (gemma4/model.rs, Q8_0 lm_head re-quantiser: 34-byte block =",
             "# fp16 scale d, little endian, in bytes 0-1, then 32 int8 values; value = d * q).",
             "# Format: 'block <34 hex bytes>' followed by 'values <32 exact decimals>'."]
    cases = [
        (0x3800, 0.5, [i - 16 for i in range(32)]),                      # d = 0.5
        (0x0001, 2.0 ** -24, [127 if i % 2 == 0 else -127 for i in range(32)]),  # subnormal d
        (0x7BFF, 65504.0, [-127 + 8 * i if -127 + 8 * i <= 127 else 0 for i in range(32)]),
        (0xBC00, -1.0, [(i * 37) % 255 - 127 for i in range(32)]),       # negative d
        (0x0000, 0.0, [100 - i for i in range(32)]),                     # d = 0
    ]
    for dbits, d, qs in cases:
        lines.append("block " + block(dbits, qs))
        lines.append("values " + " ".join(repr(d * q) for q in qs))
    with open(os.path.join(HERE, "q8_0_blocks.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
