"""Writes tests/golden/handbuilt_blocks.txt: hand-built blocks whose weights have
closed forms.  Block bytes come from the oracle's packer; every expected value
is the closed form written below (exact small rationals), not a decoder output.

Fields follow the k-quant definitions (Q4_K/Q5_K: w = d*sc_j*q - dmin*m_j over
32-weight sub-blocks j; Q6_K: w = d*sc_j*(q-32) over 16-weight sub-blocks).

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

CASES = []

# Q4_K: d = 1.0 (0x3C00), dmin = 0.5 (0x3800), sc_j = j+1, m_j = 2j, q_i = i mod 16
#   w_i = (j+1)*(i mod 16) - 0.5*2j = (j+1)*(i mod 16) - j,  j = i // 32
CASES.append(("Q4_K", "d=1 dmin=0.5 sc_j=j+1 m_j=2j q_i=i%16 -> w_i=(j+1)*(i%16)-j",
              oracle.pack(oracle.Q4_K, 0x3C00, [j + 1 for j in range(8)], [i % 16 for i in range(256)],
                          0x3800, [2 * j for j in range(8)]),
              [(i // 32 + 1) * (i % 16) - i // 32 for i in range(256)]))

# Q4_K with the largest fields: d = 2^-24 (0x0001, smallest fp16 subnormal), dmin = 0,
#   sc_j = 63, m_j = 63, q_i = 15  ->  w_i = 2^-24 * 63 * 15
CASES.append(("Q4_K", "d=2^-24 (subnormal) dmin=0 sc=63 m=63 q=15 -> w=945*2^-24",
              oracle.pack(oracle.Q4_K, 0x0001, [63] * 8, [15] * 256, 0x0000, [63] * 8),
              [945.0 * 2.0 ** -24] * 256))

# Q5_K: d = 0.25 (0x3400), dmin = 1.0 (0x3C00), sc_j = 4, m_j = j, q_i = i mod 32
#   w_i = 0.25*4*(i mod 32) - j = (i mod 32) - j
CASES.append(("Q5_K", "d=0.25 dmin=1 sc=4 m_j=j q_i=i%32 -> w_i=(i%32)-j",
              oracle.pack(oracle.Q5_K, 0x3400, [4] * 8, [i % 32 for i in range(256)],
                          0x3C00, list(range(8))),
              [(i % 32) - i // 32 for i in range(256)]))

# Q6_K: d = 0.5 (0x3800), sc_j = j - 8 (j = i // 16), q_i = i mod 64
#   w_i = 0.5*(j-8)*((i mod 64) - 32)
CASES.append(("Q6_K", "d=0.5 sc_j=j-8 q_i=i%64 -> w_i=0.5*(j-8)*(i%64-32)",
              oracle.pack(oracle.Q6_K, 0x3800, [j - 8 for j in range(16)], [i % 64 for i in range(256)]),
              [0.5 * (i // 16 - 8) * ((i % 64) - 32) for i in range(256)]))

# Q6_K extremes: d = -2.0 (0xC000), sc = -128, q = 0  ->  w = -2*-128*-32 = -8192
CASES.append(("Q6_K", "d=-2 sc=-128 q=0 -> w=-8192",
              oracle.pack(oracle.Q6_K, 0xC000, [-128] * 16, [0] * 256),
              [-8192.0] * 256))


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "handbuilt_blocks.txt")
    with open(path, "w") as f:
        f.write("# Hand-built k-quant blocks with closed-form weights (see make_golden.py).\n")
        f.write("# TYPE <name> | <closed form>\n# BYTES <hex>\n# W <256 values, repr of float>\n")
        for name, desc, blk, w in CASES:
            f.write(f"TYPE {name} | {desc}\n")
            f.write("BYTES " + bytes(blk).hex() + "\n")
            f.write("W " + " ".join(repr(float(v)) for v in w) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
