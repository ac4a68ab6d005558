"""Writes rng_frozen_vectors.txt: values of the counter-based random numbers
taken from the oracle alone, so that any later change to the generator's
layout (key folding, skip draws, fine bits, the uniform and Gumbel maps) shows
up as a changed value, even when both implementations change together.

Run from the repository root:  python tests/golden/make_rng_vectors.py

Coverage: every stream (ACCEPT, SAMPLE, DRAFT, TREE), seeds near 0 and near
2^64, large absolute positions and call indices, ids at both ends of a block
of 256, ids in the last (partial, 128-id) block of a 151,936-id vocabulary,
and top ids (the ids whose uniform lies in the top 1/256), found by scanning
the row with the oracle.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

OUT = os.path.join(HERE, "rng_frozen_vectors.txt")
V_BIG = 151936

# (seed, stream, seq, pos, iter)
KEYS = [
    (0, oracle.ST_ACCEPT, 0, 0, 0),
    (1, oracle.ST_ACCEPT, 63, 15, 0),
    (2**64 - 1, oracle.ST_ACCEPT, 5, 2**40 + 7, 0),
    (3, oracle.ST_SAMPLE, 0, 16, 0),
    (99, oracle.ST_SAMPLE, 127, 123456789, 0),
    (4, oracle.ST_DRAFT, 255, 31, 1),
    (4, oracle.ST_DRAFT, 255, 31, 2**33 + 5),
    (3, oracle.ST_TREE, 31, 7, 0),
    (0xDEADBEEFCAFEF00D, oracle.ST_TREE, 2**31, 2**62, 0),
]
# ordinary ids: block ends, the last partial block of V = 151,936
IDS = [0, 1, 255, 256, 65535, 151807, 151808, 151935]


def main():
    lines = [
        "# Frozen values of the counter RNG, written by make_rng_vectors.py from",
        "# the oracle alone.  Each 'key' line gives the fields and the row key;",
        "# each 'id' line that follows gives, for that key, a vocabulary id, its",
        "# top flag, its 52 fine bits, and the uniform and Gumbel values as the",
        "# exact hex of the fp64 number.",
    ]
    for (seed, st, seq, pos, it) in KEYS:
        k = oracle.key(seed, st, seq, pos, it)
        lines.append("key %d %d %d %d %d 0x%016X" % (seed, st, seq, pos, it, k))
        _, top = oracle.row_uniforms(k, V_BIG)
        tops = [int(v) for v in top.nonzero()[0]]
        # the first and last top ids of the row and one from the last block
        pick = [tops[0], tops[len(tops) // 2], tops[-1]]
        pick += [v for v in tops if v >= 151808][:1]
        for v in sorted(set(IDS + pick)):
            lines.append("id %d %d 0x%013X %s %s" % (
                v, int(oracle.is_top(k, v)), oracle.fine52(k, v),
                float.hex(oracle.uniform(k, v)), float.hex(oracle.gumbel(k, v))))
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
