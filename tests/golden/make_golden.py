"""Writes the stored expected values under tests/golden/ that come from the
oracle.  It calls only the oracle and the synthetic-input module.

    python tests/golden/make_golden.py

tiny_g_table.txt: the greedy next-token table g[x] for every id x of the
tiny instance (2 layers, d=64, 8 experts of 32, top-2, 1 shared expert,
vocab 512, weights N(0, 0.05) from seed 0).
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle as O  # noqa: E402
from moe_speculative_decoding_router_gb300 import synth as S  # noqa: E402


def main():
    o = O.Oracle(S.TINY, S.make_weights(S.TINY))
    g = o.g_table(range(S.TINY.vocab), nthreads=4)
    np.savetxt(os.path.join(HERE, "tiny_g_table.txt"), g, fmt="%d",
               header="greedy next id g[x] for x = 0..511, tiny instance, written by make_golden.py")


if __name__ == "__main__":
    main()
