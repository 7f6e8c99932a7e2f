"""Writes tests/golden/tiny_fp32_8x8.txt from the oracle alone (a drift guard, not a pin).

Run: python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
import workloads as W  # noqa: E402


def main():
    w = W.decoder_weights(W.TINY, seed=1)
    m = O.OracleDecoder(W.TINY, w, max_seq=32)
    out = O.generate(m, W.prompt_uniform(8, W.TINY.vocab, seed=0), 8)
    with open(os.path.join(HERE, "tiny_fp32_8x8.txt"), "w") as f:
        f.write("# Oracle output for the tiny FP32 decoder: weights seed 1, 8 uniform prompt tokens\n")
        f.write("# from seed 0, 8 greedy outputs. Written by make_golden.py (oracle only).\n")
        f.write("tokens = " + " ".join(str(t) for t in out["tokens"]) + "\n")
        f.write("logits0_head = " + " ".join(repr(float(v)) for v in out["logits"][0][:16]) + "\n")


if __name__ == "__main__":
    main()
