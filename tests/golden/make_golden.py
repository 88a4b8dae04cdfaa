"""Write tests/golden/tiny_decode.txt from the CPU oracle alone.

The pages print no worked example, so this fixture is a regression record of
the oracle on the tiny decode workload (2 requests, seq_lens 300 and 700, one
query token, one head, topk 4, init 1, local 1, sm_scale 1/sqrt(128), 16
pages).  It calls only ``oracle`` and the seeded input generator.

    python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402


def main():
    wl = workloads.make("tiny")
    s, ids = oracle.problem(wl)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.txt")
    with open(out, "w") as f:
        f.write("# oracle output on the tiny decode workload; written by make_golden.py\n")
        f.write("# row ids <topk ids> | row scores <visible block scores>\n")
        for r in range(wl.rows):
            f.write(f"{r} ids " + " ".join(str(int(x)) for x in ids[0, r]) + "\n")
            nb = (int(wl.seq_lens[r]) - 1) // 128 + 1
            f.write(f"{r} scores " + " ".join(repr(float(x)) for x in s[0, r, :nb]) + "\n")


if __name__ == "__main__":
    main()
