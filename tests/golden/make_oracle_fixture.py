"""Write oracle_small_5x4x3x2.txt: the fp64 oracle's output on a small seeded case.

A regression fixture: it is written by this script, which calls only the
oracle and the seeded input generator, and it lets a later change to the
oracle that alters its results (on any host) show up as a test failure.

    python tests/golden/make_oracle_fixture.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

DIMS, R, SEED = (5, 4, 3, 2), 3, 4242


def main():
    Y, A = synth.random_case(SEED, DIMS, R)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_5x4x3x2.txt")
    with open(path, "w") as f:
        f.write("# fp64 oracle MTTKRP of synth.random_case(4242, (5, 4, 3, 2), R=3) (fp32 inputs)\n")
        f.write("# written by tests/golden/make_oracle_fixture.py; format: mode row r value\n")
        for k in range(len(DIMS)):
            M = oracle.mttkrp(Y, A, k)
            for i in range(DIMS[k]):
                for r in range(R):
                    f.write(f"{k} {i} {r} {float(M[i, r])!r}\n")


if __name__ == "__main__":
    main()
