"""Write the oracle regression fixture tests/golden/bob_N6_d3_seed5.txt.

Calls only the fp64 oracle.  The pages print no worked numerical example of
the operator, so this fixture pins the oracle to its own earlier output,
which the finite-difference, symbolic and brute-force tests pin in turn.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import bob as orc  # noqa: E402


def main():
    rng = np.random.default_rng(5)
    args = [rng.standard_normal((6, 3)) for _ in range(7)]
    r = orc.bob(*args, 0.5)
    path = os.path.join(HERE, "bob_N6_d3_seed5.txt")
    with open(path, "w") as fh:
        fh.write("# oracle.bob on N=6, d=3, tau=0.5; inputs Q,K,V,dO,U_Q,U_K,U_V drawn in that\n")
        fh.write("# order as numpy default_rng(5).standard_normal((6, 3)); values row-major.\n")
        for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
            fh.write(key + " " + " ".join(repr(float(v)) for v in r[key].ravel()) + "\n")


if __name__ == "__main__":
    main()
