"""Write tests/golden/tiny_layer.txt from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The file holds, for the 16-token tiny workload (seed 0), every token's top-4
expert ids and its 512 output BF16 bit patterns.  Only the oracle and the
seeded input generator are called.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from block_scaled_fp4_router_gb300 import workloads as W  # noqa: E402
from oracle import moe as M  # noqa: E402


def main():
    wl = W.WORKLOADS["tiny"]
    lay = W.generate(wl)
    r = M.layer_forward(lay, wl.top_k, wl.fmt)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_layer.txt")
    with open(path, "w") as f:
        f.write("# tiny workload (T=16, H=512, I=256, E=16, k=4, MXFP4, seed 0)\n")
        f.write("# written by tests/golden/make_golden.py from the oracle only\n")
        f.write("# ids <token> <e0..e3> / out <token> <H bf16 bit patterns, hex>\n")
        for t in range(wl.T):
            f.write("ids %d %s\n" % (t, " ".join(str(int(v)) for v in r["ids"][t])))
        for t in range(wl.T):
            f.write("out %d %s\n" % (t, " ".join("%04x" % int(v) for v in r["out_bits"][t])))


if __name__ == "__main__":
    main()
