"""Writes the stored expected values under tests/golden/.

Calls only the oracle (and the seeded input generator); nothing here comes from
the CUDA path.  Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from kimi_delta_attention_18_gb300.inputs import WORKLOADS, make_prefill_inputs  # noqa: E402

TOKENS = [0, 1, 15, 16, 31, 47, 63]


def main():
    w = WORKLOADS["kda_fwd_f32_h2_t64_d16"]
    x = make_prefill_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], seed=0)
    f = lambda t: t.double().numpy()
    o, S = oracle.kda_forward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]),
                              None, x["cu_seqlens"].numpy())
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "kda_fwd_f32_h2_t64_d16.txt")
    with open(path, "w") as fh:
        fh.write("# KDA forward, fp32 inputs, B=1 H=2 T=64 dk=dv=16, S0=0, seed 0.\n")
        fh.write("# Written by tests/golden/make_golden.py from the fp64 oracle only.\n")
        fh.write("# Recurrence: decay, erase, write, read ('Kimi K3 Architecture\n")
        fh.write("# Explained', section 3); g = -5 sigmoid(x) (Kimi K3 technical-report\n")
        fh.write("# digest, section 2.1 (1)).\n")
        fh.write("# lines: 'o t h j value' for t in %s, then 'S h i j value'.\n" % TOKENS)
        for t in TOKENS:
            for h in range(2):
                for j in range(16):
                    fh.write("o %d %d %d %.17g\n" % (t, h, j, o[t, h, j]))
        for h in range(2):
            for i in range(16):
                for j in range(16):
                    fh.write("S %d %d %d %.17g\n" % (h, i, j, S[0, h, i, j]))
    print("wrote", path)


if __name__ == "__main__":
    main()
