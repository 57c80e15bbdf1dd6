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
from kimi_delta_attention_18_gb300.inputs import (WORKLOADS, make_backward_adjoints,  # noqa: E402
                                                  make_prefill_inputs)

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
    backward(w, x, f)


def backward(w, x, f):
    """Gradients of the same problem for d_out and d_S_final drawn with seed 1."""
    T, H, d = sum(w["lengths"]), w["H"], w["dk"]
    d_out, d_sf = make_backward_adjoints(T, 1, H, d, d, w["act"], seed=1)
    grads = oracle.kda_backward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]),
                                np.zeros((1, H, d, d)), x["cu_seqlens"].numpy(), f(d_out),
                                f(d_sf))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "kda_bwd_f32_h2_t64_d16.txt")
    names = ("dq", "dk", "dv", "dg", "dbeta")
    header = [
        "KDA backward, fp32 inputs, B=1 H=2 T=64 dk=dv=16, S0=0, seed 0; adjoints",
        "d_out, d_S_final from make_backward_adjoints(seed=1).  Written by",
        "tests/golden/make_golden.py from the fp64 oracle only: gradients of",
        "<d_out, o> + <d_S_final, S_final> for the recurrence of 'Kimi K3",
        "Architecture Explained', section 3.",
        "lines: 'name t h j value' (dbeta: j = 0) for t in %s, then" % TOKENS,
        "'dS0 h i j value'.",
    ]
    with open(path, "w") as fh:
        for line in header:
            fh.write("# " + line + "\n")
        for name, arr in zip(names, grads[:5]):
            for t in TOKENS:
                for h in range(H):
                    if arr.ndim == 2:
                        fh.write("%s %d %d 0 %.17g\n" % (name, t, h, arr[t, h]))
                    else:
                        for j in range(arr.shape[2]):
                            fh.write("%s %d %d %d %.17g\n" % (name, t, h, j, arr[t, h, j]))
        for h in range(H):
            for i in range(d):
                for j in range(d):
                    fh.write("dS0 %d %d %d %.17g\n" % (h, i, j, grads[5][0, h, i, j]))
    print("wrote", path)


if __name__ == "__main__":
    main()
