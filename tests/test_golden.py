"""The stored config-0 values (written by tests/golden/make_golden.py from the
oracle alone) still come out of the oracle and the seeded generator: catches an
accidental change to either."""
import os

import numpy as np

import oracle
from kimi_delta_attention_18_gb300.inputs import WORKLOADS, make_prefill_inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(path):
    o, S = {}, {}
    with open(path) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            tag, a, b, c, val = line.split()
            (o if tag == "o" else S)[(int(a), int(b), int(c))] = float(val)
    return o, S


def test_config0_golden_values():
    w = WORKLOADS["kda_fwd_f32_h2_t64_d16"]
    x = make_prefill_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], seed=0)
    f = lambda t: t.double().numpy()
    o, S = oracle.kda_forward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]),
                              None, x["cu_seqlens"].numpy())
    go, gS = _read(os.path.join(HERE, "kda_fwd_f32_h2_t64_d16.txt"))
    assert len(go) == 7 * 2 * 16 and len(gS) == 2 * 16 * 16
    for (t, h, j), val in go.items():
        assert abs(o[t, h, j] - val) <= 1e-14 * max(1.0, abs(val))
    for (h, i, j), val in gS.items():
        assert abs(S[0, h, i, j] - val) <= 1e-14 * max(1.0, abs(val))
