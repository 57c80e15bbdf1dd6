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


def test_config0_backward_golden_values():
    """The backward oracle's gradients on the config-0 problem against the stored
    values (written by make_golden.py from the oracle only)."""
    from kimi_delta_attention_18_gb300.inputs import make_backward_adjoints
    w = WORKLOADS["kda_fwd_f32_h2_t64_d16"]
    x = make_prefill_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], seed=0)
    T, H, d = sum(w["lengths"]), w["H"], w["dk"]
    d_out, d_sf = make_backward_adjoints(T, 1, H, d, d, w["act"], seed=1)
    f = lambda t: t.double().numpy()
    grads = oracle.kda_backward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]),
                                np.zeros((1, H, d, d)), x["cu_seqlens"].numpy(), f(d_out),
                                f(d_sf))
    got = dict(zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), grads))
    seen = 0
    with open(os.path.join(HERE, "kda_bwd_f32_h2_t64_d16.txt")) as fh:
        for line in fh:
            if line.startswith("#"):
                continue
            name, a, b, c, val = line.split()
            a, b, c, val = int(a), int(b), int(c), float(val)
            if name == "dS0":
                ref = got[name][0, a, b, c]
            elif name == "dbeta":
                ref = got[name][a, b]
            else:
                ref = got[name][a, b, c]
            assert abs(ref - val) <= 1e-12 * max(1.0, abs(val)), (name, a, b, c)
            seen += 1
    assert seen == 4 * 7 * 2 * 16 + 7 * 2 + 2 * 16 * 16
