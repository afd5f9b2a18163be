"""Write oracle_small.json: small seeded inputs and the oracle's outputs for
each function of the oracle, as a regression record of its arithmetic.

The pages print no worked example with values, so no fixture here comes from
them; every expected value below is written by this script, which calls only
the oracle package.  What ties the oracle to the pages' definitions (closed
forms, invariants, brute force) is the pin suite beside these fixtures.

    python tests/golden/make_golden.py      # rewrites oracle_small.json
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def _inputs():
    rng = np.random.default_rng(2026)
    T, H, K, V = 7, 2, 4, 3
    cu = np.array([0, 3, 3, 7])
    x = dict(q=rng.standard_normal((T, H, K)), k=rng.standard_normal((T, H, K)),
             v=rng.standard_normal((T, H, V)), g=-rng.uniform(0.01, 0.5, (T, H, K)),
             beta=rng.uniform(0.1, 0.9, (T, H)), cu_seqlens=cu,
             initial_state=0.1 * rng.standard_normal((3, H, K, V)))
    gate = dict(raw_gate=rng.standard_normal((T, H, K)), raw_beta=rng.standard_normal((T, H)),
                a_log=np.log(rng.uniform(1.0, 4.0, H)), dt_bias=rng.uniform(-1.0, 1.0, (H, K)))
    epi = dict(o=rng.standard_normal((T, H, V)), gate=rng.standard_normal((T, H, V)),
               weight=rng.uniform(0.5, 1.5, V))
    conv = dict(x=rng.standard_normal((9, 5)), weight=rng.uniform(-0.5, 0.5, (4, 5)),
                cu_seqlens=np.array([0, 2, 9]), initial_states=rng.standard_normal((2, 3, 5)))
    return x, gate, epi, conv


def compute():
    x, gate, epi, conv = _inputs()
    o, s = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=x["cu_seqlens"],
                             initial_state=x["initial_state"])
    one = slice(3, 7)  # the third sequence alone, through the chunked form (chunk 3: a ragged tail)
    oc, sc = oracle.chunked_form(x["q"][one], x["k"][one], x["v"][one], x["g"][one], x["beta"][one],
                                 initial_state=x["initial_state"][2], chunk=3)
    g_lb, b_lb = oracle.gate_activation(gate["raw_gate"], gate["raw_beta"], gate["a_log"], gate["dt_bias"],
                                        lower_bound=-5.0)
    g_sp, _ = oracle.gate_activation(gate["raw_gate"], gate["raw_beta"], gate["a_log"], gate["dt_bias"])
    on = oracle.output_gate_norm(epi["o"], epi["gate"], epi["weight"], 1e-5)
    yc, fc = oracle.short_conv_prefill(conv["x"], conv["weight"], conv["cu_seqlens"],
                                       initial_states=conv["initial_states"])
    tolist = lambda a: np.asarray(a, dtype=np.float64).tolist()
    return {
        "inputs": {"kda": {k_: tolist(v_) for k_, v_ in x.items()},
                   "gate": {k_: tolist(v_) for k_, v_ in gate.items()},
                   "epilogue": {k_: tolist(v_) for k_, v_ in epi.items()},
                   "conv": {k_: tolist(v_) for k_, v_ in conv.items()}},
        "expected": {"recurrence_o": tolist(o), "recurrence_state": tolist(s),
                     "chunked_o_seq3": tolist(oc), "chunked_state_seq3": tolist(sc),
                     "gate_g_lower_bound_m5": tolist(g_lb), "gate_beta": tolist(b_lb),
                     "gate_g_softplus": tolist(g_sp), "output_gate_norm": tolist(on),
                     "short_conv_y": tolist(yc), "short_conv_final": tolist(fc)},
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(compute(), f)
    print("wrote", os.path.join(HERE, "oracle_small.json"))
