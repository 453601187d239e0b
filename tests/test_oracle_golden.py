"""The oracle reproduces its stored tiny-workload fixtures on this host.

The fixtures were written by tests/golden/make_golden.py, which calls only
the oracle; this test catches unintended oracle changes and host-dependent
results (x86_64 versus aarch64 libm and compilers).
"""
import json
import os

import numpy as np

import oracle
from gpt_transformer_forward_gb300 import inputs


def test_tiny_fixtures():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_tiny.json")
    with open(path) as f:
        gold = json.load(f)
    w = inputs.WORKLOADS["tiny"]
    for init, case in gold["cases"].items():
        params, tok = inputs.workload_inputs(w, init)
        logits, probs = oracle.forward(w.cfg, params, tok)
        for i, (b, t) in enumerate(gold["rows"]):
            np.testing.assert_allclose(logits[b, t, :8], [float(x) for x in case["logits_head"][i]],
                                       rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(logits[b, t].sum(), float(case["logits_row_sum"][i]),
                                       rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(probs[b, t].max(), float(case["probs_max"][i]), rtol=1e-12)
