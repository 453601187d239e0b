"""Writes oracle regression fixtures for the tiny GPT-2 workload.

The pages print no worked numerical example of the forward pass, so the
fixtures here are the oracle's own outputs on seeded inputs.  They pin the
oracle against unintended change and against differences between host
machines (x86_64 and aarch64 must reproduce them).  This script calls only
the oracle and the seeded input generator.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gpt_transformer_forward_gb300 import inputs  # noqa: E402

ROWS = [(0, 0), (0, 31), (1, 7), (1, 20)]


def main():
    w = inputs.WORKLOADS["tiny"]
    out = {"workload": "tiny", "rows": ROWS, "cases": {}}
    for init in ("gpt2", "perturbed"):
        params, tok = inputs.workload_inputs(w, init)
        logits, probs = oracle.forward(w.cfg, params, tok)
        out["cases"][init] = {
            "logits_head": [[repr(float(x)) for x in logits[b, t, :8]] for b, t in ROWS],
            "logits_row_sum": [repr(float(logits[b, t].sum())) for b, t in ROWS],
            "probs_max": [repr(float(probs[b, t].max())) for b, t in ROWS],
        }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
