"""Writes tests/golden/tiny_oracle.json: oracle rows of the 'tiny' workload.

The pages print no worked example with numbers, so this fixture is a
regression pin of the oracle itself: inputs come from the seeded generator
(digested so that a generator change is noticed), expected values from
``oracle`` only.  Re-run only when a commit changes the oracle's arithmetic,
naming the passage that justifies the change.
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import rpa_inputs as ri  # noqa: E402


def digest(p):
    h = hashlib.sha256()
    for a in (p.q, p.kv_pages, p.kv_lens, p.page_indices, p.cu_q_lens):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def main():
    p = ri.workload("tiny")
    o = oracle.forward(p)
    rows = [(0, 0), (0, 3), (1, 1), (3, 2), (5, 0), (6, 3), (10, 1), (21, 2), (13, 0)]
    out = {
        "source": "oracle.forward on rpa_inputs.workload('tiny') (seed 0)",
        "input_sha256": digest(p),
        "rows": [{"token": t, "q_head": h, "o": [float(v) for v in o[t, h]]} for t, h in rows],
        "row_sums": [float(v) for v in o.sum(axis=(1, 2))],
    }
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
