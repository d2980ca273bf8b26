"""Writes oracle_small_case.json: the oracle's fp64 output on one seeded small workload.

A regression fixture only (it pins the oracle to its own earlier output, so an
accidental change to the oracle's arithmetic shows up).  It calls nothing but the
oracle and the seeded input generator.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_decode_mapping_gb300 import workloads as W  # noqa: E402

SPEC = dict(B=3, Hq=8, Hkv=2, D=16, BS=4, lens=(1, 7, 13), seed=11, pool_factor=1.5)


def main():
    inp = W.make_inputs(W.small_workload(**SPEC))
    out, kc, vc = oracle.get().step(inp)
    doc = {
        "about": "oracle fp64 output of one write-then-attend step on small_workload(**spec); "
                 "written by tests/golden/make_golden.py",
        "spec": {k: list(v) if isinstance(v, tuple) else v for k, v in SPEC.items()},
        "out": [[[float(x) for x in row] for row in head] for head in out.tolist()],
    }
    with open(os.path.join(HERE, "oracle_small_case.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
