"""Write tests/golden/oracle_dense_b1_n128_h32_d64_rows.json.

The pages print no worked numerical example for the attention leaf, so the
only stored expected values are the oracle's own, written by this script
(which calls nothing but ``oracle``) on seeded inputs.  The fixture freezes
the oracle: a later change to its arithmetic shows up as a failing test and
must be justified by the definition it follows.

Run from the repository root:  python tests/golden/make_oracle_fixture.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle      # noqa: E402
import workloads   # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                   "oracle_dense_b1_n128_h32_d64_rows.json")
ROWS = [0, 1, 31, 32, 1000, 2047, 2048, 4095]


def main():
    w = workloads.WORKLOADS[1]
    q, k, v = (workloads.bf16_bits(t) for t in workloads.make_inputs(w))
    out = oracle.dense_attention_rows(q, k, v, np.array(ROWS))
    doc = {
        "what": "oracle FP64 rows of dense attention, config 1 inputs (seed 1000+i)",
        "definition": "noncausal_dense_attention_h32_d64.json, field reference",
        "workload": w.describe(),
        "rows_flat_index": ROWS,
        "row_index_rule": "r = (b*Nq + i)*H + h",
        "values": [[float(x).hex() for x in row] for row in out],
    }
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
