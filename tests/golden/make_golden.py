"""Write the regression fixtures of this folder.  Calls only ``oracle/`` and
the seeded input generators; run from the repository root:

    python tests/golden/make_golden.py

The source pages print no worked example for the attention (no inputs with
printed outputs), so nothing here is a value quoted from them.  The fixture
records the oracle's own result on the tiny dense workload (batch 2, one query
token, 64 heads, 256 cached tokens, N(0,1)*0.5 values, scale 1/sqrt(192)) so
that any later change to the oracle's arithmetic shows up as a failing test
and has to be justified.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402


def main():
    w = workloads.config(1)
    out, lse = oracle.decode_all(w)
    rec = {
        "workload": w.name,
        "seed": w.seed,
        "lse": [[float(x) for x in lse[b, :, 0]] for b in range(w.B)],
        "o_rows": {f"{b},{h}": [float(x) for x in out[b, 0, h, :8]]
                   for b, h in ((0, 0), (0, 63), (1, 17))},
        "o_abs_sum": float(abs(out).sum()),
    }
    with open(os.path.join(HERE, "tiny_dense_oracle.json"), "w") as f:
        json.dump(rec, f, indent=1)


if __name__ == "__main__":
    main()
