"""Writes tiny16.json: sparse 16-token rows and the oracle's outputs for every target.

Calls only the oracle.  The rows carry -inf outside 16 real columns, so the
same cases are also checked by exhaustive subset enumeration in
tests/test_oracle_pins.py (pin_brute_force_16).  Regenerate with
``python tests/golden/make_golden.py``.
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(1616)
    cases = []
    params = [(1.0, 0.9, -1), (0.7, 0.6, 5), (1.3, 1.0, 3), (0.5, 0.95, 12), (2.0, 0.3, -1),
              (0.0, 0.9, -1), (1.0, 1.0, -1)]
    for c in range(4):
        cols = np.sort(rng.choice(oracle.VREAL, 16, replace=False))
        if c == 3:
            cols[-1] = oracle.VREAL - 1           # last real column (shard 7 edge)
            cols[0] = 0
        vals = (np.round(rng.standard_normal(16) * (2 + c)) / 2).astype(np.float32)
        row = np.full(oracle.VPAD, 0xFF80, dtype=np.uint16)
        row[cols] = (vals.view(np.uint32) >> 16).astype(np.uint16)
        for tau, p, k in params:
            outs = []
            for t in cols:
                r = oracle.logp_row(row, tau, p, k, int(t))
                enc = lambda v: "-inf" if v == -math.inf else repr(float(v))
                outs.append([int(t), enc(r.full), enc(r.restr), int(r.support)])
            cases.append({"cols": cols.tolist(), "values": vals.tolist(), "tau": tau,
                          "top_p": p, "top_k": k, "per_target": outs})
    with open(os.path.join(HERE, "tiny16.json"), "w") as f:
        json.dump({"source": "oracle/logp_oracle.py via tests/golden/make_golden.py",
                   "vocab_padded": oracle.VPAD, "vocab_real": oracle.VREAL,
                   "fill": "-inf outside the listed columns", "cases": cases}, f, indent=0)


if __name__ == "__main__":
    main()
