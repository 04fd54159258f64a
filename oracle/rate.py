"""Time the oracle on a stored sample of rows (TEST INFRASTRUCTURE ONLY).

Run by the CPU-baseline leg of ``bench.py`` as one process per host core:

    python -m oracle.rate DIR WORKER NWORKERS SECONDS TAU TOP_P TOP_K

DIR holds ``bits.npy`` and ``ref_bits.npy`` (uint16 [n, 152576]) and
``targets.npy`` (int32 [n]), mapped read-only so that the processes share
them.  Worker w takes rows w, w + NWORKERS, ... (cycling through the sample)
until SECONDS have passed, resolving each row as the operator's step does
(policy pair, then the reference full logprob), and prints one JSON line
{"rows", "seconds"}.
"""

from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

from .logp_oracle import logp_row


def main(argv=None) -> None:
    d, worker, nworkers, seconds, tau, top_p, top_k = (argv or sys.argv[1:])[:7]
    worker, nworkers, seconds = int(worker), int(nworkers), float(seconds)
    tau, top_p, top_k = float(tau), float(top_p), int(top_k)
    bits = np.load(os.path.join(d, "bits.npy"), mmap_mode="r")
    rbits = np.load(os.path.join(d, "ref_bits.npy"), mmap_mode="r")
    tg = np.load(os.path.join(d, "targets.npy"))
    n = bits.shape[0]
    t0 = time.perf_counter()
    done = 0
    i = worker
    while time.perf_counter() - t0 < seconds:
        r = i % n
        logp_row(np.asarray(bits[r]), tau, top_p, top_k, int(tg[r]))
        logp_row(np.asarray(rbits[r]), tau, 1.0, -1, int(tg[r]))
        done += 1
        i += nworkers
    print(json.dumps({"rows": done, "seconds": time.perf_counter() - t0}), flush=True)


if __name__ == "__main__":
    main()
