"""Batch invariance: a row's outputs are bit-identical whatever the batch.

The 8192 rows of the T = 8192 workload (tau 1.3, p 0.99, k 128) are evaluated
in packings of 1, 7, 256, 1000 and 8192 rows, in original and shuffled order,
and at random row offsets inside a larger buffer with a different row
stride; every row's three outputs must match the reference batch byte for
byte (the zero-byte-mismatch criterion of "H100 rollout context
parallelism", Measured results).
"""

import numpy as np
import pytest
import torch

import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import workloads as W

pytestmark = pytest.mark.gpu
VP = pkg.VOCAB_PADDED


def _bytes(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int32).cpu().numpy()


def test_packings_and_offsets_bitwise():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    wl = W.workload_c2(device="cuda", with_ref=False)
    T = wl.T
    targets = W.structural_targets(T, wl.hot, wl.hot_n, seed=2, device="cuda")
    # per-row parameters too, so packings also move the parameter arrays
    g = torch.Generator(device="cuda").manual_seed(33)
    tau = torch.tensor([0.7, 1.0, 1.3], device="cuda")[torch.randint(0, 3, (T,), generator=g, device="cuda")]
    p = torch.tensor([0.9, 0.99, 1.0], device="cuda")[torch.randint(0, 3, (T,), generator=g, device="cuda")]
    k = torch.tensor([-1, 50, 128], dtype=torch.int32, device="cuda")[
        torch.randint(0, 3, (T,), generator=g, device="cuda")]
    ref = [_bytes(o) for o in pkg.logp_pair(wl.logits, targets, tau, p, k)]

    plans, offsets = W.packing_plan(T)
    big_rows = 2 * T
    stride = VP + 24
    big = torch.empty((big_rows, stride), dtype=torch.bfloat16, device="cuda")
    mismatches = 0
    for (order_name, size, batches), off in zip(plans, offsets.tolist()):
        out = [np.empty(T, np.int32) for _ in range(3)]
        for bi, rows in enumerate(batches):
            ridx = rows.to("cuda")
            if bi % 2 == 0:
                xs = wl.logits[ridx]
            else:
                # place the batch at a random row offset of a wider buffer
                o = (off + bi * 131) % (big_rows - len(rows))
                big[o:o + len(rows), :VP] = wl.logits[ridx]
                big[o:o + len(rows), VP:] = float("nan")
                xs = big[o:o + len(rows)]
            outs = pkg.logp_pair(xs, targets[ridx].contiguous(), tau[ridx].contiguous(),
                                 p[ridx].contiguous(), k[ridx].contiguous())
            rn = rows.numpy()
            for j in range(3):
                out[j][rn] = _bytes(outs[j])
        for j in range(3):
            mismatches += int((out[j] != ref[j]).sum())
        assert mismatches == 0, f"packing {order_name}/{size}: {mismatches} byte mismatches"
