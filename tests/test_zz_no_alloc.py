"""GPU: rlk_sample_noalloc, the sampler for callers that cannot allocate.

Such callers (code whose device memory belongs to a framework allocator or a
fixed memory plan) cannot hand rlk_sample a workspace, so the library keeps
the scratch in a fixed device array instead.  The entry point is called here
through the C ABI and must give exactly what rlk_sample gives with a
workspace of its own, on two calls in a row with different inputs (the
second call sees the first call's leftovers in the shared array).  This file
is collected last so that a failure here stops a run only after every other
test has run.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import _binding as b
from rollout_consistent_vocab_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_ROWS = 65536          # RLK_SAMPLE_NOALLOC_MAX_ROWS


@pytest.fixture(scope="module")
def lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    return pkg.load_library()


def _noalloc(lib, x, tau, p, k, seed, counter):
    T = x.shape[0]
    a = b.make_args(x, None, tau, p, k)
    tok = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    restr = torch.full((T,), 7.0, device=DEV)
    full = torch.full((T,), 7.0, device=DEV)
    sup = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    st = lib.rlk_sample_noalloc(ctypes.byref(a), seed, counter.data_ptr(), None, tok.data_ptr(),
                                restr.data_ptr(), full.data_ptr(), sup.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == b.RLK_OK, lib.rlk_last_error()
    return tok, restr, full, sup


def _same(u, v):
    assert torch.equal(u.view(torch.int32), v.view(torch.int32))


def _case(T, seed):
    rng = np.random.default_rng(seed)
    x, _, _ = W.hot_logits(T, 1, 200, seed=seed, device=DEV)
    tau = torch.as_tensor(rng.choice([0.0, 0.7, 1.0, 1.3], T).astype(np.float32), device=DEV)
    p = torch.as_tensor(rng.choice([0.9, 0.95, 1.0], T).astype(np.float32), device=DEV)
    k = torch.as_tensor(rng.choice([-1, 20, 128], T).astype(np.int32), device=DEV)
    ctr = torch.as_tensor(rng.integers(0, 2 ** 40, T), dtype=torch.int64, device=DEV)
    return x, tau, p, k, ctr


def test_noalloc_sampler_matches_rlk_sample_twice(lib):
    for T, seed in ((300, 61), (77, 62)):          # the second call reuses the scratch
        x, tau, p, k, ctr = _case(T, seed)
        got = _noalloc(lib, x, tau, p, k, seed * 1000 + 1, ctr)
        want = pkg.sample(x, tau, p, k, seed=seed * 1000 + 1, counter=ctr)
        torch.cuda.synchronize()
        for u, v in zip(got, want):
            _same(u, v)
        assert (got[0] >= 0).all()


def test_noalloc_sampler_rejects_batches_above_its_scratch(lib):
    a = b.make_args(torch.empty((1, b.VOCAB_PADDED), dtype=torch.bfloat16, device=DEV), None)
    a.T = MAX_ROWS + 1
    st = lib.rlk_sample_noalloc(ctypes.byref(a), 1, 0x1000, None, 0x2000, None, None, None, None)
    assert st == b.RLK_EINVAL
    assert b"rlk_sample_noalloc" in lib.rlk_last_error()
