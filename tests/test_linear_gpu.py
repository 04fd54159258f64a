"""GPU: the fused LM-head logprob (tensor-core GEMM + per-tile summaries)
against the oracle's exact logits.

Tolerance, per row, from the arithmetic: the tensor cores accumulate each
logit in fp32 over K/16 steps, each rounding at most 2^-24 of the running sum,
which is bounded by S = max_j sum_k |h_k W_jk|; as a random walk that is
sqrt(K/16) 2^-24 S, taken with a 4-sigma margin.  The logprob moves by at most
twice the largest logit error over tau, plus 2e-5 for the exponentials and the
logarithm (the bound of the logits path).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg

pytestmark = pytest.mark.gpu
DEV = "cuda"
VR, VP = oracle.VREAL, oracle.VPAD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    pkg.load_library()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _case(T, H, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    h = torch.randn((T, H), generator=g, device=DEV).to(torch.bfloat16)
    w = (4.0 / H ** 0.5 * torch.randn((VP, H), generator=g, device=DEV)).to(torch.bfloat16)
    tg = torch.randint(0, VR, (T,), generator=g, device=DEV, dtype=torch.int32)
    return h, w, tg


def _tolerance(hb, wb, H, tau):
    hf = np.abs(oracle.bf16_bits_to_f32(hb).astype(np.float64))
    wf = np.abs(oracle.bf16_bits_to_f32(wb[:VR]).astype(np.float64))
    S = (wf @ hf.T).max(axis=0)                        # per row: max_j sum_k |h_k W_jk|
    return 2e-5 + 2 * 4 * math.sqrt(H / 16) * 2.0 ** -24 * S / tau


@pytest.mark.parametrize("H", [256, 1024, 4096])
def test_linear_logp_matches_oracle(H):
    T = 130                                            # a ragged last row tile
    h, w, tg = _case(T, H, seed=H)
    rng = np.random.default_rng(H)
    tau = rng.choice([0.5, 0.7, 1.0, 1.3, 2.0], T).astype(np.float32)
    out = pkg.linear_logp(h, w, tg, torch.as_tensor(tau, device=DEV))
    torch.cuda.synchronize()
    rows = np.sort(rng.choice(T, 6, replace=False))
    rows[-1] = T - 1
    hb, wb = _bits(h)[rows], _bits(w)
    want = oracle.linear_logp_rows(hb, wb, tau[rows], tg.cpu().numpy()[rows])
    got = out.cpu().numpy()[rows]
    tol = _tolerance(hb, wb, H, tau[rows])
    assert np.all(np.abs(got - want) <= tol), (np.abs(got - want), tol)
    print(H, "max |d| =", float(np.max(np.abs(got - want))), "tol", float(tol.min()))


def test_linear_logp_is_batch_invariant():
    """A row's bits do not depend on the batch: its row tile, or the rows around it."""
    h, w, tg = _case(300, 512, seed=7)
    a = pkg.linear_logp(h, w, tg, 1.1)
    sub = torch.as_tensor([299, 5, 128, 127, 200], device=DEV)
    big = torch.full((9, 512 + 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    big[4:, :512] = h[sub]
    b = pkg.linear_logp(big[4:, :512], w, tg[sub].contiguous(), 1.1)
    torch.cuda.synchronize()
    assert torch.equal(a[sub].view(torch.int32), b.view(torch.int32))


def test_linear_logp_rejected_rows():
    h, w, tg = _case(8, 256, seed=9)
    tau = torch.tensor([1.0, 0.0, -1.0, float("nan"), 1.0, 1.0, 1.0, 1.0], device=DEV)
    tg[5] = VR
    tg[6] = -3
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.linear_logp(h, w, tg, tau, err_count=err)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert err.item() == 5
    assert all(math.isnan(o[i]) for i in (1, 2, 3, 5, 6))
    assert math.isfinite(o[0]) and math.isfinite(o[4]) and math.isfinite(o[7])


def test_linear_logp_full_size_sampled_rows():
    """T = 8192, H = 4096 (the Qwen3-8B hidden size), the bench's case: sampled rows."""
    T, H = 8192, 4096
    h, w, tg = _case(T, H, seed=11)
    out = pkg.linear_logp(h, w, tg, 1.3)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 4095, 4096, 8190, 8191])
    hb, wb = _bits(h[torch.as_tensor(rows, device=DEV)]), _bits(w)
    want = oracle.linear_logp_rows(hb, wb, 1.3, tg.cpu().numpy()[rows])
    got = out.cpu().numpy()[rows]
    assert np.all(np.abs(got - want) <= _tolerance(hb, wb, H, 1.3))
    assert torch.isfinite(out).all()
    del h, w
    torch.cuda.empty_cache()
