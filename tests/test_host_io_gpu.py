"""rlk_logp_kl_host: the policy pair + reference + KL step on host-resident
inputs, the copies in running beside the passes, range by range.  A row's
results do not depend on its batch, so every output must equal the device
path's (rlk_logp_kl over the whole batch) bit for bit, whatever the number of
ranges, the host row stride, or the padding's contents."""

import pytest
import torch

import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import workloads as W

pytestmark = pytest.mark.gpu

VP, VR = pkg.VOCAB_PADDED, pkg.VOCAB_REAL


def _inputs(T, seed):
    dev = torch.device("cuda")
    x, hot, n = W.hot_logits(T, 1, 256, seed=seed, device=dev)
    ref = W.perturbed_copy(x, 0.05, seed=seed + 100)
    tg = W.structural_targets(T, hot, n, seed=seed, device=dev)
    g = torch.Generator(device=dev).manual_seed(seed)
    tau = torch.tensor([0.0, 0.7, 1.0, 1.3], device=dev)[torch.randint(0, 4, (T,), generator=g, device=dev)]
    p = torch.tensor([0.9, 0.95, 0.99, 1.0], device=dev)[torch.randint(0, 4, (T,), generator=g, device=dev)]
    k = torch.tensor([-1, 1, 50, 128], dtype=torch.int32, device=dev)[torch.randint(0, 4, (T,), generator=g, device=dev)]
    return x, ref, tg, tau.contiguous(), p.contiguous(), k.contiguous()


def _host(t, extra_cols=0, pad_value=None):
    """A pinned host copy, optionally with wider rows whose padding holds pad_value."""
    if t.dim() == 1:
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h
    h = torch.empty((t.shape[0], t.shape[1] + extra_cols), dtype=t.dtype, pin_memory=True)
    h[:, :t.shape[1]].copy_(t)
    if pad_value is not None:
        h[:, VR:] = pad_value
    return h[:, :VP] if extra_cols else h


def _same(a, b):
    return all(torch.equal(u.view(torch.int32), v.cpu().view(torch.int32)) for u, v in zip(a, b))


@pytest.mark.parametrize("T,chunks,two_streams,extra", [
    (1000, 3, True, 64),     # ragged ranges, wider host rows
    (1000, 1, False, 0),     # one range, one stream
    (5, 8, True, 0),         # more ranges than rows
    (257, 16, True, 8),
])
def test_kl_host_bitwise_equals_device_path(T, chunks, two_streams, extra):
    x, ref, tg, tau, p, k = _inputs(T, seed=11 + T)
    want = pkg.logp_kl(x, ref, tg, tau, p, k)
    hx = _host(x, extra, pad_value=float("nan"))
    hr = _host(ref)
    ht = _host(tg)
    cs = torch.cuda.Stream() if two_streams else None
    got = pkg.logp_kl_host(hx, hr, ht, tau, p, k, chunks=chunks, copy_stream=cs)
    torch.cuda.synchronize()
    assert hx.stride(0) == VP + extra
    assert _same(got, want)


def test_kl_host_consecutive_calls_share_a_workspace():
    """The second call's copies wait for the first call's passes: both see their own inputs."""
    T = 600
    x, ref, tg, tau, p, k = _inputs(T, seed=5)
    y, ref2, tg2, _, _, _ = _inputs(T, seed=6)
    want1 = pkg.logp_kl(x, ref, tg, tau, p, k)
    want2 = pkg.logp_kl(y, ref2, tg2, tau, p, k)
    ws = torch.empty(pkg.logp_kl_host_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    cs = torch.cuda.Stream()
    a = (_host(x), _host(ref), _host(tg))
    b = (_host(y), _host(ref2), _host(tg2))
    got1 = pkg.logp_kl_host(*a, tau, p, k, workspace=ws, chunks=4, copy_stream=cs)
    got2 = pkg.logp_kl_host(*b, tau, p, k, workspace=ws, chunks=4, copy_stream=cs)
    torch.cuda.synchronize()
    assert _same(got1, want1)
    assert _same(got2, want2)


def test_kl_host_scalar_parameters_and_err_count():
    T = 300
    x, ref, tg, _, _, _ = _inputs(T, seed=9)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = pkg.logp_kl(x, ref, tg, 1.3, 0.99, 128)
    got = pkg.logp_kl_host(_host(x), _host(ref), _host(tg), 1.3, 0.99, 128, chunks=5,
                           copy_stream=torch.cuda.Stream(), err_count=err)
    torch.cuda.synchronize()
    assert _same(got, want)
    assert int(err.item()) == 0


def test_kl_host_rejects_device_inputs():
    x, ref, tg, _, _, _ = _inputs(4, seed=3)
    with pytest.raises(ValueError):
        pkg.logp_kl_host(x, ref, tg)
