"""GPU: the deterministic gradient norm against the oracle, bit for bit.

The bins' exact value (an integer in units of 2^-149), the NaN / infinity
counts and the two float64 results must equal the oracle's exactly: both
sides compute the same exact sum and round it once.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    pkg.load_library()


def _np_view(t):
    """The elements as the oracle takes them: float32 / float16 arrays, bf16 bit patterns."""
    c = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return c.view(torch.int16).numpy().view(np.uint16), "bf16"
    if t.dtype == torch.float16:
        return c.numpy(), "f16"
    return c.numpy(), "f32"


def _check(t, bins=None):
    bins = pkg.norm_bins(DEV) if bins is None else bins
    pkg.sqnorm_accumulate(t, bins)
    out = pkg.sqnorm_finalize(bins)
    torch.cuda.synchronize()
    x, dt = _np_view(t)
    want_bins = oracle.sqnorm_bins(x, dt)
    got_bins = bins.cpu().numpy().view(np.uint64)
    assert oracle.bins_exact(got_bins) == oracle.bins_exact(want_bins)
    assert got_bins[oracle.NAN_BIN] == want_bins[oracle.NAN_BIN]
    assert got_bins[oracle.INF_BIN] == want_bins[oracle.INF_BIN]
    s, n = oracle.norm_finalize(want_bins)
    got = out.cpu().numpy()
    for g, w in zip(got.tolist(), (s, n)):
        assert (g == w) or (math.isnan(g) and math.isnan(w)), (got, s, n)
    return got


def _values(kind, n, g):
    if kind == "normal":
        return 1e-3 * torch.randn(n, generator=g, device=DEV)
    if kind == "spread":      # squares across most of the FP32 exponent range
        e = torch.empty(n, device=DEV).uniform_(-75, 63, generator=g)
        s = torch.where(torch.rand(n, generator=g, device=DEV) < 0.5, -1.0, 1.0)
        return s * torch.exp2(e)
    if kind == "zeros_mixed":
        x = torch.randn(n, generator=g, device=DEV)
        return torch.where(torch.rand(n, generator=g, device=DEV) < 0.3, torch.zeros_like(x), x)
    raise ValueError(kind)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 4095, 65536 + 3, (1 << 20) + 5])
def test_norm_matches_oracle(dtype, n):
    g = torch.Generator(device=DEV).manual_seed(n)
    for kind in ("normal", "spread", "zeros_mixed"):
        x = _values(kind, n, g)
        if dtype == torch.float16 and kind == "spread":
            x = x.clamp(-60000.0, 60000.0)
        _check(x.to(dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("offset", [1, 2, 3, 5])
def test_norm_unaligned_start(dtype, offset):
    g = torch.Generator(device=DEV).manual_seed(offset)
    buf = torch.randn(10000 + offset, generator=g, device=DEV).to(dtype)
    _check(buf[offset:])
    _check(buf[offset:offset + 3])


def test_norm_special_values():
    f = lambda v: _check(torch.tensor(v, dtype=torch.float32, device=DEV))
    assert all(math.isnan(r) for r in f([1.0, float("nan"), 2.0]))
    assert list(f([float("inf"), 1.0])) == [math.inf, math.inf]
    assert list(f([2.0 ** 64])) == [math.inf, math.inf]
    assert f([2.0 ** -70, 3.0])[0] == 9.0 + 2.0 ** -140
    assert f([2.0 ** -75])[0] == 0.0
    assert f([1.0 + 2.0 ** -23])[0] == 1.0 + 2.0 ** -22
    assert f([2.0 ** 27, 1.0, 1.0, 1.0])[0] == 2.0 ** 54 + 4
    assert list(f([3.0, 4.0])) == [25.0, 5.0]
    # finite squares whose sum exceeds the FP32 range
    big = torch.full((1000,), 1.8e19, dtype=torch.float32, device=DEV)
    _check(big)


def test_norm_empty_and_errors():
    bins = pkg.norm_bins(DEV)
    pkg.sqnorm_accumulate(torch.empty(0, device=DEV), bins)
    assert pkg.sqnorm_finalize(bins).cpu().tolist() == [0.0, 0.0]
    with pytest.raises(TypeError):
        pkg.sqnorm_accumulate(torch.zeros(4, dtype=torch.float64, device=DEV), bins)
    with pytest.raises(ValueError):
        pkg.sqnorm_accumulate(torch.zeros(4, 4, device=DEV).t(), bins)


def test_norm_invariant_to_order_and_split():
    """Any order of the elements and any split into tensors gives the same bits."""
    g = torch.Generator(device=DEV).manual_seed(11)
    x = _values("spread", 300001, g)
    ref = pkg.grad_norm(x).cpu()
    perm = torch.randperm(x.numel(), generator=g, device=DEV)
    assert torch.equal(pkg.grad_norm(x[perm]).cpu(), ref)
    for cuts in ([1], [12345, 200000], [7, 8, 9, 100000, 299999]):
        parts = torch.tensor_split(x, cuts)
        assert torch.equal(pkg.grad_norm(list(parts)).cpu(), ref)
    _check(x)


def test_norm_many_tensors_match_concatenation():
    g = torch.Generator(device=DEV).manual_seed(12)
    ts = [_values("normal", n, g).to(dt) for n, dt in ((1000, torch.float32), (777, torch.bfloat16),
                                                        (4096, torch.float16), (1, torch.float32))]
    bins = pkg.norm_bins(DEV)
    for t in ts:
        pkg.sqnorm_accumulate(t, bins)
    got = pkg.sqnorm_finalize(bins).cpu().numpy()
    total = sum(oracle.sqnorm_bins(*_np_view(t)).astype(object) for t in ts)
    want = oracle.norm_finalize(np.array(total, dtype=np.uint64))
    assert tuple(got.tolist()) == want


def test_norm_ten_million_bf16():
    """The page's microbenchmark size: 10M BF16-derived FP32 elements."""
    g = torch.Generator(device=DEV).manual_seed(13)
    x = (1e-2 * torch.randn(10_000_000, generator=g, device=DEV)).to(torch.bfloat16)
    _check(x)


def test_norm_large_f32():
    g = torch.Generator(device=DEV).manual_seed(14)
    x = _values("spread", 1 << 26, g)
    _check(x)
    del x
    torch.cuda.empty_cache()


def test_norm_every_bf16_pattern():
    """All 65536 BF16 bit patterns (both zeros, subnormals, the exponents at the
    edges of the BF16 integer path, infinities, NaNs) in shuffled order, then
    the finite ones alone and mixed with ordinary values: bin for bin against
    the oracle."""
    g = torch.Generator(device=DEV).manual_seed(15)
    pats = torch.arange(65536, dtype=torch.int32, device=DEV).to(torch.int16).view(torch.bfloat16)
    x = pats[torch.randperm(65536, generator=g, device=DEV)]
    assert torch.isnan(x.float()).any()
    _check(x)
    finite = x[torch.isfinite(x.float())]
    _check(finite)
    mixed = torch.cat([finite, (1e-3 * torch.randn(200000, generator=g, device=DEV)).to(torch.bfloat16)])
    _check(mixed[torch.randperm(mixed.numel(), generator=g, device=DEV)])
    # exponents just inside and outside the integer path, with a window that moves
    e = torch.tensor([58, 59, 60, 61, 120, 184, 185, 186, 190, 191, 200], device=DEV, dtype=torch.float32)
    edge = torch.exp2(e.repeat(5000) - 127.0) * (1.0 + torch.rand(55000, generator=g, device=DEV))
    _check(edge.to(torch.bfloat16)[torch.randperm(55000, generator=g, device=DEV)])
