"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before touching the GPU (runs without a GPU)."""

import ctypes
import os
import re

import pytest

import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import _binding as b
from rollout_consistent_vocab_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return pkg.load_library()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(rlk_\w+)\s*\(", text, re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"rlk_logp_full", "rlk_logp_restricted", "rlk_logp_pair", "rlk_logp_kl"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(b.EXPORTS) == names


def test_abi_version_and_status_strings(lib):
    assert lib.rlk_abi_version() == 5
    assert lib.rlk_status_string(0) == b"ok"
    assert lib.rlk_status_string(2) == b"misaligned pointer or stride"


def _args(**kw):
    a = b.LogpArgs()
    a.logits = 0x10000
    a.T = 4
    a.row_stride = b.VOCAB_PADDED
    a.vocab_real = b.VOCAB_REAL
    a.vocab_padded = b.VOCAB_PADDED
    a.target = 0x20000
    a.temperature = None
    a.temperature_scalar = 0.7
    a.top_p = None
    a.top_p_scalar = 0.95
    a.top_k = None
    a.top_k_scalar = -1
    a.err_count = None
    for k, v in kw.items():
        setattr(a, k, v)
    return a


OUT = 0x30000


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), b.RLK_EINVAL),
    (dict(T=1 << 28), b.RLK_EINVAL),
    (dict(vocab_real=151935), b.RLK_EINVAL),
    (dict(vocab_padded=152577), b.RLK_EINVAL),
    (dict(logits=None), b.RLK_EINVAL),
    (dict(target=None), b.RLK_EINVAL),
    (dict(row_stride=152575), b.RLK_EINVAL),
    (dict(logits=0x10008), b.RLK_EALIGN),
    (dict(row_stride=152580), b.RLK_EALIGN),
    (dict(target=0x20002), b.RLK_EALIGN),
    (dict(temperature_scalar=-0.5), b.RLK_EINVAL),
    (dict(temperature_scalar=float("inf")), b.RLK_EINVAL),
    (dict(temperature_scalar=float("nan")), b.RLK_EINVAL),
    (dict(top_p_scalar=0.0), b.RLK_EINVAL),
    (dict(top_p_scalar=1.5), b.RLK_EINVAL),
    (dict(top_k_scalar=0), b.RLK_EINVAL),
    (dict(top_k_scalar=151937), b.RLK_EINVAL),
    (dict(top_k_scalar=-2), b.RLK_EINVAL),
    (dict(temperature=0x40001), b.RLK_EALIGN),
])
def test_pair_rejects_bad_arguments_on_host(lib, kw, status):
    a = _args(**kw)
    got = lib.rlk_logp_pair(ctypes.byref(a), OUT, OUT + 0x1000, None, None)
    assert got == status
    assert lib.rlk_last_error()


def test_null_and_misaligned_outputs(lib):
    a = _args()
    assert lib.rlk_logp_pair(ctypes.byref(a), None, None, None, None) == b.RLK_EINVAL
    assert lib.rlk_logp_pair(ctypes.byref(a), OUT + 2, None, None, None) == b.RLK_EALIGN
    assert lib.rlk_logp_full(ctypes.byref(a), None, None) == b.RLK_EINVAL
    assert lib.rlk_logp_restricted(ctypes.byref(a), None, None, None) == b.RLK_EINVAL
    assert lib.rlk_logp_full(None, OUT, None) == b.RLK_EINVAL
    assert lib.rlk_logp_kl(ctypes.byref(a), 0x50008, b.VOCAB_PADDED, OUT, None, None,
                           OUT, OUT, None) == b.RLK_EALIGN
    assert lib.rlk_logp_kl(ctypes.byref(a), 0x50000, b.VOCAB_PADDED, OUT, None, None,
                           None, OUT, None) == b.RLK_EINVAL


def test_full_ignores_top_p_top_k(lib):
    # top_p/top_k are not part of the full-vocabulary call; out-of-domain values
    # there must not be rejected (the call then fails only at the launch, on CPU).
    a = _args(top_p_scalar=7.0, top_k_scalar=0, T=0)
    assert lib.rlk_logp_full(ctypes.byref(a), OUT, None) == b.RLK_OK


def test_empty_batch_is_a_noop(lib):
    a = _args(T=0, logits=None, target=None)
    assert lib.rlk_logp_pair(ctypes.byref(a), None, None, None, None) == b.RLK_OK
    assert lib.rlk_logp_full(ctypes.byref(a), None, None) == b.RLK_OK


def test_kl_host_validation(lib):
    """The host-input step checks everything before its first CUDA call."""
    a = _args()
    WS = 0x60000                      # 256-byte aligned
    def call(args=a, ref=0x50000, stride=b.VOCAB_PADDED, outs=(OUT, None, None, OUT, OUT), ws=WS,
             chunks=4):
        return lib.rlk_logp_kl_host(ctypes.byref(args) if args is not None else None, ref, stride,
                                    *outs, ws, chunks, None, None)
    assert call(args=None) == b.RLK_EINVAL
    assert call(args=_args(T=-1)) == b.RLK_EINVAL
    assert call(args=_args(T=1 << 27)) == b.RLK_EINVAL
    assert call(args=_args(logits=None)) == b.RLK_EINVAL
    assert call(args=_args(target=None)) == b.RLK_EINVAL
    assert call(args=_args(row_stride=152575)) == b.RLK_EINVAL
    assert call(ref=None) == b.RLK_EINVAL
    assert call(stride=152575) == b.RLK_EINVAL
    assert call(args=_args(top_p_scalar=0.0)) == b.RLK_EINVAL
    assert call(args=_args(top_k_scalar=0)) == b.RLK_EINVAL
    assert call(args=_args(temperature=0x40001)) == b.RLK_EALIGN
    assert call(outs=(None, None, None, OUT, OUT)) == b.RLK_EINVAL
    assert call(outs=(OUT, None, None, None, OUT)) == b.RLK_EINVAL
    assert call(outs=(OUT, None, None, OUT, None)) == b.RLK_EINVAL
    assert call(outs=(OUT, OUT + 2, None, OUT, OUT)) == b.RLK_EALIGN
    assert call(ws=None) == b.RLK_EINVAL
    assert call(ws=WS + 16) == b.RLK_EALIGN
    assert call(chunks=0) == b.RLK_EINVAL
    # host logits need no 16-byte alignment (they are copied), and T = 0 is a no-op
    assert call(args=_args(T=0, logits=None, target=None), ref=None, ws=None) == b.RLK_OK
    assert lib.rlk_last_error()


def test_kl_ref_validation(lib):
    a = _args()
    assert lib.rlk_logp_kl_ref(ctypes.byref(a), None, OUT, OUT, None) == b.RLK_EINVAL
    assert lib.rlk_logp_kl_ref(ctypes.byref(a), OUT, OUT + 1, OUT, None) == b.RLK_EALIGN
    assert lib.rlk_logp_kl_ref(ctypes.byref(_args(T=0)), None, None, None, None) == b.RLK_OK


# ------------------------------------------------------------ vocabulary-sharded entry points

def _sargs(**kw):
    a = b.ShardArgs()
    a.logits = 0x10000
    a.T = 4
    a.row_stride = b.SHARD_WIDTH
    a.shard = 3
    a.target = 0x20000
    a.temperature = None
    a.temperature_scalar = 0.7
    a.top_p = None
    a.top_p_scalar = 0.95
    a.top_k = None
    a.top_k_scalar = -1
    a.err_count = None
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), b.RLK_EINVAL),
    (dict(T=1 << 31), b.RLK_EINVAL),
    (dict(shard=-1), b.RLK_EINVAL),
    (dict(shard=8), b.RLK_EINVAL),
    (dict(logits=None), b.RLK_EINVAL),
    (dict(target=None), b.RLK_EINVAL),
    (dict(row_stride=19064), b.RLK_EINVAL),
    (dict(logits=0x10004), b.RLK_EALIGN),
    (dict(row_stride=19076), b.RLK_EALIGN),
    (dict(target=0x20001), b.RLK_EALIGN),
    (dict(temperature_scalar=-1.0), b.RLK_EINVAL),
    (dict(top_p_scalar=0.0), b.RLK_EINVAL),
    (dict(top_k_scalar=0), b.RLK_EINVAL),
    (dict(top_k=0x40002), b.RLK_EALIGN),
    (dict(err_count=0x40002), b.RLK_EALIGN),
])
def test_shard_entry_points_reject_bad_arguments_on_host(lib, kw, status):
    a = _sargs(**kw)
    assert lib.rlk_logp_shard_summary(ctypes.byref(a), OUT, OUT, OUT, OUT, None, None) == status
    assert lib.rlk_logp_shard_counts(ctypes.byref(a), OUT, OUT, OUT, None, OUT, None) == status
    assert lib.rlk_last_error()


def test_shard_outputs_checked(lib):
    a = _sargs()
    assert lib.rlk_logp_shard_summary(ctypes.byref(a), None, OUT, OUT, OUT, None, None) == b.RLK_EINVAL
    assert lib.rlk_logp_shard_summary(ctypes.byref(a), OUT, OUT, OUT, OUT + 2, None, None) == b.RLK_EALIGN
    assert lib.rlk_logp_shard_summary(ctypes.byref(a), OUT, OUT, OUT, OUT, OUT + 2, None) == b.RLK_EALIGN
    assert lib.rlk_logp_shard_counts(ctypes.byref(a), OUT, OUT, OUT, None, None, None) == b.RLK_EINVAL
    # the count rows are copied out as 16-byte vectors
    assert lib.rlk_logp_shard_counts(ctypes.byref(a), OUT, OUT, OUT, None, OUT + 4, None) == b.RLK_EALIGN
    assert lib.rlk_logp_shard_counts(ctypes.byref(a), OUT, OUT, OUT, OUT + 2, OUT, None) == b.RLK_EALIGN
    assert lib.rlk_logp_shard_counts(ctypes.byref(a), None, OUT, OUT, None, OUT, None) == b.RLK_EINVAL
    z = _sargs(T=0, logits=None, target=None)
    assert lib.rlk_logp_shard_summary(ctypes.byref(z), None, None, None, None, None, None) == b.RLK_OK
    assert lib.rlk_logp_shard_counts(ctypes.byref(z), None, None, None, None, None, None) == b.RLK_OK


def _merge(lib, T=4, tau=0.7, p=0.95, k=-1, counts=OUT, nc=8, full=OUT, restr=OUT, sup=OUT,
           maxes=OUT, target=OUT):
    return lib.rlk_logp_merge(maxes, OUT, OUT, OUT, T, target, None, tau, None, p, None, k,
                              counts, nc, full, restr, sup, None)


def test_merge_validation(lib):
    assert _merge(lib, T=-1) == b.RLK_EINVAL
    assert _merge(lib, T=0, maxes=None, target=None, full=None) == b.RLK_OK
    assert _merge(lib, maxes=None) == b.RLK_EINVAL
    assert _merge(lib, target=OUT + 2) == b.RLK_EALIGN
    assert _merge(lib, full=None) == b.RLK_EINVAL
    assert _merge(lib, tau=float("nan")) == b.RLK_EINVAL
    assert _merge(lib, nc=2) == b.RLK_EINVAL
    assert _merge(lib, nc=0) == b.RLK_EINVAL
    assert _merge(lib, p=1.5) == b.RLK_EINVAL
    assert _merge(lib, k=151937) == b.RLK_EINVAL
    assert _merge(lib, restr=None, sup=None) == b.RLK_EINVAL
    assert _merge(lib, counts=OUT + 2) == b.RLK_EALIGN
    assert _merge(lib, restr=OUT + 1) == b.RLK_EALIGN


def _merge_res(lib, T=4, counts=OUT, nc=8, state=OUT, pending=None, full=OUT, restr=OUT, sup=OUT,
               p=0.95, k=-1):
    return lib.rlk_logp_merge_resumable(OUT, OUT, OUT, OUT, T, OUT, None, 0.7, None, p, None, k, counts,
                                        nc, state, full, restr, sup, pending, None)


def test_resumable_merge_and_window_counts_validation(lib):
    assert _merge_res(lib, T=0, state=None, counts=None) == b.RLK_OK
    assert _merge_res(lib, state=None) == b.RLK_EINVAL
    assert _merge_res(lib, state=OUT + 4) == b.RLK_EALIGN
    assert _merge_res(lib, counts=None) == b.RLK_EINVAL
    assert _merge_res(lib, pending=OUT + 2) == b.RLK_EALIGN
    assert _merge_res(lib, nc=3) == b.RLK_EINVAL
    assert _merge_res(lib, restr=None, sup=None) == b.RLK_EINVAL
    assert _merge_res(lib, p=0.0) == b.RLK_EINVAL
    a = _sargs()
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(a), None, None, OUT, None) == b.RLK_EINVAL
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(a), OUT + 4, None, OUT, None) == b.RLK_EALIGN
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(a), OUT, None, None, None) == b.RLK_EINVAL
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(a), OUT, None, OUT + 4, None) == b.RLK_EALIGN
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(a), OUT, OUT + 2, OUT, None) == b.RLK_EALIGN
    bad = _sargs(shard=9)
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(bad), OUT, None, OUT, None) == b.RLK_EINVAL
    z = _sargs(T=0, logits=None, target=None)
    assert lib.rlk_logp_shard_counts_window(ctypes.byref(z), None, None, None, None) == b.RLK_OK


def test_merge_state_layout():
    """rlk_merge_state is 40 bytes: five int64 words in the binding's state tensor."""
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "rlk_logp.h")).read()
    body = re.search(r"typedef struct rlk_merge_state \{(.*?)\} rlk_merge_state;", hdr, re.S).group(1)
    sizes = {"int32_t": 4, "uint32_t": 4, "uint64_t": 8}
    fields = re.findall(r"^\s*(int32_t|uint32_t|uint64_t)\s+([\w, ]+);", body, re.M)
    total = sum(sizes[t] * len(names.split(",")) for t, names in fields)
    assert total == 8 * b.MERGE_STATE_WORDS == 40


# ------------------------------------------------------------ backward

def _bwd(lib, a=None, gf=OUT, gr=None, grad=0x60000, stride=b.VOCAB_PADDED, dtype=0,
         full=None, restr=None, sup=None):
    a = _args() if a is None else a
    return lib.rlk_logp_backward(ctypes.byref(a), gf, gr, grad, stride, dtype, full, restr, sup, None)


def test_backward_validation(lib):
    assert _bwd(lib, gf=None, gr=None) == b.RLK_EINVAL
    assert _bwd(lib, grad=None) == b.RLK_EINVAL
    assert _bwd(lib, grad=0x60008) == b.RLK_EALIGN
    assert _bwd(lib, stride=b.VOCAB_PADDED - 8) == b.RLK_EINVAL
    assert _bwd(lib, stride=b.VOCAB_PADDED + 4) == b.RLK_EALIGN          # bf16 rows 8 bytes apart
    assert _bwd(lib, stride=b.VOCAB_PADDED + 2, dtype=1) == b.RLK_EALIGN   # f32 rows 8 bytes apart
    assert _bwd(lib, dtype=2) == b.RLK_EINVAL
    assert _bwd(lib, gf=OUT + 2) == b.RLK_EALIGN
    assert _bwd(lib, full=OUT + 1) == b.RLK_EALIGN
    # top_p / top_k are validated only when the restricted side is requested
    bad_p = _args(top_p_scalar=3.0, T=0)
    assert _bwd(lib, a=bad_p) == b.RLK_OK
    assert _bwd(lib, a=_args(top_p_scalar=3.0), gr=OUT) == b.RLK_EINVAL
    assert _bwd(lib, a=_args(top_k_scalar=0), restr=OUT) == b.RLK_EINVAL
    assert _bwd(lib, a=_args(T=0, logits=None, target=None), gf=None, gr=None, grad=None) == b.RLK_OK


def test_pair_save_and_backward_saved_validation(lib):
    a = _args()
    assert lib.rlk_logp_pair_save(ctypes.byref(a), OUT, OUT, OUT, None, None) == b.RLK_EINVAL
    assert lib.rlk_logp_pair_save(ctypes.byref(a), OUT, OUT, OUT, 0x70008, None) == b.RLK_EALIGN
    assert lib.rlk_logp_pair_save(ctypes.byref(a), None, None, OUT, 0x70000, None) == b.RLK_EINVAL
    assert lib.rlk_logp_pair_save(ctypes.byref(_args(top_k_scalar=0)), OUT, OUT, OUT, 0x70000, None) == b.RLK_EINVAL
    bs = lambda a=a, st=0x70000, gf=OUT, gr=None, grad=0x60000, stride=b.VOCAB_PADDED, dt=0: \
        lib.rlk_logp_backward_saved(ctypes.byref(a), st, gf, gr, grad, stride, dt, None)
    assert bs(st=None) == b.RLK_EINVAL
    assert bs(st=0x70004) == b.RLK_EALIGN
    assert bs(gf=None) == b.RLK_EINVAL
    assert bs(grad=0x60002) == b.RLK_EALIGN
    assert bs(dt=5) == b.RLK_EINVAL
    # top_p / top_k are not read by the saved backward
    assert bs(a=_args(top_p_scalar=9.0, T=0)) == b.RLK_OK
    assert bs(a=_args(T=0, logits=None, target=None), st=None, gf=None, grad=None) == b.RLK_OK


def test_sample_validation(lib):
    a = _args(target=None)           # the sampler has no target
    smp = lambda a=a, ctr=0x80000, uni=None, tok=OUT, ws=0x90000: lib.rlk_sample(
        ctypes.byref(a), 7, ctr, uni, tok, None, None, None, ws, None)
    assert smp(ctr=None, uni=None) == b.RLK_EINVAL
    assert smp(ctr=0x80004) == b.RLK_EALIGN
    assert smp(ctr=None, uni=0x80002) == b.RLK_EALIGN
    assert smp(tok=None) == b.RLK_EINVAL
    assert smp(a=_args(target=None, top_p_scalar=0.0)) == b.RLK_EINVAL
    assert smp(ws=None) == b.RLK_EINVAL
    assert smp(ws=0x90008) == b.RLK_EALIGN
    assert smp(a=_args(target=None, T=0, logits=None), ctr=None, tok=None, ws=None) == b.RLK_OK


def test_linear_logp_validation(lib):
    L = lambda T=4, H=256, hs=256, w=0xA0000, ws_=256, tg=OUT, tau=1.0, out=OUT, ws=0xB0000, h=0xC0000: \
        lib.rlk_linear_logp(h, T, H, hs, w, ws_, tg, None, tau, out, ws, None, None)
    assert L(T=-1) == b.RLK_EINVAL
    assert L(T=0, h=None, w=None, tg=None, out=None, ws=None) == b.RLK_OK
    assert L(H=100) == b.RLK_EINVAL             # not a multiple of 64
    assert L(H=0) == b.RLK_EINVAL
    assert L(hs=128) == b.RLK_EINVAL            # stride < H
    assert L(hs=260) == b.RLK_EALIGN            # rows 520 bytes apart
    assert L(h=0xC0008) == b.RLK_EALIGN
    assert L(w=None) == b.RLK_EINVAL
    assert L(tau=0.0) == b.RLK_EINVAL           # greedy is not a full-vocabulary logprob here
    assert L(tau=float("inf")) == b.RLK_EINVAL
    assert L(ws=None) == b.RLK_EINVAL
    assert L(ws=0xB0004) == b.RLK_EALIGN
    assert L(out=None) == b.RLK_EINVAL


def test_linear_logp_pair_validation(lib):
    f32 = ctypes.c_float

    def L(T=4, H=256, hs=256, w=0xA0000, ws_=256, tg=OUT, tau=1.0, pp=None, p=0.9, kp=None, k=50,
          full=None, restr=OUT, sup=None, ws=0xB0000, h=0xC0000, err=None):
        return lib.rlk_linear_logp_pair(h, T, H, hs, w, ws_, tg, None, f32(tau), pp, f32(p), kp, k, full,
                                        restr, sup, ws, err, None)
    assert L(T=-1) == b.RLK_EINVAL
    assert L(T=1 << 24) == b.RLK_EINVAL
    assert L(T=0, h=None, w=None, tg=None, restr=None, ws=None) == b.RLK_OK
    assert L(restr=None) == b.RLK_EINVAL        # the restricted output is required
    assert L(restr=OUT + 2) == b.RLK_EALIGN
    assert L(full=OUT + 2) == b.RLK_EALIGN
    assert L(sup=OUT + 6) == b.RLK_EALIGN
    assert L(p=0.0) == b.RLK_EINVAL
    assert L(p=1.5) == b.RLK_EINVAL
    assert L(k=0) == b.RLK_EINVAL
    assert L(k=-2) == b.RLK_EINVAL
    assert L(k=b.VOCAB_REAL + 1) == b.RLK_EINVAL
    assert L(pp=OUT + 2) == b.RLK_EALIGN
    assert L(kp=OUT + 2) == b.RLK_EALIGN
    assert L(ws=None) == b.RLK_EINVAL
    assert L(ws=0xB0010) == b.RLK_EALIGN        # the pair's workspace is 256-byte aligned
    assert L(H=100) == b.RLK_EINVAL
    assert L(hs=260) == b.RLK_EALIGN
    assert L(h=0xC0008) == b.RLK_EALIGN
    assert L(tau=0.0) == b.RLK_EINVAL
    assert L(tg=None) == b.RLK_EINVAL
    assert L(err=OUT + 2) == b.RLK_EALIGN


def _declared_param_counts():
    """Parameter count of every rlk_* function declared in include/*.h."""
    counts = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", fn)).read(), flags=re.S)
        for m in re.finditer(r"(?:rlk_status|const char\*|int)\s+(rlk_\w+)\s*\(([^)]*)\)\s*;", text):
            params = m.group(2).strip()
            counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_argument_counts_match_the_headers(lib):
    """The ctypes binding passes as many arguments as each C declaration takes."""
    counts = _declared_param_counts()
    assert set(counts) == set(b.EXPORTS)
    for name, n in counts.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes)


def test_binding_sizes_match_the_header_macros():
    """The binding's workspace sizes and constants follow the C header's macros."""
    text = open(os.path.join(ROOT, "include", "rlk_logp.h")).read()
    norm = open(os.path.join(ROOT, "include", "rlk_norm.h")).read()

    def macro(src, name):
        m = re.search(r"#define\s+" + name + r"(\([A-Za-z]+\))?\s+(.+)", src)
        assert m, name
        return m.group(2).strip()

    for T in (1, 7, 8192):
        ws = eval(re.sub(r"\(size_t\)|u\b", "", macro(text, "RLK_SAMPLE_WORKSPACE_BYTES")).replace("(T)", f"({T})"))
        assert b.sample_workspace_bytes(T) == ws
        lw = eval(re.sub(r"\(size_t\)|u\b", "", macro(text, "RLK_LINEAR_WORKSPACE_BYTES")).replace("(T)", f"({T})"))
        assert b.linear_workspace_bytes(T) == lw
        lp = eval(re.sub(r"\(size_t\)|u\b", "", macro(text, "RLK_LINEAR_PAIR_WORKSPACE_BYTES")).replace("(T)", f"({T})"))
        assert b.linear_pair_workspace_bytes(T) == lp
        kh = eval(re.sub(r"\(size_t\)|u\b", "", macro(text, "RLK_LOGP_KL_HOST_WORKSPACE_BYTES")).replace("(T)", f"({T})"))
        assert b.logp_kl_host_workspace_bytes(T) == kh
    assert int(macro(text, "RLK_SHARD_CHUNKS")) == b.SHARD_CHUNKS
    assert int(macro(norm, "RLK_NORM_BINS")) == b.NORM_BINS
    assert int(macro(text, "RLK_VOCAB_PADDED")) == b.VOCAB_PADDED
    assert int(macro(text, "RLK_VOCAB_REAL")) == b.VOCAB_REAL
